"""The workspace-free query selection (quoka_select_queries_noalloc), for callers
that cannot give the library any device scratch memory, against the workspace
entry point on the same inputs, over two calls in a row.

Collected last on purpose (file name), so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_chunked_gb300 import workloads as wl
from tests.parity import check_index_rows, f64, oracle_query_values

pytestmark = pytest.mark.gpu


def _select(quoka, x, cfg, gqa, noalloc):
    Q = x.Q.cuda()
    shape = quoka.shape_of(Q, x.K_hist.cuda())
    params = quoka.params_of(gqa)
    H_sel = cfg.H_q if gqa == "max" else cfg.H_kv
    q_idx = torch.full((H_sel, min(cfg.N_q, cfg.C)), -1, dtype=torch.int32, device="cuda")
    if noalloc:
        quoka.quoka_select_queries_noalloc(shape, Q, cfg.N_q, params, q_idx)
    else:
        ws = quoka.make_workspace(shape, cfg.N_q, cfg.B, params)
        quoka.quoka_select_queries(shape, Q, cfg.N_q, params, q_idx, ws)
    torch.cuda.synchronize()
    return q_idx.cpu().numpy()


@pytest.mark.parametrize("gqa", ["max", "mean"])
def test_noalloc_matches_workspace_entry_on_two_calls(quoka, gqa):
    cases = [wl.small_chunk(H_q=8, H_kv=2, d=128, C=300, T=64, N_q=20, B=8, dtype="bf16", seed=1),
             wl.small_chunk(H_q=4, H_kv=4, d=64, C=97, T=64, N_q=9, B=8, dtype="fp32", seed=2)]
    for cfg, x in cases:            # two calls in a row: the shared scratch keeps the first call's contents
        got = _select(quoka, x, cfg, gqa, noalloc=True)
        ref = _select(quoka, x, cfg, gqa, noalloc=False)
        assert np.array_equal(got, ref)
        check_index_rows(got, oracle_query_values(f64(x.Q), cfg.H_kv, gqa), cfg.N_q, largest=False,
                         what="noalloc q_idx")


def test_noalloc_rejects_problems_beyond_its_scratch(quoka):
    shape = quoka.Shape(0, 128, 8, 8192, 0, 128, 0)       # 128 heads x 8192 queries: more than 4 MiB of scratch
    rc = quoka.load().quoka_select_queries_noalloc(ctypes.byref(shape), ctypes.c_void_p(1 << 20), 8,
                                                   ctypes.byref(quoka.params_of("max")), ctypes.c_void_p(1 << 20),
                                                   None)
    assert rc == 2   # QUOKA_ERR_UNSUPPORTED
