"""The workspace-free query selection (quoka_select_queries_noalloc), against
the workspace entry point on the same inputs, over two calls in a row.

Some callers cannot give the library any device scratch memory (engine
plugins whose enqueue path may not allocate, runtimes that plan all device
memory up front); this entry point keeps the selection kernels' scratch in a
library-owned device array.  The cases cover every launch path: the
one-launch clustered kernel (which needs no scratch beyond the error header)
and the split of mean pooling, which writes the per-head cosines into the
array and reads them back, so a wrong array address or layout offset fails
here.

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
    """q_idx from one entry point, and how many kernels the call launched."""
    Q = x.Q.cuda()
    shape = quoka.shape_of(Q, x.K_hist.cuda())
    params = quoka.params_of(gqa)
    H_sel = cfg.H_q if gqa == "max" else cfg.H_kv
    q_idx = torch.full((H_sel, min(cfg.N_q, cfg.C)), -1, dtype=torch.int32, device="cuda")
    before = quoka.quoka_launch_count()
    if noalloc:
        quoka.quoka_select_queries_noalloc(shape, Q, cfg.N_q, params, q_idx)
    else:
        ws = quoka.make_workspace(shape, cfg.N_q, cfg.B, params)
        quoka.quoka_select_queries(shape, Q, cfg.N_q, params, q_idx, ws)
    launches = quoka.quoka_launch_count() - before
    torch.cuda.synchronize()
    return q_idx.cpu().numpy(), launches


def _check_two_calls(quoka, cases, gqa, launches_expected):
    for cfg, x in cases:            # two calls in a row: the shared scratch keeps the first call's contents
        for _ in range(2):
            got, n_launch = _select(quoka, x, cfg, gqa, noalloc=True)
            ref, _ = _select(quoka, x, cfg, gqa, noalloc=False)
            assert n_launch == launches_expected, (cfg.name, n_launch)
            assert np.array_equal(got, ref), cfg.name
            check_index_rows(got, oracle_query_values(f64(x.Q), cfg.H_kv, gqa), cfg.N_q, largest=False,
                             what="noalloc q_idx")


@pytest.mark.parametrize("gqa", ["max", "mean"])
def test_noalloc_matches_workspace_entry_clustered(quoka, gqa):
    """Chunks small enough for the clustered kernel.  Max pooling, and mean pooling with one query head
    per KV head: one launch, no scratch region used.  Mean pooling over several heads: a clustered pass
    per query head writes its cosines into the array, then the clustered group select reads them."""
    cases = [(wl.small_chunk(H_q=8, H_kv=2, d=128, C=300, T=64, N_q=20, B=8, dtype="bf16", seed=1), 1, 2),
             (wl.small_chunk(H_q=4, H_kv=4, d=64, C=97, T=64, N_q=9, B=8, dtype="fp32", seed=2), 1, 1),
             (wl.small_chunk(H_q=64, H_kv=1, d=128, C=1024, T=64, N_q=64, B=8, dtype="bf16", seed=3), 1, 2),
             (wl.small_chunk(H_q=32, H_kv=1, d=128, C=4096, T=64, N_q=64, B=8, dtype="bf16", seed=4), 1, 2)]
    for (cfg, x), n_max, n_mean in cases:
        _check_two_calls(quoka, [(cfg, x)], gqa, launches_expected=n_max if gqa == "max" else n_mean)


def test_noalloc_mean_pooling_beyond_the_array(quoka):
    """Mean pooling whose cosines would not fit the 4 MiB array (128 query heads x 8192 queries: 4 MiB
    plus the header) runs the one-launch kernel over whole groups of 8 heads, and matches the workspace
    entry point (which splits)."""
    cases = [wl.small_chunk(H_q=128, H_kv=16, d=64, C=8192, T=64, N_q=64, B=8, dtype="bf16", seed=7)]
    _check_two_calls(quoka, cases, "mean", launches_expected=1)


def test_noalloc_keeps_every_query_when_n_q_reaches_c(quoka):
    """N_q >= C keeps the positions 0..C-1 without any cosine (the workspace entry point's branch)."""
    cfg, x = wl.small_chunk(H_q=8, H_kv=2, d=128, C=40, T=64, N_q=64, B=8, dtype="bf16", seed=5)
    for gqa in ("max", "mean"):
        for _ in range(2):
            got, _ = _select(quoka, x, cfg, gqa, noalloc=True)
            ref, _ = _select(quoka, x, cfg, gqa, noalloc=False)
            assert np.array_equal(got, ref)
            assert np.array_equal(got, np.tile(np.arange(cfg.C, dtype=np.int32), (got.shape[0], 1)))


def test_noalloc_rejects_problems_beyond_its_scratch(quoka):
    """Mean pooling over 128 query heads of one KV head at C = 8192: the per-head cosines need 4 MiB
    plus the header (more than the array) and the whole-group kernel's shared memory is far above its
    limit, so the call is refused before anything is enqueued (the pointers are never dereferenced)."""
    shape = quoka.Shape(0, 128, 1, 8192, 0, 128, 0)
    rc = quoka.load().quoka_select_queries_noalloc(ctypes.byref(shape), ctypes.c_void_p(1 << 20), 8,
                                                   ctypes.byref(quoka.params_of("mean")), ctypes.c_void_p(1 << 20),
                                                   None)
    assert rc == 2   # QUOKA_ERR_UNSUPPORTED
