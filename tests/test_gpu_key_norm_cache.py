"""GPU parity of the key-norm cache: 1/|k| written when keys enter the cache and
read by the scorer instead of being recomputed from every key tile.

The cached norms are checked against float64 norms of the same keys; scores
read through the cache against the oracle (and against the recomputing path,
to fp32 rounding); the 64K-token chunked sweep keeps the cache up to date
with quoka_append_kv_norms and checks sampled chunks against the oracle.
"""
import numpy as np
import pytest
import torch

from oracle import quoka_oracle as qo
from sparse_attention_chunked_gb300 import workloads as wl
from tests.parity import SCORE_ATOL, check_index_rows, check_output, f64, oracle_query_values

pytestmark = pytest.mark.gpu
DEV = "cuda"


def inv_norms_ref(K: np.ndarray) -> np.ndarray:
    return 1.0 / np.maximum(np.linalg.norm(K, axis=-1), qo.EPS)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("fp32", 128)])
def test_key_inv_norms_match_float64(quoka, dtype, d):
    cfg, x = wl.small_chunk(H_q=4, H_kv=2, d=d, C=16, T=1000, N_q=4, B=64, dtype=dtype)
    Kh = x.K_hist.to(DEV)
    Kh[1, 7] = 0                                      # a zero key: clamped norm
    shape = quoka.shape_of(x.Q.to(DEV), Kh)
    inv = torch.full((cfg.H_kv, 1100), -1.0, dtype=torch.float32, device=DEV)
    quoka.quoka_key_inv_norms(shape, Kh, 0, 300, inv)
    quoka.quoka_key_inv_norms(shape, Kh, 300, cfg.T, inv)
    torch.cuda.synchronize()
    ref = inv_norms_ref(f64(Kh))
    got = f64(inv[:, :cfg.T])
    assert np.max(np.abs(got - ref) / ref) < 1e-6
    assert torch.all(inv[:, cfg.T:] == -1.0)          # nothing written past t1


@pytest.mark.parametrize("gqa", ["max", "mean"])
@pytest.mark.parametrize("cfg_name", ["small", "gqa32k"])
def test_cached_scores_and_chunk(quoka, gqa, cfg_name):
    if cfg_name == "small":
        cfg, x = wl.small_chunk(H_q=8, H_kv=2, d=128, C=200, T=3000, N_q=12, B=300, dtype="bf16")
    else:
        cfg = wl.GQA_32K_BF16
        x = wl.make_chunk(cfg, 0)
    Q, Kh, Vh, Kc, Vc = (t.to(DEV) for t in (x.Q, x.K_hist, x.V_hist, x.K_chunk, x.V_chunk))
    shape = quoka.shape_of(Q, Kh)
    params = quoka.params_of(gqa)
    ws = quoka.make_workspace(shape, cfg.N_q, cfg.B, params)
    inv = torch.empty((cfg.H_kv, cfg.T + 64), dtype=torch.float32, device=DEV)   # a cache with spare room
    quoka.quoka_key_inv_norms(shape, Kh, 0, cfg.T, inv)
    H_sel = cfg.H_q if gqa == "max" else cfg.H_kv
    q_idx = torch.empty((H_sel, min(cfg.N_q, cfg.C)), dtype=torch.int32, device=DEV)
    quoka.quoka_select_queries(shape, Q, cfg.N_q, params, q_idx, ws)
    s_plain = torch.empty((cfg.H_kv, cfg.T), dtype=torch.float32, device=DEV)
    s_cached = torch.empty_like(s_plain)
    quoka.quoka_score_keys(shape, Q, q_idx, cfg.N_q, Kh, params, s_plain, ws)
    quoka.quoka_score_keys_cached(shape, Q, q_idx, cfg.N_q, Kh, inv, params, s_cached, ws)
    O = torch.empty_like(Q)
    sel = torch.empty((cfg.H_kv, cfg.B), dtype=torch.int32, device=DEV)
    quoka.quoka_chunk_attend_cached(shape, Q, Kh, Vh, Kc, Vc, inv, cfg.N_q, cfg.B, params, O, None, sel, ws)
    torch.cuda.synchronize()
    assert quoka.quoka_get_last_device_error(ws) == 0
    q_idx = q_idx.cpu().numpy()
    ref = qo.score_keys(f64(x.Q), f64(x.K_hist), q_idx, gqa)
    assert np.max(np.abs(f64(s_cached) - ref)) <= SCORE_ATOL
    assert np.max(np.abs(f64(s_cached) - f64(s_plain))) <= 1e-6
    sel = sel.cpu().numpy()
    check_index_rows(sel, ref, cfg.B, largest=True, what="cached sel")
    s = sel.astype(np.int64)
    O_ref, _ = qo.attend(f64(x.Q), qo.gather(f64(x.K_hist), s), qo.gather(f64(x.V_hist), s), f64(x.K_chunk),
                         f64(x.V_chunk))
    check_output(O, O_ref, "cached O")


def test_sweep_keeps_the_norm_cache_with_append(quoka):
    """The 64K-token prompt in 32 chunks, the norm cache written by quoka_append_kv_norms after every chunk."""
    cfg = wl.SWEEP_64K_BF16
    sw = wl.make_sweep(cfg, 0)
    K_all, V_all = sw.K_all.to(DEV), sw.V_all.to(DEV)
    Kcache, Vcache = torch.zeros_like(K_all), torch.zeros_like(V_all)
    inv = torch.zeros((cfg.H_kv, cfg.total), dtype=torch.float32, device=DEV)
    params = quoka.params_of("max")
    ws = quoka.make_workspace(quoka.shape_of(sw.Q[0].to(DEV), Kcache, T=cfg.total - cfg.C), cfg.N_q, cfg.B, params)
    check, results = {2, 17, 31}, {}
    for i in range(cfg.n_chunks):
        T = i * cfg.C
        Q = sw.Q[i].to(DEV)
        Kc, Vc = K_all[:, T:T + cfg.C].contiguous(), V_all[:, T:T + cfg.C].contiguous()
        shape = quoka.shape_of(Q, Kcache, T=T)
        O = torch.empty_like(Q)
        sel = torch.empty((cfg.H_kv, min(cfg.B, T)), dtype=torch.int32, device=DEV) if T else None
        quoka.quoka_chunk_attend_cached(shape, Q, Kcache, Vcache, Kc, Vc, inv, cfg.N_q, cfg.B, params, O, None,
                                        sel, ws)
        quoka.quoka_append_kv_norms(shape, Kcache, Vcache, Kc, Vc, inv)
        if i in check:
            results[i] = (O, sel.cpu().numpy())
    torch.cuda.synchronize()
    assert torch.equal(Kcache, K_all)
    assert np.max(np.abs(f64(inv) / inv_norms_ref(f64(K_all)) - 1.0)) < 1e-6
    for i, (O, sel) in results.items():
        T = i * cfg.C
        Qn = f64(sw.Q[i])
        Kh, Vh = f64(sw.K_all[:, :T]), f64(sw.V_all[:, :T])
        Qd = sw.Q[i].to(DEV)
        q_idx = torch.empty((cfg.H_q, cfg.N_q), dtype=torch.int32, device=DEV)
        quoka.quoka_select_queries(quoka.shape_of(Qd, Kcache, T=T), Qd, cfg.N_q, params, q_idx, ws)
        q_idx = q_idx.cpu().numpy()
        check_index_rows(q_idx, oracle_query_values(Qn, cfg.H_kv, "max"), cfg.N_q, largest=False, what="q_idx")
        check_index_rows(sel, qo.score_keys(Qn, Kh, q_idx, "max"), cfg.B, largest=True, what=f"chunk {i} sel")
        s = sel.astype(np.int64)
        O_ref, _ = qo.attend(Qn, qo.gather(Kh, s), qo.gather(Vh, s), f64(sw.K_all[:, T:T + cfg.C]),
                             f64(sw.V_all[:, T:T + cfg.C]))
        check_output(O, O_ref, f"chunk {i} O")
