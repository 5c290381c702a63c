"""GPU parity: every C-ABI stage and the fused chunk call against the CPU oracle.

Index sets must equal the oracle's modulo ties (see tests/parity.py), scores
and outputs must be within the stated tolerances, and the gather is byte-exact.
The oracle's later stages are run on the GPU's own earlier results, so a tie
resolved differently upstream does not cascade into a false failure.
"""
import numpy as np
import pytest
import torch

from oracle import quoka_oracle as qo
from sparse_attention_chunked_gb300 import workloads as wl
from tests.parity import (SCORE_ATOL, check_index_rows, check_output, f64, oracle_query_values)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_stages(q, cfg, x, gqa, engine="auto", score_fn="cos", query_agg="max"):
    """Every stage through its own entry point, then the fused call on the same inputs."""
    Q, Kh, Vh = x.Q.to(DEV), x.K_hist.to(DEV), x.V_hist.to(DEV)
    Kc, Vc = x.K_chunk.to(DEV), x.V_chunk.to(DEV)
    shape = q.shape_of(Q, Kh, H_kv=cfg.H_kv, T=cfg.T)
    params = q.params_of(gqa, engine, score_fn=score_fn, query_agg=query_agg)
    ws = q.make_workspace(shape, cfg.N_q, cfg.B, params)
    n = min(cfg.N_q, cfg.C)
    H_sel = cfg.H_q if gqa == "max" else cfg.H_kv
    out = {"shape": shape, "params": params, "ws": ws}
    q_idx = torch.empty((H_sel, n), dtype=torch.int32, device=DEV)
    q.quoka_select_queries(shape, Q, cfg.N_q, params, q_idx, ws)
    scores = torch.empty((cfg.H_kv, cfg.T), dtype=torch.float32, device=DEV)
    q.quoka_score_keys(shape, Q, q_idx, cfg.N_q, Kh, params, scores, ws)
    B_e = min(cfg.B, cfg.T)
    sel = torch.empty((cfg.H_kv, B_e), dtype=torch.int32, device=DEV)
    q.quoka_topk(shape, scores, cfg.B, sel, ws)
    Ks = torch.empty((cfg.H_kv, B_e, cfg.d), dtype=Q.dtype, device=DEV)
    Vs = torch.empty_like(Ks)
    q.quoka_gather(shape, Kh, Vh, sel, B_e, Ks, Vs)
    O = torch.empty_like(Q)
    lse = torch.empty((cfg.H_q, cfg.C), dtype=torch.float32, device=DEV)
    q.quoka_sparse_attend(shape, Q, Ks, Vs, B_e, Kc, Vc, params, O, lse, ws)
    O2 = torch.empty_like(Q)
    sel2 = torch.empty_like(sel)
    q.quoka_chunk_attend(shape, Q, Kh, Vh, Kc, Vc, cfg.N_q, cfg.B, params, O2, None, sel2, ws)
    torch.cuda.synchronize()
    assert q.quoka_get_last_device_error(ws) == 0
    out.update(q_idx=q_idx.cpu().numpy(), scores=scores, sel=sel.cpu().numpy(), Ks=Ks, Vs=Vs, O=O, lse=lse,
               O_fused=O2, sel_fused=sel2.cpu().numpy())
    return out


def check_stages(cfg, x, gqa, r, score_fn="cos", query_agg="max"):
    Q, Kh, Vh = f64(x.Q), f64(x.K_hist), f64(x.V_hist)
    Kc, Vc = f64(x.K_chunk), f64(x.V_chunk)
    # a1/a2: query subselection, modulo ties of the (group-averaged) cosine
    check_index_rows(r["q_idx"], oracle_query_values(Q, cfg.H_kv, gqa), cfg.N_q, largest=False, what="q_idx")
    # a3: scores of the oracle on the GPU's selected queries; a dot-product score carries the
    # norms, so its rounding scales with the largest |row| * |key|
    ref_scores = qo.score_keys(Q, Kh, r["q_idx"], gqa, score_fn, query_agg)
    mag = 1.0
    if score_fn == "dot" and cfg.T > 0:
        rows = qo.scoring_queries(Q, r["q_idx"], cfg.H_kv, gqa, "dot")
        mag = max(1.0, max(np.linalg.norm(rw, axis=1).max() for rw in rows) * np.linalg.norm(Kh, axis=2).max())
    err = np.max(np.abs(f64(r["scores"]) - ref_scores))
    assert err <= SCORE_ATOL * mag, f"scores: max-abs error {err} (scale {mag})"
    # a4: top-B on the oracle's scores, modulo ties
    check_index_rows(r["sel"], ref_scores, cfg.B, largest=True, what="sel")
    # a5: gather is a byte-exact copy
    sel = r["sel"].astype(np.int64)
    for g in range(cfg.H_kv):
        assert torch.equal(r["Ks"][g].cpu(), x.K_hist[g, sel[g]])
        assert torch.equal(r["Vs"][g].cpu(), x.V_hist[g, sel[g]])
    # a6: attention of the oracle over the GPU's kept set
    O_ref, lse_ref = qo.attend(Q, qo.gather(Kh, sel), qo.gather(Vh, sel), Kc, Vc)
    check_output(r["O"], O_ref, "O")
    lse_err = np.max(np.abs(f64(r["lse"]) - lse_ref))
    assert lse_err <= (1e-3 if cfg.dtype == "bf16" else 1e-4), f"lse error {lse_err}"
    # the fused call runs the same kernels: identical results
    assert np.array_equal(r["sel_fused"], r["sel"])
    assert torch.equal(r["O_fused"], r["O"])


SMALL = [
    # name, kwargs for wl.small_chunk
    ("mha_fp32_ragged", dict(H_q=4, H_kv=4, d=64, C=77, T=333, N_q=9, B=50, dtype="fp32")),
    ("gqa4_bf16_d128", dict(H_q=8, H_kv=2, d=128, C=200, T=1000, N_q=12, B=300, dtype="bf16")),
    ("gqa4_bf16_d64", dict(H_q=8, H_kv=2, d=64, C=130, T=4099, N_q=16, B=129, dtype="bf16")),
    ("gqa8_fp32_d128", dict(H_q=16, H_kv=2, d=128, C=64, T=700, N_q=7, B=65, dtype="fp32")),
    ("gqa2_bf16_one_query", dict(H_q=4, H_kv=2, d=128, C=96, T=513, N_q=1, B=1, dtype="bf16")),
    ("nq_above_C", dict(H_q=4, H_kv=1, d=64, C=20, T=300, N_q=64, B=31, dtype="fp32")),
    ("single_row_chunk", dict(H_q=4, H_kv=2, d=128, C=1, T=257, N_q=4, B=17, dtype="bf16")),
    ("iid_recipe_bf16", dict(H_q=4, H_kv=4, d=64, C=128, T=1024, N_q=16, B=256, dtype="bf16", recipe="iid_outliers")),
    # max pooling with 320 scoring rows: two accumulator chunks, the second 64 wide
    ("gqa5_bf16_320_rows", dict(H_q=10, H_kv=2, d=128, C=256, T=2000, N_q=64, B=300, dtype="bf16")),
    # max pooling with 384 and 512 scoring rows: two accumulator chunks of 192 and 256 columns
    ("gqa4_bf16_384_rows", dict(H_q=8, H_kv=2, d=128, C=256, T=1500, N_q=96, B=200, dtype="bf16")),
    ("gqa4_bf16_512_rows", dict(H_q=8, H_kv=2, d=64, C=300, T=2100, N_q=128, B=333, dtype="bf16")),
    # max pooling with 576 scoring rows: wider than TMEM, the CUDA-core scorer takes it
    ("gqa8_bf16_576_rows", dict(H_q=16, H_kv=2, d=64, C=100, T=900, N_q=72, B=111, dtype="bf16")),
    # decode-size chunks (G * C <= 32): the split-key attention, 64-key blocks with ragged tails
    ("decode_c3_g8", dict(H_q=16, H_kv=2, d=128, C=3, T=700, N_q=2, B=100, dtype="bf16")),
    ("decode_c8_g4_fp32_d64", dict(H_q=8, H_kv=2, d=64, C=8, T=500, N_q=4, B=64, dtype="fp32")),
    ("decode_c1_g1", dict(H_q=3, H_kv=3, d=128, C=1, T=129, N_q=1, B=65, dtype="bf16")),
]


@pytest.mark.parametrize("gqa", ["max", "mean"])
@pytest.mark.parametrize("engine", ["auto", "simt"])
@pytest.mark.parametrize("name,kw", SMALL, ids=[s[0] for s in SMALL])
def test_small_cases(quoka, name, kw, gqa, engine):
    cfg, x = wl.small_chunk(**kw)
    r = run_stages(quoka, cfg, x, gqa, engine)
    check_stages(cfg, x, gqa, r)


VARIANT_CASES = [
    ("gqa4_bf16_d128", dict(H_q=8, H_kv=2, d=128, C=200, T=1000, N_q=12, B=300, dtype="bf16")),
    ("gqa5_bf16_320_rows", dict(H_q=10, H_kv=2, d=128, C=256, T=2000, N_q=64, B=300, dtype="bf16")),
    ("mha_fp32_ragged", dict(H_q=4, H_kv=4, d=64, C=77, T=333, N_q=9, B=50, dtype="fp32")),
]


@pytest.mark.parametrize("score_fn,query_agg", [("dot", "max"), ("cos", "mean"), ("dot", "mean")])
@pytest.mark.parametrize("gqa", ["max", "mean"])
@pytest.mark.parametrize("name,kw", VARIANT_CASES, ids=[c[0] for c in VARIANT_CASES])
def test_score_variants(quoka, name, kw, gqa, score_fn, query_agg):
    """The ablations of the key score (dot product, mean over the selected queries) against the oracle."""
    cfg, x = wl.small_chunk(**kw)
    r = run_stages(quoka, cfg, x, gqa, score_fn=score_fn, query_agg=query_agg)
    check_stages(cfg, x, gqa, r, score_fn, query_agg)


@pytest.mark.parametrize("score_fn,query_agg", [("dot", "max"), ("cos", "mean")])
def test_score_variants_full_size(quoka, score_fn, query_agg):
    """32K history, GQA 32/8, per-head max pooling: the variants on the tensor-core scorer at size."""
    cfg = wl.GQA_32K_BF16
    x = wl.make_chunk(cfg, 0)
    r = run_stages(quoka, cfg, x, "max", score_fn=score_fn, query_agg=query_agg)
    check_stages(cfg, x, "max", r, score_fn, query_agg)


@pytest.mark.parametrize("gqa", ["max", "mean"])
def test_tiny_mha_fp32_config(quoka, gqa):
    cfg = wl.TINY_MHA_FP32
    x = wl.make_chunk(cfg, 0)
    r = run_stages(quoka, cfg, x, gqa)
    check_stages(cfg, x, gqa, r)


@pytest.mark.parametrize("gqa", ["max", "mean"])
@pytest.mark.parametrize("cfg", [wl.GQA_32K_BF16, wl.GQA_128K_BF16, wl.DECODE_32K_BF16], ids=lambda c: c.name)
def test_full_size_configs(quoka, cfg, gqa):
    x = wl.make_chunk(cfg, 0)
    r = run_stages(quoka, cfg, x, gqa)
    check_stages(cfg, x, gqa, r)
    # planted needles whose source query was selected are kept (max pooling)
    if gqa == "max":
        sel = [set(row.tolist()) for row in r["sel"]]
        for g, t, h, c in x.needles:
            if c in set(r["q_idx"][h].tolist()):
                assert t in sel[g]


@pytest.mark.parametrize("C", [1, 4])
@pytest.mark.parametrize("T,B", [(0, 64), (300, 300), (1000, 5000)])
def test_decode_budget_covers_history_is_dense(quoka, C, T, B):
    """Decode-size chunks with no history or a budget covering it: dense attention, split over the keys."""
    cfg, x = wl.small_chunk(H_q=8, H_kv=2, d=128, C=C, T=T, N_q=4, B=B, dtype="bf16")
    Q, Kh, Vh, Kc, Vc = (t.to(DEV) for t in (x.Q, x.K_hist, x.V_hist, x.K_chunk, x.V_chunk))
    O, lse, _ = quoka.chunk_attend(Q, Kh, Vh, Kc, Vc, cfg.N_q, B, gqa="max", with_lse=True)
    O_ref, lse_ref = qo.dense_attend(f64(x.Q), f64(x.K_hist), f64(x.V_hist), f64(x.K_chunk), f64(x.V_chunk))
    check_output(O, O_ref, "O")
    assert np.max(np.abs(f64(lse) - lse_ref)) <= 1e-3


@pytest.mark.parametrize("T,B", [(0, 64), (300, 300), (300, 5000)])
def test_budget_covers_history_is_dense(quoka, T, B):
    """T = 0 is causal self-attention of the chunk; B >= T keeps every history key."""
    cfg, x = wl.small_chunk(H_q=8, H_kv=2, d=128, C=150, T=T, N_q=8, B=B, dtype="bf16")
    Q, Kh, Vh = x.Q.to(DEV), x.K_hist.to(DEV), x.V_hist.to(DEV)
    Kc, Vc = x.K_chunk.to(DEV), x.V_chunk.to(DEV)
    O, lse, sel = quoka.chunk_attend(Q, Kh, Vh, Kc, Vc, cfg.N_q, B, gqa="max", with_lse=True, with_sel=True)
    O_ref, lse_ref = qo.dense_attend(f64(x.Q), f64(x.K_hist), f64(x.V_hist), f64(x.K_chunk), f64(x.V_chunk))
    check_output(O, O_ref, "O")
    if T > 0:
        assert np.array_equal(sel.cpu().numpy(), np.tile(np.arange(T), (cfg.H_kv, 1)))
    else:
        assert sel is None


def test_dense_attend_matches_oracle(quoka):
    cfg, x = wl.small_chunk(H_q=8, H_kv=2, d=128, C=190, T=2100, dtype="bf16")
    Q, Kh, Vh = x.Q.to(DEV), x.K_hist.to(DEV), x.V_hist.to(DEV)
    Kc, Vc = x.K_chunk.to(DEV), x.V_chunk.to(DEV)
    shape = quoka.shape_of(Q, Kh)
    params = quoka.params_of()
    ws = quoka.make_workspace(shape, 1, 1, params)
    O = torch.empty_like(Q)
    lse = torch.empty((cfg.H_q, cfg.C), dtype=torch.float32, device=DEV)
    quoka.quoka_dense_attend(shape, Q, Kh, Vh, Kc, Vc, params, O, lse, ws)
    O_ref, lse_ref = qo.dense_attend(f64(x.Q), f64(x.K_hist), f64(x.V_hist), f64(x.K_chunk), f64(x.V_chunk))
    check_output(O, O_ref, "dense O")
    assert np.max(np.abs(f64(lse) - lse_ref)) < 1e-3


def test_dense_attend_full_size_sampled_heads(quoka):
    """The dense reference at the 32K-history workload, checked on three query heads."""
    cfg = wl.GQA_32K_BF16
    x = wl.make_chunk(cfg, 0)
    Q, Kh, Vh = x.Q.to(DEV), x.K_hist.to(DEV), x.V_hist.to(DEV)
    Kc, Vc = x.K_chunk.to(DEV), x.V_chunk.to(DEV)
    shape = quoka.shape_of(Q, Kh)
    params = quoka.params_of()
    ws = quoka.make_workspace(shape, 1, 1, params)
    O = torch.empty_like(Q)
    quoka.quoka_dense_attend(shape, Q, Kh, Vh, Kc, Vc, params, O, None, ws)
    torch.cuda.synchronize()
    G = cfg.G
    for h in (0, 13, 31):
        g = h // G
        O_ref, _ = qo.dense_attend(f64(x.Q[h:h + 1]), f64(x.K_hist[g:g + 1]), f64(x.V_hist[g:g + 1]),
                                   f64(x.K_chunk[g:g + 1]), f64(x.V_chunk[g:g + 1]))
        check_output(O[h:h + 1], O_ref, f"dense O head {h}")


def test_append_kv_grows_cache_in_place(quoka):
    H_kv, cap, d, T, C = 2, 1000, 128, 300, 77
    cache_k = torch.zeros((H_kv, cap, d), dtype=torch.bfloat16, device=DEV)
    cache_v = torch.zeros_like(cache_k)
    Kc = torch.randn((H_kv, C, d), device=DEV).to(torch.bfloat16)
    Vc = torch.randn((H_kv, C, d), device=DEV).to(torch.bfloat16)
    Q = torch.empty((4, C, d), dtype=torch.bfloat16, device=DEV)
    shape = quoka.shape_of(Q, cache_k, T=T)
    assert shape.kv_head_stride == cap * d
    quoka.quoka_append_kv(shape, cache_k, cache_v, Kc, Vc)
    torch.cuda.synchronize()
    assert torch.equal(cache_k[:, T:T + C], Kc) and torch.equal(cache_v[:, T:T + C], Vc)
    assert not cache_k[:, :T].any() and not cache_k[:, T + C:].any()


def test_history_inside_larger_cache(quoka):
    """A strided history (preallocated cache) gives the same result as a compact copy."""
    cfg, x = wl.small_chunk(H_q=8, H_kv=2, d=64, C=64, T=500, N_q=6, B=70, dtype="bf16")
    cap = 900
    Kcache = torch.zeros((cfg.H_kv, cap, cfg.d), dtype=torch.bfloat16, device=DEV)
    Vcache = torch.zeros_like(Kcache)
    Kcache[:, :cfg.T] = x.K_hist.to(DEV)
    Vcache[:, :cfg.T] = x.V_hist.to(DEV)
    Q, Kc, Vc = x.Q.to(DEV), x.K_chunk.to(DEV), x.V_chunk.to(DEV)
    for gqa in ("max", "mean"):
        O1, _, s1 = quoka.chunk_attend(Q, Kcache, Vcache, Kc, Vc, cfg.N_q, cfg.B, gqa=gqa, T=cfg.T, with_sel=True)
        O2, _, s2 = quoka.chunk_attend(Q, x.K_hist.to(DEV), x.V_hist.to(DEV), Kc, Vc, cfg.N_q, cfg.B, gqa=gqa,
                                       with_sel=True)
        assert torch.equal(s1, s2) and torch.equal(O1, O2)


def test_topk_ties_go_to_lower_positions(quoka):
    """Many exactly equal scores (and -0.0 vs 0.0): the lowest positions win, output ascending."""
    H_kv, T, B = 3, 5000, 700
    rng = np.random.default_rng(7)
    s = rng.integers(-3, 4, (H_kv, T)).astype(np.float32) * 0.125
    s[1, ::7] = -0.0
    s[2] = 0.0
    scores = torch.from_numpy(s).to(DEV)
    Q = torch.empty((H_kv, 4, 64), dtype=torch.float32, device=DEV)
    shape = quoka.Shape(0, H_kv, H_kv, 4, T, 64, 1)
    ws = quoka.make_workspace(shape, 1, B, quoka.params_of())
    sel = torch.empty((H_kv, B), dtype=torch.int32, device=DEV)
    quoka.quoka_topk(shape, scores, B, sel, ws)
    got = sel.cpu().numpy()
    for g in range(H_kv):
        assert list(got[g]) == list(qo.top_b(s[g].astype(np.float64), B))


def test_chunked_prefill_sweep_sampled_chunks(quoka):
    """The 64K-token prompt in 32 chunks of 2048, appending to a preallocated cache;
    chunks 0 (no history), 1 (budget covers history), 2, 17 and 31 are checked."""
    cfg = wl.SWEEP_64K_BF16
    sw = wl.make_sweep(cfg, 0)
    K_all, V_all = sw.K_all.to(DEV), sw.V_all.to(DEV)
    Kcache = torch.zeros_like(K_all)
    Vcache = torch.zeros_like(V_all)
    check = {0, 1, 2, 17, 31}
    results = {}
    shape0 = quoka.shape_of(sw.Q[0].to(DEV), Kcache, T=cfg.total - cfg.C)
    params = quoka.params_of("max")
    ws = quoka.make_workspace(shape0, cfg.N_q, cfg.B, params)
    for i in range(cfg.n_chunks):
        T = i * cfg.C
        Q = sw.Q[i].to(DEV)
        Kc, Vc = K_all[:, T:T + cfg.C].contiguous(), V_all[:, T:T + cfg.C].contiguous()
        O, _, sel = quoka.chunk_attend(Q, Kcache, Vcache, Kc, Vc, cfg.N_q, cfg.B, gqa="max", T=T, ws=ws,
                                       with_sel=True)
        shape = quoka.shape_of(Q, Kcache, T=T)
        quoka.quoka_append_kv(shape, Kcache, Vcache, Kc, Vc)
        if i in check:
            results[i] = (O, None if sel is None else sel.cpu().numpy())
    torch.cuda.synchronize()
    assert torch.equal(Kcache, K_all) and torch.equal(Vcache, V_all)
    for i, (O, sel) in results.items():
        T = i * cfg.C
        Qn = f64(sw.Q[i])
        Kh, Vh = f64(sw.K_all[:, :T]), f64(sw.V_all[:, :T])
        Kc, Vc = f64(sw.K_all[:, T:T + cfg.C]), f64(sw.V_all[:, T:T + cfg.C])
        if T > cfg.B:
            Qd = sw.Q[i].to(DEV)
            shape = quoka.shape_of(Qd, Kcache, T=T)
            q_idx = torch.empty((cfg.H_q, cfg.N_q), dtype=torch.int32, device=DEV)
            quoka.quoka_select_queries(shape, Qd, cfg.N_q, params, q_idx, ws)
            q_idx = q_idx.cpu().numpy()
            check_index_rows(q_idx, oracle_query_values(Qn, cfg.H_kv, "max"), cfg.N_q, largest=False,
                             what=f"chunk {i} q_idx")
            ref_scores = qo.score_keys(Qn, Kh, q_idx, "max")
            check_index_rows(sel, ref_scores, cfg.B, largest=True, what=f"chunk {i} sel")
        else:
            sel = np.tile(np.arange(T), (cfg.H_kv, 1))
        O_ref, _ = qo.attend(Qn, qo.gather(Kh, sel.astype(np.int64)), qo.gather(Vh, sel.astype(np.int64)), Kc, Vc)
        check_output(O, O_ref, f"chunk {i} O")


@pytest.mark.parametrize("gqa", ["max", "mean"])
def test_ragged_batch(quoka, gqa):
    """Eight sequences with log-uniform histories in [4K, 64K], GQA 64/8, one chunk each."""
    cfg = wl.RAGGED_8x_BF16
    seqs = wl.make_ragged(cfg, 0)
    for s, x in enumerate(seqs):
        T = x.K_hist.shape[1]
        sub = wl.ChunkConfig(f"seq{s}", cfg.H_q, cfg.H_kv, cfg.d, cfg.C, T, cfg.N_q, cfg.B, cfg.dtype, "massive_act")
        r = run_stages(quoka, sub, x, gqa)
        if s in (0, 3, 7):
            check_stages(sub, x, gqa, r)


@pytest.mark.parametrize("T,B", [(400_000, 5000), (90_000, 3000), (70_000, 4096), (12_288, 2048), (9, 8)])
def test_topk_sizes_and_slices(quoka, T, B):
    """Slices that do and do not fit in shared memory, and tiny rows, with frequent exact ties."""
    H_kv = 2
    rng = np.random.default_rng(T)
    s = (rng.integers(-200, 200, (H_kv, T)) * 0.01).astype(np.float32)
    scores = torch.from_numpy(s).to(DEV)
    shape = quoka.Shape(0, H_kv, H_kv, 4, T, 64, 1)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    sel = torch.empty((H_kv, B), dtype=torch.int32, device=DEV)
    quoka.quoka_topk(shape, scores, B, sel, ws)
    got = sel.cpu().numpy()
    for g in range(H_kv):
        assert np.array_equal(got[g], qo.top_b(s[g].astype(np.float64), B))


@pytest.mark.parametrize("T,B,n_big,n_tie", [(60_000, 3000, 1000, 59_000), (20_000, 2000, 500, 6000)])
def test_topk_ties_inside_and_beyond_the_candidate_list(quoka, T, B, n_big, n_tie):
    """A threshold bin with more keys than the select's candidate list (the general radix select
    takes over) and one with fewer (resolved from the list), both ending in exact ties."""
    H_kv = 2
    rng = np.random.default_rng(T + B)
    s = np.full((H_kv, T), -0.75, dtype=np.float32)
    for g in range(H_kv):
        perm = rng.permutation(T)
        s[g, perm[:n_tie]] = 1.0
        s[g, perm[n_tie:n_tie + n_big]] = 1.5 + rng.integers(0, 200, n_big).astype(np.float32) / 512
    scores = torch.from_numpy(s).to(DEV)
    shape = quoka.Shape(0, H_kv, H_kv, 4, T, 64, 1)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    sel = torch.empty((H_kv, B), dtype=torch.int32, device=DEV)
    quoka.quoka_topk(shape, scores, B, sel, ws)
    got = sel.cpu().numpy()
    for g in range(H_kv):
        assert np.array_equal(got[g], qo.top_b(s[g].astype(np.float64), B))


@pytest.mark.parametrize("T,distinct", [(3000, 7), (20_000, 2), (30_000, 2)])
def test_fused_topk_with_duplicate_keys(quoka, T, distinct):
    """History keys repeating a few rows give exactly equal scores: the fused select (fed by the
    scorer's histogram) keeps the lowest positions, as the oracle's top-B does on the GPU's scores;
    with two distinct rows of 30000 the threshold bin overflows the candidate list."""
    cfg, x = wl.small_chunk(H_q=8, H_kv=2, d=128, C=64, T=T, N_q=8, B=1500, dtype="bf16")
    x.K_hist[:] = x.K_hist[:, torch.arange(T) % distinct]
    r = run_stages(quoka, cfg, x, "max")
    sc = r["scores"].cpu().numpy().astype(np.float64)
    for g in range(cfg.H_kv):
        want = qo.top_b(sc[g], cfg.B)
        assert np.array_equal(r["sel"][g], want)
        assert np.array_equal(r["sel_fused"][g], want)


def test_fused_topk_one_slice_full_of_ties(quoka):
    """The first eighth of every head's history repeats the head's best key: one CTA of the fused
    select holds more candidates than it can stage, and every CTA takes the general select."""
    cfg, x = wl.small_chunk(H_q=8, H_kv=2, d=128, C=64, T=40_000, N_q=8, B=3000, dtype="bf16")
    r0 = run_stages(quoka, cfg, x, "max")
    best = r0["scores"].argmax(dim=1).cpu()
    for g in range(cfg.H_kv):
        x.K_hist[g, :5000] = x.K_hist[g, int(best[g])]
    r = run_stages(quoka, cfg, x, "max")
    sc = r["scores"].cpu().numpy().astype(np.float64)
    for g in range(cfg.H_kv):
        want = qo.top_b(sc[g], cfg.B)
        assert np.array_equal(want, np.arange(cfg.B))
        assert np.array_equal(r["sel"][g], want)
        assert np.array_equal(r["sel_fused"][g], want)
