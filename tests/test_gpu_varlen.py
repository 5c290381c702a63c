"""GPU parity of the ragged-batch entry point, quoka_chunk_attend_varlen.

Every sequence of the packed batch must come out exactly as a single-sequence
quoka_chunk_attend call on that sequence's tensors gives it (the same kernels
run on the same inputs), and those single calls are held to the oracle here
as well: stage by stage where keys are selected, against dense chunked
attention where the budget covers the history or there is none.
"""
import numpy as np
import pytest
import torch

from oracle import quoka_oracle as qo
from sparse_attention_chunked_gb300 import workloads as wl
from tests.parity import check_output, f64
from tests.test_gpu_parity import check_stages, run_stages

pytestmark = pytest.mark.gpu
DEV = "cuda"


def empty_chunk(H_q, H_kv, d, T, dtype):
    """A sequence with no queries this step (C = 0): it must be skipped."""
    t = torch.float32 if dtype == "fp32" else torch.bfloat16
    z = lambda h, n: torch.zeros((h, n, d), dtype=t)
    return wl.ChunkInputs(z(H_q, 0), torch.randn((H_kv, T, d)).to(t), torch.randn((H_kv, T, d)).to(t),
                          z(H_kv, 0), z(H_kv, 0), np.zeros((H_q, 0), dtype=np.int64))


def run_varlen(q, seqs, H_q, H_kv, d, N_q, B, gqa, dtype):
    pk = wl.pack_varlen(seqs)
    t = {k: v.to(DEV) for k, v in pk.items() if isinstance(v, torch.Tensor)}
    vshape = q.varlen_shape_of(len(seqs), H_q, H_kv, d, t["Q"].dtype)
    params = q.params_of(gqa)
    n_ws = q.quoka_workspace_size_varlen(vshape, pk["cu_T"], pk["cu_C"], N_q, B, params)
    ws = torch.zeros(max(n_ws, 256), dtype=torch.uint8, device=DEV)
    O = torch.full_like(t["Q"], float("nan"))
    lse = torch.full((H_q * pk["cu_C"][-1],), float("nan"), dtype=torch.float32, device=DEV)
    B_s = [min(B, t1 - t0) for t0, t1 in zip(pk["cu_T"], pk["cu_T"][1:])]
    sel = torch.full((H_kv * sum(B_s),), -7, dtype=torch.int32, device=DEV)
    q.quoka_chunk_attend_varlen(vshape, pk["cu_T"], pk["cu_C"], t["Q"], t["K_hist"], t["V_hist"], t["K_chunk"],
                                t["V_chunk"], N_q, B, params, O, lse, sel, ws)
    torch.cuda.synchronize()
    assert q.quoka_get_last_device_error(ws) == 0
    out, cb = [], 0
    for s, x in enumerate(seqs):
        c0, c1 = pk["cu_C"][s], pk["cu_C"][s + 1]
        out.append(dict(O=O[H_q * d * c0:H_q * d * c1].view(H_q, c1 - c0, d),
                        lse=lse[H_q * c0:H_q * c1].view(H_q, c1 - c0),
                        sel=sel[H_kv * cb:H_kv * (cb + B_s[s])].view(H_kv, B_s[s])))
        cb += B_s[s]
    return out


def single(q, x, N_q, B, gqa):
    """quoka_chunk_attend on one sequence."""
    Q, Kh, Vh, Kc, Vc = (a.to(DEV) for a in (x.Q, x.K_hist, x.V_hist, x.K_chunk, x.V_chunk))
    shape = q.shape_of(Q, Kh, H_kv=Kc.shape[0])
    params = q.params_of(gqa)
    ws = q.make_workspace(shape, N_q, B, params)
    O = torch.empty_like(Q)
    lse = torch.empty(Q.shape[:2], dtype=torch.float32, device=DEV)
    B_e = min(B, shape.T)
    sel = torch.empty((shape.H_kv, B_e), dtype=torch.int32, device=DEV)
    q.quoka_chunk_attend(shape, Q, Kh, Vh, Kc, Vc, N_q, B, params, O, lse, sel if B_e > 0 else None, ws)
    torch.cuda.synchronize()
    return dict(O=O, lse=lse, sel=sel)


def check_against_oracle(q, x, H_q, H_kv, d, N_q, B, gqa, dtype, got):
    C, T = x.Q.shape[1], x.K_hist.shape[1]
    if 0 < B < T:
        cfg = wl.ChunkConfig("seq", H_q, H_kv, d, C, T, N_q, B, dtype, "massive_act")
        r = run_stages(q, cfg, x, gqa)
        check_stages(cfg, x, gqa, r)
        assert torch.equal(got["O"], r["O_fused"])
        assert np.array_equal(got["sel"].cpu().numpy(), r["sel_fused"])
    else:   # the budget covers the history, or there is none: dense chunked attention
        O_ref, lse_ref = qo.attend(f64(x.Q), f64(x.K_hist), f64(x.V_hist), f64(x.K_chunk), f64(x.V_chunk))
        check_output(got["O"], O_ref, "O (dense)")
        assert np.max(np.abs(f64(got["lse"]) - lse_ref)) <= (1e-3 if dtype == "bf16" else 1e-4)
        if T > 0:
            assert np.array_equal(got["sel"].cpu().numpy(), np.tile(np.arange(T), (H_kv, 1)))


# (C_s, T_s) per sequence: ragged chunks including 1 and 0 queries, a history
# shorter than the budget, an empty history, several tiles and ragged tails.
SEQS = [(77, 333), (0, 50), (1, 700), (130, 1000), (64, 20), (33, 0), (200, 2100)]


@pytest.mark.parametrize("gqa", ["max", "mean"])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("fp32", 64)])
def test_varlen_small_batch(quoka, gqa, dtype, d):
    H_q, H_kv, N_q, B = 8, 2, 9, 40
    seqs = []
    for s, (C, T) in enumerate(SEQS):
        if C == 0:
            seqs.append(empty_chunk(H_q, H_kv, d, T, dtype))
        else:
            seqs.append(wl.small_chunk(H_q=H_q, H_kv=H_kv, d=d, C=C, T=T, N_q=N_q, B=B, dtype=dtype, seed=s)[1])
    got = run_varlen(quoka, seqs, H_q, H_kv, d, N_q, B, gqa, dtype)
    for s, x in enumerate(seqs):
        if x.Q.shape[1] == 0:
            continue
        ref = single(quoka, x, N_q, B, gqa)
        assert torch.equal(got[s]["O"], ref["O"]), f"sequence {s}: O differs from the single-sequence call"
        assert torch.equal(got[s]["lse"], ref["lse"]), f"sequence {s}: lse differs"
        if ref["sel"].numel():
            assert torch.equal(got[s]["sel"], ref["sel"]), f"sequence {s}: sel differs"
        check_against_oracle(quoka, x, H_q, H_kv, d, N_q, B, gqa, dtype, got[s])


@pytest.mark.parametrize("gqa", ["max", "mean"])
def test_varlen_ragged8_full_size(quoka, gqa):
    """Eight sequences, GQA 64/8, C = 1024 each, log-uniform histories in [4K, 64K], one call."""
    cfg = wl.RAGGED_8x_BF16
    seqs = wl.make_ragged(cfg, 0)
    got = run_varlen(quoka, seqs, cfg.H_q, cfg.H_kv, cfg.d, cfg.N_q, cfg.B, gqa, cfg.dtype)
    for s, x in enumerate(seqs):
        ref = single(quoka, x, cfg.N_q, cfg.B, gqa)
        assert torch.equal(got[s]["O"], ref["O"]), f"sequence {s}"
        assert torch.equal(got[s]["sel"], ref["sel"]), f"sequence {s}"
        if s in (1, 6):
            check_against_oracle(quoka, x, cfg.H_q, cfg.H_kv, cfg.d, cfg.N_q, cfg.B, gqa, cfg.dtype, got[s])


def test_varlen_more_sequences_than_one_joint_launch(quoka):
    """Twenty-five sequences: the bf16 chunks above decode size (G * C_s > 32) attend in joint
    launches of at most 16 sequences each; decode-size chunks, histories within the budget and
    empty histories mixed in.  Every sequence must match its single-sequence call bit for bit."""
    H_q, H_kv, d, N_q, B = 8, 2, 128, 9, 40
    Cs = [130, 1, 77, 9, 256, 8, 33, 200, 2, 129, 64]
    Ts = [300, 1000, 0, 50, 2100, 129, 40, 777, 0, 128]
    shapes = [(Cs[i % len(Cs)], Ts[i % len(Ts)]) for i in range(25)]
    assert sum(4 * C > 32 for C, _ in shapes) > 16
    seqs = [wl.small_chunk(H_q=H_q, H_kv=H_kv, d=d, C=C, T=T, N_q=N_q, B=B, dtype="bf16", seed=60 + i)[1]
            for i, (C, T) in enumerate(shapes)]
    for gqa in ("max", "mean"):
        got = run_varlen(quoka, seqs, H_q, H_kv, d, N_q, B, gqa, "bf16")
        for s, x in enumerate(seqs):
            ref = single(quoka, x, N_q, B, gqa)
            assert torch.equal(got[s]["O"], ref["O"]), f"{gqa}: sequence {s} {shapes[s]}: O differs"
            assert torch.equal(got[s]["lse"], ref["lse"]), f"{gqa}: sequence {s}: lse differs"
            if ref["sel"].numel():
                assert torch.equal(got[s]["sel"], ref["sel"]), f"{gqa}: sequence {s}: sel differs"
            if s in (4, 17, 20):
                check_against_oracle(quoka, x, H_q, H_kv, d, N_q, B, gqa, "bf16", got[s])


@pytest.mark.parametrize("H_q,H_kv", [(4, 4), (10, 2)], ids=["mha", "gqa5"])
def test_varlen_joint_attention_head_layouts(quoka, H_q, H_kv):
    """One query head per KV group, and an odd group size (the last head pair of a group is a
    single slot): the joint attention launch against per-sequence calls, bit for bit."""
    d, N_q, B = 128, 9, 40
    shapes = [(77, 300), (200, 1000), (130, 0), (33, 20)]
    seqs = [wl.small_chunk(H_q=H_q, H_kv=H_kv, d=d, C=C, T=T, N_q=N_q, B=B, dtype="bf16", seed=90 + i)[1]
            for i, (C, T) in enumerate(shapes)]
    for gqa in ("max", "mean"):
        got = run_varlen(quoka, seqs, H_q, H_kv, d, N_q, B, gqa, "bf16")
        for s, x in enumerate(seqs):
            ref = single(quoka, x, N_q, B, gqa)
            assert torch.equal(got[s]["O"], ref["O"]), f"{gqa}: sequence {s} {shapes[s]}: O differs"
            assert torch.equal(got[s]["lse"], ref["lse"]), f"{gqa}: sequence {s}: lse differs"
        check_against_oracle(quoka, seqs[1], H_q, H_kv, d, N_q, B, gqa, "bf16", got[1])


def test_sparse_attend_varlen_matches_single_calls(quoka):
    """quoka_sparse_attend_varlen on packed kept rows: every sequence's O and lse equal
    quoka_sparse_attend (tensor-core engine) on that sequence bit for bit, and the oracle's
    attention within the bf16 tolerance.  Kept-row counts include 0 and ragged tails; one
    chunk is empty; twenty sequences take two launches."""
    q = quoka
    H_q, H_kv, d = 8, 2, 128
    shapes = [(130, 40), (1, 0), (77, 300), (0, 50), (256, 129), (33, 128), (200, 7), (5, 2048), (129, 1000),
              (64, 64)] * 2
    g = torch.Generator().manual_seed(7)
    mk = lambda h, n: (torch.randn((h, n, d), generator=g) * 0.5).to(torch.bfloat16)
    seqs = [(mk(H_q, C), mk(H_kv, B), mk(H_kv, B), mk(H_kv, C), mk(H_kv, C)) for C, B in shapes]
    cu_C = [0] + list(np.cumsum([C for C, _ in shapes]))
    cu_B = [0] + list(np.cumsum([B for _, B in shapes]))
    cat = lambda i: torch.cat([x[i].reshape(-1) for x in seqs]).to(DEV)
    Q, Ks, Vs, Kc, Vc = (cat(i) for i in range(5))
    O = torch.full_like(Q, float("nan"))
    lse = torch.full((H_q * cu_C[-1],), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    vs = q.varlen_shape_of(len(shapes), H_q, H_kv, d, torch.bfloat16)
    params = q.params_of("max")
    q.quoka_sparse_attend_varlen(vs, cu_B, cu_C, Q, Ks, Vs, Kc, Vc, params, O, lse, ws)
    torch.cuda.synchronize()
    assert q.quoka_get_last_device_error(ws) == 0
    tensor = q.params_of("max")
    tensor.engine = 2
    for s, (C, B) in enumerate(shapes):
        if C == 0:
            continue
        x = [t.to(DEV) for t in seqs[s]]
        shape = q.shape_of(x[0], x[1], H_kv=H_kv)
        O1 = torch.empty_like(x[0])
        lse1 = torch.empty((H_q, C), dtype=torch.float32, device=DEV)
        ws1 = q.make_workspace(shape, 1, max(B, 1), tensor)
        q.quoka_sparse_attend(shape, x[0], x[1] if B else None, x[2] if B else None, B, x[3], x[4], tensor, O1,
                              lse1, ws1)
        torch.cuda.synchronize()
        c0, c1 = cu_C[s], cu_C[s + 1]
        Ov = O[H_q * d * c0:H_q * d * c1].view(H_q, C, d)
        assert torch.equal(Ov, O1), f"sequence {s} {shapes[s]}: O differs from quoka_sparse_attend"
        assert torch.equal(lse[H_q * c0:H_q * c1].view(H_q, C), lse1), f"sequence {s}: lse differs"
        if s in (0, 4, 8):
            O_ref, _ = qo.attend(*(f64(t) for t in seqs[s]))
            check_output(Ov, O_ref, f"O (sequence {s})")


def test_varlen_decode_batch(quoka):
    """Batched decode: twelve sequences of one new token each over histories of 1 to 3000 keys."""
    H_q, H_kv, d, N_q, B = 8, 2, 128, 1, 64
    Ts = [1, 63, 64, 65, 300, 1000, 3000, 7, 129, 2048, 511, 0]
    seqs = [wl.small_chunk(H_q=H_q, H_kv=H_kv, d=d, C=1, T=T, N_q=N_q, B=B, dtype="bf16", seed=40 + i)[1]
            for i, T in enumerate(Ts)]
    for gqa in ("max", "mean"):
        got = run_varlen(quoka, seqs, H_q, H_kv, d, N_q, B, gqa, "bf16")
        for s, x in enumerate(seqs):
            ref = single(quoka, x, N_q, B, gqa)
            assert torch.equal(got[s]["O"], ref["O"]), f"sequence {s}"
            check_against_oracle(quoka, x, H_q, H_kv, d, N_q, B, gqa, "bf16", got[s])
