"""The C ABI without a GPU: the library loads, exports what include/quoka.h declares,
and rejects bad arguments on the host before anything is enqueued."""
import ctypes
import re
from pathlib import Path

import pytest

HEADER = Path(__file__).resolve().parent.parent / "include" / "quoka.h"

# A fake, 256-byte aligned device address: every call below fails its host-side
# checks before any pointer is used, so the address is never dereferenced.
FAKE = 1 << 20


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(quoka_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_stage_entry_points():
    names = declared_functions()
    for fn in ("quoka_select_queries", "quoka_score_keys", "quoka_topk", "quoka_gather", "quoka_sparse_attend",
               "quoka_chunk_attend", "quoka_dense_attend", "quoka_append_kv", "quoka_workspace_size",
               "quoka_get_last_device_error", "quoka_status_string"):
        assert fn in names


def test_library_exports_every_declared_symbol(quoka):
    lib = ctypes.CDLL(str(quoka.lib_path()))
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_missing_library_fails_loudly(quoka, tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        quoka.load(tmp_path / "nope.so")


def _shape(q, **kw):
    base = dict(kv_head_stride=0, H_q=8, H_kv=2, C=128, T=1000, d=128, dtype=0)
    base.update(kw)
    return q.Shape(**base)


def test_status_strings(quoka):
    assert quoka.status_string(0) == "QUOKA_OK"
    assert quoka.status_string(3) == "QUOKA_ERR_WORKSPACE"
    assert quoka.status_string(99) == "QUOKA_ERR_UNKNOWN"


def test_workspace_size_grows_with_problem(quoka):
    p = quoka.params_of("max")
    small = quoka.workspace_size(_shape(quoka), 16, 64, p)
    big = quoka.workspace_size(_shape(quoka, T=100000), 16, 4096, p)
    assert 256 < small < big
    assert small % 256 == 0 and big % 256 == 0
    # mean pooling scores with fewer rows than max pooling
    assert quoka.workspace_size(_shape(quoka), 16, 64, quoka.params_of("mean")) < small


@pytest.mark.parametrize("kw,code", [
    (dict(H_q=6, H_kv=4), 1),          # H_q not a multiple of H_kv
    (dict(H_kv=0), 1),
    (dict(C=0), 1),
    (dict(T=-1), 1),
    (dict(dtype=7), 1),
    (dict(d=96), 2),                   # head dim outside 64/128
    (dict(C=9000), 2),
    (dict(kv_head_stride=1000 * 128 - 1), 1),   # stride below T*d
    (dict(kv_head_stride=1001 * 128 + 4), 4),   # stride not a multiple of 16 bytes
])
def test_shape_checks(quoka, kw, code):
    n = ctypes.c_size_t(0)
    rc = quoka.load().quoka_workspace_size(ctypes.byref(_shape(quoka, **kw)), 4, 16,
                                           ctypes.byref(quoka.params_of()), ctypes.byref(n))
    assert rc == code, quoka.status_string(rc)


def _chunk_call(q, shape, N_q=4, B=16, ws=FAKE, ws_bytes=None, params=None, Q=FAKE, O=FAKE, sel=None):
    p = params or q.params_of("max")
    if ws_bytes is None:
        ws_bytes = 1 << 30
    P = ctypes.c_void_p
    return q.load().quoka_chunk_attend(ctypes.byref(shape), P(Q), P(FAKE), P(FAKE), P(FAKE), P(FAKE), N_q, B,
                                       ctypes.byref(p), P(O), None, P(sel) if sel else None, P(ws), ws_bytes, None)


def test_chunk_attend_argument_errors(quoka):
    q = quoka
    s = _shape(q)
    assert _chunk_call(q, s, N_q=0) == 1
    assert _chunk_call(q, s, B=0) == 1
    assert _chunk_call(q, s, Q=0) == 1                       # NULL query
    assert _chunk_call(q, s, Q=FAKE + 8) == 4                # misaligned query
    assert _chunk_call(q, s, sel=FAKE + 2) == 4              # sel_out not 4-byte aligned (int32 elements)
    assert _chunk_call(q, s, ws=0) == 3                      # no workspace
    assert _chunk_call(q, s, ws=FAKE + 16) == 3              # workspace not 256-byte aligned
    need = q.workspace_size(s, 4, 16, q.params_of("max"))
    assert _chunk_call(q, s, ws_bytes=need - 1) == 3         # workspace too small
    assert _chunk_call(q, s, params=q.Params(5, 0, 0.0, 0)) == 1     # unknown pooling
    assert _chunk_call(q, s, params=q.Params(0, 9, 0.0, 0)) == 1     # unknown engine
    assert _chunk_call(q, s, params=q.Params(0, 0, 0.0, 4)) == 1     # undefined flag bit
    assert _chunk_call(q, s, params=q.Params(0, 0, float("nan"), 0)) == 1


def test_stage_argument_errors(quoka):
    q = quoka
    lib = q.load()
    s = _shape(q)
    P = ctypes.c_void_p
    p = q.params_of("max")
    assert lib.quoka_select_queries(ctypes.byref(s), P(FAKE), 0, ctypes.byref(p), P(FAKE), P(FAKE), 1 << 30, None) == 1
    assert lib.quoka_select_queries(ctypes.byref(s), P(FAKE), 4, ctypes.byref(p), P(FAKE), P(FAKE), 16, None) == 3
    assert lib.quoka_score_keys(ctypes.byref(s), P(FAKE), P(FAKE), 4, P(FAKE + 2), ctypes.byref(p), P(FAKE), P(FAKE),
                                1 << 30, None) == 4
    assert lib.quoka_topk(ctypes.byref(s), P(FAKE), 0, P(FAKE), P(FAKE), 1 << 30, None) == 1
    assert lib.quoka_topk(ctypes.byref(s), P(FAKE), 8, P(FAKE), P(0), 1 << 30, None) == 3
    assert lib.quoka_gather(ctypes.byref(s), P(FAKE), P(FAKE), P(FAKE), 1001, P(FAKE), P(FAKE), None) == 1
    assert lib.quoka_gather(ctypes.byref(s), P(FAKE), P(FAKE), P(FAKE), -1, P(FAKE), P(FAKE), None) == 1
    assert lib.quoka_sparse_attend(ctypes.byref(s), P(FAKE), P(0), P(0), 5, P(FAKE), P(FAKE), ctypes.byref(p), P(FAKE),
                                   None, P(FAKE), 1 << 30, None) == 1
    # appending needs room for T + C rows per head
    assert lib.quoka_append_kv(ctypes.byref(s), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None) == 1
    assert lib.quoka_get_last_device_error(None, None) == 3


# ---------------------------------------------------------------- ragged batch entry point

def _vshape(q, **kw):
    base = dict(nseq=3, H_q=8, H_kv=2, d=128, dtype=0, reserved=0)
    base.update(kw)
    return q.VarlenShape(**base)


def _ws_varlen(q, vshape, cu_T, cu_C, N_q=16, B=64, gqa="max"):
    n = ctypes.c_size_t(0)
    rc = q.load().quoka_workspace_size_varlen(ctypes.byref(vshape), q._cu(cu_T), q._cu(cu_C), N_q, B,
                                              ctypes.byref(q.params_of(gqa)), ctypes.byref(n))
    return rc, n.value


def test_varlen_workspace_layout(quoka):
    """Header, then the kept K/V rows of the sequences that attend in the joint tensor-core
    launch and select keys, then one slice per stream lane (up to 8, one per non-empty
    sequence), each for the largest sequence without the joint sequences' kept rows."""
    al = lambda x: (x + 255) // 256 * 256
    H_kv, d, G, B = 2, 128, 4, 64
    for cu_T, cu_C, lanes in (([0, 1000, 1000, 41000], [0, 128, 200, 201], 3),
                              ([0, 1000, 1000, 41000], [0, 128, 128, 201], 2),
                              ([0, 50, 1050], [0, 40, 80], 2),
                              ([0, 5, 9, 13, 17, 21, 25], [0, 1, 2, 3, 4, 5, 6], 6),
                              (list(range(0, 55, 5)), list(range(0, 11)), 8)):
        rc, n = _ws_varlen(quoka, _vshape(quoka, nseq=len(cu_T) - 1), cu_T, cu_C, B=B)
        assert rc == 0
        per_lane, kept = [], 0
        for (c0, c1, t0, t1) in zip(cu_C, cu_C[1:], cu_T, cu_T[1:]):
            C, T = c1 - c0, t1 - t0
            if C == 0:
                continue
            single = quoka.workspace_size(_shape(quoka, C=C, T=T), 16, B, quoka.params_of("max"))
            joint = G * C > 32                       # bf16 above decode size: the joint attention launch
            rows = 2 * al(H_kv * min(B, T) * d * 2)  # the gathered K and V rows of a single call
            per_lane.append(single - 256 - (rows if joint else 0))
            if joint and 0 < B < T:
                kept += rows
        assert n == 256 + kept + lanes * max(per_lane)


@pytest.mark.parametrize("cu_T,cu_C,kw,code", [
    ([1, 10, 20, 30], [0, 1, 2, 3], {}, 1),          # prefix sums must start at 0
    ([0, 10, 5, 30], [0, 1, 2, 3], {}, 1),           # decreasing history offsets
    ([0, 10, 20, 30], [0, 2, 1, 3], {}, 1),          # decreasing chunk offsets
    ([0, 10, 20, 30], [0, 1, 9002, 9003], {}, 2),    # a chunk longer than 8192
    ([0, 10, 20, 30], [0, 1, 2, 3], dict(reserved=1), 1),
    ([0, 10, 20, 30], [0, 1, 2, 3], dict(H_q=6, H_kv=4), 1),
    ([0, 10, 20, 30], [0, 1, 2, 3], dict(d=96), 2),
])
def test_varlen_checks(quoka, cu_T, cu_C, kw, code):
    rc, _ = _ws_varlen(quoka, _vshape(quoka, **kw), cu_T, cu_C)
    assert rc == code, quoka.status_string(rc)


def test_varlen_checks_every_sequence_before_enqueueing(quoka):
    """Sequence 0 (no history) is valid; sequence 1 has history but K/V_hist are NULL: nothing may be enqueued."""
    q = quoka
    vs = _vshape(q, nseq=2)
    cu_T, cu_C = [0, 0, 500], [0, 64, 128]
    P = ctypes.c_void_p
    rc = q.load().quoka_chunk_attend_varlen(
        ctypes.byref(vs), q._cu(cu_T), q._cu(cu_C), P(FAKE), None, None, P(FAKE), P(FAKE), 16, 64,
        ctypes.byref(q.params_of("max")), P(FAKE), None, None, P(FAKE), 1 << 30, None)
    assert rc == 1, q.status_string(rc)
    _, need = _ws_varlen(q, vs, cu_T, cu_C)
    rc = q.load().quoka_chunk_attend_varlen(
        ctypes.byref(vs), q._cu(cu_T), q._cu(cu_C), *([P(FAKE)] * 5), 16, 64,
        ctypes.byref(q.params_of("max")), P(FAKE), None, None, P(FAKE), need - 1, None)
    assert rc == 3, q.status_string(rc)


def test_varlen_alignment_of_packed_offsets(quoka):
    """lse of sequence 1 starts at H_q * C_0 floats: 4-byte alignment is all it needs."""
    q = quoka
    vs = _vshape(q, nseq=2)
    cu_T, cu_C = [0, 500, 1000], [0, 3, 6]
    rc = q.load().quoka_chunk_attend_varlen(
        ctypes.byref(vs), q._cu(cu_T), q._cu(cu_C), *([ctypes.c_void_p(FAKE)] * 5), 16, 64,
        ctypes.byref(q.params_of("max")), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + 2), None, None, 0, None)
    assert rc == 4, q.status_string(rc)   # lse not 4-byte aligned
    rc = q.load().quoka_chunk_attend_varlen(
        ctypes.byref(vs), q._cu(cu_T), q._cu(cu_C), *([ctypes.c_void_p(FAKE)] * 5), 16, 64,
        ctypes.byref(q.params_of("max")), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + 4), None, None, 0, None)
    assert rc == 3, q.status_string(rc)   # offsets fine; fails on the missing workspace


def test_key_norm_cache_argument_errors(quoka):
    q = quoka
    lib = q.load()
    s = _shape(q)                       # T = 1000
    P = ctypes.c_void_p
    assert lib.quoka_key_inv_norms(ctypes.byref(s), P(FAKE), 0, 1001, P(FAKE), 2000, None) == 1    # t1 > T
    assert lib.quoka_key_inv_norms(ctypes.byref(s), P(FAKE), 5, 4, P(FAKE), 2000, None) == 1       # t1 < t0
    assert lib.quoka_key_inv_norms(ctypes.byref(s), P(FAKE), 0, 1000, P(FAKE), 999, None) == 1     # row too short
    assert lib.quoka_key_inv_norms(ctypes.byref(s), P(FAKE), 0, 1000, None, 2000, None) == 1        # no cache
    assert lib.quoka_key_inv_norms(ctypes.byref(s), P(FAKE), 0, 1000, P(FAKE + 2), 2000, None) == 4 # misaligned
    p = q.params_of("max")
    assert lib.quoka_chunk_attend_cached(ctypes.byref(s), *([P(FAKE)] * 5), P(FAKE), 999, 4, 16, ctypes.byref(p),
                                         P(FAKE), None, None, P(FAKE), 1 << 30, None) == 1         # stride < T
    assert lib.quoka_score_keys_cached(ctypes.byref(s), P(FAKE), P(FAKE), 4, P(FAKE), None, 1000, ctypes.byref(p),
                                       P(FAKE), P(FAKE), 1 << 30, None) == 1
    # appending C = 128 keys needs room for T + C norms per row
    assert lib.quoka_append_kv_norms(ctypes.byref(_shape(q, kv_head_stride=2000 * 128)), *([P(FAKE)] * 4), P(FAKE),
                                     1100, None) == 1


def test_sparse_attend_varlen_checks(quoka):
    """The ragged attention entry point: prefix sums, element type, engine, alignment, workspace."""
    q = quoka
    P = ctypes.c_void_p
    fn = q.load().quoka_sparse_attend_varlen
    cu_B, cu_C = [0, 100, 100], [0, 64, 200]

    def call(vs, cuB=cu_B, cuC=cu_C, params=None, lse=None, ws_bytes=256, ksel=P(FAKE)):
        return fn(ctypes.byref(vs), q._cu(cuB), q._cu(cuC), P(FAKE), ksel, ksel, P(FAKE), P(FAKE),
                  ctypes.byref(params or q.params_of("max")), P(FAKE), lse, P(FAKE), ws_bytes, None)

    vs = _vshape(q, nseq=2)
    assert call(vs, cuB=[1, 100, 100]) == 1                     # prefix sums must start at 0
    assert call(vs, cuC=[0, 64, 9000]) == 2                     # a chunk longer than 8192
    assert call(_vshape(q, nseq=2, dtype=1)) == 2               # fp32: no tensor-core attention
    simt = q.params_of("max")
    simt.engine = 1
    assert call(vs, params=simt) == 2                           # the CUDA-core engine is not offered
    assert call(vs, ksel=None) == 1                             # kept rows but no K_sel / V_sel
    assert call(vs, lse=P(FAKE + 2)) == 4                       # lse needs 4-byte alignment
    assert call(vs, ws_bytes=255) == 3                          # the error header

