"""Python binding of libquoka.so (ctypes).

Argument marshalling only: every function here turns torch tensors into the
pointers and sizes of the C entry point with the same name and raises
QuokaError on a non-OK status.  All compute runs in the library's CUDA
kernels; there is no Python or CPU fallback.  Tensors must be CUDA tensors,
contiguous, in the dtype of the shape (bf16 or fp32); the history K/V may be a
larger preallocated cache (see ``shape_of``'s ``kv_head_stride``).
"""
from __future__ import annotations

import ctypes
import os
from pathlib import Path

import torch

_LIB_PATH = Path(__file__).resolve().parent / "libquoka.so"
_lib = None

QUOKA_OK = 0
STATUS = {0: "QUOKA_OK", 1: "QUOKA_ERR_INVALID_ARG", 2: "QUOKA_ERR_UNSUPPORTED", 3: "QUOKA_ERR_WORKSPACE",
          4: "QUOKA_ERR_ALIGNMENT", 5: "QUOKA_ERR_CUDA", 6: "QUOKA_ERR_TIMEOUT", 7: "QUOKA_ERR_DEVICE"}
DTYPE = {torch.bfloat16: 0, torch.float32: 1}
GQA = {"mean": 0, "max": 1}
ENGINE = {"auto": 0, "simt": 1, "tensor": 2}


class QuokaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


class Shape(ctypes.Structure):
    _fields_ = [("kv_head_stride", ctypes.c_int64), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
                ("C", ctypes.c_int32), ("T", ctypes.c_int32), ("d", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class Params(ctypes.Structure):
    _fields_ = [("gqa_pool", ctypes.c_int32), ("engine", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("flags", ctypes.c_int32)]


class VarlenShape(ctypes.Structure):
    _fields_ = [("nseq", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("d", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_P = ctypes.c_void_p
_I64P = ctypes.POINTER(ctypes.c_int64)
_SIG = {
    "quoka_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "quoka_workspace_size": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_int, ctypes.c_int,
                                            ctypes.POINTER(Params), ctypes.POINTER(ctypes.c_size_t)]),
    "quoka_select_queries": (ctypes.c_int, [ctypes.POINTER(Shape), _P, ctypes.c_int, ctypes.POINTER(Params), _P,
                                            _P, ctypes.c_size_t, _P]),
    "quoka_select_queries_noalloc": (ctypes.c_int, [ctypes.POINTER(Shape), _P, ctypes.c_int, ctypes.POINTER(Params),
                                                    _P, _P]),
    "quoka_score_keys": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, ctypes.c_int, _P, ctypes.POINTER(Params), _P,
                                        _P, ctypes.c_size_t, _P]),
    "quoka_topk": (ctypes.c_int, [ctypes.POINTER(Shape), _P, ctypes.c_int, _P, _P, ctypes.c_size_t, _P]),
    "quoka_gather": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, _P, ctypes.c_int, _P, _P, _P]),
    "quoka_sparse_attend": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, _P, ctypes.c_int, _P, _P,
                                           ctypes.POINTER(Params), _P, _P, _P, ctypes.c_size_t, _P]),
    "quoka_chunk_attend": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(Params), _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "quoka_workspace_size_varlen": (ctypes.c_int, [ctypes.POINTER(VarlenShape), _I64P, _I64P, ctypes.c_int,
                                                   ctypes.c_int, ctypes.POINTER(Params),
                                                   ctypes.POINTER(ctypes.c_size_t)]),
    "quoka_chunk_attend_varlen": (ctypes.c_int, [ctypes.POINTER(VarlenShape), _I64P, _I64P, _P, _P, _P, _P, _P,
                                                 ctypes.c_int, ctypes.c_int, ctypes.POINTER(Params), _P, _P, _P, _P,
                                                 ctypes.c_size_t, _P]),
    "quoka_sparse_attend_varlen": (ctypes.c_int, [ctypes.POINTER(VarlenShape), _I64P, _I64P, _P, _P, _P, _P, _P,
                                                  ctypes.POINTER(Params), _P, _P, _P, ctypes.c_size_t, _P]),
    "quoka_key_inv_norms": (ctypes.c_int, [ctypes.POINTER(Shape), _P, ctypes.c_int, ctypes.c_int, _P, ctypes.c_int64,
                                           _P]),
    "quoka_score_keys_cached": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, ctypes.c_int, _P, _P, ctypes.c_int64,
                                               ctypes.POINTER(Params), _P, _P, ctypes.c_size_t, _P]),
    "quoka_chunk_attend_cached": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, _P, ctypes.c_int64,
                                                 ctypes.c_int, ctypes.c_int, ctypes.POINTER(Params), _P, _P, _P, _P,
                                                 ctypes.c_size_t, _P]),
    "quoka_append_kv_norms": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, ctypes.c_int64, _P]),
    "quoka_dense_attend": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P, ctypes.POINTER(Params), _P, _P,
                                          _P, ctypes.c_size_t, _P]),
    "quoka_append_kv": (ctypes.c_int, [ctypes.POINTER(Shape), _P, _P, _P, _P, _P]),
    "quoka_get_last_device_error": (ctypes.c_int, [_P, _P]),
    "quoka_launch_count": (ctypes.c_uint64, []),
    "quoka_last_cuda_error_string": (ctypes.c_char_p, []),
    "quoka_selftest_expire_wait": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_longlong, _P]),
    "quoka_stage_engine": (ctypes.c_int, [ctypes.POINTER(Shape), ctypes.POINTER(Params), ctypes.c_int]),
}


def lib_path() -> Path:
    return _LIB_PATH


def load(path: str | os.PathLike | None = None):
    """Load libquoka.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path is not None else _LIB_PATH
    if not p.exists():
        raise RuntimeError(f"{p} is missing: build it first (python -m sparse_attention_chunked_gb300.build)")
    lib = ctypes.CDLL(str(p))
    for name, (res, args) in _SIG.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(fn, rc):
    if rc != QUOKA_OK:
        err = QuokaError(fn, rc)
        if rc == 5:   # QUOKA_ERR_CUDA: say which CUDA error
            err.args = (f"{err.args[0]} ({load().quoka_last_cuda_error_string().decode()})",)
        raise err


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libquoka takes CUDA tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def shape_of(Q: torch.Tensor, K_hist: torch.Tensor | None, H_kv: int | None = None, T: int | None = None,
             kv_head_stride: int = 0) -> Shape:
    """Shape of a chunk: Q [H_q, C, d]; K_hist [H_kv, >=T, d] (T defaults to its length)."""
    H_q, C, d = Q.shape
    if K_hist is not None:
        H_kv = K_hist.shape[0] if H_kv is None else H_kv
        if T is None:
            T = K_hist.shape[1]
        if kv_head_stride == 0 and K_hist.shape[1] != T:
            kv_head_stride = K_hist.stride(0)
    return Shape(kv_head_stride, H_q, H_kv, C, T or 0, d, DTYPE[Q.dtype])


SCORE_FLAGS = {"cos": 0, "dot": 1}        # QUOKA_FLAG_SCORE_DOT
QUERY_AGG_FLAGS = {"max": 0, "mean": 2}   # QUOKA_FLAG_QUERY_MEAN


def params_of(gqa: str = "mean", engine: str = "auto", softmax_scale: float = 0.0, score_fn: str = "cos",
              query_agg: str = "max") -> Params:
    return Params(GQA[gqa], ENGINE[engine], softmax_scale, SCORE_FLAGS[score_fn] | QUERY_AGG_FLAGS[query_agg])


def workspace_size(shape: Shape, N_q: int, B: int, params: Params) -> int:
    n = ctypes.c_size_t(0)
    _check("quoka_workspace_size", load().quoka_workspace_size(ctypes.byref(shape), N_q, B, ctypes.byref(params),
                                                               ctypes.byref(n)))
    return n.value


def make_workspace(shape: Shape, N_q: int, B: int, params: Params, device="cuda") -> torch.Tensor:
    """A zeroed workspace tensor (uint8) of the size quoka_workspace_size asks for (256-byte aligned)."""
    n = workspace_size(shape, N_q, B, params)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def status_string(status: int) -> str:
    return load().quoka_status_string(status).decode()


def quoka_select_queries(shape, Q, N_q, params, q_idx, ws, stream=None):
    _check("quoka_select_queries", load().quoka_select_queries(
        ctypes.byref(shape), _ptr(Q), N_q, ctypes.byref(params), _ptr(q_idx), _ptr(ws), ws.numel(), _stream(stream)))


def quoka_select_queries_noalloc(shape, Q, N_q, params, q_idx, stream=None):
    _check("quoka_select_queries_noalloc", load().quoka_select_queries_noalloc(
        ctypes.byref(shape), _ptr(Q), N_q, ctypes.byref(params), _ptr(q_idx), _stream(stream)))


def quoka_score_keys(shape, Q, q_idx, N_q, K_hist, params, scores, ws, stream=None):
    _check("quoka_score_keys", load().quoka_score_keys(
        ctypes.byref(shape), _ptr(Q), _ptr(q_idx), N_q, _ptr(K_hist), ctypes.byref(params), _ptr(scores), _ptr(ws),
        ws.numel(), _stream(stream)))


def quoka_topk(shape, scores, B, sel, ws, stream=None):
    _check("quoka_topk", load().quoka_topk(ctypes.byref(shape), _ptr(scores), B, _ptr(sel), _ptr(ws), ws.numel(),
                                           _stream(stream)))


def quoka_gather(shape, K_hist, V_hist, sel, B_e, K_sel, V_sel, stream=None):
    _check("quoka_gather", load().quoka_gather(ctypes.byref(shape), _ptr(K_hist), _ptr(V_hist), _ptr(sel), B_e,
                                               _ptr(K_sel), _ptr(V_sel), _stream(stream)))


def quoka_sparse_attend(shape, Q, K_sel, V_sel, B_e, K_chunk, V_chunk, params, O, lse, ws, stream=None):
    _check("quoka_sparse_attend", load().quoka_sparse_attend(
        ctypes.byref(shape), _ptr(Q), _ptr(K_sel), _ptr(V_sel), B_e, _ptr(K_chunk), _ptr(V_chunk),
        ctypes.byref(params), _ptr(O), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))


def quoka_chunk_attend(shape, Q, K_hist, V_hist, K_chunk, V_chunk, N_q, B, params, O, lse, sel_out, ws,
                       stream=None):
    _check("quoka_chunk_attend", load().quoka_chunk_attend(
        ctypes.byref(shape), _ptr(Q), _ptr(K_hist), _ptr(V_hist), _ptr(K_chunk), _ptr(V_chunk), N_q, B,
        ctypes.byref(params), _ptr(O), _ptr(lse), _ptr(sel_out), _ptr(ws), ws.numel(), _stream(stream)))


def _cu(offsets):
    """Host int64 prefix-sum array for the ragged entry points."""
    arr = (ctypes.c_int64 * len(offsets))(*[int(v) for v in offsets])
    return arr


def varlen_shape_of(nseq: int, H_q: int, H_kv: int, d: int, dtype) -> VarlenShape:
    return VarlenShape(nseq, H_q, H_kv, d, DTYPE[dtype] if isinstance(dtype, torch.dtype) else dtype, 0)


def quoka_workspace_size_varlen(vshape, cu_T, cu_C, N_q, B, params) -> int:
    n = ctypes.c_size_t(0)
    _check("quoka_workspace_size_varlen", load().quoka_workspace_size_varlen(
        ctypes.byref(vshape), _cu(cu_T), _cu(cu_C), N_q, B, ctypes.byref(params), ctypes.byref(n)))
    return n.value


def quoka_chunk_attend_varlen(vshape, cu_T, cu_C, Q, K_hist, V_hist, K_chunk, V_chunk, N_q, B, params, O, lse,
                              sel_out, ws, stream=None):
    """cu_T, cu_C: host sequences of nseq + 1 prefix sums; tensors packed sequence-major (see quoka.h)."""
    _check("quoka_chunk_attend_varlen", load().quoka_chunk_attend_varlen(
        ctypes.byref(vshape), _cu(cu_T), _cu(cu_C), _ptr(Q), _ptr(K_hist), _ptr(V_hist), _ptr(K_chunk),
        _ptr(V_chunk), N_q, B, ctypes.byref(params), _ptr(O), _ptr(lse), _ptr(sel_out), _ptr(ws),
        ws.numel() if ws is not None else 0, _stream(stream)))


def quoka_sparse_attend_varlen(vshape, cu_B, cu_C, Q, K_sel, V_sel, K_chunk, V_chunk, params, O, lse, ws,
                               stream=None):
    """cu_B, cu_C: host sequences of nseq + 1 prefix sums; tensors packed sequence-major (see quoka.h)."""
    _check("quoka_sparse_attend_varlen", load().quoka_sparse_attend_varlen(
        ctypes.byref(vshape), _cu(cu_B), _cu(cu_C), _ptr(Q), _ptr(K_sel), _ptr(V_sel), _ptr(K_chunk), _ptr(V_chunk),
        ctypes.byref(params), _ptr(O), _ptr(lse), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def quoka_dense_attend(shape, Q, K_hist, V_hist, K_chunk, V_chunk, params, O, lse, ws, stream=None):
    _check("quoka_dense_attend", load().quoka_dense_attend(
        ctypes.byref(shape), _ptr(Q), _ptr(K_hist), _ptr(V_hist), _ptr(K_chunk), _ptr(V_chunk), ctypes.byref(params),
        _ptr(O), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))


def quoka_key_inv_norms(shape, K_hist, t0, t1, k_inv_norm, stream=None):
    """k_inv_norm: fp32 [H_kv, >= t1] (its row stride is the cache's head stride)."""
    _check("quoka_key_inv_norms", load().quoka_key_inv_norms(
        ctypes.byref(shape), _ptr(K_hist), t0, t1, _ptr(k_inv_norm), k_inv_norm.stride(0), _stream(stream)))


def quoka_score_keys_cached(shape, Q, q_idx, N_q, K_hist, k_inv_norm, params, scores, ws, stream=None):
    _check("quoka_score_keys_cached", load().quoka_score_keys_cached(
        ctypes.byref(shape), _ptr(Q), _ptr(q_idx), N_q, _ptr(K_hist), _ptr(k_inv_norm), k_inv_norm.stride(0),
        ctypes.byref(params), _ptr(scores), _ptr(ws), ws.numel(), _stream(stream)))


def quoka_chunk_attend_cached(shape, Q, K_hist, V_hist, K_chunk, V_chunk, k_inv_norm, N_q, B, params, O, lse,
                              sel_out, ws, stream=None):
    _check("quoka_chunk_attend_cached", load().quoka_chunk_attend_cached(
        ctypes.byref(shape), _ptr(Q), _ptr(K_hist), _ptr(V_hist), _ptr(K_chunk), _ptr(V_chunk), _ptr(k_inv_norm),
        k_inv_norm.stride(0), N_q, B, ctypes.byref(params), _ptr(O), _ptr(lse), _ptr(sel_out), _ptr(ws), ws.numel(),
        _stream(stream)))


def quoka_append_kv_norms(shape, K_hist, V_hist, K_chunk, V_chunk, k_inv_norm, stream=None):
    _check("quoka_append_kv_norms", load().quoka_append_kv_norms(
        ctypes.byref(shape), _ptr(K_hist), _ptr(V_hist), _ptr(K_chunk), _ptr(V_chunk), _ptr(k_inv_norm),
        k_inv_norm.stride(0), _stream(stream)))


def quoka_append_kv(shape, K_hist, V_hist, K_chunk, V_chunk, stream=None):
    _check("quoka_append_kv", load().quoka_append_kv(ctypes.byref(shape), _ptr(K_hist), _ptr(V_hist), _ptr(K_chunk),
                                                     _ptr(V_chunk), _stream(stream)))


def quoka_stage_engine(shape, params, stage: int) -> int:
    rc = load().quoka_stage_engine(ctypes.byref(shape), ctypes.byref(params), stage)
    if rc < 0:
        raise QuokaError("quoka_stage_engine", -rc)
    return rc


def uses_tensor_cores(stage: str, shape, params) -> bool:
    """True if the library runs `stage` ("score" or "attend") on tcgen05 tensor cores for this problem."""
    return quoka_stage_engine(shape, params, {"score": 0, "attend": 1}[stage]) == ENGINE["tensor"]


def quoka_selftest_expire_wait(ws, cycles: int, stream=None):
    _check("quoka_selftest_expire_wait", load().quoka_selftest_expire_wait(_ptr(ws), ws.numel(), cycles,
                                                                           _stream(stream)))


def quoka_launch_count() -> int:
    return int(load().quoka_launch_count())


def quoka_get_last_device_error(ws, stream=None) -> int:
    return load().quoka_get_last_device_error(_ptr(ws), _stream(stream))


# ---------------------------------------------------------------- convenience wrappers

def chunk_attend(Q, K_hist, V_hist, K_chunk, V_chunk, N_q, B, gqa="mean", engine="auto", T=None, ws=None,
                 with_lse=False, with_sel=False, stream=None):
    """Allocate outputs (and a workspace unless given) and run quoka_chunk_attend."""
    shape = shape_of(Q, K_hist, H_kv=K_chunk.shape[0], T=T)
    params = params_of(gqa, engine)
    if ws is None:
        ws = make_workspace(shape, N_q, B, params, device=Q.device)
    O = torch.empty_like(Q)
    lse = torch.empty(Q.shape[:2], dtype=torch.float32, device=Q.device) if with_lse else None
    B_e = min(B, shape.T)
    sel = torch.empty((shape.H_kv, B_e), dtype=torch.int32, device=Q.device) if with_sel and B_e > 0 else None
    quoka_chunk_attend(shape, Q, K_hist, V_hist, K_chunk, V_chunk, N_q, B, params, O, lse, sel, ws, stream)
    return O, lse, sel
