"""Block-quantized-weight matmul on GB300 (sm_103a): Python binding.

A thin ctypes layer over libcq.so: each function takes torch tensors (or
numpy arrays for host-side helpers), checks nothing itself, and passes
pointers and sizes to the C entry point of the same name.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback,
and the functions raise if the library is missing.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcq.so")
INCLUDE = os.path.join(os.path.dirname(_HERE), "include", "cq.h")

CQ_F16, CQ_BF16, CQ_F32 = 0, 1, 2
CQ_OPT_SMALL_T_MAX, CQ_OPT_FORCE_PATH, CQ_OPT_WAIT_NS, CQ_OPT_TEST_STALL, CQ_OPT_TRACE, CQ_OPT_TC_BN, CQ_OPT_TC_KSPLIT, \
    CQ_OPT_TC_AMODE, CQ_OPT_TC_PAIR, CQ_OPT_STREAM_KERNEL = 0, 1, 2, 3, 4, 5, 6, 7, 8, 9
STATUS = {0: "CQ_OK", 1: "CQ_ERR_NULL", 2: "CQ_ERR_DTYPE", 3: "CQ_ERR_SHAPE", 4: "CQ_ERR_ALIGN",
          5: "CQ_ERR_INDEX", 6: "CQ_ERR_WORKSPACE", 7: "CQ_ERR_CUDA", 8: "CQ_ERR_TIMEOUT", 9: "CQ_ERR_ARCH",
          10: "CQ_ERR_ARG"}

_lib = None

_c_p, _c_i64, _c_int, _c_sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "cq_gemm_q4_workspace_bytes": (_c_sz, [_c_i64, _c_i64]),
    "cq_gemm_q4": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_p, _c_p, _c_i64, _c_p, _c_int, _c_p, _c_sz, _c_p]),
    "cq_gemm_q4_noalloc": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_p, _c_p, _c_i64, _c_p, _c_int, _c_p]),
    "cq_gemm_q8row": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_p, _c_p, _c_i64, _c_p, _c_int, _c_p]),
    "cq_moe_workspace_bytes": (_c_sz, [_c_i64] * 5),
    "cq_ffn_q4_workspace_bytes": (_c_sz, [_c_i64] * 3),
    "cq_gemm_q8b_workspace_bytes": (_c_sz, [_c_i64, _c_i64]),
    "cq_gemm_q8b": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_p, _c_p, _c_i64, _c_p, _c_int, _c_p, _c_sz, _c_p]),
    "cq_gemm_q4a_workspace_bytes": (_c_sz, [_c_i64] * 4),
    "cq_gemm_q4a": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_p, _c_int, _c_p, _c_sz,
                             _c_p]),
    "cq_gemm_q8_2f_workspace_bytes": (_c_sz, [_c_i64, _c_i64]),
    "cq_gemm_q8_2f": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_int, _c_p, _c_sz, _c_p]),
    "cq_gemm_q4_batched_workspace_bytes": (_c_sz, [_c_i64, _c_i64, _c_int]),
    "cq_gemm_q4_batched": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_p, _c_int, _c_i64, _c_p, _c_int, _c_i64,
                                    _c_p, _c_sz, _c_p]),
    "cq_ffn_q4": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_p, _c_sz,
                           _c_p]),
    "cq_moe_panels": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_p,
                               _c_p, _c_p, _c_p, _c_int, _c_p, _c_sz, _c_p]),
    "cq_moe_route": (_c_int, [_c_p, _c_i64, _c_i64, _c_i64, _c_int, _c_p, _c_p, _c_p]),
    "cq_moe_layout": (_c_int, [_c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_p]),
    "cq_dequant_q4": (_c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_p, _c_p]),
    "cq_dequant_q8row": (_c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_p, _c_p]),
    "cq_get_device_error": (_c_int, [_c_p]),
    "cq_last_error": (ctypes.c_char_p, []),
    "cq_last_launches": (_c_int, []),
    "cq_set_option": (_c_int, [_c_int, _c_i64]),
    "cq_get_option": (_c_i64, [_c_int]),
    "cq_version": (_c_int, []),
}


class CQError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


def lib():
    """The loaded libcq.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libcq.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(st: int):
    if st != 0:
        raise CQError(st, lib().cq_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _xt(t):
    import torch
    if t.dtype == torch.float16:
        return CQ_F16
    if t.dtype == torch.bfloat16:
        return CQ_BF16
    if t.dtype == torch.float32:
        return CQ_F32
    return -1


# ---- entry points (same names as the C ABI) -----------------------------

def cq_gemm_q4_workspace_bytes(T: int, K: int) -> int:
    return lib().cq_gemm_q4_workspace_bytes(T, K)


def cq_gemm_q4(X, Wq, Ws, Y, ws, stream=None, raise_on_error=True):
    """Y[T][N] = X[T][K] . dequant(Wq, Ws)^T.  X fp16/bf16, Wq uint8 [N][K/2],
    Ws int16/uint16-bits fp16 [N][K/32], Y f32/bf16 [T][N], ws uint8."""
    T, K = X.shape
    N = Wq.shape[0]
    st = lib().cq_gemm_q4(_ptr(X), _xt(X), T, K, _ptr(Wq), _ptr(Ws), N, _ptr(Y), _xt(Y), _ptr(ws),
                          0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    if raise_on_error:
        _check(st)
    return st


def cq_gemm_q4_noalloc(X, Wq, Ws, Y, stream=None, raise_on_error=True):
    """cq_gemm_q4 without a caller workspace: for callers that cannot
    allocate device memory; the scratch is a fixed array inside the library
    (see include/cq.h for the size limit and the sharing rules)."""
    T, K = X.shape
    N = Wq.shape[0]
    st = lib().cq_gemm_q4_noalloc(_ptr(X), _xt(X), T, K, _ptr(Wq), _ptr(Ws), N, _ptr(Y), _xt(Y), _stream(stream))
    if raise_on_error:
        _check(st)
    return st


def cq_gemm_q8row(X, Wq, rs, Y, stream=None, raise_on_error=True):
    T, K = X.shape
    N = Wq.shape[0]
    st = lib().cq_gemm_q8row(_ptr(X), _xt(X), T, K, _ptr(Wq), _ptr(rs), N, _ptr(Y), _xt(Y), _stream(stream))
    if raise_on_error:
        _check(st)
    return st


def cq_moe_workspace_bytes(T, H, I, E, topk) -> int:
    return lib().cq_moe_workspace_bytes(T, H, I, E, topk)


def cq_moe_panels(X, idx, w, Wgu_q, Wgu_s, Wd_q, Wd_s, Y, ws, stream=None, raise_on_error=True):
    T, H = X.shape
    E, twoI = Wgu_q.shape[0], Wgu_q.shape[1]
    topk = idx.shape[1]
    st = lib().cq_moe_panels(_ptr(X), _xt(X), T, H, E, twoI // 2, topk, _ptr(idx), _ptr(w), _ptr(Wgu_q),
                             _ptr(Wgu_s), _ptr(Wd_q), _ptr(Wd_s), _ptr(Y), _xt(Y), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream))
    if raise_on_error:
        _check(st)
    return st


class cq_q4_job(ctypes.Structure):
    """One job of cq_gemm_q4_batched (the C struct of the same name)."""
    _fields_ = [("Wq", ctypes.c_void_p), ("Ws", ctypes.c_void_p), ("x_off", ctypes.c_int64), ("y_off", ctypes.c_int64)]


def cq_gemm_q4_batched_workspace_bytes(T, K, z) -> int:
    return lib().cq_gemm_q4_batched_workspace_bytes(T, K, z)


def cq_gemm_q4_batched(X, K, jobs, N, Y, ws, stream=None, raise_on_error=True):
    """jobs: list of (Wq, Ws, x_off, y_off) with device tensors; X [T][ldx],
    Y [T][ldy] (the pitches are the tensors' row strides)."""
    T = X.shape[0]
    arr = (cq_q4_job * len(jobs))(*[cq_q4_job(Wq.data_ptr(), Ws.data_ptr(), xo, yo) for Wq, Ws, xo, yo in jobs])
    st = lib().cq_gemm_q4_batched(_ptr(X), _xt(X), T, K, X.stride(0), ctypes.cast(arr, ctypes.c_void_p), len(jobs), N,
                                  _ptr(Y), _xt(Y), Y.stride(0), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream))
    if raise_on_error:
        _check(st)
    return st


def cq_gemm_q8b_workspace_bytes(T, K) -> int:
    return lib().cq_gemm_q8b_workspace_bytes(T, K)


def cq_gemm_q8b(X, Wq, Ws, Y, ws, stream=None, raise_on_error=True):
    """Q8 per 32-k block: Wq int8 [N][K], Ws f32 [N][K/32]."""
    T, K = X.shape
    st = lib().cq_gemm_q8b(_ptr(X), _xt(X), T, K, _ptr(Wq), _ptr(Ws), Wq.shape[0], _ptr(Y), _xt(Y), _ptr(ws),
                           ws.numel() * ws.element_size(), _stream(stream))
    if raise_on_error:
        _check(st)
    return st


def cq_gemm_q4a_workspace_bytes(T, K, N, gk) -> int:
    return lib().cq_gemm_q4a_workspace_bytes(T, K, N, gk)


def cq_gemm_q4a(X, Wq, Ws, Wo, gk, Y, ws, stream=None, raise_on_error=True):
    """Affine Q4: the Q4 split plane plus Wo bf16-bit offsets [N][K/32/gk]."""
    T, K = X.shape
    st = lib().cq_gemm_q4a(_ptr(X), _xt(X), T, K, _ptr(Wq), _ptr(Ws), _ptr(Wo), gk, Wq.shape[0], _ptr(Y), _xt(Y),
                           _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    if raise_on_error:
        _check(st)
    return st


def cq_gemm_q8_2f_workspace_bytes(T, K) -> int:
    return lib().cq_gemm_q8_2f_workspace_bytes(T, K)


def cq_gemm_q8_2f(X, Wq, rs, col, Y, ws, stream=None, raise_on_error=True):
    """q8_2f: Wq int8 [N][K], rs f32 [N], col f32 [K]."""
    T, K = X.shape
    st = lib().cq_gemm_q8_2f(_ptr(X), _xt(X), T, K, _ptr(Wq), _ptr(rs), _ptr(col), Wq.shape[0], _ptr(Y), _xt(Y),
                             _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    if raise_on_error:
        _check(st)
    return st


def cq_ffn_q4_workspace_bytes(T, H, I) -> int:
    return lib().cq_ffn_q4_workspace_bytes(T, H, I)


def cq_ffn_q4(X, Wgu_q, Wgu_s, Wd_q, Wd_s, Y, ws, stream=None, raise_on_error=True):
    """Y[T][H] = Wd . (silu(Wg . x) * (Wu . x)) per token; Wgu_q uint8 [2I][H/2]
    (gate rows then up rows), Wd_q uint8 [H][I/2], fp16-bit scales."""
    T, H = X.shape
    I = Wgu_q.shape[0] // 2
    st = lib().cq_ffn_q4(_ptr(X), _xt(X), T, H, I, _ptr(Wgu_q), _ptr(Wgu_s), _ptr(Wd_q), _ptr(Wd_s), _ptr(Y), _xt(Y),
                         _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    if raise_on_error:
        _check(st)
    return st


def cq_moe_route(logits, topk, idx, w, shared=False, stream=None):
    """idx [T][topk + shared] int32, w [T][topk + shared] f32 from logits [T][E + shared] f32."""
    T, cols = logits.shape
    E = cols - (1 if shared else 0)
    _check(lib().cq_moe_route(_ptr(logits), T, E, topk, 1 if shared else 0, _ptr(idx), _ptr(w), _stream(stream)))


def cq_moe_layout(ws, T, H, I, E, topk, perm_out, seg_out, stream=None):
    _check(lib().cq_moe_layout(_ptr(ws), T, H, I, E, topk, _ptr(perm_out), _ptr(seg_out), _stream(stream)))


def cq_dequant_q4(Wq, Ws, W, stream=None):
    N, K = W.shape
    _check(lib().cq_dequant_q4(_ptr(Wq), _ptr(Ws), N, K, _ptr(W), _stream(stream)))


def cq_dequant_q8row(Wq, rs, W, stream=None):
    N, K = W.shape
    _check(lib().cq_dequant_q8row(_ptr(Wq), _ptr(rs), N, K, _ptr(W), _stream(stream)))


def cq_get_device_error(stream=None) -> int:
    return lib().cq_get_device_error(_stream(stream))


def cq_last_error() -> str:
    return lib().cq_last_error().decode(errors="replace")


def cq_last_launches() -> int:
    """Kernel launches of the calling thread's most recent library call."""
    return lib().cq_last_launches()


def cq_set_option(option: int, value: int):
    _check(lib().cq_set_option(option, value))


def cq_get_option(option: int) -> int:
    return lib().cq_get_option(option)


def cq_version() -> int:
    return lib().cq_version()
