"""CPU oracle for the block-quantized-weight matmul (test infrastructure).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It wraps ``oracle.c`` (plain C, f64 accumulation),
which shares nothing with the CUDA library.  See ``oracle.c`` for the
passages each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (plain C, OpenMP, no FP contraction)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.or_f64_to_bf16.restype = ctypes.c_uint16
        _lib.or_f16_to_f64.restype = ctypes.c_double
        _lib.or_bf16_to_f64.restype = ctypes.c_double
        _lib.or_f64_to_bf16.argtypes = [ctypes.c_double]
        _lib.or_f16_to_f64.argtypes = [ctypes.c_uint16]
        _lib.or_bf16_to_f64.argtypes = [ctypes.c_uint16]
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def _i(v):
    return ctypes.c_int64(int(v))


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ---- formats -------------------------------------------------------------

def f16_to_f64(bits) -> float:
    return _load().or_f16_to_f64(int(bits))


def bf16_to_f64(bits) -> float:
    return _load().or_bf16_to_f64(int(bits))


def f64_to_bf16(v: np.ndarray) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().or_f64_to_bf16_array(_p(v), _i(v.size), _p(out))
    return out


def f64_to_f32(v: np.ndarray) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.float32)
    _load().or_f64_to_f32_array(_p(v), _i(v.size), _p(out))
    return out


def x_to_f64(x_bits: np.ndarray, dtype: str) -> np.ndarray:
    x = _c(x_bits, np.uint16)
    out = np.empty(x.shape, np.float64)
    _load().or_x_to_f64(_p(x), ctypes.c_int(1 if dtype == "bf16" else 0), _i(x.size), _p(out))
    return out


def round_out(y: np.ndarray, out_dtype: str) -> np.ndarray:
    """One rounding of the f64 result to the output type ('f32' or 'bf16' bits)."""
    return f64_to_f32(y) if out_dtype == "f32" else f64_to_bf16(y)


# ---- Q4 / Q8-row ---------------------------------------------------------

def pack_q4(codes: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    N, K = codes.shape
    out = np.empty((N, K // 2), np.uint8)
    _load().or_pack_q4(_p(codes), _i(N), _i(K), _p(out))
    return out


def dequant_q4(wq: np.ndarray, ws: np.ndarray, N: int, K: int) -> np.ndarray:
    wq = _c(wq, np.uint8)
    ws = _c(ws, np.uint16)
    assert wq.size == N * K // 2 and ws.size == N * K // 32
    out = np.empty((N, K), np.float32)
    _load().or_dequant_q4(_p(wq), _p(ws), _i(N), _i(K), _p(out))
    return out


def dequant_q8row(q: np.ndarray, rs: np.ndarray) -> np.ndarray:
    q = _c(q, np.int8)
    rs = _c(rs, np.float32)
    N, K = q.shape
    out = np.empty((N, K), np.float32)
    _load().or_dequant_q8row(_p(q), _p(rs), _i(N), _i(K), _p(out))
    return out


def gemm(W: np.ndarray, X: np.ndarray, rowscale=None):
    """(Y, S) in f64: Y = X . W^T with f64 sums in k order, S = sum |w x|."""
    W = _c(W, np.float32)
    X = _c(X, np.float64)
    N, K = W.shape
    T = X.shape[0]
    Y = np.empty((T, N), np.float64)
    S = np.empty((T, N), np.float64)
    rsp = None
    if rowscale is not None:
        rowscale = _c(rowscale, np.float32)
        rsp = _p(rowscale)
    _load().or_gemm(_p(W), _p(X), _i(T), _i(N), _i(K), rsp, _p(Y), _p(S))
    return Y, S


def gemm_q4(wq, ws, N, K, X):
    return gemm(dequant_q4(wq, ws, N, K), X)


def gemm_q8row(q, rs, X):
    """Integer weights, f64 sums, row scale applied to the sum."""
    return gemm(_c(q, np.int8).astype(np.float32), X, rowscale=rs)


def gemm_q4_sampled(wq, ws, N, K, X, tn):
    wq = _c(wq, np.uint8)
    ws = _c(ws, np.uint16)
    X = _c(X, np.float64)
    tn = _c(tn, np.int64)
    cnt = tn.shape[0]
    Y = np.empty(cnt, np.float64)
    S = np.empty(cnt, np.float64)
    _load().or_gemm_q4_sampled(_p(wq), _p(ws), _p(X), _i(N), _i(K), _p(tn), _i(cnt), _p(Y), _p(S))
    return Y, S


def gemm_q8_sampled(q, rs, X, tn):
    q = _c(q, np.int8)
    rs = _c(rs, np.float32)
    X = _c(X, np.float64)
    tn = _c(tn, np.int64)
    N, K = q.shape
    cnt = tn.shape[0]
    Y = np.empty(cnt, np.float64)
    S = np.empty(cnt, np.float64)
    _load().or_gemm_q8_sampled(_p(q), _p(rs), _p(X), _i(N), _i(K), _p(tn), _i(cnt), _p(Y), _p(S))
    return Y, S


# ---- MoE -----------------------------------------------------------------

def moe_layout(idx: np.ndarray, E: int):
    idx = _c(idx, np.int32)
    T, topk = idx.shape
    perm = np.empty(T * topk, np.int32)
    seg = np.empty(E + 1, np.int32)
    rc = _load().or_moe_layout(_p(idx), _i(T), _i(topk), _i(E), _p(perm), _p(seg))
    if rc != 0:
        raise ValueError("routing index out of range")
    return perm, seg


def moe_pair(wgu: np.ndarray, wd: np.ndarray, x: np.ndarray):
    """One routed pair on dequantized f32 weights: (a, o, sabs)."""
    wgu = _c(wgu, np.float32)
    wd = _c(wd, np.float32)
    x = _c(x, np.float64)
    H = x.shape[0]
    I = wd.shape[1]
    a = np.empty(I, np.float64)
    o = np.empty(H, np.float64)
    s = np.empty(H, np.float64)
    _load().or_moe_pair(_p(wgu), _p(wd), _p(x), _i(H), _i(I), _p(a), _p(o), _p(s))
    return a, o, s


def moe(X, idx, w, gu_q, gu_s, d_q, d_s, E, I):
    """(Y, S) f64 for the routed MoE block. X [T][H] f64."""
    X = _c(X, np.float64)
    idx = _c(idx, np.int32)
    w = _c(w, np.float32)
    T, H = X.shape
    topk = idx.shape[1]
    gu_q = _c(gu_q, np.uint8)
    gu_s = _c(gu_s, np.uint16)
    d_q = _c(d_q, np.uint8)
    d_s = _c(d_s, np.uint16)
    Y = np.empty((T, H), np.float64)
    S = np.empty((T, H), np.float64)
    rc = _load().or_moe(_p(X), _i(T), _i(H), _i(E), _i(I), _i(topk), _p(idx), _p(w),
                        _p(gu_q), _p(gu_s), _p(d_q), _p(d_s), _p(Y), _p(S))
    if rc != 0:
        raise ValueError("routing index out of range")
    return Y, S


# ---- dense FFN chain -------------------------------------------------------

def ffn(X, gu_q, gu_s, d_q, d_s, I, want_a=False):
    """(Y, S[, A]) f64 for the dense gate/up -> SwiGLU -> down chain over every
    token of X [T][H] (f64): gu_q/gu_s the Q4 gate|up rows [2I][H/2], [2I][H/32];
    d_q/d_s the Q4 down rows [H][I/2], [H][I/32]."""
    X = _c(X, np.float64)
    T, H = X.shape
    gu_q = _c(gu_q, np.uint8)
    gu_s = _c(gu_s, np.uint16)
    d_q = _c(d_q, np.uint8)
    d_s = _c(d_s, np.uint16)
    assert gu_q.size == 2 * I * H // 2 and d_q.size == H * I // 2
    Y = np.empty((T, H), np.float64)
    S = np.empty((T, H), np.float64)
    A = np.empty((T, I), np.float64) if want_a else None
    _load().or_ffn(_p(X), _i(T), _i(H), _i(I), _p(gu_q), _p(gu_s), _p(d_q), _p(d_s), _p(Y), _p(S),
                   _p(A) if want_a else None)
    return (Y, S, A) if want_a else (Y, S)


# ---- MoE routing from router logits ----------------------------------------

def route(logits, topk, shared=False):
    """(idx, w): top-k by logit (descending, lower index first on ties),
    weights p_e / sum over the picked experts from an f64 softmax, rounded to
    f32; with `shared` the last logit column is the shared expert's gate and
    slot topk is expert E with weight sigmoid(gate).  logits [T][E (+1)] f32."""
    lg = _c(logits, np.float32)
    T, cols = lg.shape
    E = cols - (1 if shared else 0)
    assert 1 <= topk <= min(E, 64)
    slots = topk + (1 if shared else 0)
    idx = np.empty((T, slots), np.int32)
    w = np.empty((T, slots), np.float32)
    _load().or_route(_p(lg), _i(T), _i(E), _i(topk), ctypes.c_int(1 if shared else 0), _p(idx), _p(w))
    return idx, w


# ---- format variants -------------------------------------------------------

def dequant_q8b(q, s):
    """Q8 per 32-k block: W = f32(q) * s[n][k/32] (f32 scales)."""
    q = _c(q, np.int8)
    s = _c(s, np.float32)
    N, K = q.shape
    assert s.shape == (N, K // 32)
    out = np.empty((N, K), np.float32)
    _load().or_dequant_q8b(_p(q), _p(s), _i(N), _i(K), _p(out))
    return out


def dequant_q4a(wq, ws, off, gk, N, K):
    """Affine Q4: (nibble - 8) * d + bf16 offset of the group of gk blocks."""
    wq = _c(wq, np.uint8)
    ws = _c(ws, np.uint16)
    off = _c(off, np.uint16)
    assert off.size == N * (K // 32 // gk)
    out = np.empty((N, K), np.float32)
    _load().or_dequant_q4a(_p(wq), _p(ws), _p(off), _i(gk), _i(N), _i(K), _p(out))
    return out


def gemm_q8b(q, s, X):
    return gemm(dequant_q8b(q, s), X)


def gemm_q4a(wq, ws, off, gk, N, K, X):
    return gemm(dequant_q4a(wq, ws, off, gk, N, K), X)


def gemm_q8_2f(q, rs, col, X):
    """(Y, S) f64: Y[t][n] = rs[n] * sum_k q[n][k] col[k] X[t][k]."""
    q = _c(q, np.int8)
    rs = _c(rs, np.float32)
    col = _c(col, np.float32)
    X = _c(X, np.float64)
    N, K = q.shape
    T = X.shape[0]
    Y = np.empty((T, N), np.float64)
    S = np.empty((T, N), np.float64)
    _load().or_gemm_q8_2f(_p(q), _p(rs), _p(col), _p(X), _i(T), _i(N), _i(K), _p(Y), _p(S))
    return Y, S
