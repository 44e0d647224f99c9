"""Seeded synthetic inputs for the quantized-weight GEMM and MoE workloads.

This module only draws numbers and rounds them to their storage types. It
holds none of the computation under test (no dequantization, no packing, no
matmul), so the CUDA path and the CPU oracle can both consume what it makes.

Recipe (one ``numpy.random.default_rng(seed)`` per workload, draws in a fixed
order): X first, then Q4 codes, then scale magnitudes, then scale signs (only
where the workload asks for signed scales), then Q8 int8 values and row
scales, then router logits.  Floating values are drawn in f64; they reach f32
by numpy's RNE cast, fp16 by numpy's RNE cast, bf16 by RNE from that f32.

Routing for the MoE workload is part of the input recipe (the expert panel
entry point takes the routing indices and weights as inputs): per row a
softmax in f64 over the logits, the top-k experts by descending probability
with the lower index first on ties (cortiq-engine src/clover.rs, the
coreset's top-k rule), and weights renormalised over the chosen experts
(cortiq-engine src/clover.rs, the ``route`` closure: ``p[e] / wsum``).
"""
from __future__ import annotations

import numpy as np


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round f32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(a)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_storage(v: np.ndarray, dtype: str) -> np.ndarray:
    """f64 values -> uint16 bit patterns of ``dtype`` ('f16' or 'bf16')."""
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return f32_to_bf16_bits(v.astype(np.float32))
    raise ValueError(dtype)


def draw_x(rng, T, K, std=1.0, dtype="bf16"):
    return to_storage(rng.standard_normal((T, K)) * std, dtype)


def draw_q4(rng, N, K, lo=0.005, hi=0.02, signed=False):
    """Codes uniform in 0..15 ([N][K] uint8) and fp16 block scales ([N][K/32] bits)."""
    codes = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    mag = rng.uniform(lo, hi, size=(N, K // 32))
    if signed:
        mag = mag * np.where(rng.integers(0, 2, size=mag.shape) == 1, -1.0, 1.0)
    return codes, mag.astype(np.float16).view(np.uint16)


def draw_q8row(rng, N, K, lo=1e-3, hi=1e-2):
    """int8 uniform in -127..127 ([N][K]) and f32 row scales ([N])."""
    q = rng.integers(-127, 128, size=(N, K), dtype=np.int16).astype(np.int8)
    rs = rng.uniform(lo, hi, size=N).astype(np.float32)
    return q, rs


def route_topk(logits: np.ndarray, topk: int):
    """Softmax (f64) -> top-k (desc, lower index first on ties) -> renormalise.

    Returns idx [T][topk] int32 (in that order) and w [T][topk] f32.
    """
    lg = np.asarray(logits, dtype=np.float64)
    T, E = lg.shape
    m = lg.max(axis=1, keepdims=True)
    p = np.exp(lg - m)
    p = p / p.sum(axis=1, keepdims=True)
    idx = np.empty((T, topk), dtype=np.int32)
    w = np.empty((T, topk), dtype=np.float32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-p[t, e], e))[:topk]
        ws = sum(p[t, e] for e in order)
        idx[t] = order
        w[t] = [p[t, e] / ws for e in order]
    return idx, w


# ---------------------------------------------------------------------------
# The five workloads (shapes and distributions as the configurations state).
# ---------------------------------------------------------------------------

def gemm_q4_case(seed, T, K, N, x_dtype="bf16", x_std=1.0, signed=False):
    rng = np.random.default_rng(seed)
    x = draw_x(rng, T, K, x_std, x_dtype)
    codes, scales = draw_q4(rng, N, K, signed=signed)
    return {"x": x, "x_dtype": x_dtype, "codes": codes, "scales": scales, "T": T, "K": K, "N": N}


def gemm_q8_case(seed, T, K, N, x_dtype="bf16", x_std=1.0):
    rng = np.random.default_rng(seed)
    x = draw_x(rng, T, K, x_std, x_dtype)
    q, rs = draw_q8row(rng, N, K)
    return {"x": x, "x_dtype": x_dtype, "q": q, "rs": rs, "T": T, "K": K, "N": N}


def moe_case(seed, T=32, H=2048, I=768, E=128, topk=8, x_dtype="bf16"):
    """Router logits are drawn first, then X, then expert codes/scales.

    Expert order of draws: for each expert, gate|up codes+scales then down.
    """
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = draw_x(rng, T, H, 1.0, x_dtype)
    gu_codes = np.empty((E, 2 * I, H), np.uint8)
    gu_scales = np.empty((E, 2 * I, H // 32), np.uint16)
    d_codes = np.empty((E, H, I), np.uint8)
    d_scales = np.empty((E, H, I // 32), np.uint16)
    for e in range(E):
        gu_codes[e], gu_scales[e] = draw_q4(rng, 2 * I, H)
        d_codes[e], d_scales[e] = draw_q4(rng, H, I)
    idx, w = route_topk(logits, topk)
    return {"x": x, "x_dtype": x_dtype, "logits": logits, "idx": idx, "w": w,
            "gu_codes": gu_codes, "gu_scales": gu_scales, "d_codes": d_codes, "d_scales": d_scales,
            "T": T, "H": H, "I": I, "E": E, "topk": topk}


def c1():
    """Q4 smallest case: X[16,512] fp16 N(0,1), N=256, signed scales, f32 out, seed 0."""
    return gemm_q4_case(0, 16, 512, 256, x_dtype="f16", signed=True)


def c2_q4():
    return gemm_q4_case(1, 512, 4096, 4096)


def c2_q8():
    return gemm_q8_case(2, 512, 4096, 4096)


def c3():
    """Denoiser block: gate/up then down, independent X draws from one seed."""
    rng = np.random.default_rng(3)
    x_gu = draw_x(rng, 1024, 3072, 0.5)
    gu_codes, gu_scales = draw_q4(rng, 24576, 3072)
    x_d = draw_x(rng, 1024, 12288, 0.5)
    d_codes, d_scales = draw_q4(rng, 3072, 12288)
    return ({"x": x_gu, "x_dtype": "bf16", "codes": gu_codes, "scales": gu_scales, "T": 1024, "K": 3072, "N": 24576},
            {"x": x_d, "x_dtype": "bf16", "codes": d_codes, "scales": d_scales, "T": 1024, "K": 12288, "N": 3072})


def c4():
    return moe_case(4)


def c5_q4(T):
    return gemm_q4_case(5, T, 8192, 8192)


def c5_q8(T):
    return gemm_q8_case(5, T, 8192, 8192)
