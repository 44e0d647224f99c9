"""Host-side packer for the Q4 split-plane format (not timed).

codes[N][K] in 0..15 -> Wq[N][K/2] bytes, where byte 16*b + i of row n
holds codes[n][32b+i] in its low nibble and codes[n][32b+16+i] in its high
nibble ("oxinfer 0.0.5 src/metal.rs", shader section "Dequantizers",
struct Q4W / load(Q4W ...)).  The fp16 block scales are stored as they are,
[N][K/32].  MoE experts stack along a leading axis:
gate|up [E][2I][H/2] (rows 0..I-1 gate, I..2I-1 up), down [E][H][I/2].
"""
from __future__ import annotations

import numpy as np


def pack_q4(codes: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    if c.ndim < 2 or c.shape[-1] % 32:
        raise ValueError("codes must be [..., K] with K % 32 == 0")
    *lead, K = c.shape
    blk = c.reshape(*lead, K // 32, 2, 16)          # [..., block, half, i]
    lo = blk[..., 0, :] & 0x0F
    hi = blk[..., 1, :] & 0x0F
    return (lo | (hi << 4)).astype(np.uint8).reshape(*lead, K // 2)


def unpack_q4_codes(wq: np.ndarray) -> np.ndarray:
    """Inverse of pack_q4 (codes, not values)."""
    b = np.ascontiguousarray(wq, dtype=np.uint8)
    *lead, Kh = b.shape
    blk = b.reshape(*lead, Kh // 16, 16)
    out = np.stack([blk & 0x0F, blk >> 4], axis=-2)    # [..., block, half, i]
    return out.reshape(*lead, Kh * 2)


def widen_f16_row_scales(rs_f16_bits: np.ndarray) -> np.ndarray:
    """Q8-row scales stored as fp16 (as the pages store them) -> f32, exact."""
    return np.asarray(rs_f16_bits, dtype=np.uint16).view(np.float16).astype(np.float32)
