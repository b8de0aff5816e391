"""3-bit block codec (oracle; test infrastructure only).

Source: "Quasar" (q27 wiki), "turbo3 3-bit KV cache" bullet and the "KV cache"
bullet of the stack list -- K and V are Walsh-Hadamard rotated and stored as
3-bit codes in fixed-size blocks, symmetric for K and V.  The pages give no
bit-level format; this library fixes its own (a stated substitute for turbo3,
112 bytes per 256-dim vector instead of turbo3's 100):

1. y = H x                      (``wht.fwht_f32``: pinned float32 butterfly)
2. split y into 8 blocks of 32 elements
3. per block:  s = fp16( fp32(absmax) / 3.5f )          (IEEE fp32 divide, then
                                                          round-to-nearest-even to fp16)
4. per element: q = clamp( rint( fp32(y / s) + 3.5f ), 0, 7 )
               with s taken back to fp32, an IEEE fp32 divide (not a multiply by
               1/s), an fp32 add, and rint rounding half to even
5. dequantised value: (q - 3.5) * s     (exact in fp32 and fp64: <= 14 bits)

Edge rules (a reading of the plainest kind; the pages are silent):
* s == 0 (all-zero block or fp16 underflow): every code is 4, which is also what
  y = 0 gives for any s > 0 (rint(3.5) = 4), and dequantises to 0.
* fp32(absmax)/3.5 that rounds to +inf in fp16 is a precondition violation: the
  vector is flagged FLAG_SCALE_OVERFLOW; the codes follow the same formula
  (y / inf = 0, so code 4).
* non-finite input is flagged FLAG_NONFINITE; its codes and scales are
  unspecified and are never compared.
"""
from __future__ import annotations

import numpy as np

from .wht import fwht_f32

BLOCK = 32
BLOCKS_PER_VECTOR = 8
FLAG_NONFINITE = 1
FLAG_SCALE_OVERFLOW = 2


def block_scales(y: np.ndarray) -> np.ndarray:
    """fp16 scale of each 32-element block of rotated vectors y (float32 [..., 256])."""
    y = np.asarray(y, dtype=np.float32)
    blocks = y.reshape(y.shape[:-1] + (BLOCKS_PER_VECTOR, BLOCK))
    absmax = np.max(np.abs(blocks), axis=-1)                      # float32
    with np.errstate(over="ignore"):
        return (absmax / np.float32(3.5)).astype(np.float16)      # fp32 divide, RNE to fp16


def quantize_rotated(y: np.ndarray):
    """Codes (uint8 [..., 256]) and scales (float16 [..., 8]) of already-rotated vectors."""
    y = np.asarray(y, dtype=np.float32)
    s16 = block_scales(y)
    s32 = s16.astype(np.float32)
    blocks = y.reshape(y.shape[:-1] + (BLOCKS_PER_VECTOR, BLOCK))
    with np.errstate(divide="ignore", invalid="ignore"):
        t = blocks / s32[..., None] + np.float32(3.5)             # fp32 divide, fp32 add
    q = np.clip(np.rint(t), 0.0, 7.0)                             # rint: half to even
    q = np.where((s32 == 0)[..., None], 4.0, q)
    q = np.where(np.isfinite(q), q, 4.0)
    return q.astype(np.uint8).reshape(y.shape), s16


def vector_flags(x: np.ndarray, s16: np.ndarray) -> np.ndarray:
    """Per-vector status bits for raw inputs x [..., 256] and their scales [..., 8]."""
    flags = np.zeros(x.shape[:-1], dtype=np.int32)
    flags |= np.where(np.all(np.isfinite(x), axis=-1), 0, FLAG_NONFINITE).astype(np.int32)
    over = np.any(np.isinf(s16.astype(np.float32)), axis=-1) & np.all(np.isfinite(x), axis=-1)
    flags |= np.where(over, FLAG_SCALE_OVERFLOW, 0).astype(np.int32)
    return flags


def encode(x: np.ndarray):
    """Raw float32 head vectors [..., 256] -> (codes uint8 [..., 256], scales float16 [..., 8], flags int32 [...])."""
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        y = fwht_f32(x)
    codes, s16 = quantize_rotated(y)
    return codes, s16, vector_flags(x, s16)


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """(q - 3.5) * s in float64, [..., 256] (rotated basis)."""
    c = np.asarray(codes, dtype=np.float64)
    s = np.asarray(scales, dtype=np.float64)
    c = c.reshape(c.shape[:-1] + (BLOCKS_PER_VECTOR, BLOCK))
    return ((c - 3.5) * s[..., None]).reshape(codes.shape)
