"""turbo5k-style cache: 5-bit Lloyd-Max K, 3-bit V (oracle; test infrastructure only).

Source: "Quasar" (q27 wiki), the turbo5k bullet of the stack list: 5-bit K
with 32 Lloyd-Max centroids over the same WHT rotation turbo3 uses, 82-byte K
blocks per 128 dims, and the 3-bit V of turbo3 -- the pages' own fix for
turbo3's tail errors.  The pages give the centroid count, the rotation and the
block size, nothing bit-level.  The reading taken here:

K, per head vector x (256 dims):
1. y = H x, the 3-bit codec's pinned float32 butterfly (``wht.fwht_f32``);
2. two blocks of 128 dims; per block a scale s = fp16_rn(sqrt(sum y^2 / 128))
   (the root mean square: Lloyd-Max centroids are those of a unit normal, so
   y / s is put on that scale).  The float32 sum of squares runs in this order:
   each group of 8 consecutive elements is summed from its first element on
   (each square rounded, then added), and the 16 group sums of a block are
   added pairwise (groups 2k and 2k+1, then pairs of pairs, ...); then the
   float32 square root of sum * (1/128);
3. codes: v = fp32(y / s) (IEEE divide), code = the number of boundaries b_j
   (j = 0..30) with v > b_j, where b_j = fp32(c_j + c_{j+1}) * 0.5 over the
   float32 centroids c_0 < ... < c_31 (so a tie with a boundary takes the lower
   code).  s == 0: every code is 16 (the value is 0 for any code).
4. value: c_code * s.

The centroids: the 32-level Lloyd-Max quantizer of N(0, 1) (each centroid the
mean of the normal over its cell, each boundary the midpoint of its two
centroids), symmetric about 0, found by Max's shooting method (the first
positive centroid fixes all others cell by cell; bisection on it until the
last cell's centroid condition holds) in float64, then rounded to float32.

V: the 3-bit codec of ``codec`` (112-byte record), unchanged.

K record (164 bytes; the pages' two 82-byte blocks, fields grouped so that the
code bytes stay 4-byte aligned): bytes 0..127 the low 4 bits of the 256 codes,
two per byte, element 2j in the low nibble of byte j; bytes 128..159 the 5th
bits, element d at bit d % 8 of byte 128 + d // 8; bytes 160..163 the two fp16
scales.  Pool: per (page, layer, kv head) 256 K records (41,984 bytes) then 256
V records (28,672 bytes):
  K: ((page * layers + layer) * kv_heads + head) * 70,656 + row * 164
  V: ((page * layers + layer) * kv_heads + head) * 70,656 + 41,984 + row * 112

Parity status: pinned against this reading (Lloyd-Max conditions, brute force,
closed forms); *parity unpinned* against the pages' turbo5k, which has no
bit-level specification.
"""
from __future__ import annotations

import math

import numpy as np

from . import codec as q3codec
from . import packing as q3packing
from .attention import verify_attention
from .wht import fwht_f32

LEVELS = 32
HALF = 128
K_RECORD_BYTES = 164
V_RECORD_BYTES = 112
PAGE_SIZE = 256
CHUNK_BYTES = PAGE_SIZE * (K_RECORD_BYTES + V_RECORD_BYTES)   # 70,656


def _upper_tail(x: float) -> float:
    return 0.5 * math.erfc(x / math.sqrt(2.0))


def _pdf(x: float) -> float:
    return math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def _cell_mean(a: float, b: float) -> float:
    """E[X | a < X < b] for X ~ N(0, 1), 0 <= a < b <= inf."""
    if math.isinf(b):
        return _pdf(a) / _upper_tail(a)
    return (_pdf(a) - _pdf(b)) / (_upper_tail(a) - _upper_tail(b))


def _shoot(y0: float):
    """Positive half from its first centroid: (centroids, boundaries, excess of the last centroid)."""
    ys, ts = [y0], [0.0]
    for k in range(LEVELS // 2 - 1):
        a, y = ts[-1], ys[-1]
        if _cell_mean(a, math.inf) <= y:          # no upper boundary can bring the mean up to y
            return ys, ts, math.inf
        lo, hi = a, a + 1.0
        while _cell_mean(a, hi) < y:
            hi = a + 2.0 * (hi - a)
        for _ in range(200):                      # bisection to the float64 resolution
            mid = 0.5 * (lo + hi)
            if mid <= lo or mid >= hi:
                break
            if _cell_mean(a, mid) < y:
                lo = mid
            else:
                hi = mid
        t = 0.5 * (lo + hi)
        ts.append(t)
        ys.append(2.0 * t - y)
    return ys, ts, ys[-1] - _cell_mean(ts[-1], math.inf)


def lloyd_max_gaussian_f64() -> np.ndarray:
    """The 32 Lloyd-Max centroids of N(0, 1), float64, ascending."""
    lo, hi = 1e-3, 0.5
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if mid <= lo or mid >= hi:
            break
        _, _, excess = _shoot(mid)
        if excess > 0:
            hi = mid
        else:
            lo = mid
    ys, _, _ = _shoot(0.5 * (lo + hi))
    pos = np.array(ys, np.float64)
    return np.concatenate([-pos[::-1], pos])


_TABLE = None


def table():
    """(float32 centroids [32], float32 boundaries [31])."""
    global _TABLE
    if _TABLE is None:
        c = lloyd_max_gaussian_f64().astype(np.float32)
        b = ((c[:-1] + c[1:]) * np.float32(0.5)).astype(np.float32)
        _TABLE = (c, b)
    return _TABLE


def half_scales(y: np.ndarray) -> np.ndarray:
    """fp16 root-mean-square scale of each 128-dim half of rotated vectors y (float32 [..., 256])."""
    y = np.asarray(y, np.float32)
    g = y.reshape(y.shape[:-1] + (2, 16, 8))                     # half, group of 8, element
    sq = g * g                                                    # float32 squares
    acc = sq[..., 0]
    for e in range(1, 8):
        acc = acc + sq[..., e]                                    # sequential within a group
    while acc.shape[-1] > 1:                                      # pairwise over the 16 groups
        acc = acc[..., 0::2] + acc[..., 1::2]
    mean_sq = acc[..., 0] * np.float32(1.0 / 128.0)
    with np.errstate(over="ignore"):
        return np.sqrt(mean_sq).astype(np.float32).astype(np.float16)


def encode_k(x: np.ndarray):
    """Raw K vectors [..., 256] -> (codes uint8 [..., 256], scales fp16 [..., 2], flags int32 [...])."""
    x = np.asarray(x, np.float32)
    y = fwht_f32(x)
    s16 = half_scales(y)
    s32 = s16.astype(np.float32)
    _, b = table()
    yh = y.reshape(y.shape[:-1] + (2, HALF))
    with np.errstate(divide="ignore", invalid="ignore"):
        v = yh / s32[..., None]                                   # IEEE float32 divide
    codes = (v[..., None] > b).sum(axis=-1)
    codes = np.where((s32 == 0)[..., None], 16, codes).astype(np.uint8).reshape(y.shape)
    flags = np.zeros(x.shape[:-1], np.int32)
    flags |= np.where(np.all(np.isfinite(x), axis=-1), 0, q3codec.FLAG_NONFINITE)
    flags |= np.where(np.any(np.isinf(s16.astype(np.float32)), axis=-1) & (flags == 0),
                      q3codec.FLAG_SCALE_OVERFLOW, 0)
    return codes, s16, flags


def decode_k(codes: np.ndarray, s16: np.ndarray) -> np.ndarray:
    """Rotated K values c_code * s, float64 (exact)."""
    c, _ = table()
    vals = c.astype(np.float64)[np.asarray(codes, np.int64)]
    s = np.repeat(np.asarray(s16, np.float16).astype(np.float64), HALF, axis=-1)
    return vals * s


def pack_k(codes: np.ndarray, s16: np.ndarray) -> np.ndarray:
    """K records uint8 [..., 164]."""
    codes = np.asarray(codes, np.uint8)
    lo = codes & 0xF
    nib = (lo[..., 0::2] | (lo[..., 1::2] << 4)).astype(np.uint8)                  # [..., 128]
    hi = ((codes >> 4) & 1).reshape(codes.shape[:-1] + (32, 8))
    plane = (hi << np.arange(8, dtype=np.uint8)).sum(axis=-1).astype(np.uint8)    # [..., 32]
    sc = np.ascontiguousarray(np.asarray(s16, np.float16)).view(np.uint8).reshape(codes.shape[:-1] + (4,))
    return np.concatenate([nib, plane, sc], axis=-1)


def unpack_k(rec: np.ndarray):
    rec = np.asarray(rec, np.uint8)
    nib = rec[..., :128]
    lo = np.stack([nib & 0xF, nib >> 4], axis=-1).reshape(rec.shape[:-1] + (256,))
    plane = rec[..., 128:160]
    hi = ((plane[..., :, None] >> np.arange(8, dtype=np.uint8)) & 1).reshape(rec.shape[:-1] + (256,))
    s16 = np.ascontiguousarray(rec[..., 160:164]).view(np.float16).reshape(rec.shape[:-1] + (2,))
    return (lo | (hi << 4)).astype(np.uint8), s16


def k_offset(num_layers, num_kv_heads, page, layer, head, row):
    return (((page * num_layers + layer) * num_kv_heads + head) * CHUNK_BYTES) + row * K_RECORD_BYTES


def v_offset(num_layers, num_kv_heads, page, layer, head, row):
    return (((page * num_layers + layer) * num_kv_heads + head) * CHUNK_BYTES) + PAGE_SIZE * K_RECORD_BYTES + \
        row * V_RECORD_BYTES


class T5kPagedCache:
    def __init__(self, num_pages: int, num_layers: int, num_kv_heads: int):
        self.num_pages, self.num_layers, self.num_kv_heads = num_pages, num_layers, num_kv_heads
        self.pool = np.zeros(num_pages * num_layers * num_kv_heads * CHUNK_BYTES, np.uint8)

    def _pages(self, page_table_row, positions):
        positions = np.asarray(positions, np.int64)
        pages = np.asarray(page_table_row, np.int64)[positions // PAGE_SIZE]
        if np.any(pages < 0) or np.any(pages >= self.num_pages):
            raise IndexError("page id out of range")
        return pages, positions % PAGE_SIZE

    def append(self, page_table_row, start: int, layer: int, k_raw: np.ndarray, v_raw: np.ndarray) -> np.ndarray:
        n = k_raw.shape[0]
        flags = np.zeros((n, self.num_kv_heads, 2), np.int32)
        pages, rows = self._pages(page_table_row, np.arange(start, start + n))
        L, H = self.num_layers, self.num_kv_heads
        for g in range(H):
            codes, s16, f = encode_k(k_raw[:, g, :])
            off = k_offset(L, H, pages, layer, g, rows)
            self.pool[off[:, None] + np.arange(K_RECORD_BYTES)[None, :]] = pack_k(codes, s16)
            flags[:, g, 0] = f
            vc, vs, vf = q3codec.encode(v_raw[:, g, :])
            off = v_offset(L, H, pages, layer, g, rows)
            self.pool[off[:, None] + np.arange(V_RECORD_BYTES)[None, :]] = q3packing.pack_records(vc, vs)
            flags[:, g, 1] = vf
        return flags

    def k_records(self, page_table_row, layer, head, count):
        pages, rows = self._pages(page_table_row, np.arange(count))
        off = k_offset(self.num_layers, self.num_kv_heads, pages, layer, head, rows)
        return self.pool[off[:, None] + np.arange(K_RECORD_BYTES)[None, :]]

    def v_records(self, page_table_row, layer, head, count):
        pages, rows = self._pages(page_table_row, np.arange(count))
        off = v_offset(self.num_layers, self.num_kv_heads, pages, layer, head, rows)
        return self.pool[off[:, None] + np.arange(V_RECORD_BYTES)[None, :]]

    def verify(self, page_table_row, layer: int, n_ctx: int, q: np.ndarray, group: int) -> np.ndarray:
        L = n_ctx + q.shape[0]
        kh = np.stack([decode_k(*unpack_k(self.k_records(page_table_row, layer, g, L)))
                       for g in range(self.num_kv_heads)])
        vh = np.stack([q3codec.dequantize(*q3packing.unpack_records(self.v_records(page_table_row, layer, g, L)))
                       for g in range(self.num_kv_heads)])
        return verify_attention(q, kh, vh, n_ctx, group)


def encode_dequantized_k(x_raw: np.ndarray) -> np.ndarray:
    codes, s16, _ = encode_k(x_raw)
    return decode_k(codes, s16)
