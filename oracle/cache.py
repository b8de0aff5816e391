"""Paged per-slot cache and the full verify step (oracle; test infrastructure only).

Source: "Quasar" (q27 wiki), "turbo3 3-bit KV cache" bullet (per-slot KV, "two
full 131K tenants at once"), the vLLM paragraph of the prefix-reuse section
(attention KV is an append-only, position-addressed log kept in fixed-size
blocks) and "Continuous batching" (several slots per round).

A slot's position p lives in page ``page_table[p // 256]`` at row ``p % 256``.
Appending T tokens at positions [len, len + T) encodes each raw K and V head
vector with ``codec.encode`` and writes its 112-byte record (``packing``).
Rolling back rejected drafts is only a smaller length: later appends overwrite.
"""
from __future__ import annotations

import numpy as np

from . import codec, packing
from .attention import verify_attention


class PagedCache:
    def __init__(self, num_pages: int, num_layers: int, num_kv_heads: int):
        self.num_pages = num_pages
        self.num_layers = num_layers
        self.num_kv_heads = num_kv_heads
        self.pool = np.zeros(packing.pool_bytes(num_pages, num_layers, num_kv_heads), dtype=np.uint8)

    def _offsets(self, page_table_row, positions, layer, kv_head, kv):
        positions = np.asarray(positions, dtype=np.int64)
        pages = np.asarray(page_table_row, dtype=np.int64)[positions // packing.PAGE_SIZE]
        if np.any(pages < 0) or np.any(pages >= self.num_pages):
            raise IndexError("page id out of range")
        rows = positions % packing.PAGE_SIZE
        L, H = self.num_layers, self.num_kv_heads
        return ((((pages * L + layer) * H + kv_head) * 2 + kv) * packing.PAGE_SIZE + rows) * packing.RECORD_BYTES

    def append(self, page_table_row, start: int, layer: int, k_raw: np.ndarray, v_raw: np.ndarray) -> np.ndarray:
        """Encode and store raw K, V [n, Hkv, 256] at positions [start, start + n). Returns flags [n, Hkv, 2]."""
        n = k_raw.shape[0]
        flags = np.zeros((n, self.num_kv_heads, 2), dtype=np.int32)
        pos = np.arange(start, start + n)
        for kv, x in ((0, k_raw), (1, v_raw)):
            for g in range(self.num_kv_heads):
                codes, s16, f = codec.encode(x[:, g, :])
                rec = packing.pack_records(codes, s16)
                off = self._offsets(page_table_row, pos, layer, g, kv)
                self.pool[off[:, None] + np.arange(packing.RECORD_BYTES)[None, :]] = rec
                flags[:, g, kv] = f
        return flags

    def records(self, page_table_row, layer: int, kv_head: int, kv: int, start: int, count: int) -> np.ndarray:
        off = self._offsets(page_table_row, np.arange(start, start + count), layer, kv_head, kv)
        return self.pool[off[:, None] + np.arange(packing.RECORD_BYTES)[None, :]]

    def dequantized(self, page_table_row, layer: int, kv_head: int, kv: int, count: int) -> np.ndarray:
        codes, s16 = packing.unpack_records(self.records(page_table_row, layer, kv_head, kv, 0, count))
        return codec.dequantize(codes, s16)

    def verify(self, page_table_row, layer: int, n_ctx: int, q: np.ndarray, group: int) -> np.ndarray:
        """Verify attention of T = q.shape[0] tokens over positions [0, n_ctx + T)."""
        L = n_ctx + q.shape[0]
        kh = np.stack([self.dequantized(page_table_row, layer, g, 0, L) for g in range(self.num_kv_heads)])
        vh = np.stack([self.dequantized(page_table_row, layer, g, 1, L) for g in range(self.num_kv_heads)])
        return verify_attention(q, kh, vh, n_ctx, group)


def encode_dequantized(x_raw: np.ndarray) -> np.ndarray:
    """Raw vectors [..., 256] -> dequantised rotated vectors (float64), no pool."""
    codes, s16, _ = codec.encode(x_raw)
    return codec.dequantize(codes, s16)
