"""Paged per-slot cache and the full verify step (oracle; test infrastructure only).

Source: "Quasar" (q27 wiki), "turbo3 3-bit KV cache" bullet (per-slot KV, "two
full 131K tenants at once"), the vLLM paragraph of the prefix-reuse section
(attention KV is an append-only, position-addressed log kept in fixed-size
blocks) and "Continuous batching" (several slots per round).

A slot's position p lives in page ``page_table[p // 256]`` at row ``p % 256``.
Appending T tokens at positions [len, len + T) encodes each raw K and V head
vector with ``codec.encode``; a K vector is written as its 112-byte record, a V
vector into the page's value page (its codes and scales at the row's places in
the per-dimension planes, ``packing``).  Rolling back rejected drafts is only
a smaller length: later appends overwrite.
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

    def _value_page_offset(self, page_table_row, page_index, layer, kv_head):
        page = int(np.asarray(page_table_row)[page_index])
        if page < 0 or page >= self.num_pages:
            raise IndexError("page id out of range")
        return packing.record_offset(self.num_layers, self.num_kv_heads, page, layer, kv_head, 1, 0)

    def append(self, page_table_row, start: int, layer: int, k_raw: np.ndarray, v_raw: np.ndarray) -> np.ndarray:
        """Encode and store raw K, V [n, Hkv, 256] at positions [start, start + n). Returns flags [n, Hkv, 2]."""
        n = k_raw.shape[0]
        flags = np.zeros((n, self.num_kv_heads, 2), dtype=np.int32)
        pos = np.arange(start, start + n)
        for g in range(self.num_kv_heads):
            codes, s16, f = codec.encode(k_raw[:, g, :])
            off = self._offsets(page_table_row, pos, layer, g, 0)
            self.pool[off[:, None] + np.arange(packing.RECORD_BYTES)[None, :]] = packing.pack_records(codes, s16)
            flags[:, g, 0] = f
            codes, s16, f = codec.encode(v_raw[:, g, :])
            flags[:, g, 1] = f
            for pi in np.unique(pos // packing.PAGE_SIZE):
                sel = (pos // packing.PAGE_SIZE) == pi
                base = self._value_page_offset(page_table_row, pi, layer, g)
                pc, ps = packing.unpack_value_page(self.pool[base:base + packing.VALUE_PAGE_BYTES])
                rows = pos[sel] % packing.PAGE_SIZE
                pc[rows] = codes[sel]
                ps[rows] = s16[sel]
                self.pool[base:base + packing.VALUE_PAGE_BYTES] = packing.pack_value_page(pc, ps)
        return flags

    def records(self, page_table_row, layer: int, kv_head: int, start: int, count: int) -> np.ndarray:
        """The K records of positions [start, start + count)."""
        off = self._offsets(page_table_row, np.arange(start, start + count), layer, kv_head, 0)
        return self.pool[off[:, None] + np.arange(packing.RECORD_BYTES)[None, :]]

    def value_codes(self, page_table_row, layer: int, kv_head: int, count: int):
        """Codes [count, 256] and scales [count, 8] of the V vectors at positions [0, count)."""
        codes = np.zeros((count, 256), np.uint8)
        scales = np.zeros((count, 8), np.float16)
        for pi in range((count + packing.PAGE_SIZE - 1) // packing.PAGE_SIZE):
            base = self._value_page_offset(page_table_row, pi, layer, kv_head)
            pc, ps = packing.unpack_value_page(self.pool[base:base + packing.VALUE_PAGE_BYTES])
            n = min(packing.PAGE_SIZE, count - pi * packing.PAGE_SIZE)
            codes[pi * packing.PAGE_SIZE:pi * packing.PAGE_SIZE + n] = pc[:n]
            scales[pi * packing.PAGE_SIZE:pi * packing.PAGE_SIZE + n] = ps[:n]
        return codes, scales

    def dequantized(self, page_table_row, layer: int, kv_head: int, kv: int, count: int) -> np.ndarray:
        if kv == 0:
            codes, s16 = packing.unpack_records(self.records(page_table_row, layer, kv_head, 0, count))
        else:
            codes, s16 = self.value_codes(page_table_row, layer, kv_head, count)
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
