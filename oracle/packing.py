"""Byte layout of coded vectors and cache pages (oracle; test infrastructure only).

The layout is this library's choice (the pages give turbo3's size, "50-byte
blocks per 128 dims", but not its bits).  It is chosen so that a GPU thread can
turn a 32-bit word into two fp16 values with one shift and one mask.

Record of one vector (112 bytes, 16-byte aligned):
  bytes  0..95  : 24 little-endian uint32 words, three per 32-element block
                  (block b owns words 3b, 3b+1, 3b+2)
  bytes 96..111 : 8 fp16 scales, block 0 first

Inside block b (codes q[0..31], 3 bits each):
  element e < 30: pair m = e // 2, half = e % 2
                  word 3b + m // 5, bit offset 16*half + 3*(m % 5), bits [off, off+3)
                  (a word holds 5 even elements in bits 0..14 and the 5 odd
                   partners in bits 16..30, so (w >> 3j) & 0x00070007 is a pair)
  element 30    : code bit k in bit 15 of word 3b + k   (k = 0, 1, 2)
  element 31    : code bit k in bit 31 of word 3b + k

Page pool: page p holds positions [256*i, 256*i + 256) of whichever slot's page
table names p at index i.  Inside the pool the record of
(page, layer, kv_head, kv in {0: K, 1: V}, row r = position % 256) starts at byte

  ((((page * num_layers + layer) * num_kv_heads + kv_head) * 2 + kv) * 256 + r) * 112

so one (page, layer, kv head) is a 28,672-byte K chunk followed by its V chunk.
"""
from __future__ import annotations

import numpy as np

RECORD_BYTES = 112
CODE_WORDS = 24
PAGE_SIZE = 256


def _field(e: int):
    """(word index within the block, list of (bit position, code bit)) for element e."""
    if e < 30:
        m, half = divmod(e, 2)
        off = 16 * half + 3 * (m % 5)
        return [(m // 5, off + k, k) for k in range(3)]
    top = 15 if e == 30 else 31
    return [(k, top, k) for k in range(3)]


def pack_records(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes uint8 [..., 256], scales float16 [..., 8] -> uint8 [..., 112]."""
    codes = np.asarray(codes, dtype=np.uint32)
    lead = codes.shape[:-1]
    words = np.zeros(lead + (CODE_WORDS,), dtype=np.uint32)
    for b in range(8):
        for e in range(32):
            c = codes[..., 32 * b + e]
            for wi, bit, k in _field(e):
                words[..., 3 * b + wi] |= ((c >> np.uint32(k)) & np.uint32(1)) << np.uint32(bit)
    out = np.empty(lead + (RECORD_BYTES,), dtype=np.uint8)
    out[..., :96] = words.astype("<u4").view(np.uint8).reshape(lead + (96,))
    out[..., 96:] = np.asarray(scales, dtype="<f2").view(np.uint8).reshape(lead + (16,))
    return out


def unpack_records(rec: np.ndarray):
    """uint8 [..., 112] -> (codes uint8 [..., 256], scales float16 [..., 8])."""
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    lead = rec.shape[:-1]
    words = rec[..., :96].copy().view("<u4").reshape(lead + (CODE_WORDS,)).astype(np.uint32)
    codes = np.zeros(lead + (256,), dtype=np.uint32)
    for b in range(8):
        for e in range(32):
            for wi, bit, k in _field(e):
                codes[..., 32 * b + e] |= ((words[..., 3 * b + wi] >> np.uint32(bit)) & np.uint32(1)) << np.uint32(k)
    scales = rec[..., 96:].copy().view("<f2").reshape(lead + (8,)).astype(np.float16)
    return codes.astype(np.uint8), scales


def record_offset(num_layers: int, num_kv_heads: int, page: int, layer: int, kv_head: int, kv: int, row: int) -> int:
    return ((((page * num_layers + layer) * num_kv_heads + kv_head) * 2 + kv) * PAGE_SIZE + row) * RECORD_BYTES


def pool_bytes(num_pages: int, num_layers: int, num_kv_heads: int) -> int:
    return num_pages * num_layers * num_kv_heads * 2 * PAGE_SIZE * RECORD_BYTES
