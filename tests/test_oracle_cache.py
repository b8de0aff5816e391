"""Pins of the oracle's paged cache: records land where the layout says,
scattered page tables read back what was appended, rollback overwrites, and a
full step agrees with the un-paged definition.  Also pins the input generator's
addressing (page-wise regeneration equals a range draw)."""
import numpy as np
import pytest

import q3kv_inputs as qi
from oracle import codec, packing
from oracle.attention import verify_attention
from oracle.cache import PagedCache, encode_dequantized


def test_append_lands_at_layout_offset():
    c = PagedCache(num_pages=4, num_layers=2, num_kv_heads=2)
    pt = np.array([3, 1], np.int32)
    rng = np.random.default_rng(0)
    k = rng.standard_normal((3, 2, 256)).astype(np.float32)
    v = rng.standard_normal((3, 2, 256)).astype(np.float32)
    c.append(pt, 255, 1, k, v)              # positions 255 (page 3 row 255), 256, 257 (page 1 rows 0, 1)
    for i, pos in enumerate([255, 256, 257]):
        page = pt[pos // 256]
        for g in range(2):
            for kv, x in ((0, k), (1, v)):
                off = packing.record_offset(2, 2, page, 1, g, kv, pos % 256)
                codes, s16, _ = codec.encode(x[i, g][None])
                assert np.array_equal(c.pool[off:off + 112], packing.pack_records(codes, s16)[0])
    # nothing else was written
    touched = np.zeros_like(c.pool, dtype=bool)
    for pos in (255, 256, 257):
        for g in range(2):
            for kv in range(2):
                off = packing.record_offset(2, 2, pt[pos // 256], 1, g, kv, pos % 256)
                touched[off:off + 112] = True
    assert not np.any(c.pool[~touched])


def test_rollback_is_overwrite():
    c = PagedCache(num_pages=2, num_layers=1, num_kv_heads=2)
    pt = np.array([1, 0], np.int32)
    rng = np.random.default_rng(1)
    a = rng.standard_normal((10, 2, 256)).astype(np.float32)
    b = rng.standard_normal((4, 2, 256)).astype(np.float32)
    c.append(pt, 0, 0, a, a)
    c.append(pt, 6, 0, b, b)                 # drafts 6..9 rejected, new tokens written over them
    want = np.concatenate([a[:6], b])
    for g in range(2):
        got = c.dequantized(pt, 0, g, 0, 10)
        np.testing.assert_array_equal(got, encode_dequantized(want[:, g]))


def test_out_of_range_page_raises():
    c = PagedCache(num_pages=2, num_layers=1, num_kv_heads=2)
    with pytest.raises(IndexError):
        c.append(np.array([5], np.int32), 0, 0, np.zeros((1, 2, 256), np.float32), np.zeros((1, 2, 256), np.float32))


def test_step_matches_unpaged_definition():
    w = qi.WORKLOADS[1]
    n_ctx, T = 300, 4
    pt = qi.random_page_table(1, [2], 5, seed=1)[0]
    c = PagedCache(num_pages=5, num_layers=1, num_kv_heads=2)
    k = np.stack([qi.kv_rows(w, 0, 0, g, 0, 0, n_ctx + T) for g in range(2)], axis=1)
    v = np.stack([qi.kv_rows(w, 0, 0, g, 1, 0, n_ctx + T) for g in range(2)], axis=1)
    c.append(pt, 0, 0, k[:n_ctx], v[:n_ctx])
    c.append(pt, n_ctx, 0, k[n_ctx:], v[n_ctx:])
    q = qi.q_rows(w, 0, 0, 0, T)
    got = c.verify(pt, 0, n_ctx, q, 8)
    kh = np.stack([encode_dequantized(k[:, g]) for g in range(2)])
    vh = np.stack([encode_dequantized(v[:, g]) for g in range(2)])
    np.testing.assert_array_equal(got, verify_attention(q, kh, vh, n_ctx, 8))


def test_inputs_pagewise_addressing():
    w = qi.WORKLOADS[2]
    whole = qi.kv_rows(w, 0, 3, 1, 0, 200, 400)
    assert np.array_equal(whole[:56], qi.kv_page(w, 0, 3, 1, 0, 0)[200:])
    assert np.array_equal(whole[56:312], qi.kv_page(w, 0, 3, 1, 0, 1))
    # bf16 workloads hand out bf16-representable values
    assert np.all((whole.view(np.uint32) & 0xFFFF) == 0)
    s = qi.draw_shapes(qi.WORKLOADS[3])
    assert all(8192 <= c <= 131072 for c in s.ctx) and all(3 <= t <= 8 for t in s.n_new[0])
    s4 = qi.draw_shapes(qi.WORKLOADS[4])
    assert len(s4.n_new) == 32 and all(4 <= t <= 8 for row in s4.n_new for t in row)


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9], np.float32)
    r = qi.round_to_bf16(x)
    assert r.tolist() == [1.0, 1.0 + 2.0 ** -6, 1.0]
