"""Pins of the turbo5k-style K codec (oracle/turbo5k.py).

* Lloyd-Max: every centroid is the normal mean over its cell (numerical
  integration), boundaries are midpoints, exact symmetry; an independent
  algorithm (plain Lloyd iteration) lands on the same table, and the table is a
  fixed point of k-means on normal samples;
* scale: closed forms where every partial sum is exact (constant blocks,
  1..128), an all-zero block;
* codes: brute-force nearest float32 centroid with ties to the lower code;
* packing: a hand-built record, round trip; decoding is exact;
* cache: records at the layout's offsets; the paged verify equals the
  un-paged definition.
"""
import math

import numpy as np
import pytest

from oracle import codec as q3codec
from oracle import turbo5k as t
from oracle.attention import verify_attention
from oracle.wht import fwht_f32


def test_lloyd_max_conditions():
    integrate = pytest.importorskip("scipy.integrate")
    c = t.lloyd_max_gaussian_f64()
    assert c.shape == (32,) and np.all(np.diff(c) > 0)
    assert np.array_equal(c[:16], -c[16:][::-1])
    b = np.concatenate([[-np.inf], (c[:-1] + c[1:]) / 2, [np.inf]])
    pdf = lambda x: math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)
    for j in range(32):
        num = integrate.quad(lambda x: x * pdf(x), b[j], b[j + 1], epsabs=1e-14, epsrel=1e-12)[0]
        den = integrate.quad(pdf, b[j], b[j + 1], epsabs=1e-14, epsrel=1e-12)[0]
        assert abs(num / den - c[j]) < 1e-9


def test_plain_lloyd_iteration_agrees():
    from scipy.special import ndtr
    pdf = lambda x: np.exp(-0.5 * x * x) / np.sqrt(2 * np.pi)
    c = np.linspace(-3, 3, 32)
    for _ in range(20000):
        b = np.concatenate([[-np.inf], (c[:-1] + c[1:]) / 2, [np.inf]])
        c = (pdf(b[:-1]) - pdf(b[1:])) / (ndtr(b[1:]) - ndtr(b[:-1]))
    assert np.max(np.abs(c - t.lloyd_max_gaussian_f64())) < 1e-4


def test_table_is_a_fixed_point_of_sample_kmeans():
    # the table, as the starting point of k-means on normal samples, stays put
    x = np.random.default_rng(0).standard_normal(2_000_000)
    c0 = t.lloyd_max_gaussian_f64()
    c = c0.copy()
    for _ in range(5):
        idx = np.searchsorted((c[:-1] + c[1:]) / 2, x)
        c = np.bincount(idx, weights=x, minlength=32) / np.bincount(idx, minlength=32)
    assert np.max(np.abs(c - c0)) < 0.02


def test_table_boundaries_are_float32_midpoints():
    c, b = t.table()
    assert c.dtype == np.float32 and b.dtype == np.float32 and b[15] == 0.0
    assert np.array_equal(b, (c[:-1] + c[1:]) * np.float32(0.5))


def test_half_scale_closed_forms():
    y = np.zeros((3, 256), np.float32)
    y[0, :128] = 4.0                      # rms 4
    y[0, 128:] = -0.5
    y[1, :128] = np.arange(1, 129)        # sum of squares 707,264, exact in float32
    s = t.half_scales(y)
    assert s[0, 0] == 4.0 and s[0, 1] == 0.5
    assert s[1, 0] == np.float16(np.sqrt(np.float32(707264.0 / 128.0)))
    assert s[1, 1] == 0.0 and s[2, 0] == 0.0 and s[2, 1] == 0.0


def test_codes_are_nearest_centroid_ties_down():
    c, b = t.table()
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((40, 256)) * rng.uniform(0.1, 10, size=(40, 1))).astype(np.float32)
    codes, s16, flags = t.encode_k(x)
    assert not flags.any()
    y = fwht_f32(x).reshape(40, 2, 128)
    v = (y / s16.astype(np.float32)[..., None]).astype(np.float32)
    d = np.abs(v[..., None].astype(np.float64) - c.astype(np.float64))
    want = np.argmin(d, axis=-1)           # the first (lower) index on ties
    assert np.array_equal(codes.reshape(40, 2, 128), want)
    # exact boundary values take the lower code
    vb = b.astype(np.float32)
    assert np.array_equal((vb[:, None] > b).sum(axis=-1), np.arange(31))


def test_zero_block_and_flags():
    x = np.zeros((2, 256), np.float32)
    x[1, 3] = np.nan
    codes, s16, flags = t.encode_k(x)
    assert np.all(codes[0] == 16) and np.all(s16[0] == 0)
    assert flags[0] == 0 and flags[1] == q3codec.FLAG_NONFINITE


def test_hand_record_and_round_trip():
    codes = np.tile(np.arange(32, dtype=np.uint8), 8)[None]
    s16 = np.array([[1.0, 2.0]], np.float16)
    rec = t.pack_k(codes, s16)[0]
    assert rec.shape == (164,)
    assert list(rec[:4]) == [0x10, 0x32, 0x54, 0x76] and rec[8] == 0x10
    assert list(rec[128:136]) == [0, 0, 0xFF, 0xFF, 0, 0, 0xFF, 0xFF]
    assert list(rec[160:164]) == [0x00, 0x3C, 0x00, 0x40]
    c2, s2 = t.unpack_k(rec[None])
    assert np.array_equal(c2, codes) and np.array_equal(s2, s16)
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 32, size=(50, 256)).astype(np.uint8)
    s16 = rng.uniform(0.01, 100, size=(50, 2)).astype(np.float16)
    c2, s2 = t.unpack_k(t.pack_k(codes, s16))
    assert np.array_equal(c2, codes) and np.array_equal(s2, s16)


def test_decode_is_exact():
    c, _ = t.table()
    codes = np.arange(256, dtype=np.int64)[None] % 32
    s16 = np.array([[3.25, 0.0078125]], np.float16)
    val = t.decode_k(codes.astype(np.uint8), s16)
    assert np.array_equal(val[0, :128], c[codes[0, :128]].astype(np.float64) * 3.25)
    assert np.array_equal(val[0, 128:], c[codes[0, 128:]].astype(np.float64) * 0.0078125)


def test_cache_offsets_and_verify():
    rng = np.random.default_rng(3)
    cache = t.T5kPagedCache(num_pages=4, num_layers=2, num_kv_heads=2)
    pt = np.array([3, 1], np.int32)
    n_ctx, T = 290, 4
    k = rng.standard_normal((n_ctx + T, 2, 256)).astype(np.float32)
    v = rng.standard_normal((n_ctx + T, 2, 256)).astype(np.float32)
    assert not cache.append(pt, 0, 1, k, v).any()
    # position 257 of layer 1, head 0: page 1, row 1
    off = t.k_offset(2, 2, 1, 1, 0, 1)
    assert np.array_equal(cache.pool[off:off + 164], t.pack_k(*t.encode_k(k[257, 0])[:2]))
    off = t.v_offset(2, 2, 1, 1, 1, 1)
    vc, vs, _ = q3codec.encode(v[257, 1])
    from oracle import packing
    assert np.array_equal(cache.pool[off:off + 112], packing.pack_records(vc, vs))
    q = rng.standard_normal((T, 16, 256))
    kh = np.stack([t.encode_dequantized_k(k[:, g]) for g in range(2)])
    vh = np.stack([q3codec.dequantize(*q3codec.encode(v[:, g])[:2]) for g in range(2)])
    assert np.array_equal(cache.verify(pt, 1, n_ctx, q, 8), verify_attention(q, kh, vh, n_ctx, 8))
