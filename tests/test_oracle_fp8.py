"""Pins of the fp8 E4M3 comparison format (oracle/fp8.py).

* the format's published facts: largest finite 448, smallest normal 2^-6,
  smallest subnormal 2^-9, NaN patterns, monotone positive codes;
* round trip: every finite byte decodes to a value that encodes back to it;
* brute force: encoding picks the nearest representable value, ties to the
  even mantissa, against a scan over the whole value table;
* saturation above 448 and signed zero below the smallest subnormal;
* the library routine: torch's float8_e4m3fn cast agrees on in-range inputs;
* attention: constant V gives V; a single visible position gives its V; the
  plain formula equals the rotated-basis oracle on rotated inputs.
"""
import numpy as np
import pytest

from oracle import fp8
from oracle.attention import verify_attention
from oracle.wht import rotate_f64


def test_published_format_facts():
    v = fp8.decode(np.arange(256, dtype=np.uint8))
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x00] == 0.0 and np.signbit(v[0x80]) and v[0x80] == 0.0
    assert v[0x38] == 1.0                                   # exponent field 7 = bias
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                         # strictly increasing magnitudes
    assert np.array_equal(v[0x80:0xFF], -pos)


def test_round_trip_every_finite_byte():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    back, nf = fp8.encode(fp8.decode(codes).astype(np.float32))
    assert np.array_equal(back, codes) and not nf.any()


def _nearest_even_bruteforce(x):
    table = fp8.decode(np.arange(0x7F, dtype=np.uint8))    # non-negative finite values, index = code
    a = abs(float(x))
    if a >= 448.0:
        c = 0x7E
    else:
        d = np.abs(table - a)
        best = np.flatnonzero(d == d.min())
        c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return c | (0x80 if np.signbit(x) else 0)


def test_nearest_ties_even_bruteforce():
    rng = np.random.default_rng(0)
    table = fp8.decode(np.arange(0x7F, dtype=np.uint8))
    mids = (table[:-1] + table[1:]) / 2                     # every tie, both signs
    xs = np.concatenate([
        rng.standard_normal(3000) * 30, rng.uniform(-500, 500, 2000), rng.uniform(-0.02, 0.02, 2000),
        mids, -mids, table, np.nextafter(mids, 0), np.nextafter(mids, 1000),
    ]).astype(np.float32)
    got, _ = fp8.encode(xs)
    want = np.array([_nearest_even_bruteforce(x) for x in xs], np.uint8)
    assert np.array_equal(got, want)


def test_saturation_underflow_and_non_finite():
    got, nf = fp8.encode(np.array([448, 464, 480, 1e30, -470, 2.0 ** -10, -2.0 ** -10, 2.0 ** -10 * 1.01,
                                   np.inf, -np.inf, np.nan], np.float32))
    assert list(got[:8]) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x00, 0x80, 0x01]
    assert list(got[8:]) == [0x7E, 0xFE, 0x7F]
    assert list(nf) == [0] * 8 + [1, 1, 1]


def test_matches_torch_float8_cast_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 10, rng.uniform(-447, 447, 5000),
                        rng.standard_normal(5000) * 1e-3]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got, _ = fp8.encode(x)
    assert np.array_equal(got, ref)


def test_attention_constant_v_and_single_position():
    rng = np.random.default_rng(2)
    T, Hq, L = 3, 16, 20
    q = rng.standard_normal((T, Hq, 256))
    k = rng.standard_normal((2, L, 256))
    v = np.broadcast_to(rng.standard_normal(256), (2, L, 256))
    out = fp8.attention(q, k, v, L - T, 8)
    assert np.allclose(out, v[0, 0][None, None, :], atol=1e-12)
    v2 = rng.standard_normal((2, 1, 256))
    out1 = fp8.attention(q[:1], k[:, :1], v2, 0, 8)
    for h in range(Hq):
        assert np.allclose(out1[0, h], v2[h // 8, 0], atol=1e-12)


def test_plain_attention_equals_rotated_oracle():
    # the rotated-basis oracle on (H k, H v) is the same attention: H is orthonormal
    rng = np.random.default_rng(3)
    T, L = 4, 37
    q = rng.standard_normal((T, 16, 256))
    k = rng.standard_normal((2, L, 256))
    v = rng.standard_normal((2, L, 256))
    plain = fp8.attention(q, k, v, L - T, 8)
    rot = verify_attention(q, rotate_f64(k), rotate_f64(v), L - T, 8)
    assert np.max(np.abs(plain - rot)) < 1e-10


def test_cache_layout_and_decode():
    cache = fp8.Fp8PagedCache(num_pages=3, num_layers=2, num_kv_heads=2)
    rng = np.random.default_rng(4)
    pt = np.array([2, 0], np.int32)
    k = (rng.standard_normal((300, 2, 256)) * 50).astype(np.float32)
    v = (rng.standard_normal((300, 2, 256)) * 50).astype(np.float32)
    flags = cache.append(pt, 0, 1, k, v)
    assert not flags.any()
    # position 257 of layer 1, head 1, V: page pt[1] = 0, row 1
    off = ((((0 * 2 + 1) * 2 + 1) * 2 + 1) * 256 + 1) * 256
    assert np.array_equal(cache.pool[off:off + 256], fp8.encode(v[257, 1])[0])
    dec = cache.decoded(pt, 1, 0, 0, 300)
    assert np.array_equal(dec, fp8.decode(fp8.encode(k[:, 0])[0]))
