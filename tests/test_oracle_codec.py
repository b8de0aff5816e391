"""Pins of the oracle's 3-bit codec.

* hand-derived blocks (tests/golden/codec_hand_examples.json);
* the fp16 scale against an independent computation with Python floats and the
  struct module's IEEE half packing;
* brute force: each code is the nearest of the 8 levels (ties to the even
  code), except where float32 rounding of y/s crosses a half-integer;
* the error bound |y - (q - 3.5)s| <= s/2 (1 + 2^-10);
* dequantisation is exact in float32;
* flags for non-finite input and scale overflow.
"""
import json
import os
import struct

import numpy as np
import pytest

from oracle import codec
from oracle.wht import fwht_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "codec_hand_examples.json")


def _block(case):
    y = list(case["y"]) + [case["pad"]] * (32 - len(case["y"]))
    return np.array(y, dtype=np.float32)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"][:40])
def test_hand_examples(case):
    y = np.zeros(256, np.float32)
    y[64:96] = _block(case)             # put it in block 2 so the block index matters
    codes, s16 = codec.quantize_rotated(y[None, :])
    assert s16[0, 2].tobytes().hex() == bytes.fromhex(case["scale_f16_hex"])[::-1].hex()
    want = list(case["codes"]) + [case["codes_pad"]] * (32 - len(case["codes"]))
    assert codes[0, 64:96].tolist() == want
    # the other (all-zero) blocks
    assert np.all(codes[0, :64] == 4) and np.all(codes[0, 96:] == 4)
    assert np.all(s16[0, [0, 1, 3, 4, 5, 6, 7]] == 0)


def _scale_independent(absmax_f32: float) -> float:
    q = struct.unpack("<f", struct.pack("<f", absmax_f32 / 3.5))[0]   # correctly rounded fp32 quotient
    return struct.unpack("<e", struct.pack("<e", q))[0]               # IEEE RNE to half


def test_scale_matches_independent_rounding():
    rng = np.random.default_rng(1)
    y = (rng.standard_normal((400, 256)) * 10 ** rng.uniform(-6, 4, (400, 1))).astype(np.float32)
    s16 = codec.block_scales(y)
    absmax = np.max(np.abs(y.reshape(400, 8, 32)), axis=-1)
    for i in range(400):
        for b in range(8):
            assert float(s16[i, b]) == _scale_independent(float(absmax[i, b]))


def _levels_brute(y, s):
    """Nearest of (q - 3.5)s for q in 0..7, ties to even q (float64)."""
    lv = (np.arange(8) - 3.5) * s
    d = np.abs(y - lv)
    best = np.min(d)
    cand = [q for q in range(8) if d[q] == best]
    return [q for q in cand if q % 2 == 0][0] if len(cand) > 1 else cand[0]


def test_codes_are_nearest_levels():
    rng = np.random.default_rng(2)
    y = (rng.standard_normal((300, 256)) * np.where(rng.random(256) < 0.05, 8.0, 1.0)).astype(np.float32)
    codes, s16 = codec.quantize_rotated(y)
    s = s16.astype(np.float64)
    mismatches = 0
    for i in range(300):
        for e in range(256):
            b = e // 32
            want = _levels_brute(float(y[i, e]), float(s[i, b]))
            if codes[i, e] != want:
                mismatches += 1
                assert abs(int(codes[i, e]) - want) == 1
    assert mismatches <= 300 * 256 * 1e-4


def test_exact_ties_go_to_even_code():
    s = np.float32(0.5)
    y = np.zeros(256, np.float32)
    # y/s + 3.5 = k + 0.5 exactly for k = 0..6  ->  even neighbour
    y[:7] = (np.arange(7) + 0.5 - 3.5) * s
    y[7] = 3.5 * s
    codes, s16 = codec.quantize_rotated(y[None, :])
    assert float(s16[0, 0]) == 0.5
    assert codes[0, :8].tolist() == [0, 2, 2, 4, 4, 6, 6, 7]


def test_error_bound():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((256, 256)) * 10 ** rng.uniform(0, 1, 256)).astype(np.float32)
    y = fwht_f32(x)
    codes, s16 = codec.quantize_rotated(y)
    deq = codec.dequantize(codes, s16)
    s = np.repeat(s16.astype(np.float64), 32, axis=-1)
    assert np.all(np.abs(y - deq) <= s / 2 * (1 + 2.0 ** -10))


def test_dequant_exact_in_float32():
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 8, (64, 256)).astype(np.uint8)
    s16 = (rng.standard_normal((64, 8)) * 10).astype(np.float16)
    d64 = codec.dequantize(codes, s16)
    d32 = ((codes.astype(np.float32).reshape(64, 8, 32) - np.float32(3.5)) * s16.astype(np.float32)[..., None]).reshape(64, 256)
    assert np.array_equal(d64, d32.astype(np.float64))


def test_encode_rotates_first():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((4, 256)).astype(np.float32)
    c1, s1, f = codec.encode(x)
    c2, s2 = codec.quantize_rotated(fwht_f32(x))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2) and np.all(f == 0)


def test_flags():
    x = np.zeros((3, 256), np.float32)
    x[0, 5] = np.nan
    x[1, 0] = 4.0e6    # rotates to 250000 everywhere; 250000 / 3.5 > 65504 -> fp16 overflow
    _, s16, flags = codec.encode(x)
    assert flags[0] & codec.FLAG_NONFINITE
    assert flags[1] & codec.FLAG_SCALE_OVERFLOW
    assert flags[2] == 0
