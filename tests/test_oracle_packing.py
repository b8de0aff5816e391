"""Pins of the oracle's record and page layout: hand-derived words, round trip, offsets."""
import json
import os

import numpy as np

from oracle import packing

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "packing_hand_examples.json")


def test_hand_examples():
    for case in json.load(open(GOLDEN))["cases"]:
        codes = np.zeros(256, np.uint8)
        for e, c in case["codes"].items():
            codes[int(e)] = c
        scales = np.zeros(8, np.float16)
        for b, hx in case["scales_hex"].items():
            scales[int(b)] = np.frombuffer(bytes.fromhex(hx)[::-1], dtype="<f2")[0]
        rec = packing.pack_records(codes[None], scales[None])[0]
        assert rec.shape == (112,)
        words = rec[:96].view("<u4")
        want = np.zeros(24, np.uint32)
        for w, hx in case["words_hex"].items():
            want[int(w)] = int(hx, 16)
        assert np.array_equal(words, want), case
        for b, hx in case["scales_hex"].items():
            assert rec[96 + 2 * int(b):98 + 2 * int(b)].tobytes() == bytes.fromhex(hx)[::-1]
        c2, s2 = packing.unpack_records(rec[None])
        assert np.array_equal(c2[0], codes) and np.array_equal(s2[0].view(np.uint16), scales.view(np.uint16))


def test_every_bit_used_once():
    # 256 codes x 3 bits fill the 768 code bits exactly
    seen = np.zeros(24 * 32, np.int32)
    for e in range(256):
        for k in range(3):
            codes = np.zeros(256, np.uint8)
            codes[e] = 1 << k
            words = packing.pack_records(codes[None], np.zeros((1, 8), np.float16))[0, :96].view("<u4")
            bits = np.unpackbits(words.view(np.uint8), bitorder="little")
            assert bits.sum() == 1
            seen[np.argmax(bits)] += 1
    assert np.all(seen == 1)


def test_pairs_extract_with_shift_and_mask():
    # the property the layout exists for: (w >> 3j) & 0x00070007 holds elements (2m, 2m+1)
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 8, 256).astype(np.uint8)
    words = packing.pack_records(codes[None], np.zeros((1, 8), np.float16))[0, :96].view("<u4")
    for b in range(8):
        for m in range(15):
            w = int(words[3 * b + m // 5]) >> (3 * (m % 5))
            assert (w & 7) == codes[32 * b + 2 * m]
            assert ((w >> 16) & 7) == codes[32 * b + 2 * m + 1]
        w0, w1, w2 = (int(words[3 * b + k]) for k in range(3))
        lo = ((w0 >> 15) & 1) | (((w1 >> 15) & 1) << 1) | (((w2 >> 15) & 1) << 2)
        hi = ((w0 >> 31) & 1) | (((w1 >> 31) & 1) << 1) | (((w2 >> 31) & 1) << 2)
        assert lo == codes[32 * b + 30] and hi == codes[32 * b + 31]


def test_round_trip_random():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 8, (50, 3, 256)).astype(np.uint8)
    scales = rng.standard_normal((50, 3, 8)).astype(np.float16)
    c, s = packing.unpack_records(packing.pack_records(codes, scales))
    assert np.array_equal(c, codes) and np.array_equal(s.view(np.uint16), scales.view(np.uint16))


def test_record_offsets():
    L, H = 16, 2
    assert packing.record_offset(L, H, 0, 0, 0, 0, 0) == 0
    assert packing.record_offset(L, H, 0, 0, 0, 0, 1) == 112
    assert packing.record_offset(L, H, 0, 0, 0, 1, 0) == 256 * 112          # V chunk follows K chunk
    assert packing.record_offset(L, H, 0, 0, 1, 0, 0) == 2 * 256 * 112
    assert packing.record_offset(L, H, 0, 1, 0, 0, 0) == 2 * 2 * 256 * 112
    assert packing.record_offset(L, H, 1, 0, 0, 0, 0) == 16 * 2 * 2 * 256 * 112
    assert packing.pool_bytes(3, L, H) == 3 * 16 * 2 * 2 * 256 * 112
    assert packing.record_offset(L, H, 2, 15, 1, 1, 255) + 112 == packing.pool_bytes(3, L, H)
