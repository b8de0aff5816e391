"""The operand-precision ladder behind the tensor-core leg's design (tests/precision_ladder.py).

On a reduced workload-2 case (4,096 cached positions, 6 tokens, log-uniform
channel scales) the ladder must show what the design rests on: any single
fp16 operand for Q or K̂ misses the 2e-3 tolerance, while the kernel's split
scheme (exact K̂/V̂ pairs, round-to-nearest Q/P pairs, three products) and the
fp8 leg's two-product scheme stay far inside it.  The ladder's exact row is
tied to the oracle's attention first, so the emulation measures against the
oracle's definition.
"""
import numpy as np

import precision_ladder as pl
from oracle import attention, fp8
from oracle.cache import encode_dequantized

MAX_ABS, REL_L2 = 2e-3, 1e-3


def _case():
    return pl.Case(2, 0, 1, 4096, 6)


def test_ladder_reference_is_the_oracle():
    case = _case()
    res = pl.ladder_q3(case)
    kh = encode_dequantized(case.k_raw)[None]
    vh = encode_dequantized(case.v_raw)[None]
    q = case.q_raw.reshape(6, 8, 256)
    want = attention.verify_attention(q, kh, vh, 4096, 8).reshape(48, 256)
    np.testing.assert_allclose(res["reference"], want, rtol=0, atol=1e-10)
    ref8 = pl.ladder_fp8(case)["reference"]
    k8 = fp8.decode(fp8.encode_vectors(case.k_raw)[0])[None]
    v8 = fp8.decode(fp8.encode_vectors(case.v_raw)[0])[None]
    np.testing.assert_allclose(ref8, fp8.attention(q, k8, v8, 4096, 8).reshape(48, 256), rtol=0, atol=1e-10)


def test_exact_split_is_exact_in_fp16():
    x = _case().k_raw[:300]
    for mask in (pl.K_HI_MASK, pl.V_HI_MASK):
        val, hi, lo = pl.exact_split_q3(x, mask)
        assert np.array_equal(hi + lo, val)
        assert np.array_equal(pl.f16(hi), hi) and np.array_equal(pl.f16(lo), lo)


def test_outlier_heavy_queries_and_keys_need_the_8_bit_key_split():
    """Queries and cache both with 10x channels: scores reach ~100 (log2 units).

    The dropped Qlo.Klo product with a 6-bit key split then costs more than
    half the tolerance; with the 8-bit split it stays far inside it.
    """
    import q3kv_inputs as qi
    base = qi.WORKLOADS[1]
    w = qi.Workload(base.key, "small", 17, 1, 2, (0, 0), (0, 0), 1, "bf16", "loguniform10", "loguniform10")
    worst6 = worst8 = 0.0
    for g in range(2):
        err = pl.errors(pl.ladder_q3(pl.Case(w, 0, g, 0, 300)))
        worst6 = max(worst6, err["kernel_q3_k6"][0])
        worst8 = max(worst8, err["kernel_q3"][0])
    assert worst6 > MAX_ABS / 2, worst6
    assert worst8 < MAX_ABS / 4, worst8


def test_single_fp16_operands_miss_and_the_split_schemes_meet_the_tolerance():
    case = _case()
    err = pl.errors(pl.ladder_q3(case))
    err.update(pl.errors(pl.ladder_fp8(case)))
    for name in ("all_f16", "q_f16", "k_f16"):
        assert err[name][0] > MAX_ABS, (name, err[name])
    assert err["kernel_q3"][0] < MAX_ABS / 5 and err["kernel_q3"][1] < REL_L2 / 10, err["kernel_q3"]
    assert err["kernel_fp8"][0] < MAX_ABS / 20 and err["kernel_fp8"][1] < REL_L2 / 100, err["kernel_fp8"]


def test_one_fused_multiply_add_per_half_is_exact_for_every_scale():
    """The tensor-core leg's dequantisation, for every fp16 scale it accepts.

    From x = 8.5 + c (exact in fp16), each half (c - 3.5) s_part is formed as
    one fused multiply-add x * s_part + (-12 s_part).  It is exact when -12
    s_part is exact in fp16 and the result is: checked exhaustively over all
    positive fp16 scales from 2^-13 up to the leg's limit 65504 / 12, all
    eight codes, with the fused operation's single rounding emulated in
    float64 (the product of two fp16 numbers is exact there).  A smaller scale
    (a block whose largest value is below 4.3e-4) can leave the lo half off by
    at most 2^-25.
    """
    s16 = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16)
    s16 = s16[s16.astype(np.float64) <= 65504.0 / 12.0]
    s = s16.astype(np.float64)
    s_hi16 = (s16.view(np.uint16) & np.uint16(pl.K_HI_MASK)).view(np.float16)
    s_hi = s_hi16.astype(np.float64)
    s_lo = s - s_hi
    assert np.array_equal(pl.f16(s_lo), s_lo)                       # s_lo exact in fp16
    normal = s >= 2.0 ** -13          # s_lo is then a multiple of 2^-23
    for part in (s_hi, s_lo):
        const = -12.0 * part
        assert np.array_equal(pl.f16(const), const)                 # the FMA's addend is exact
        for c in range(8):
            fused = pl.f16((8.5 + c) * part + const)                # one rounding
            assert np.array_equal(fused[normal], (c - 3.5) * part[normal]), c
            assert np.abs(fused - (c - 3.5) * part).max() <= 2.0 ** -25
    # and the pair adds up to the decoded value
    for c in range(8):
        assert np.array_equal((c - 3.5) * s_hi + (c - 3.5) * s_lo, (c - 3.5) * s)
