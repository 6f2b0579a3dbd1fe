"""Pins for the oracle's quantize-on-write.

Formula (#3084 qwen35: FP16 K/V cache by default, int8 with --kv-q8, section
"What changed"): per group of 64 dims, scale = fp16(max|x| / 127) and
code = clamp(rint(x / scale), -127, 127).  Readings: both divisions are IEEE
fp32, x / scale uses the stored fp16 scale, rint rounds half to even, a zero
scale gives zero codes.

The expected values below are worked out by hand from exact arithmetic (each
case says how), not produced by any implementation; the invariants hold for
every input whatever its distribution.
"""
import numpy as np
import pytest

import oracle


def _group(values):
    g = np.zeros(64, dtype=np.float32)
    g[: len(values)] = np.asarray(values, dtype=np.float32)
    return g


def _q(values):
    codes, scales = oracle.quantize_rows_q8(_group(values))
    return codes, int(scales[0])


def _f16(bits):
    return float(np.array([bits], np.uint16).view(np.float16)[0])


def test_scale_one_ties_round_half_even():
    # max|x| = 127 -> 127/127 = 1 exactly -> scale 1.0 (0x3C00); x / 1 = x.
    codes, s = _q([127.0, 0.5, 1.5, 2.5, -2.5, 126.5, -0.5, -1.5, 3.5, 0.49999997])
    assert s == 0x3C00
    assert codes[:10].tolist() == [127, 0, 2, 2, -2, 126, 0, -2, 4, 0]
    assert not codes[10:].any()


def test_scale_two_and_half():
    # max 254 -> scale 2.0 (0x4000): 3/2 = 1.5 -> 2, 1/2 -> 0, 5/2 -> 2,
    # 7/2 = 3.5 -> 4, -3/2 -> -2.
    codes, s = _q([254.0, 3.0, 1.0, 5.0, 7.0, -3.0])
    assert s == 0x4000
    assert codes[:6].tolist() == [127, 2, 0, 2, 4, -2]
    # max 63.5 -> 63.5/127 = 0.5 exactly -> scale 0.5 (0x3800): x / 0.5 = 2x.
    codes, s = _q([63.5, 0.25, 0.75, -0.25, -63.5])
    assert s == 0x3800
    assert codes[:5].tolist() == [127, 0, 2, 0, -127]


def test_negative_maximum_uses_absolute_value():
    # max|x| is taken over magnitudes: -127 dominates 1.0 -> scale 1.0.
    codes, s = _q([1.0, -127.0, 2.5])
    assert s == 0x3C00
    assert codes[:3].tolist() == [1, -127, 2]


def test_zero_group_and_underflowing_scale():
    codes, s = _q([])
    assert s == 0 and not codes.any()
    # 1e-7 / 127 ~ 7.9e-10 is below half the smallest fp16 subnormal (2^-25):
    # the scale rounds to +0 and every code is 0.
    codes, s = _q([1e-7, -5e-8])
    assert s == 0 and not codes.any()


def test_scale_is_rounded_to_fp16_before_dividing():
    # a = 127 * (1 + 2^-11) = 260223/2048 (exact in fp32); a/127 = 1 + 2^-11,
    # the midpoint between fp16 1.0 and 1.0009765625 -> ties to even -> 1.0.
    # x = 65.51: x / 1.0 = 65.51 -> 66.  (Dividing by the unrounded 1 + 2^-11
    # would give 65.478 -> 65.)
    a = 260223.0 / 2048.0
    codes, s = _q([a, 65.51, -65.51])
    assert s == 0x3C00
    assert codes[:3].tolist() == [127, 66, -66]
    # a = 127 * (1 + 3 * 2^-11) -> a/127 is the midpoint between 1 + 2^-10
    # (odd mantissa) and 1 + 2^-9 (even) -> 1 + 2^-9 = 0x3C02.  x = 2.5 * s is
    # exact, x / s = 2.5 -> 2.  a / s = 127 * 2051/2052 = 126.94 -> 127.
    a = 127.0 * (1.0 + 3.0 * 2.0 ** -11)
    s_val = 1.0 + 2.0 ** -9
    codes, s = _q([a, 2.5 * s_val, 3.5 * s_val])
    assert s == 0x3C02
    assert codes[:3].tolist() == [127, 2, 4]


def test_subnormal_scale_and_clamp():
    # a = 127 * 2^-20 -> scale 2^-20, an fp16 subnormal (16 * 2^-24, bits 0x0010).
    codes, s = _q([127.0 * 2.0 ** -20, 3.5 * 2.0 ** -20, -2.5 * 2.0 ** -20])
    assert s == 0x0010
    assert codes[:3].tolist() == [127, 4, -2]
    # a = 127 * 1.4 * 2^-24: a/127 = 1.4 * 2^-24 rounds to the smallest
    # subnormal 2^-24 (bits 1); a / 2^-24 = 177.8 -> clamped to 127 / -127.
    a = np.float32(127.0 * 1.4 * 2.0 ** -24)
    codes, s = _q([a, -a, 2.0 ** -24])
    assert s == 1
    assert codes[:3].tolist() == [127, -127, 1]


def test_overflowing_scale_gives_zero_codes():
    # a / 127 > 65520 -> fp16 overflows to +inf (0x7C00); x / inf = 0.
    codes, s = _q([1.0e7, -3.0, 5.0e6])
    assert s == 0x7C00
    assert not codes.any()


def _division_tie_cases():
    """Groups whose exact quotients x / s are ties k + 0.5 while x * fl(1/s)
    is not: rounding half-even of the true quotient is the only right answer
    and multiplying by the reciprocal would move some codes."""
    cases = []
    for s_bits in range(0x3C01, 0x4400, 37):   # fp16 scales in (1, 4)
        s = _f16(s_bits)
        a = np.float32(127.0 * s)               # 18 significant bits: exact
        assert float(a) == 127.0 * s
        recip = np.float32(1.0) / np.float32(s)
        for k in range(0, 127):
            x = np.float32((k + 0.5) * s)       # exact
            if np.float32(x * recip) != np.float32(k + 0.5):
                expect = k if k % 2 == 0 else k + 1
                cases.append((a, s_bits, x, expect))
    return cases


def test_division_is_by_the_scale_not_times_its_reciprocal():
    cases = _division_tie_cases()
    assert len(cases) > 50
    for a, s_bits, x, expect in cases:
        codes, s = _q([a, x, -x])
        assert s == s_bits
        assert codes[1] == expect and codes[2] == -expect, (a, s_bits, x)


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_invariants_on_random_rows(hd):
    rng = np.random.default_rng(hd)
    n = 4000
    x = rng.standard_normal((n, hd)).astype(np.float32)
    # magnitudes from 1e-6 to 1e4 per row, plus outlier channels x20
    x *= (10.0 ** rng.uniform(-6, 4, size=(n, 1))).astype(np.float32)
    x[:, rng.integers(0, hd, 4)] *= 20.0
    codes, scales = oracle.quantize_rows_q8(x)
    assert codes.dtype == np.int8 and scales.shape == (n, hd // 64)
    c = codes.astype(np.int64)
    assert np.abs(c).max() <= 127
    sf = scales.view(np.float16).astype(np.float64)              # library decode
    xg = x.astype(np.float64).reshape(n, hd // 64, 64)
    cg = c.reshape(n, hd // 64, 64)
    a = np.abs(xg).max(axis=2)
    normal = sf >= 2.0 ** -14
    # fp16 rounding of max|x|/127: relative error at most 2^-11 (normal range)
    rel = np.abs(sf - a / 127.0) / (a / 127.0)
    assert (rel[normal] <= 2.0 ** -11 * (1 + 2.0 ** -20)).all()
    # reconstruction error |x - c s| <= s / 2 (normal scales; the quotient is
    # rounded once in fp32, hence the 2^-22 slack)
    err = np.abs(xg - cg * sf[..., None])
    bound = sf[..., None] / 2 * (1 + 2.0 ** -22)
    assert (err[normal] <= bound[normal]).all()
    # the group maximum maps to +-127: a/s lies in 127 * [1 - 2^-11, 1 + 2^-11]
    assert (np.abs(cg).max(axis=2)[normal] == 127).all()
    # codes carry the sign of x
    assert ((cg * np.sign(xg)) >= 0).all()
