"""Pins for the oracle's own IEEE binary16 conversion.

The oracle implements fp16 rounding from the IEEE-754 definition (nearest,
ties to even, subnormals kept, overflow to infinity).  These tests check it
against two independent library conversions (numpy's float16 cast and
torch's Tensor.half), which both round to nearest-even, on every fp16 value,
every midpoint between neighbouring fp16 values (the ties), the values one
float32 ulp either side of each midpoint, and a wide random sample.
"""
import numpy as np
import torch

import oracle


def _lib_fp16(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return x.astype(np.float16).view(np.uint16)


def _torch_fp16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).half().view(torch.int16).numpy().view(np.uint16)


def _same_bits_or_both_nan(ours, ref):
    ref_f = ref.view(np.float16)
    nan = np.isnan(ref_f)
    assert np.array_equal(np.isnan(ours.view(np.float16)), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.fp16_value(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_encode_grid_points_midpoints_and_neighbours():
    pos = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)  # finite >= 0
    vals = pos.view(np.float16).astype(np.float64)
    mids = (vals[:-1] + vals[1:]) / 2.0          # ties (exact in float32)
    top_mid = np.array([65520.0])                # tie between 65504 and 2^16
    m32 = np.concatenate([mids, top_mid]).astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), np.concatenate([mids, top_mid]))
    up = np.nextafter(m32, np.float32(np.inf))
    down = np.nextafter(m32, np.float32(0))
    xs = np.concatenate([vals.astype(np.float32), m32, up, down])
    xs = np.concatenate([xs, -xs])
    ours = oracle.fp16_bits(xs)
    _same_bits_or_both_nan(ours, _lib_fp16(xs))
    _same_bits_or_both_nan(ours, _torch_fp16(xs))


def test_encode_wide_random_sample_and_specials():
    rng = np.random.default_rng(7)
    # random float32 bit patterns whose exponent spans fp16 underflow .. overflow
    exp = rng.integers(127 - 30, 127 + 18, size=1_000_000).astype(np.uint32)
    man = rng.integers(0, 1 << 23, size=exp.size).astype(np.uint32)
    sign = rng.integers(0, 2, size=exp.size).astype(np.uint32)
    xs = ((sign << 31) | (exp << 23) | man).view(np.float32)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 65504.0, 65519.996,
                         65520.0, 65536.0, 1e30, 2.0 ** -24, 2.0 ** -25,
                         np.float32(2.0 ** -25) * np.float32(1.0000001), 2.0 ** -26,
                         6.1e-5, 2.0 ** -14, 0.1, 1 / 3], dtype=np.float32)
    xs = np.concatenate([xs, specials])
    ours = oracle.fp16_bits(xs)
    _same_bits_or_both_nan(ours, _lib_fp16(xs))
    _same_bits_or_both_nan(ours, _torch_fp16(xs))
