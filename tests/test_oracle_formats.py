"""Pins of the oracle's E2M1 / E4M3 codecs against what the formats fix."""

import numpy as np
import pytest
import torch

from oracle import formats
from tests.conftest import read_golden


def test_e2m1_value_set():
    # OCP E2M1: magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}; codes 8..15 mirror 0..7
    np.testing.assert_array_equal(formats.e2m1_magnitudes(), [0, 0.5, 1, 1.5, 2, 3, 4, 6])
    neg = formats.e2m1_decode(np.arange(8, 16, dtype=np.uint8))
    np.testing.assert_array_equal(neg, -formats.e2m1_magnitudes())
    assert np.signbit(neg[0])


def test_e2m1_rne_midpoints_golden():
    for a, val, code in read_golden("e2m1_rne_ties.txt"):
        a, val, code = float(a), float(val), int(code)
        got = formats.e2m1_encode_rne(np.float32(a))
        assert int(got) == code, (a, got)
        assert formats.e2m1_decode(got) == val
        gotn = formats.e2m1_encode_rne(np.float32(-a))
        assert int(gotn) == code | 8


def _bf16_grid_positive(limit):
    bits = np.arange(0, 0x7F80, dtype=np.uint16)  # all finite non-negative bf16
    vals = formats.bf16_bits_to_float32(bits)
    return vals[vals <= limit]


def test_e2m1_rne_brute_force_all_bf16():
    """Every finite bf16 magnitude up to 16: nearest grid value by exhaustive
    search over the 8 codes, ties to the code with mantissa bit 0."""
    vals = _bf16_grid_positive(16.0)
    got = formats.e2m1_encode_rne(vals)
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for v, g in zip(vals.tolist(), got.tolist()):
        best = None
        for c, q in enumerate(grid):
            d = abs(q - v)
            if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
                best = (d, c)
        assert g == best[1], (v, g, best)
    # negative inputs mirror, including -0 for values that round to zero
    gotn = formats.e2m1_encode_rne(-vals)
    np.testing.assert_array_equal(gotn, got | 8)


def test_e2m1_saturates_and_roundtrips():
    big = np.array([6.0, 6.5, 7.9, 100.0, 3e38, np.inf], dtype=np.float32)
    np.testing.assert_array_equal(formats.e2m1_encode_rne(big), 7)
    np.testing.assert_array_equal(formats.e2m1_encode_rne(-big), 15)
    codes = np.arange(16, dtype=np.uint8)
    back = formats.e2m1_encode_rne(formats.e2m1_decode(codes).astype(np.float32))
    np.testing.assert_array_equal(back, codes)


def test_pack_nibble_order():
    codes = np.array([[1, 2, 15, 0]], dtype=np.uint8)
    np.testing.assert_array_equal(formats.pack_nibbles(codes), [[0x21, 0x0F]])
    rng = np.random.default_rng(5)
    c = rng.integers(0, 16, size=(7, 64)).astype(np.uint8)
    np.testing.assert_array_equal(formats.unpack_nibbles(formats.pack_nibbles(c)), c)


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = formats.e4m3_decode(codes.numpy())
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert formats.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert formats.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9


def test_e4m3_encode_matches_torch_in_range():
    """RNE in [0, 448] against torch's float8_e4m3fn cast (a library routine)."""
    table = formats.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (table[:-1] + table[1:]) / 2
    pts = np.concatenate([table, mids]).astype(np.float32)
    near = np.concatenate([np.nextafter(pts, np.float32(0)), np.nextafter(pts, np.float32(1e9))])
    rng = np.random.default_rng(11)
    rnd = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 200000)).astype(np.float32)
    x = np.concatenate([pts, near, rnd, np.float32([0.0])])
    x = x[(x >= 0) & (x <= 448.0)]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(formats.e4m3_encode_rne_sat(x), ref)


def test_e4m3_saturation():
    x = np.array([448.0, 449.0, 464.0, 480.0, 1e6, 3e38], dtype=np.float32)
    np.testing.assert_array_equal(formats.e4m3_encode_rne_sat(x), 0x7E)


def test_bf16_rounding_helper():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -3.14159, 1e-40, 0.0])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(formats.float64_to_bf16_rne(x), ref)
