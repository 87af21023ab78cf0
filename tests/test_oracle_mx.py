"""Pins of the MXFP4 oracle (oracle/mx.py) against what the format fixes,
independently of the oracle's own code: a library decode of UE8M0, the
power-of-two placement of each block's largest value, brute-force nearest
search, the dequantization error bound, and a closed-form GEMM."""

import numpy as np
import pytest
import torch

from oracle import formats, mx


def test_e8m0_decode_matches_library_cast():
    codes = np.arange(255, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    np.testing.assert_array_equal(mx.e8m0_decode(codes), lib)
    assert np.isnan(mx.e8m0_decode(np.array([255], np.uint8))[0])


def test_scale_places_block_max_in_4_to_8():
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.uniform(1e-30, 1e30, 20000), np.exp2(rng.uniform(-120, 120, 20000))]).astype(np.float32)
    E = mx.block_scale_codes(a)
    X = mx.e8m0_decode(E)
    r = a.astype(np.float64) / X
    assert np.all((r >= 4.0) & (r < 8.0))
    # exact powers of two land on 4
    p = np.exp2(np.arange(-100, 100)).astype(np.float32)
    np.testing.assert_array_equal(p.astype(np.float64) / mx.e8m0_decode(mx.block_scale_codes(p)), 4.0)


def test_scale_clamps_and_zero():
    assert mx.block_scale_codes(np.float32(0.0)) == 0
    tiny = np.float32(2.0 ** -130)  # floor(log2) - 2 + 127 < 0
    assert mx.block_scale_codes(tiny) == 0
    big = np.float32(3.0e38)  # floor(log2) = 127 -> 252
    assert mx.block_scale_codes(big) == 252


def test_multiplier_is_the_exact_power_of_two():
    E = np.arange(255, dtype=np.uint8)
    m = mx.scale_multiplier(E).astype(np.float64)
    np.testing.assert_array_equal(m, np.exp2(127.0 - E.astype(np.float64)))


def test_codes_are_nearest_grid_values_brute_force():
    """Every code is the nearest E2M1 value to the scaled element (ties to
    the even mantissa), saturating at 6 -- checked by searching all eight
    magnitudes, with the scaled value recomputed in float64 from the scale
    definition."""
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((16, 256)) * np.exp2(rng.integers(-20, 20, (16, 1)))).astype(np.float32)
    x[3, :32] = 0.0
    x[4, 40] = 1e-30
    q = mx.quantize_mx(x)
    codes = formats.unpack_nibbles(q["codes"])
    amax_b = np.abs(x.reshape(16, 8, 32)).max(-1).astype(np.float64)
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    for r in range(16):
        for b in range(8):
            e = 0 if amax_b[r, b] == 0 else max(0, int(np.floor(np.log2(amax_b[r, b]))) - 2 + 127)
            assert q["scales"][r, b] == e
            for j in range(32):
                xv = float(x[r, 32 * b + j])
                v = np.float64(np.float32(xv * 2.0 ** (127 - e)))
                a = min(abs(v), 6.0)
                d = np.abs(mags - a)
                best = np.flatnonzero(d == d.min())
                mag = best[0] if len(best) == 1 else best[np.argmax((best % 2) == 0)]  # even mantissa
                want = (8 if np.signbit(v) else 0) | int(mag)
                assert codes[r, 32 * b + j] == want, (r, b, j, xv)


def test_dequant_error_bound_and_saturation():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    q = mx.quantize_mx(x)
    deq = mx.dequantize_mx(q)
    X = np.repeat(mx.e8m0_decode(q["scales"]), 32, axis=-1)
    a = np.abs(x.astype(np.float64)) / X
    # within range: half a grid step; above 6: saturated to 6 X
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    inside = a <= 6
    assert np.all(np.abs(deq - x)[inside] <= 0.5 * step[inside] * X[inside])
    np.testing.assert_array_equal(np.abs(deq)[~inside], 6.0 * X[~inside])
    assert np.any(~inside)  # MXFP4's saturation does occur on Gaussian blocks


def test_gemm_mx_closed_form():
    """All codes 1.0 (0x2) and scales E: D = K * 2^(Ea-127) * 2^(Eb-127)."""
    M, N, K = 4, 3, 64
    a = dict(codes=formats.pack_nibbles(np.full((M, K), 2, np.uint8)), scales=np.full((M, K // 32), 125, np.uint8))
    b = dict(codes=formats.pack_nibbles(np.full((N, K), 2, np.uint8)), scales=np.full((N, K // 32), 130, np.uint8))
    np.testing.assert_array_equal(mx.gemm_mx_ref(a, b), np.full((M, N), K * 2.0 ** -2 * 2.0 ** 3))
    # one-hot orientation
    ac = np.zeros((M, K), np.uint8)
    ac[2, 37] = 0x7  # +6
    bc = np.zeros((N, K), np.uint8)
    bc[1, 37] = 0xB  # -1.5
    a = dict(codes=formats.pack_nibbles(ac), scales=np.full((M, 2), 127, np.uint8))
    b = dict(codes=formats.pack_nibbles(bc), scales=np.full((N, 2), 128, np.uint8))
    d = mx.gemm_mx_ref(a, b)
    assert np.argwhere(d != 0).tolist() == [[2, 1]] and d[2, 1] == 6 * -1.5 * 2.0
