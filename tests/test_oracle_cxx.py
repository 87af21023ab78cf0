"""Pins of the plain C++ oracle (oracle/cxx): the same facts the formats, the
Philox paper and the mathematics fix, checked on the C++ functions, and the
C++ oracle equal bit for bit to the numpy oracle on seeded inputs (two
independent restatements of the same definitions)."""

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import cxx, formats, gemm, linear, quant, rht
from nvfp4_bit_numerics_gb300 import workloads
from tests.conftest import read_golden


def _data(shape, seed=0, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    if outliers:
        x.reshape(-1)[rng.choice(x.size, max(1, x.size // 500), replace=False)] *= 40
    return formats.float64_to_bf16_rne(x).astype(np.float32)


# ---------------------------------------------------------------------------
# formats
# ---------------------------------------------------------------------------
def test_e2m1_value_set_and_sign():
    vals = cxx.e2m1_decode(np.arange(16, dtype=np.uint8))
    np.testing.assert_array_equal(vals[:8], [0, 0.5, 1, 1.5, 2, 3, 4, 6])
    np.testing.assert_array_equal(vals[8:], -vals[:8])
    assert np.signbit(vals[8])


def test_e2m1_rne_midpoints_golden():
    for a, val, code in read_golden("e2m1_rne_ties.txt"):
        a, code = float(a), int(code)
        assert int(cxx.e2m1_encode_rne(np.float32(a))) == code, a
        assert int(cxx.e2m1_encode_rne(np.float32(-a))) == code | 8, a


def test_e2m1_rne_brute_force_all_bf16():
    """Every finite non-negative BF16 value up to 16: the nearest of the eight
    magnitudes, ties to the code whose mantissa bit is 0, saturating at 6."""
    bits = np.arange(0, 0x7F80, dtype=np.uint16)
    vals = formats.bf16_bits_to_float32(bits)
    vals = vals[vals <= 16.0]
    got = cxx.e2m1_encode_rne(vals)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    d = np.abs(vals[:, None].astype(np.float64) - grid[None, :])
    best = np.argmin(d, axis=1)
    ties = (d == d.min(axis=1, keepdims=True)).sum(axis=1) > 1
    # at a tie the even code of the two wins
    best = np.where(ties & (best % 2 == 1), best + 1, best)
    np.testing.assert_array_equal(got, best)
    np.testing.assert_array_equal(cxx.e2m1_encode_rne(-vals), got | 8)


def test_e4m3_decode_and_encode_match_library_cast():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = cxx.e4m3_decode(codes.numpy())
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    rng = np.random.default_rng(3)
    table = ref[:127]
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    x = np.concatenate([table.astype(np.float32), mids, np.nextafter(mids, np.float32(0)),
                        np.nextafter(mids, np.float32(1e9)),
                        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 50000)).astype(np.float32)])
    x = x[(x >= 0) & (x <= 448.0)]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(cxx.e4m3_encode_rne_sat(x), lib)
    np.testing.assert_array_equal(cxx.e4m3_encode_rne_sat(np.float32([448, 449, 1e6, 3e38])), 0x7E)


# ---------------------------------------------------------------------------
# Philox, stochastic rounding, Hadamard transform
# ---------------------------------------------------------------------------
def test_philox_known_answers():
    for row in read_golden("philox4x32_10_kat.txt"):
        v = [int(t, 16) for t in row]
        assert [int(w) for w in cxx.philox4x32_10(*v[:6])] == v[6:10]


def test_sr_uniforms_are_the_halves_of_one_call_per_eight_elements():
    seed = 0xDEADBEEF12345678
    u = cxx.sr_uniform16(seed, 1, np.arange(64, dtype=np.uint64))
    k0, k1 = seed & 0xFFFFFFFF, seed >> 32
    for g in range(8):
        w = [int(x) for x in cxx.philox4x32_10(g, 0, 1, 0, k0, k1)]
        exp = [h for word in w for h in (word & 0xFFFF, word >> 16)]
        assert [int(x) for x in u[8 * g:8 * g + 8]] == exp


def test_sr_exact_probability_exhaustive():
    """Over all 2^16 uniforms the value rounds up exactly ceil(frac * 2^16)
    times, frac its fractional distance above the lower grid neighbour."""
    u = np.arange(1 << 16, dtype=np.uint32)
    for v, lo, hi in [(0.3, 0.0, 0.5), (1.2, 1.0, 1.5), (2.7, 2.0, 3.0), (5.1, 4.0, 6.0), (0.5 + 2 ** -20, 0.5, 1.0)]:
        v32 = np.float32(v)
        codes = cxx.e2m1_encode_sr(np.full(u.shape, v32), u)
        vals = cxx.e2m1_decode(codes)
        assert set(np.unique(vals)) <= {lo, hi}
        frac = Fraction(float(v32) - lo) / Fraction(hi - lo)
        expect = -(-frac * (1 << 16) // 1)  # ceil
        assert int((vals == hi).sum()) == expect, v


def test_rht_closed_forms_and_orthogonality():
    seed = 9
    s = cxx.rht_signs(seed).astype(np.float32)
    # c * s -> (4c, 0, ..., 0)
    y = cxx.rht16(np.float32(3.0) * s, s)
    np.testing.assert_array_equal(y, np.float32([12.0] + [0.0] * 15))
    assert not np.signbit(y).any()  # exact zeros are +0
    # one-hot columns: Q = 1/4 H diag(s) has orthonormal columns
    Q = np.stack([cxx.rht16(np.eye(16, dtype=np.float32)[k], s) for k in range(16)], axis=1).astype(np.float64)
    np.testing.assert_array_equal(Q.T @ Q, np.eye(16))
    H = np.array([[(-1) ** bin(i & j).count("1") for j in range(16)] for i in range(16)], np.float64)
    np.testing.assert_array_equal(Q, 0.25 * H * s[None, :])


def test_amax_rht_closed_form_along_tokens():
    seed = 31
    s = cxx.rht_signs(seed).astype(np.float32)
    x = np.zeros((48, 80), np.float32)
    x[16:32, 5] = np.float32(3.0) * s
    assert cxx.amax_rht(x, seed, 0) == np.float32(12.0)
    assert cxx.amax_rht(x, seed, 1) != np.float32(12.0)


# ---------------------------------------------------------------------------
# quantization and GEMM
# ---------------------------------------------------------------------------
def test_tensor_max_block_gets_448_and_block_max_is_six():
    x = _data((256, 256), 2)
    q = cxx.quantize_1d(x)
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert q["scales"][r, c // 16] == 0x7E
    assert q["ts"] == np.float32(np.float32(1) / np.float32(np.float32(2688) / np.float32(np.abs(x).max())))
    codes = formats.unpack_nibbles(q["codes"]).reshape(256, 16, 16)
    arg = np.argmax(np.abs(x).reshape(256, 16, 16), axis=2)
    top = np.take_along_axis(codes, arg[..., None], axis=2)[..., 0]
    normal = (q["scales"] >> 3) > 0
    assert np.all((top[normal] & 7) == 7)


def test_quant2d_transpose_identity():
    w = _data((96, 160), 4)
    a = cxx.quantize_2d(w)
    b = cxx.quantize_2d(np.ascontiguousarray(w.T))
    np.testing.assert_array_equal(a["codes_t"], b["codes"])
    np.testing.assert_array_equal(a["scales_t"], b["scales"])
    np.testing.assert_array_equal(formats.unpack_nibbles(a["codes"]).T, formats.unpack_nibbles(a["codes_t"]))


def test_gemm_closed_form_and_exact_rational():
    codes = formats.pack_nibbles(np.full((8, 64), 2, np.uint8))   # 1.0
    d = cxx.gemm_ref(codes, np.full((8, 4), 0x38, np.uint8), np.float32(0.5),
                     formats.pack_nibbles(np.full((16, 64), 2, np.uint8)), np.full((16, 4), 0x40, np.uint8),
                     np.float32(3.0))
    np.testing.assert_array_equal(d, np.full((8, 16), 64 * 2.0 * 0.5 * 3.0))
    rng = np.random.default_rng(1)
    ac = rng.integers(0, 16, (3, 48)).astype(np.uint8)
    bc = rng.integers(0, 16, (4, 48)).astype(np.uint8)
    sa = rng.integers(0, 127, (3, 3)).astype(np.uint8)
    sb = rng.integers(0, 127, (4, 3)).astype(np.uint8)
    d = cxx.gemm_ref(formats.pack_nibbles(ac), sa, np.float32(0.37), formats.pack_nibbles(bc), sb, np.float32(1e-3))
    e2 = [Fraction(float(v)) for v in formats.e2m1_decode(np.arange(16, dtype=np.uint8))]
    e4 = [Fraction(float(v)) for v in formats.e4m3_decode(np.arange(127, dtype=np.uint8))]
    for i in range(3):
        for j in range(4):
            exact = sum(e2[ac[i, k]] * e4[sa[i, k // 16]] * e2[bc[j, k]] * e4[sb[j, k // 16]] for k in range(48))
            exact *= Fraction(float(np.float32(0.37))) * Fraction(float(np.float32(1e-3)))
            assert abs(Fraction(d[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)


def test_thread_count_does_not_change_results():
    x = _data((256, 512), 7)
    a = cxx.quantize_transpose(x, "sr", seed=3, stream_id=1, rht_seed=3, threads=1)
    b = cxx.quantize_transpose(x, "sr", seed=3, stream_id=1, rht_seed=3, threads=7)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_array_equal(a["scales"], b["scales"])


# ---------------------------------------------------------------------------
# the two oracles agree bit for bit
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("kw", [dict(), dict(rounding="sr", seed=3, stream_id=1), dict(rht_seed=9),
                                dict(rounding="sr", seed=5, stream_id=0, rht_seed=9)])
def test_cxx_equals_numpy_quantize(kw):
    x = _data((256, 320), 1)
    for fn_c, fn_n in ((cxx.quantize_1d, quant.quantize_1d), (cxx.quantize_transpose, quant.quantize_transpose)):
        a, b = fn_c(x, **kw), fn_n(x, **kw)
        np.testing.assert_array_equal(a["codes"], b["codes"])
        np.testing.assert_array_equal(a["scales"], b["scales"])
        assert a["ts"] == b["ts"] and a["amax"] == b["amax"]
    a, b = cxx.quantize_2d(x), quant.quantize_2d(x)
    for k in ("codes", "scales", "codes_t", "scales_t", "scales_2d"):
        np.testing.assert_array_equal(a[k], b[k])
    for axis in (0, 1):
        assert cxx.amax_rht(x, 11, axis) == quant.amax_rht(x, 11, axis)


def test_cxx_equals_numpy_layer():
    x, w, dy = (workloads.bf16_to_f32_numpy(t) for t in workloads.tiny_layer())
    f1, f2 = linear.linear_fwd(x, w, 77), cxx.linear_fwd(x, w, 77)
    b1, b2 = linear.linear_bwd(dy, f1, 77), cxx.linear_bwd(dy, f2, 77)
    for d1, d2, keys in ((f1, f2, ("xq", "xtq")), (b1, b2, ("dyq", "dytq"))):
        for k in keys:
            np.testing.assert_array_equal(d1[k]["codes"], d2[k]["codes"])
            np.testing.assert_array_equal(d1[k]["scales"], d2[k]["scales"])
    # the float64 sums differ only in summation order (BLAS vs a k-ordered loop)
    for r1, r2 in ((f1["y"], f2["y"]), (b1["dx"], b2["dx"]), (b1["dw"], b2["dw"])):
        np.testing.assert_allclose(r2, r1, rtol=1e-12, atol=1e-12 * np.abs(r1).max())
    np.testing.assert_array_equal(formats.float64_to_bf16_rne(f2["y"]), formats.float64_to_bf16_rne(f1["y"]))
