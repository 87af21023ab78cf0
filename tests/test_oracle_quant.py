"""Pins of the oracle's NVFP4 quantization (scales, codes, 2D, SR, layout)."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import formats, quant, rht


def _data(shape, seed=0, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    if outliers:
        x.reshape(-1)[rng.choice(x.size, max(1, x.size // 500), replace=False)] *= 40
    # bf16-representable values, as the path's inputs are
    return formats.float64_to_bf16_rne(x).astype(np.float32)


def test_tensor_scale_maps_tensor_max_to_448():
    x = _data((64, 128), 1)
    q = quant.quantize_1d(x)
    E = q["scales"]
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert E[r, c // 16] == 0x7E  # 448
    assert np.all(E <= 0x7E)
    # ts = 1/s_enc, s_enc = 2688/amax, both float32
    amax = np.float32(np.max(np.abs(x)))
    assert q["amax"] == amax
    assert q["ts"] == np.float32(np.float32(1) / np.float32(np.float32(2688) / amax))


def test_block_max_encodes_to_six():
    """Each block whose E4M3 scale is normal stores its largest element as
    +-6: the largest 1 of 16 values (6.25%) sits at the top of the grid."""
    x = _data((256, 256), 2)
    q = quant.quantize_1d(x)
    codes = formats.unpack_nibbles(q["codes"])
    E = q["scales"]
    xb = np.abs(x).reshape(256, 16, 16)
    cb = codes.reshape(256, 16, 16)
    arg = np.argmax(xb, axis=2)
    top = np.take_along_axis(cb, arg[..., None], axis=2)[..., 0]
    normal = (E >> 3) > 0
    assert normal.sum() > 4000
    assert np.all((top[normal] & 7) == 7)


def test_dequant_error_bound():
    """|deq - x| <= (half the E2M1 spacing at v, or the saturation excess)
    times the decode scale, up to float32 rounding of the scale chain."""
    x = _data((128, 512), 3)
    q = quant.quantize_1d(x)
    deq = quant.dequantize(q)
    E = np.repeat(formats.e4m3_decode(q["scales"]), 16, axis=1)
    unit = E * np.float64(q["ts"])
    a = np.abs(x.astype(np.float64)) / np.where(unit == 0, 1, unit)
    half = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))
    bound = np.where(a > 6, a - 6, half) * unit
    err = np.abs(deq - x)
    assert np.all(err <= bound * (1 + 1e-5) + 1e-30)
    rel = np.linalg.norm(deq - x) / np.linalg.norm(x)
    assert rel < 0.12


def test_brute_force_codes_tiny():
    """Exact rational recomputation of the scale chain's decisions on a tiny
    tensor: for every element the chosen code is the nearest grid point to
    v = fl32(x * enc) (ties to even), and E is the nearest E4M3 value to
    fl32(fl32(amax_b / 6) * s_enc)."""
    x = _data((16, 64), 4)
    q = quant.quantize_1d(x)
    codes = formats.unpack_nibbles(q["codes"])
    amax = np.float32(np.max(np.abs(x)))
    s_enc = np.float32(np.float32(2688) / amax)
    grid = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    e4 = [Fraction(float(v)) for v in formats.e4m3_decode(np.arange(127, dtype=np.uint8))]
    for r in range(16):
        for b in range(4):
            blk = x[r, 16 * b:16 * b + 16]
            sd = np.float32(np.float32(np.max(np.abs(blk))) / np.float32(6))
            t = Fraction(float(np.float32(sd * s_enc)))
            best = min(range(127), key=lambda c: (abs(e4[c] - t), c % 2))
            assert q["scales"][r, b] == best
            enc = np.float32(0) if best == 0 else np.float32(s_enc / np.float32(float(e4[best])))
            for i in range(16):
                v = Fraction(float(np.float32(blk[i] * enc)))
                m = min(range(8), key=lambda c: (abs(grid[c] - abs(v)), c % 2))
                exp = m | (8 if np.signbit(np.float32(blk[i] * enc)) else 0)
                assert codes[r, 16 * b + i] == exp


def test_quant2d_transpose_identity():
    w = _data((96, 160), 5)
    a = quant.quantize_2d(w)
    b = quant.quantize_2d(np.ascontiguousarray(w.T))
    np.testing.assert_array_equal(a["codes_t"], b["codes"])
    np.testing.assert_array_equal(a["scales_t"], b["scales"])
    np.testing.assert_array_equal(a["codes"], b["codes_t"])
    np.testing.assert_array_equal(a["scales_2d"], b["scales_2d"].T)
    # one scale per 16x16 block: the block's largest element encodes to +-6
    E = a["scales_2d"]
    codes = formats.unpack_nibbles(a["codes"]).reshape(6, 16, 10, 16)
    blk = np.abs(w).reshape(6, 16, 10, 16)
    for i in range(6):
        for j in range(10):
            r, c = np.unravel_index(np.argmax(blk[i, :, j, :]), (16, 16))
            if E[i, j] >> 3:
                assert codes[i, r, j, c] & 7 == 7


def test_transpose_quant_equals_quant_of_transposed_rht():
    x = _data((64, 48), 6)
    seed = 1234
    got = quant.quantize_transpose(x, "rne", rht_seed=seed)
    s = rht.rht_signs(seed)
    xt = np.ascontiguousarray(x.T)
    manual = np.stack([rht.rht16_chunks(row.reshape(-1, 16), s).reshape(-1) for row in xt])
    ref = quant.quantize_1d(manual, "rne")
    np.testing.assert_array_equal(got["codes"], ref["codes"])
    np.testing.assert_array_equal(got["scales"], ref["scales"])
    assert got["ts"] == ref["ts"]
    # selecting output rows with the whole tensor's amax gives the same rows
    sub = quant.quantize_transpose(x, "sr", seed=9, stream_id=1, rht_seed=seed, amax=got["amax"],
                                   col_ids=[3, 17, 40])
    full = quant.quantize_transpose(x, "sr", seed=9, stream_id=1, rht_seed=seed)
    np.testing.assert_array_equal(sub["codes"], full["codes"][[3, 17, 40]])


def test_sr_exact_probability_exhaustive():
    """Over all 2^16 uniforms, a value rounds up exactly ceil(frac*2^16) times."""
    u = np.arange(65536, dtype=np.uint32)
    for v in (0.1, 0.3333, 0.75, 1.2, 1.5, 1.9, 2.01, 2.5, 3.999, 4.7, 5.5, 5.99):
        v32 = np.float32(v)
        codes = formats.e2m1_encode_sr(np.full(65536, v32), u)
        vals = formats.e2m1_decode(codes)
        lo_code, lo, hi = formats.e2m1_sr_bracket(np.float64(v32))
        frac = (Fraction(float(v32)) - Fraction(float(lo))) / (Fraction(float(hi)) - Fraction(float(lo)))
        n_up = int(np.sum(vals == hi))
        assert n_up + int(np.sum(vals == lo)) == 65536
        expect = -((-frac * 65536).numerator // (frac * 65536).denominator)  # ceil
        assert n_up == expect, (v, n_up, expect)
    # grid points never move; saturation
    for g in (0.0, 0.5, 1.0, 3.0, 6.0, 6.5, 100.0):
        codes = formats.e2m1_encode_sr(np.full(65536, np.float32(g)), u)
        assert len(set(formats.e2m1_decode(codes).tolist())) == 1


def test_sr_unbiased_over_seeds():
    """E[dequantized] = x over 10^4 seeds (5 sigma), the unbiasedness the
    method wants from stochastic rounding of gradients."""
    x = _data((1, 64), 7)
    amax = np.float32(np.max(np.abs(x)))
    n = 10000
    acc = np.zeros(64)
    acc2 = np.zeros(64)
    for s in range(n):
        d = quant.dequantize(quant.quantize_1d(x, "sr", seed=s, stream_id=0, amax=amax))[0]
        acc += d
        acc2 += d * d
    mean = acc / n
    sd = np.sqrt(np.maximum(acc2 / n - mean ** 2, 0)) / np.sqrt(n)
    # target: v * E * ts (the exact value the codes straddle)
    q = quant.quantize_1d(x, "rne", amax=amax)
    unit = np.repeat(formats.e4m3_decode(q["scales"][0]), 16) * np.float64(q["ts"])
    s_enc, _ = quant.tensor_scales(amax)
    _, enc = quant.block_scale_codes(np.max(np.abs(x.reshape(4, 16)), axis=1), s_enc)
    v = (x.reshape(4, 16) * enc[:, None]).astype(np.float32).reshape(-1).astype(np.float64)
    target = np.clip(v, -6, 6) * unit
    assert np.all(np.abs(mean - target) <= 5 * sd + 1e-12)
    assert np.abs(mean - x[0]).max() < 0.05 * np.abs(x).max()


def test_sr_deterministic_and_seed_dependent():
    x = _data((32, 64), 8)
    a = quant.quantize_1d(x, "sr", seed=5, stream_id=0)
    b = quant.quantize_1d(x, "sr", seed=5, stream_id=0)
    c = quant.quantize_1d(x, "sr", seed=6, stream_id=0)
    d = quant.quantize_1d(x, "sr", seed=5, stream_id=1)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    assert not np.array_equal(a["codes"], c["codes"])
    assert not np.array_equal(a["codes"], d["codes"])
    np.testing.assert_array_equal(a["scales"], c["scales"])  # SR touches codes only


def test_zero_tensor_and_nonfinite():
    z = np.zeros((16, 32), np.float32)
    q = quant.quantize_1d(z)
    assert q["ts"] == 1.0 and q["amax"] == 0.0
    assert np.all(q["scales"] == 0) and np.all(q["codes"] == 0)
    zn = -z
    qn = quant.quantize_1d(zn)
    assert np.all(formats.unpack_nibbles(qn["codes"]) == 8)
    bad = z.copy()
    bad[3, 4] = np.inf
    with pytest.raises(FloatingPointError):
        quant.quantize_1d(bad)
    bad[3, 4] = np.nan
    with pytest.raises(FloatingPointError):
        quant.quantize_1d(bad)


def test_storage_is_4p5_bits_per_element():
    x = _data((128, 1024), 9)
    q = quant.quantize_1d(x)
    assert q["codes"].nbytes + q["scales"].nbytes == int(0.5625 * x.size)


def test_swizzle_is_a_padded_bijection():
    rng = np.random.default_rng(10)
    for R, C in ((256, 8), (130, 5), (128, 4), (1, 1)):
        E = rng.integers(1, 255, size=(R, C)).astype(np.uint8)
        buf = quant.swizzle_scales(E)
        assert buf.size == quant.swizzled_scale_bytes(R, C)
        np.testing.assert_array_equal(quant.unswizzle_scales(buf, R, C), E)
        assert np.count_nonzero(buf) == R * C
    # the layout rule at one point: 256 x 8 scales, row 33, column 5 ->
    # tile (row tile 0, column tile 1) = bytes 512..1023, + 1*16 + 1*4 + 1
    E = np.zeros((256, 8), np.uint8)
    E[33, 5] = 7
    assert np.flatnonzero(quant.swizzle_scales(E)).tolist() == [533]


def _ulp_close(a, b, ulps=4):
    a, b = np.float32(a), np.float32(b)
    return abs(float(a) - float(b)) <= ulps * float(np.spacing(max(abs(a), abs(b))))


def test_amax_rht_closed_forms_pin_the_axis():
    """Q = 1/4 H diag(s) maps a 16-chunk equal to c*s to (4c, 0, ..., 0)
    (the first row of H is all ones, every other row sums to zero) and a
    one-hot chunk v*e_k to values of magnitude |v|/4.  Both shapes are laid
    along axis 0 (tokens) of a tensor whose two sizes differ, so the transform
    along the wrong axis gives a different amax."""
    seed = 31
    s = rht.rht_signs(seed).astype(np.float32)
    M, C = 48, 80
    x = np.zeros((M, C), np.float32)
    x[16:32, 5] = np.float32(3.0) * s          # chunk 1 of column 5: c = 3 -> 4c = 12
    x[32 + 9, 70] = np.float32(-20.0)          # one-hot in chunk 2 of column 70: 20/4 = 5
    assert quant.amax_rht(x, seed, axis=0) == np.float32(12.0)
    assert quant.amax_rht(x, seed, axis=1) != np.float32(12.0)
    # the one-hot alone: |v|/4 along either axis
    y = np.zeros((M, C), np.float32)
    y[32 + 9, 70] = np.float32(-20.0)
    assert quant.amax_rht(y, seed, axis=0) == np.float32(5.0)
    assert quant.amax_rht(y, seed, axis=1) == np.float32(5.0)
    # a sign vector other than the layer's does not reach 4c
    assert quant.amax_rht(x, seed + 1, axis=0) < np.float32(12.0)


@pytest.mark.parametrize("axis", [0, 1])
def test_amax_rht_slicing_and_independent_product(axis):
    """The chunked loop (slices of whole 16-chunks along the other axis) gives
    the same amax for every slice size, and it matches the transform written
    as an explicit float64 matrix product on every 16-chunk, to a few float32
    ulps (the oracle sums in float32)."""
    x = _data((64, 96), 11)
    seed = 5
    ref = quant.amax_rht(x, seed, axis)
    for chunk in (16, 100, 1000, 1 << 21):
        assert quant.amax_rht(x, seed, axis, chunk_elems=chunk) == ref
    Q = rht.rht_matrix_f64(rht.rht_signs(seed))
    xm = np.moveaxis(x.astype(np.float64), axis, -1)
    v = xm.reshape(xm.shape[:-1] + (xm.shape[-1] // 16, 16)) @ Q.T
    assert _ulp_close(ref, np.max(np.abs(v)))
    # the maximum sits somewhere else than the untransformed tensor's
    assert ref != quant.tensor_amax(x)
    # a closed-form chunk (c*s -> 4c) in the last line along the other axis,
    # which the last slice of every slice size must reach
    s = rht.rht_signs(seed).astype(np.float32)
    z = x.copy()
    if axis == 0:
        z[16:32, -1] = np.float32(1000.0) * s
    else:
        z[-1, 32:48] = np.float32(1000.0) * s
    for chunk in (16, 100, 1000, 1 << 21):
        assert quant.amax_rht(z, seed, axis, chunk_elems=chunk) == np.float32(4000.0)
