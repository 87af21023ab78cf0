"""Pins of the oracle's FP64 GEMM on dequantized operands and of the layer."""

from fractions import Fraction

import numpy as np

from oracle import formats, gemm, linear, quant, rht
from nvfp4_bit_numerics_gb300 import workloads


def _ones(rows, K, code=2, scale=0x38):
    codes = np.full((rows, K), code, np.uint8)
    return formats.pack_nibbles(codes), np.full((rows, K // 16), scale, np.uint8)


def test_gemm_closed_form_constant_operands():
    # code 2 = 1.0, E4M3 0x38 = 1.0, 0x40 = 2.0
    a, sa = _ones(8, 64)
    b, sb = _ones(16, 64, scale=0x40)
    d = gemm.gemm_ref(a, sa, np.float32(0.5), b, sb, np.float32(3.0))
    np.testing.assert_array_equal(d, np.full((8, 16), 64 * 2.0 * 0.5 * 3.0))


def test_gemm_one_hot_pins_orientation():
    """A single nonzero at (i, k) in A and (j, k) in B lands at D[i, j] only;
    catches transposed operands and nibble-order mismatches."""
    M, N, K = 5, 7, 64
    for k in (0, 1, 30, 63):
        ac = np.zeros((M, K), np.uint8)
        bc = np.zeros((N, K), np.uint8)
        ac[3, k] = 7      # 6.0
        bc[4, k] = 0xB    # -1.5
        sa = np.full((M, K // 16), 0x38, np.uint8)
        sb = np.full((N, K // 16), 0x38, np.uint8)
        sa[3, k // 16] = 0x48  # 4.0
        d = gemm.gemm_ref(formats.pack_nibbles(ac), sa, 1.0, formats.pack_nibbles(bc), sb, 1.0)
        exp = np.zeros((M, N))
        exp[3, 4] = 6.0 * 4.0 * -1.5
        np.testing.assert_array_equal(d, exp)
        bc[4, k] = 0
        bc[4, (k + 1) % K] = 0xB
        d = gemm.gemm_ref(formats.pack_nibbles(ac), sa, 1.0, formats.pack_nibbles(bc), sb, 1.0)
        assert not d.any()


def test_gemm_matches_exact_rational_brute_force():
    rng = np.random.default_rng(1)
    M, N, K = 3, 4, 48
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sa = rng.integers(0, 127, (M, K // 16)).astype(np.uint8)
    sb = rng.integers(0, 127, (N, K // 16)).astype(np.uint8)
    ta, tb = np.float32(0.37), np.float32(1e-3)
    d = gemm.gemm_ref(formats.pack_nibbles(ac), sa, ta, formats.pack_nibbles(bc), sb, tb)
    e2 = [Fraction(float(v)) for v in formats.e2m1_decode(np.arange(16, dtype=np.uint8))]
    e4 = [Fraction(float(v)) for v in formats.e4m3_decode(np.arange(127, dtype=np.uint8))]
    for i in range(M):
        for j in range(N):
            s = sum(e2[ac[i, k]] * e4[sa[i, k // 16]] * e2[bc[j, k]] * e4[sb[j, k // 16]] for k in range(K))
            exact = s * Fraction(float(ta)) * Fraction(float(tb))
            assert abs(Fraction(d[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)


def test_linear_layer_composition_tiny():
    x, w, dy = workloads.tiny_layer()
    x, w, dy = (workloads.bf16_to_f32_numpy(t) for t in (x, w, dy))
    seed = 77
    f = linear.linear_fwd(x, w, seed)
    b = linear.linear_bwd(dy, f, seed)
    X, W, DY = (t.astype(np.float64) for t in (x, w, dy))

    def rel(a, r):
        return np.linalg.norm(a - r) / np.linalg.norm(r)

    # NVFP4 keeps the layer's products close to the exact ones (stochastic
    # rounding of dY trades a larger error for unbiasedness)
    assert rel(f["y"], X @ W.T) < 0.15
    assert rel(b["dx"], DY @ W) < 0.25
    assert rel(b["dw"], DY.T @ X) < 0.25
    # the saved X^T and the gradient's dY^T carry the same sign vector:
    # with quantization removed the transform cancels exactly (to fp64 rounding)
    s = rht.rht_signs(seed)
    xt = rht.rht_along_axis(x, s, axis=0).astype(np.float64)
    dyt = rht.rht_along_axis(dy, s, axis=0).astype(np.float64)
    assert rel(dyt.T @ xt, DY.T @ X) < 1e-6
    # Fprop's W and Dgrad's W^T are the same quantized tensor
    np.testing.assert_array_equal(formats.unpack_nibbles(f["wq"]["codes"]).T,
                                  formats.unpack_nibbles(f["wq"]["codes_t"]))


def test_workload_generator_is_deterministic():
    a = workloads.tiny_layer()
    b = workloads.tiny_layer()
    for t, u in zip(a, b):
        assert t.dtype.is_floating_point and (t == u).all()
    x = workloads.bf16_to_f32_numpy(a[0])
    big_cols = np.flatnonzero(np.abs(x).max(axis=0) > 20)
    assert len(big_cols) == 2


def test_linear_bf16_closed_form_and_one_hot_orientation():
    """The BF16 layer step: constant operands give K, N and M times the
    products; one-hot inputs pin which operand is transposed in each of the
    three products."""
    M, K, N = 3, 4, 5
    y, dx, dw = gemm.linear_bf16_ref(np.full((M, K), 0.5), np.full((N, K), 3.0), np.full((M, N), -2.0))
    np.testing.assert_array_equal(y, np.full((M, N), K * 1.5))
    np.testing.assert_array_equal(dx, np.full((M, K), N * -6.0))
    np.testing.assert_array_equal(dw, np.full((N, K), M * -1.0))
    x = np.zeros((M, K)); x[2, 1] = 2.0
    w = np.zeros((N, K)); w[4, 1] = 3.0
    dy = np.zeros((M, N)); dy[2, 4] = 5.0
    y, dx, dw = gemm.linear_bf16_ref(x, w, dy)
    assert np.argwhere(y).tolist() == [[2, 4]] and y[2, 4] == 6.0
    assert np.argwhere(dx).tolist() == [[2, 1]] and dx[2, 1] == 15.0   # row 2 of dY picks row 4 of W
    assert np.argwhere(dw).tolist() == [[4, 1]] and dw[4, 1] == 10.0   # dY^T X: column 4 of dY, row 2 of X


def test_linear_bf16_matches_loop_brute_force():
    """Element-by-element sums in exact rationals on small random BF16
    operands (independent of the matrix-product routine)."""
    rng = np.random.default_rng(7)
    M, K, N = 3, 5, 4
    bf = lambda a: workloads.bf16_to_f32_numpy(workloads.to_bf16(a.astype(np.float32)))  # noqa: E731
    x, w, dy = bf(rng.standard_normal((M, K))), bf(rng.standard_normal((N, K))), bf(rng.standard_normal((M, N)))
    y, dx, dw = gemm.linear_bf16_ref(x, w, dy)
    F = lambda v: Fraction(float(v))  # noqa: E731
    for i in range(M):
        for j in range(N):
            assert Fraction(y[i, j]) == sum(F(x[i, k]) * F(w[j, k]) for k in range(K))
        for k in range(K):
            assert Fraction(dx[i, k]) == sum(F(dy[i, j]) * F(w[j, k]) for j in range(N))
    for j in range(N):
        for k in range(K):
            assert Fraction(dw[j, k]) == sum(F(dy[i, j]) * F(x[i, k]) for i in range(M))


def test_linear_layer_amax_is_the_quantized_tensors_own():
    """The per-tensor scale of every operand is set from the amax of the
    tensor actually quantized -- after the Hadamard transform for the two
    Wgrad operands -- so the block holding that tensor's largest value gets
    the largest E4M3 scale, 448 (code 0x7E), and ts = 1 / (2688 / amax).
    The transformed amax is checked against an explicit float64 product of
    Q = 1/4 H diag(s) on every 16-token chunk (not the oracle's tree)."""
    x, w, dy = workloads.tiny_layer()
    x, w, dy = (workloads.bf16_to_f32_numpy(t) for t in (x, w, dy))
    seed = 77
    f = linear.linear_fwd(x, w, seed)
    b = linear.linear_bwd(dy, f, seed)
    Q = rht.rht_matrix_f64(rht.rht_signs(seed))

    def transformed_t(t):
        # Q along the token axis (axis 0) in float64, returned transposed [cols, M]
        tt = t.astype(np.float64).T
        return (tt.reshape(tt.shape[0], -1, 16) @ Q.T).reshape(tt.shape)

    def check(q, plain, blocks_2d=False):
        amax = np.float32(np.max(np.abs(plain)))
        assert abs(float(q["amax"]) - float(amax)) <= 4 * float(np.spacing(amax)), (q["amax"], amax)
        assert q["ts"] == np.float32(np.float32(1) / np.float32(np.float32(2688) / q["amax"]))
        r, c = np.unravel_index(np.argmax(np.abs(plain)), plain.shape)
        E = q["scales_2d"][r // 16, c // 16] if blocks_2d else q["scales"][r, c // 16]
        assert E == 0x7E, (r, c, E)

    check(f["xq"], x)
    check(f["wq"], w, blocks_2d=True)
    check(f["xtq"], transformed_t(x))
    check(b["dyq"], dy)
    check(b["dytq"], transformed_t(dy))
    # the transform moves the maximum: the untransformed amax is not the one used
    assert b["dytq"]["amax"] != np.float32(np.max(np.abs(dy)))
    assert f["xtq"]["amax"] != np.float32(np.max(np.abs(x)))
