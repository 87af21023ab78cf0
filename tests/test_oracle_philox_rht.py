"""Pins of the oracle's Philox4x32-10 and 16x16 random Hadamard transform."""

import numpy as np
import pytest

from oracle import philox, rht
from tests.conftest import read_golden


def test_philox_known_answers():
    for row in read_golden("philox4x32_10_kat.txt"):
        v = [int(t, 16) for t in row]
        out = philox.philox4x32_10(v[0], v[1], v[2], v[3], v[4], v[5])
        assert [int(w) for w in out] == v[6:10]


def test_philox_vectorised_matches_scalar():
    c0 = np.arange(100, dtype=np.uint32)
    vec = philox.philox4x32_10(c0, 7, 3, 0, 0x1234, 0x5678)
    for i in (0, 1, 57, 99):
        sc = philox.philox4x32_10(i, 7, 3, 0, 0x1234, 0x5678)
        assert [int(w[i]) for w in vec] == [int(w) for w in sc]


def test_sr_uniform_uses_eight_elements_per_call():
    seed = 0xDEADBEEF12345678
    e = np.arange(64, dtype=np.uint64)
    u = philox.sr_uniform16(seed, 1, e)
    k0, k1 = philox.seed_key(seed)
    for g in range(8):
        w = [int(x) for x in philox.philox4x32_10(g, 0, 1, 0, k0, k1)]
        exp = []
        for word in w:
            exp += [word & 0xFFFF, word >> 16]
        assert [int(x) for x in u[8 * g:8 * g + 8]] == exp


def test_sr_uniform_statistics():
    u = philox.sr_uniform16(3, 0, np.arange(1 << 20, dtype=np.uint64)).astype(np.float64)
    n = u.size
    mean_sd = np.sqrt((65536.0 ** 2 - 1) / 12.0 / n)
    assert abs(u.mean() - 32767.5) < 5 * mean_sd
    bits = ((u.astype(np.uint32)[:, None] >> np.arange(16)) & 1).mean(axis=0)
    assert np.all(np.abs(bits - 0.5) < 5 * 0.5 / np.sqrt(n))


def test_hadamard_orthogonality():
    H = rht.hadamard16()
    np.testing.assert_array_equal(H @ H.T, 16 * np.eye(16, dtype=np.int64))
    assert np.all(H[0] == 1) and np.all(H[:, 0] == 1)
    s = rht.rht_signs(42)
    Q = rht.rht_matrix_f64(s)
    np.testing.assert_allclose(Q.T @ Q, np.eye(16), atol=0, rtol=0)


def test_sign_vector_from_philox_word0():
    seed = 987654321
    s = rht.rht_signs(seed)
    k0, k1 = philox.seed_key(seed)
    w0 = int(philox.philox4x32_10(0, 0, 2, 0, k0, k1)[0])
    assert all((s[j] == -1) == bool((w0 >> j) & 1) for j in range(16))
    assert set(np.unique(s)) <= {-1, 1}
    assert not np.array_equal(rht.rht_signs(seed), rht.rht_signs(seed + 1))


def test_rht_one_hot_columns():
    """Q e_j is column j of Q: entries +-1/4 with signs H[i][j]·s_j."""
    s = rht.rht_signs(7)
    H = rht.hadamard16()
    for j in range(16):
        e = np.zeros(16, np.float32)
        e[j] = 1.0
        y = rht.rht16_chunks(e[None, :], s)[0]
        np.testing.assert_array_equal(y, 0.25 * H[:, j] * s[j])


def test_rht_fp32_tree_within_bound_of_fp64():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((4096, 16)) * np.exp(rng.uniform(-8, 8, (4096, 1)))).astype(np.float32)
    x[::7, 3] *= 1000
    s = rht.rht_signs(5)
    y32 = rht.rht16_chunks(x, s).astype(np.float64)
    y64 = x.astype(np.float64) @ rht.rht_matrix_f64(s).T
    # four levels of float32 additions: |err| <= 4 u sum|terms| (u = 2^-24), times 1/4
    bound = 4 * 2.0 ** -24 * 0.25 * np.sum(np.abs(x.astype(np.float64)), axis=1, keepdims=True)
    assert np.all(np.abs(y32 - y64) <= bound * 1.0001)


def test_fwht_butterfly_equals_tree_ordered_product():
    """The in-register butterfly (strides 1, 2, 4, 8) computes exactly the
    tree-ordered sums the oracle defines, bit for bit."""
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((20000, 16)) * np.exp(rng.uniform(-20, 20, (20000, 16)))).astype(np.float32)
    # exact zeros, signed zeros and exactly cancelling pairs
    x[:2000] = 0.0
    x[1000:2000, ::3] = -0.0
    x[2000:4000, 1::2] = x[2000:4000, 0::2]
    x[4000:5000, 8:] = -x[4000:5000, :8]
    s = rht.rht_signs(11)
    t = (x * s.astype(np.float32)).astype(np.float32)
    for h in (1, 2, 4, 8):
        t = t.copy()
        for i in range(16):
            if i & h == 0:
                a, b = t[:, i].copy(), t[:, i + h].copy()
                t[:, i] = a + b
                t[:, i + h] = a - b
    t = (t * np.float32(0.25)).astype(np.float32)
    t = (t + np.float32(0.0)).astype(np.float32)  # an exact zero is +0
    np.testing.assert_array_equal(t.view(np.uint32), rht.rht16_chunks(x, s).view(np.uint32))
    assert not np.any(np.signbit(rht.rht16_chunks(x, s)) & (rht.rht16_chunks(x, s) == 0))


def test_rht_cancels_in_wgrad():
    """(Q dY)^T (Q X) over 16-token chunks equals dY^T X (unquantized)."""
    rng = np.random.default_rng(3)
    dy = rng.standard_normal((64, 24)).astype(np.float32)
    x = rng.standard_normal((64, 40)).astype(np.float32)
    s = rht.rht_signs(99)
    dyt = rht.rht_along_axis(dy, s, axis=0).astype(np.float64)
    xt = rht.rht_along_axis(x, s, axis=0).astype(np.float64)
    ref = dy.astype(np.float64).T @ x.astype(np.float64)
    got = dyt.T @ xt
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-6


def test_rht_spreads_outliers():
    """Informational property from the pages: the transform spreads an
    outlier channel over its 16-chunk, lowering the block max/RMS ratio."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((256, 64)).astype(np.float32)
    x[5::16, :] *= 50  # one outlier token per 16-token chunk
    s = rht.rht_signs(1)
    y = rht.rht_along_axis(x, s, axis=0)

    def crest(a):
        b = a.T.reshape(-1, 16)
        return np.mean(np.max(np.abs(b), axis=1) / np.sqrt(np.mean(b ** 2, axis=1)))

    assert crest(y) < 0.6 * crest(x)
