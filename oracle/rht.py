"""16x16 random Hadamard transform.  TEST INFRASTRUCTURE ONLY.

Pretraining Large Language Models with NVFP4, Resumo técnico §2, item 2: a
random Hadamard transform is applied to the inputs of the weight-gradient
(Wgrad) GEMM, spreading outliers toward a Gaussian; NVIDIA cria método para
treinar redes neurais com precisão de 4 bits, "Como funciona", gives its size
as 16x16.  The transform is a fixed Hadamard matrix times a seeded random sign
vector; applied to both Wgrad operands along the reduction (token) dimension
it cancels in the product because it is orthogonal.

Readings (the pages give no formula):
* H is the 16x16 Sylvester matrix, H[i][j] = (-1)^popcount(i & j);
* the sign vector s (16 entries of +-1) is bit j of word 0 of
  Philox(key = seed, counter = (0, 0, 2, 0)): set bit -> -1;
* Q = (1/4)·H·diag(s) acts on each contiguous chunk of 16 along the
  transformed axis, so Q^T Q = I;
* float32 arithmetic: the products H[i][j]·s[j]·x[j] are exact sign flips,
  they are summed as a pairwise tree in index order (pairs (0,1), (2,3), ...,
  then pairs of pairs), and the sum is multiplied by 0.25;
* a zero has no sign in Q x: an output that is exactly zero is +0 (any
  summation order gives the same nonzero results bit for bit, but the sign of
  an exact zero depends on where negations are applied).
"""

import numpy as np

from .philox import philox4x32_10, seed_key

RHT_STREAM = 2


def hadamard16():
    i = np.arange(16)[:, None]
    j = np.arange(16)[None, :]
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def rht_signs(seed):
    """The 16 random signs (+-1, int64) for a layer step's seed."""
    k0, k1 = seed_key(seed)
    w0 = int(philox4x32_10(0, 0, RHT_STREAM, 0, k0, k1)[0])
    return np.array([-1 if (w0 >> j) & 1 else 1 for j in range(16)], dtype=np.int64)


def _tree_sum_f32(terms):
    """Pairwise float32 sum over the last axis (length 16), index order."""
    t = terms
    while t.shape[-1] > 1:
        t = (t[..., 0::2] + t[..., 1::2]).astype(np.float32)
    return t[..., 0]


def rht16_chunks(x, signs):
    """Apply Q = 1/4·H·diag(s) to each length-16 vector on the last axis.

    x: float32 array [..., 16].  Returns float32 [..., 16].
    """
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] == 16
    H = hadamard16()
    coef = (H * signs[None, :]).astype(np.float32)  # entries +-1
    # terms[..., i, j] = H[i][j]·s[j]·x[j], exact
    terms = coef * x[..., None, :]
    y = _tree_sum_f32(terms)
    y = (y * np.float32(0.25)).astype(np.float32)
    return (y + np.float32(0.0)).astype(np.float32)  # -0 -> +0


def rht_along_axis(x, signs, axis):
    """Apply the 16-point transform to consecutive 16-chunks along ``axis``."""
    x = np.asarray(x, dtype=np.float32)
    xm = np.moveaxis(x, axis, -1)
    n = xm.shape[-1]
    assert n % 16 == 0
    y = rht16_chunks(xm.reshape(xm.shape[:-1] + (n // 16, 16)), signs)
    return np.moveaxis(y.reshape(xm.shape), -1, axis)


def rht_matrix_f64(signs):
    """Q = 1/4·H·diag(s) in float64 (for error-bound checks only)."""
    return 0.25 * hadamard16().astype(np.float64) * signs[None, :].astype(np.float64)
