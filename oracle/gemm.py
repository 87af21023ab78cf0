"""FP64-accumulated GEMM on dequantized NVFP4 operands.  TEST INFRASTRUCTURE ONLY.

Pretraining Large Language Models with NVFP4, Resumo técnico §3 ("Suporte de
Hardware"): the GEMMs run on Blackwell tensor cores that consume NVFP4
natively, i.e. block-scaled FP4 operands with FP32 accumulation.  The oracle's
definition of the product is exact arithmetic on the decoded values:

    D[i, j] = ts_A * ts_B * sum_k e2m1(A[i,k]) e4m3(SA[i,k//16]) e2m1(B[j,k]) e4m3(SB[j,k//16])

Both operands are K-major ([rows, K/2] packed codes, [rows, K/16] scales).
Every decoded value is exact in float64; the sum is a float64 matrix product.
"""

import numpy as np

from . import formats


def dequant_operand(codes, scales, rows=None):
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    if rows is not None:
        codes, scales = codes[rows], scales[rows]
    vals = formats.e2m1_decode(formats.unpack_nibbles(codes))
    sc = np.repeat(formats.e4m3_decode(scales), 16, axis=-1)
    return vals * sc


def gemm_ref(a_codes, a_scales, ts_a, b_codes, b_scales, ts_b, rows=None):
    """D = A·B^T in float64 for K-major NVFP4 A [M, K] and B [N, K].

    ``rows`` selects a subset of D's rows (A's rows)."""
    A = dequant_operand(a_codes, a_scales, rows)
    B = dequant_operand(b_codes, b_scales)
    return (A @ B.T) * (np.float64(ts_a) * np.float64(ts_b))


def linear_bf16_ref(x, w, dy):
    """The layer step of a linear layer kept in BF16 (Resumo técnico §2,
    item 1, "Precisão Mista Seletiva"): Y = X W^T, dX = dY W, dW = dY^T X for
    X [M, K], W [N, K], dY [M, N] given as float arrays holding BF16 values.
    Products of BF16 values are exact in float64; the sums are float64
    matrix products.  Returns (Y, dX, dW) in float64."""
    x, w, dy = (np.asarray(a, dtype=np.float64) for a in (x, w, dy))
    return x @ w.T, dy @ w, dy.T @ x
