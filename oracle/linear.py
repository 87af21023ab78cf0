"""NVFP4 linear layer: Fprop, Dgrad and Wgrad.  TEST INFRASTRUCTURE ONLY.

Pretraining Large Language Models with NVFP4, Resumo técnico §2 (Técnicas de
Treinamento Integradas), for a layer Y = X W^T with X [M, K] (M tokens),
W [N, K] and the incoming gradient dY [M, N]:

* Fprop  Y  = X W^T       X quantized 1x16 along K, RNE; W with 16x16 blocks.
* Dgrad  dX = dY W        dY quantized 1x16 along N with stochastic rounding
                          (item 4); W^T is the same 16x16 quantization as
                          in Fprop, transposed (item 3).
* Wgrad  dW = dY^T X      both operands go through the 16x16 random Hadamard
                          transform along the token dimension M (item 2), then
                          are quantized 1x16 along M: dY^T with stochastic
                          rounding, X^T with RNE.  The same sign vector is
                          used for both, so the transform cancels.

Random streams (a reading; the pages do not fix them): with the layer step's
seed as Philox key, stream 0 rounds dY (Dgrad operand), stream 1 rounds the
transformed dY^T (Wgrad operand), stream 2 draws the Hadamard signs.
"""

import numpy as np

from . import quant
from .gemm import gemm_ref

SR_STREAM_DY = 0
SR_STREAM_DYT = 1


def linear_fwd(x, w, seed, rows=None):
    """Quantize X (row-wise, and transposed with the Hadamard transform for
    Wgrad) and W (2D), and compute Y = X W^T in float64.

    ``rows`` restricts Y (and X's row-wise quantization) to a subset of
    tokens; the transposed X and W are always complete.
    """
    x = np.asarray(x, dtype=np.float32)
    xq = quant.quantize_1d(x, "rne", amax=quant.tensor_amax(x), row_ids=rows)
    wq = quant.quantize_2d(w)
    xtq = quant.quantize_transpose(x, "rne", rht_seed=seed)
    y = gemm_ref(xq["codes"], xq["scales"], xq["ts"], wq["codes"], wq["scales"], wq["ts"])
    return dict(y=y, xq=xq, wq=wq, xtq=xtq)


def linear_bwd(dy, fwd, seed, rows_dx=None, rows_dw=None):
    """Quantize dY (row-wise SR, and transposed + Hadamard + SR) and compute
    dX = dY W and dW = dY^T X in float64 from the saved forward operands."""
    dy = np.asarray(dy, dtype=np.float32)
    dyq = quant.quantize_1d(dy, "sr", seed=seed, stream_id=SR_STREAM_DY,
                            amax=quant.tensor_amax(dy), row_ids=rows_dx)
    amax_t = quant.amax_rht(dy, seed, axis=0)
    dytq = quant.quantize_transpose(dy, "sr", seed=seed, stream_id=SR_STREAM_DYT, rht_seed=seed,
                                    amax=amax_t, col_ids=rows_dw)
    wq, xtq = fwd["wq"], fwd["xtq"]
    dx = gemm_ref(dyq["codes"], dyq["scales"], dyq["ts"], wq["codes_t"], wq["scales_t"], wq["ts"])
    dw = gemm_ref(dytq["codes"], dytq["scales"], dytq["ts"], xtq["codes"], xtq["scales"], xtq["ts"])
    return dict(dx=dx, dw=dw, dyq=dyq, dytq=dytq)
