"""Seeded synthetic inputs for the NVFP4 linear-layer workloads.

This module only draws random numbers and rounds them to BF16; it holds none
of the quantization or GEMM arithmetic, so both the CUDA path and the CPU
oracle can take their inputs from it.

Every tensor is drawn with numpy's PCG64 generator (``default_rng(seed)``) in
float64, in the order the functions below list, then rounded to BF16 with
round-to-nearest-even.  N(mu, sigma) takes sigma as the standard deviation.

Workloads (shapes of the layers the method trains; the pages use a 12B hybrid
Mamba-Transformer, whose MLP and attention projections these stand in for):

* ``tiny_layer``      M=128, K=256, N=256: X ~ N(0,1) with 2 input channels
                      x50, W ~ N(0, 0.02), dY ~ N(0, 1e-3)
* ``quant_sweep``     [8192, 5120] and [8192, 20480] ~ N(0,1), 0.1% of entries
                      replaced by 20 * Student-t(nu=2)
* ``mlp_up``          M=8192, K=5120, N=20480: X ~ N(0,1) with 8 outlier
                      channels x30, W ~ N(0, 0.014), dY ~ N(0, 1e-4)
* ``mlp_down`` / ``qkv``  M=8192, (K, N) = (20480, 5120) / (5120, 7168), same
                      distributions as ``mlp_up``
* ``gemm_sweep``      M=16384, X ~ Student-t(nu=3), W ~ N(0, 0.02),
                      dY ~ N(0, 1e-4)
"""

import numpy as np
import torch


def to_bf16(a):
    """float64/float32 numpy -> torch.bfloat16 (CPU), round-to-nearest-even."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bf16_to_f32_numpy(t):
    return t.to(torch.float32).numpy()


def _normal(rng, shape, sigma):
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma)


def layer_inputs(M, K, N, seed, outlier_cols, outlier_scale, w_sigma, dy_sigma, x_dist="normal"):
    """(X [M,K], W [N,K], dY [M,N]) as CPU bf16 tensors.

    Draw order: X, the outlier channel indices, W, dY."""
    rng = np.random.default_rng(seed)
    if x_dist == "normal":
        x = rng.standard_normal((M, K), dtype=np.float32)
    elif x_dist == "t3":
        x = rng.standard_t(3, size=(M, K)).astype(np.float32)
    else:
        raise ValueError(x_dist)
    if outlier_cols:
        cols = rng.choice(K, outlier_cols, replace=False)
        x[:, cols] *= np.float32(outlier_scale)
    w = _normal(rng, (N, K), w_sigma)
    dy = _normal(rng, (M, N), dy_sigma)
    return to_bf16(x), to_bf16(w), to_bf16(dy)


def tiny_layer(M=128, K=256, N=256, seed=0):
    return layer_inputs(M, K, N, seed, 2, 50.0, 0.02, 1e-3)


def mlp_up(M=8192, K=5120, N=20480, seed=2):
    return layer_inputs(M, K, N, seed, 8, 30.0, 0.014, 1e-4)


def mlp_down(M=8192, K=20480, N=5120, seed=3):
    return layer_inputs(M, K, N, seed, 8, 30.0, 0.014, 1e-4)


def qkv(M=8192, K=5120, N=7168, seed=3):
    return layer_inputs(M, K, N, seed, 8, 30.0, 0.014, 1e-4)


def gemm_sweep(K, N, M=16384, seed=4):
    return layer_inputs(M, K, N, seed, 0, 1.0, 0.02, 1e-4, x_dist="t3")


def heavy_tailed(rows, cols, seed=1, frac=0.001, scale=20.0):
    """[rows, cols] ~ N(0,1) with ``frac`` of the entries (drawn uniformly
    without replacement) replaced by scale * Student-t(nu=2)."""
    rng = np.random.default_rng(seed)
    t = rng.standard_normal((rows, cols), dtype=np.float32)
    n_out = int(round(frac * rows * cols))
    if n_out:
        idx = rng.choice(rows * cols, n_out, replace=False)
        t.reshape(-1)[idx] = (scale * rng.standard_t(2, size=n_out)).astype(np.float32)
    return to_bf16(t)


def quant_sweep(seed=1):
    """The two tensors of the quantize-only sweep, drawn in this order."""
    rng_seed = np.random.SeedSequence(seed).spawn(2)
    a = heavy_tailed(8192, 5120, seed=rng_seed[0])
    b = heavy_tailed(8192, 20480, seed=rng_seed[1])
    return a, b
