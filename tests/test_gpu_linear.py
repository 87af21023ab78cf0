"""GPU parity of the whole NVFP4 linear layer (Fprop, Dgrad, Wgrad) against
the oracle: every quantized operand bit-exact, every GEMM output within a
relative Frobenius error of 1e-3 of the BF16-rounded FP64 oracle."""

import numpy as np
import pytest
import torch

from nvfp4_bit_numerics_gb300 import binding as B
from nvfp4_bit_numerics_gb300 import workloads
from oracle import formats, gemm, linear, quant
from tests.gpu_util import assert_q_equal, ensure_lib, f32, rel_fro

pytestmark = pytest.mark.gpu

TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_lib()


def run_layer(x, w, dy, seed):
    M, K = x.shape
    N = w.shape[0]
    ws = B.linear_workspace(M, K, N)
    xg, wg, dyg = x.cuda(), w.cuda(), dy.cuda()
    y = B.nvfp4_linear_fwd(xg, wg, seed, ws)
    dx, dw = B.nvfp4_linear_bwd(dyg, K, seed, ws)
    torch.cuda.synchronize()
    assert B.nvfp4_get_status() == B.NVFP4_OK
    return y, dx, dw, B.nvfp4_linear_get_views(ws, M, K, N)


def test_tiny_layer_full_parity():
    """The single-layer case with outlier channels: X [128,256], W [256,256],
    dY [128,256], all three GEMMs and all six quantized operands."""
    x, w, dy = workloads.tiny_layer()
    seed = 0xC0FFEE
    y, dx, dw, v = run_layer(x, w, dy, seed)
    xf, wf, dyf = f32(x), f32(w), f32(dy)
    f = linear.linear_fwd(xf, wf, seed)
    b = linear.linear_bwd(dyf, f, seed)
    assert_q_equal(v["xq"], f["xq"], what="xq")
    wq = f["wq"]
    assert_q_equal(v["wq"], dict(codes=wq["codes"], scales=wq["scales"], amax=wq["amax"], ts=wq["ts"]), what="wq")
    assert_q_equal(v["wtq"], dict(codes=wq["codes_t"], scales=wq["scales_t"], amax=wq["amax"], ts=wq["ts"]),
                   what="wtq")
    assert_q_equal(v["xtq"], f["xtq"], what="xtq")
    assert_q_equal(v["dyq"], b["dyq"], what="dyq")
    assert_q_equal(v["dytq"], b["dytq"], what="dytq")
    for name, got, ref in (("y", y, f["y"]), ("dx", dx, b["dx"]), ("dw", dw, b["dw"])):
        g = got.float().cpu().numpy()
        assert rel_fro(g, formats.float64_to_bf16_rne(ref)) <= TOL, name
    # and the layer is close to the unquantized one
    X, W, DY = (a.astype(np.float64) for a in (xf, wf, dyf))
    assert rel_fro(y.float().cpu().numpy(), X @ W.T) < 0.15
    assert rel_fro(dw.float().cpu().numpy(), DY.T @ X) < 0.25


def test_layer_step_is_deterministic():
    x, w, dy = workloads.tiny_layer(M=256, K=512, N=384, seed=5)
    r1 = run_layer(x, w, dy, 17)
    r2 = run_layer(x, w, dy, 17)
    for a, b in zip(r1[:3], r2[:3]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("shape", [(8192, 5120, 20480), (512, 256, 768), (768, 512, 256), (256, 256, 2048),
                                   (2048, 256, 256), (256, 1024, 512), (384, 256, 128)])
def test_bwd_one_launch_equals_separate_gemms(shape):
    """nvfp4_linear_bwd runs Dgrad and Wgrad as one launch of the CTA-pair
    kernel over a shared tile schedule when both shapes take that kernel: its
    dX and dW equal two separate nvfp4_gemm calls on the same quantized
    operands bit for bit (the last shape, M % 256 != 0, takes two launches)."""
    M, K, N = shape
    x, w, dy = workloads.tiny_layer(M=M, K=K, N=N, seed=9)
    ws = B.linear_workspace(M, K, N)
    B.nvfp4_linear_fwd(x.cuda(), w.cuda(), 5, ws)
    dyg = dy.cuda()
    # outputs pre-filled with NaN: a tile the schedule skipped would show
    dx = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    dw = torch.full((N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    n0 = B.nvfp4_kernel_launch_count()
    dx, dw = B.nvfp4_linear_bwd(dyg, K, 5, ws, dx=dx, dw=dw)
    torch.cuda.synchronize()
    launches = B.nvfp4_kernel_launch_count() - n0
    assert B.nvfp4_get_status() == B.NVFP4_OK
    v = B.nvfp4_linear_get_views(ws, M, K, N)
    dx2 = B.nvfp4_gemm(v["dyq"], v["wtq"])
    dw2 = B.nvfp4_gemm(v["dytq"], v["xtq"])
    torch.cuda.synchronize()
    assert torch.equal(dx, dx2)
    assert torch.equal(dw, dw2)
    # amax, the fused quantize, then one GEMM launch (two when M % 256 != 0)
    assert launches == (3 if M % 256 == 0 else 4)


@pytest.mark.parametrize("layer", ["mlp_up", "mlp_down", "qkv"])
def test_layer_full_size_sampled(layer):
    """The full-size layers: MLP up-projection (M=8192, K=5120, N=20480, the
    benchmark's workload, launched as the benchmark launches it), MLP
    down-projection (K=20480, N=5120) and the QKV projection (K=5120,
    N=7168).  The oracle recomputes the amaxes and the quantized operands it
    needs and the GEMM outputs of sampled rows of Y, dX and dW."""
    x, w, dy = getattr(workloads, layer)()
    M, K = x.shape
    N = w.shape[0]
    seed = 2 if layer == "mlp_up" else 3
    y, dx, dw, v = run_layer(x, w, dy, seed)
    xf, wf, dyf = f32(x), f32(w), f32(dy)
    rng = np.random.default_rng(1)
    rm = np.sort(rng.choice(M, 12, replace=False))
    rn = np.sort(rng.choice(N, 12, replace=False))
    # forward operands
    xq = quant.quantize_1d(xf, "rne", amax=quant.tensor_amax(xf), row_ids=rm)
    assert_q_equal(v["xq"], xq, rows=rm, what="xq")
    wq = quant.quantize_2d(wf)
    assert_q_equal(v["wq"], dict(codes=wq["codes"], scales=wq["scales"], amax=wq["amax"], ts=wq["ts"]), what="wq")
    xtq = quant.quantize_transpose(xf, "rne", rht_seed=seed)
    assert_q_equal(v["xtq"], xtq, what="xtq")
    yr = gemm.gemm_ref(xq["codes"], xq["scales"], xq["ts"], wq["codes"], wq["scales"], wq["ts"])
    assert rel_fro(y[rm].float().cpu().numpy(), formats.float64_to_bf16_rne(yr)) <= TOL
    # backward operands
    dyq = quant.quantize_1d(dyf, "sr", seed=seed, stream_id=linear.SR_STREAM_DY, amax=quant.tensor_amax(dyf),
                            row_ids=rm)
    assert_q_equal(v["dyq"], dyq, rows=rm, what="dyq")
    amax_t = quant.amax_rht(dyf, seed, axis=0)
    dytq = quant.quantize_transpose(dyf, "sr", seed=seed, stream_id=linear.SR_STREAM_DYT, rht_seed=seed,
                                    amax=amax_t, col_ids=rn)
    assert_q_equal(v["dytq"], dytq, rows=rn, what="dytq")
    dxr = gemm.gemm_ref(dyq["codes"], dyq["scales"], dyq["ts"], wq["codes_t"], wq["scales_t"], wq["ts"])
    assert rel_fro(dx[rm].float().cpu().numpy(), formats.float64_to_bf16_rne(dxr)) <= TOL
    dwr = gemm.gemm_ref(dytq["codes"], dytq["scales"], dytq["ts"], xtq["codes"], xtq["scales"], xtq["ts"])
    assert rel_fro(dw[rn].float().cpu().numpy(), formats.float64_to_bf16_rne(dwr)) <= TOL


def test_layer_full_size_every_operand_cxx_oracle():
    """The benchmark's layer (MLP up-projection, M=8192, K=5120, N=20480) with
    every element of all six quantized operands -- X and X^T (Hadamard, RNE),
    W and W^T (16x16 blocks), dY (stochastic) and dY^T (Hadamard, stochastic)
    -- codes, block scales, amax and tensor scale compared bit for bit with the
    plain C++ oracle, which runs the whole tensors on the host's cores."""
    from oracle import cxx

    x, w, dy = workloads.mlp_up()
    M, K = x.shape
    N = w.shape[0]
    seed = 2
    _, _, _, v = run_layer(x, w, dy, seed)
    xf, wf, dyf = f32(x), f32(w), f32(dy)
    assert_q_equal(v["xq"], cxx.quantize_1d(xf, "rne"), what="xq")
    assert_q_equal(v["xtq"], cxx.quantize_transpose(xf, "rne", rht_seed=seed), what="xtq")
    wq = cxx.quantize_2d(wf)
    assert_q_equal(v["wq"], dict(codes=wq["codes"], scales=wq["scales"], amax=wq["amax"], ts=wq["ts"]), what="wq")
    assert_q_equal(v["wtq"], dict(codes=wq["codes_t"], scales=wq["scales_t"], amax=wq["amax"], ts=wq["ts"]),
                   what="wtq")
    assert_q_equal(v["dyq"], cxx.quantize_1d(dyf, "sr", seed=seed, stream_id=linear.SR_STREAM_DY), what="dyq")
    assert_q_equal(v["dytq"], cxx.quantize_transpose(dyf, "sr", seed=seed, stream_id=linear.SR_STREAM_DYT,
                                                     rht_seed=seed), what="dytq")
