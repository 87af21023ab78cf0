"""GPU parity of the GEMM with a quantized output (nvfp4_gemm_quant): the
NVFP4 codes, scales and tensor scale its epilogue writes equal, bit for bit,
(a) the library's two-pass path -- the BF16 output of the plain GEMM, then the
rowwise RNE quantizer with the same amax -- and (b) the oracle's 1x16 RNE
quantization of that same BF16 output.  The BF16 output and the epilogue amax
it also writes equal the plain GEMM's."""

import numpy as np
import pytest
import torch

from nvfp4_bit_numerics_gb300 import binding as B
from nvfp4_bit_numerics_gb300 import workloads
from oracle import quant
from tests.gpu_util import assert_q_equal, ensure_lib, f32
from tests.test_gpu_gemm import make_q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_lib()


def random_operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    asc = rng.integers(0x28, 0x48, size=(M, K // 16)).astype(np.uint8)
    bsc = rng.integers(0x28, 0x48, size=(N, K // 16)).astype(np.uint8)
    return make_q(ac, asc, 0.75), make_q(bc, bsc, 1.5)


def qtensor_with_amax(M, N, amax):
    yq = B.empty_qtensor(M, N)
    yq.amax.copy_(amax.reshape(1))
    return yq


def assert_same_q(a, b, what):
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes), what + ": codes"
    assert torch.equal(a.scales, b.scales), what + ": scales"
    assert torch.equal(a.tensor_scale, b.tensor_scale), what + ": tensor scale"


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (512, 768, 512), (256, 512, 1024), (768, 256, 320)])
@pytest.mark.parametrize("amax_factor", [1.0, 1.7, 0.3])
def test_gemm_quant_equals_two_pass_and_oracle(M, N, K, amax_factor):
    """amax_factor 1: the output's own amax; 1.7: a stale larger amax;
    0.3: a stale smaller one, so the largest blocks saturate."""
    qa, qb = random_operands(M, N, K, M + N + K)
    y, amax = B.nvfp4_gemm_amax(qa, qb)
    amax_in = amax * amax_factor
    yq = qtensor_with_amax(M, N, amax_in)
    y2 = torch.empty_like(y)
    amax2 = torch.empty(1, dtype=torch.float32, device="cuda")
    B.nvfp4_gemm_quant(qa, qb, yq, out=y2, amax_out=amax2)
    assert B.nvfp4_get_status() == B.NVFP4_OK
    assert torch.equal(y2, y) and torch.equal(amax2, amax)
    # (a) the library's two-pass path on the same BF16 output
    q2 = B.empty_qtensor(M, N)
    q2.amax.copy_(amax_in)
    B.nvfp4_quantize(y, B.NVFP4_Q_ROWWISE, B.NVFP4_ROUND_RNE, compute_amax=False, out=q2)
    assert_same_q(yq, q2, "two-pass")
    # (b) the oracle on the same BF16 output
    ref = quant.quantize_1d(f32(y), "rne", amax=np.float32(amax_in.item()), row_ids=np.arange(M))
    assert_q_equal(yq, ref, what="oracle")
    # without a BF16 output: the same quantized output
    yq3 = qtensor_with_amax(M, N, amax_in)
    B.nvfp4_gemm_quant(qa, qb, yq3)
    assert_same_q(yq3, yq, "no BF16 output")


def test_gemm_quant_full_size_fprop_sampled():
    """The MLP up-projection Fprop (8192x5120 by 20480x5120): Y quantized in
    the epilogue with the amax of the previous (identical) step, against the
    oracle's quantization of sampled rows of the stored BF16 Y."""
    x, w, _ = workloads.mlp_up()
    qx, _ = B.nvfp4_quantize(x.cuda(), B.NVFP4_Q_ROWWISE, B.NVFP4_ROUND_RNE)
    qw, _ = B.nvfp4_quantize(w.cuda(), B.NVFP4_Q_2D)
    y, amax = B.nvfp4_gemm_amax(qx, qw)
    yq = qtensor_with_amax(8192, 20480, amax)
    y2 = torch.empty_like(y)
    B.nvfp4_gemm_quant(qx, qw, yq, out=y2)
    assert B.nvfp4_get_status() == B.NVFP4_OK
    assert torch.equal(y, y2)
    rows = np.sort(np.random.default_rng(0).choice(8192, 32, replace=False))
    yf = f32(y[torch.from_numpy(rows).cuda()])
    ref = quant.quantize_1d(yf, "rne", amax=np.float32(amax.item()), row_ids=np.arange(32))
    codes = yq.codes.cpu().numpy()[rows]
    sc = quant.unswizzle_scales(yq.scales.cpu().numpy(), 8192, 20480 // 16)[rows]
    assert np.array_equal(sc, ref["scales"])
    assert np.array_equal(codes, ref["codes"])
    assert yq.tensor_scale.item() == np.float32(ref["ts"])


def test_gemm_quant_nonfinite_amax_sets_status():
    qa, qb = random_operands(256, 256, 256, 3)
    yq = qtensor_with_amax(256, 256, torch.tensor([float("inf")], device="cuda"))
    B.nvfp4_gemm_quant(qa, qb, yq)
    assert B.nvfp4_get_status() == B.NVFP4_ERR_NONFINITE
    assert B.nvfp4_get_status() == B.NVFP4_OK
