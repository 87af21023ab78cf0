"""GPU parity of the BF16 layer step (nvfp4_linear_bf16_fwd/_bwd, the layers
the method keeps in high precision) against the oracle's float64 products:
each output within one BF16 unit in the last place of the exactly rounded
result, and the relative Frobenius error of the NVFP4 GEMM tests."""

import numpy as np
import pytest
import torch

from nvfp4_bit_numerics_gb300 import binding as B
from nvfp4_bit_numerics_gb300 import workloads
from oracle import formats, gemm
from tests.gpu_util import ensure_lib, f32, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_lib()


def assert_bf16_close(got, ref, absmag, k, what):
    """got: BF16 results as float32; ref: float64 exact products; absmag: the
    same products of |operands|.  FP32 accumulation of k terms errs by at
    most k 2^-24 absmag (a standard worst-case bound), and the BF16 rounding
    adds at most one BF16 ulp (2^-7 of the magnitude)."""
    r16 = formats.float64_to_bf16_rne(ref)
    err = np.abs(got.astype(np.float64) - r16)
    bound = np.abs(r16) * 2.0 ** -7 + k * 2.0 ** -24 * absmag + 1e-30
    bad = np.argwhere(err > bound)
    assert bad.size == 0, "%s: %d elements beyond the bound, first %s got=%r ref=%r" % (
        what, len(bad), bad[0], got[tuple(bad[0])], ref[tuple(bad[0])])
    assert rel_fro(got, r16) <= 1e-3, what


@pytest.mark.parametrize("M,K,N", [(100, 64, 72), (128, 256, 256), (257, 520, 136), (1, 8, 8), (640, 1024, 384)])
def test_bf16_layer_step(M, K, N):
    x, w, dy = workloads.tiny_layer(M, K, N, seed=M + K + N)
    y = B.nvfp4_linear_bf16_fwd(x.cuda(), w.cuda())
    dx, dw = B.nvfp4_linear_bf16_bwd(dy.cuda(), x.cuda(), w.cuda())
    torch.cuda.synchronize()
    xf, wf, dyf = f32(x), f32(w), f32(dy)
    ry, rdx, rdw = gemm.linear_bf16_ref(xf, wf, dyf)
    ay, adx, adw = gemm.linear_bf16_ref(np.abs(xf), np.abs(wf), np.abs(dyf))
    assert_bf16_close(f32(y), ry, ay, K, "Y")
    assert_bf16_close(f32(dx), rdx, adx, N, "dX")
    assert_bf16_close(f32(dw), rdw, adw, M, "dW")


def test_bf16_layer_full_size_sampled():
    """The MLP up-projection shapes (X 8192x5120, W 20480x5120, dY
    8192x20480): sampled blocks of Y, dX and dW against the oracle on the
    sampled rows and columns."""
    x, w, dy = workloads.mlp_up()
    xg, wg, dyg = x.cuda(), w.cuda(), dy.cuda()
    y = B.nvfp4_linear_bf16_fwd(xg, wg)
    dx, dw = B.nvfp4_linear_bf16_bwd(dyg, xg, wg)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    rs = np.sort(rng.choice(8192, 12, replace=False))
    ns = np.sort(rng.choice(20480, 12, replace=False))
    ks = np.sort(rng.choice(5120, 12, replace=False))
    xf, wf, dyf = f32(x), f32(w), f32(dy)
    z = np.zeros((12, 12), np.float32)
    pick = lambda t, r, c: f32(t)[np.ix_(r, c)]  # noqa: E731

    def ref(i, xs, ws, dys):
        """Output i of the oracle's layer step on sliced operands, and the
        same for |operands|."""
        return (gemm.linear_bf16_ref(xs, ws, dys)[i],
                gemm.linear_bf16_ref(np.abs(xs), np.abs(ws), np.abs(dys))[i])

    # Y[rs, ns] = X[rs] W[ns]^T;  dX[rs, ks] = dY[rs] W[:, ks];  dW[ns, ks] = dY[:, ns]^T X[:, ks]
    assert_bf16_close(pick(y, rs, ns), *ref(0, xf[rs], wf[ns], z), 5120, "Y")
    assert_bf16_close(pick(dx, rs, ks), *ref(1, z, wf[:, ks], dyf[rs]), 20480, "dX")
    assert_bf16_close(pick(dw, ns, ks), *ref(2, xf[:, ks], z, dyf[:, ns]), 8192, "dW")
