"""GPU parity of the MXFP4 path (nvfp4_quantize_mx and nvfp4_gemm on MXFP4
operands) against the oracle's MXFP4 definition (oracle/mx.py): codes and
UE8M0 scales bit for bit, GEMMs within the FP32/BF16 tolerances of the NVFP4
GEMM tests.  One-hot probes pin which scale byte the tensor cores apply to
which 32-element half of a 64-element chunk."""

import numpy as np
import pytest
import torch

from nvfp4_bit_numerics_gb300 import binding as B
from nvfp4_bit_numerics_gb300 import workloads
from oracle import formats, mx, quant
from tests.gpu_util import assert_q_equal, ensure_lib, f32, outlier_tensor, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_lib()


def mx_to_numpy(q):
    """MXFP4 QTensor -> (codes [rows, cols/2], scales [rows, cols/32]); for
    the MMA layout also checks that the two padding bytes of every word are
    zero."""
    torch.cuda.synchronize()
    codes = q.codes.cpu().numpy()
    sc = q.scales.cpu().numpy()
    if q.layout == B.NVFP4_SCALES_MMA:
        words = quant.unswizzle_scales(sc, q.rows, q.cols // 16).reshape(q.rows, q.cols // 64, 4)
        assert not words[:, :, 2:].any(), "nonzero padding bytes in MMA scale words"
        sc = words[:, :, :2].reshape(q.rows, q.cols // 32)
    else:
        sc = sc.reshape(q.rows, q.cols // 32)
    return codes, sc


def assert_mx_equal(q, ref, rows=None, what=""):
    codes, sc = mx_to_numpy(q)
    if rows is not None:
        codes, sc = codes[rows], sc[rows]
    bad_s = np.argwhere(sc != ref["scales"])
    assert bad_s.size == 0, "%s: %d scale mismatches, first %s gpu=%d ref=%d" % (
        what, len(bad_s), bad_s[0], sc[tuple(bad_s[0])], ref["scales"][tuple(bad_s[0])])
    bad = np.argwhere(codes != ref["codes"])
    assert bad.size == 0, "%s: %d code-byte mismatches of %d, first %s gpu=%#x ref=%#x" % (
        what, len(bad), codes.size, bad[0], codes[tuple(bad[0])], ref["codes"][tuple(bad[0])])


def mx_edge_tensor(rows, cols, seed):
    """bf16 tensor with Gaussian blocks, outliers, zero blocks, blocks of
    tiny (subnormal-range) and huge values, exact powers of two and values on
    the E2M1 rounding ties after scaling."""
    x = f32(outlier_tensor(rows, cols, seed))
    rng = np.random.default_rng(seed + 100)
    x[0, :32] = 0.0                                  # zero block
    x[1, 32:64] = rng.standard_normal(32) * 1e-38    # amax in the BF16 subnormal range
    x[2, :32] = rng.standard_normal(32) * 1e37       # E near the top of the range
    x[3, :32] = np.exp2(rng.integers(-20, 20, 32))   # exact powers of two
    # block max 5 -> E = 127, multiplier 1: the ties 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, both signs
    x[4, :32] = np.tile([4.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], 4) * np.repeat([1, -1, 1, -1], 8)
    x[5, :32] = 7.9375                               # above 6 after scaling: saturation
    if rows > 64:
        x[64:96, 7] = rng.standard_normal(32) * 1e-30  # a column block of the transposed output
    return workloads.to_bf16(x)


SHAPES = [(64, 64), (128, 256), (192, 320), (256, 1024), (384, 128)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", [B.NVFP4_SCALES_LINEAR, B.NVFP4_SCALES_MMA])
def test_quantize_mx_rowwise(shape, layout):
    rows, cols = shape
    if layout == B.NVFP4_SCALES_MMA and rows % 128:
        pytest.skip("the MMA scale layout needs rows % 128 == 0")
    x = mx_edge_tensor(rows, cols, rows + cols)
    out, _ = B.nvfp4_quantize_mx(x.cuda(), B.NVFP4_Q_ROWWISE, layout=layout)
    assert_mx_equal(out, mx.quantize_mx(f32(x)), what="mx rowwise %s" % (shape,))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", [B.NVFP4_SCALES_LINEAR, B.NVFP4_SCALES_MMA])
def test_quantize_mx_transpose(shape, layout):
    rows, cols = shape
    if layout == B.NVFP4_SCALES_MMA and cols % 128:
        pytest.skip("the MMA scale layout needs the transposed rows % 128 == 0")
    x = mx_edge_tensor(rows, cols, 3 * rows + cols)
    out, _ = B.nvfp4_quantize_mx(x.cuda(), B.NVFP4_Q_TRANSPOSE, layout=layout)
    assert (out.rows, out.cols) == (cols, rows)
    assert_mx_equal(out, mx.quantize_mx(np.ascontiguousarray(f32(x).T)), what="mx transpose %s" % (shape,))


@pytest.mark.parametrize("shape", [(128, 128), (192, 256), (512, 384)])
def test_quantize_mx_rowwise_and_transpose(shape):
    """One read, two outputs; the ragged last tile (192 rows: 128 + 64) too."""
    rows, cols = shape
    lay = B.NVFP4_SCALES_LINEAR if rows % 128 else B.NVFP4_SCALES_MMA
    x = mx_edge_tensor(rows, cols, 5 * rows + cols)
    o, ot = B.nvfp4_quantize_mx(x.cuda(), B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, layout=lay)
    xf = f32(x)
    assert_mx_equal(o, mx.quantize_mx(xf), what="fused rowwise")
    assert_mx_equal(ot, mx.quantize_mx(np.ascontiguousarray(xf.T)), what="fused transpose")


def test_quantize_mx_all_zero_and_deterministic():
    x = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    o, ot = B.nvfp4_quantize_mx(x, B.NVFP4_Q_ROWWISE_AND_TRANSPOSE)
    codes, sc = mx_to_numpy(o)
    assert not codes.any() and not sc.any()
    y = mx_edge_tensor(256, 512, 7).cuda()
    a, _ = B.nvfp4_quantize_mx(y)
    b, _ = B.nvfp4_quantize_mx(y)
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)


# ---------------------------------------------------------------------------
# GEMM
# ---------------------------------------------------------------------------
def make_mx(codes_u4, scales_lin):
    """Device MXFP4 QTensor from unpacked codes [rows, K] and UE8M0 codes
    [rows, K/32], put in the MMA layout: words (E0, E1, 0, 0) of the NVFP4
    tile layout (the oracle's tile-layout definition on the padded words)."""
    rows, K = codes_u4.shape
    words = np.zeros((rows, K // 64, 4), np.uint8)
    words[:, :, :2] = scales_lin.reshape(rows, K // 64, 2)
    sc = quant.swizzle_scales(words.reshape(rows, K // 16))
    return B.QTensor(torch.from_numpy(formats.pack_nibbles(codes_u4)).cuda(), torch.from_numpy(sc).cuda(), None,
                     None, rows, K, B.NVFP4_SCALES_MMA, B.NVFP4_FORMAT_MXFP4)


def ref_mx(ac, asc, bc, bsc):
    return mx.gemm_mx_ref(dict(codes=formats.pack_nibbles(ac), scales=asc),
                          dict(codes=formats.pack_nibbles(bc), scales=bsc))


@pytest.mark.parametrize("M,N", [(128, 128), (128, 256), (256, 256)])
def test_mx_one_hot_layout_probe(M, N):
    """A single nonzero in A (row i, element k) and B (row j, element k) must
    land at D[i, j] only, scaled by exactly 2^(SA[i,k/32]-127) and
    2^(SB[j,k/32]-127), with every other block given another scale; k covers
    both halves of a 64-element chunk and both nibbles of a byte.  (128x128:
    1-CTA kernel, BN 128; 128x256: BN 256; 256x256: CTA-pair kernel.)"""
    K = 512
    rng = np.random.default_rng(M + N)
    positions = [(0, 0, 0), (1, 33, 1), (37, 63, 100), (127, 64, N - 1), (64, 255, 5), (33, 256, 7),
                 (96, 511, N // 2 + 3), (31, 300, 32), (32, 31, 31), (M - 1, 480, 64)]
    for (i, k, j) in positions:
        j = j % N
        ac = np.zeros((M, K), np.uint8)
        bc = np.zeros((N, K), np.uint8)
        ac[i, k] = 7        # +6
        bc[j, k] = 0xB      # -1.5
        asc = rng.integers(110, 120, size=(M, K // 32)).astype(np.uint8)
        bsc = rng.integers(135, 145, size=(N, K // 32)).astype(np.uint8)
        asc[i, k // 32] = 130  # 2^3
        bsc[j, k // 32] = 125  # 2^-2
        d = B.nvfp4_gemm(make_mx(ac, asc), make_mx(bc, bsc), out_dtype=torch.float32).cpu().numpy()
        nz = np.argwhere(d != 0)
        assert nz.tolist() == [[i, j]], ((i, k, j), nz[:5].tolist())
        assert d[i, j] == 6.0 * -1.5 * 2.0 ** 3 * 2.0 ** -2, ((i, k, j), d[i, j])


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 1024), (384, 384, 320), (128, 128, 192),
                                   (512, 768, 2048), (256, 256, 64)])
def test_mx_random_gemm(M, N, K):
    rng = np.random.default_rng(M * 5 + N * 11 + K)
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    asc = rng.integers(115, 135, size=(M, K // 32)).astype(np.uint8)
    bsc = rng.integers(115, 135, size=(N, K // 32)).astype(np.uint8)
    qa, qb = make_mx(ac, asc), make_mx(bc, bsc)
    ref = ref_mx(ac, asc, bc, bsc)
    d32 = B.nvfp4_gemm(qa, qb, out_dtype=torch.float32).cpu().numpy()
    assert B.nvfp4_get_status() == B.NVFP4_OK
    assert rel_fro(d32, ref) <= 1e-5
    d16 = B.nvfp4_gemm(qa, qb).float().cpu().numpy()
    assert rel_fro(d16, formats.float64_to_bf16_rne(ref)) <= 1e-3


def test_mx_quantize_then_gemm():
    """Quantize X and W on the GPU, multiply; the same through the oracle."""
    M, K, N = 256, 512, 384
    x, w, _ = workloads.tiny_layer(M, K, N, seed=11)
    qx, _ = B.nvfp4_quantize_mx(x.cuda())
    qw, _ = B.nvfp4_quantize_mx(w.cuda())
    d = B.nvfp4_gemm(qx, qw, out_dtype=torch.float32).cpu().numpy()
    ref = mx.gemm_mx_ref(mx.quantize_mx(f32(x)), mx.quantize_mx(f32(w)))
    assert rel_fro(d, ref) <= 1e-5


def test_mx_gemm_amax_and_mixed_formats_rejected():
    rng = np.random.default_rng(2)
    M, N, K = 256, 256, 256
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    asc = rng.integers(120, 130, size=(M, K // 32)).astype(np.uint8)
    bsc = rng.integers(120, 130, size=(N, K // 32)).astype(np.uint8)
    qa, qb = make_mx(ac, asc), make_mx(bc, bsc)
    d, amax = B.nvfp4_gemm_amax(qa, qb)
    torch.cuda.synchronize()
    assert amax.item() == float(d.float().abs().max().item())
    nv = B.empty_qtensor(N, K)
    with pytest.raises(B.Nvfp4Error):
        B.nvfp4_gemm(qa, nv)


def test_mx_gemm2_one_launch():
    """nvfp4_gemm2 on two MXFP4 products of different K (the Dgrad + Wgrad
    pattern): one launch, each product bit-identical to its own nvfp4_gemm and
    within the BF16 tolerance of the oracle's MXFP4 GEMM."""
    rng = np.random.default_rng(23)
    shapes = ((512, 768, 256), (256, 512, 1024))  # (M, N, K) of each product
    ops, refs = [], []
    for M, N, K in shapes:
        ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
        bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
        asc = rng.integers(115, 135, size=(M, K // 32)).astype(np.uint8)
        bsc = rng.integers(115, 135, size=(N, K // 32)).astype(np.uint8)
        ops += [make_mx(ac, asc), make_mx(bc, bsc)]
        refs.append(ref_mx(ac, asc, bc, bsc))
    a0, b0, a1, b1 = ops
    # outputs pre-filled with NaN: a tile the schedule skipped would show
    d0 = torch.full((shapes[0][0], shapes[0][1]), float("nan"), dtype=torch.bfloat16, device="cuda")
    d1 = torch.full((shapes[1][0], shapes[1][1]), float("nan"), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    n_before = B.nvfp4_kernel_launch_count()
    d0, d1 = B.nvfp4_gemm2(a0, b0, a1, b1, out0=d0, out1=d1)
    torch.cuda.synchronize()
    assert B.nvfp4_kernel_launch_count() - n_before == 1
    assert B.nvfp4_get_status() == B.NVFP4_OK
    assert torch.equal(d0, B.nvfp4_gemm(a0, b0))
    assert torch.equal(d1, B.nvfp4_gemm(a1, b1))
    for d, ref in ((d0, refs[0]), (d1, refs[1])):
        assert rel_fro(d.float().cpu().numpy(), formats.float64_to_bf16_rne(ref)) <= 1e-3


def test_mx_full_size_sampled():
    """The MXFP4 layer-shape Fprop (X 8192x5120, W 20480x5120, the 16x
    inter-layer MLP up-projection): sampled rows of the quantized X, its
    transpose and W bit for bit, and a sampled 32x32 block of Y = X W^T
    against the oracle's GEMM of the sampled quantized rows."""
    x, w, _ = workloads.mlp_up()
    xg, wg = x.cuda(), w.cuda()
    qx, qxt = B.nvfp4_quantize_mx(xg, B.NVFP4_Q_ROWWISE_AND_TRANSPOSE)
    qw, _ = B.nvfp4_quantize_mx(wg)
    y = B.nvfp4_gemm(qx, qw)
    assert B.nvfp4_get_status() == B.NVFP4_OK
    rng = np.random.default_rng(0)
    rs = np.sort(rng.choice(x.shape[0], 32, replace=False))
    cs = np.sort(rng.choice(w.shape[0], 32, replace=False))
    ks = np.sort(rng.choice(x.shape[1], 24, replace=False))
    xf, wf = f32(x), f32(w)
    rx = mx.quantize_mx(xf[rs])
    rw = mx.quantize_mx(wf[cs])
    assert_mx_equal(qx, rx, rows=rs, what="full X")
    assert_mx_equal(qw, rw, rows=cs, what="full W")
    assert_mx_equal(qxt, mx.quantize_mx(np.ascontiguousarray(xf[:, ks].T)), rows=ks, what="full X^T")
    ys = y[torch.from_numpy(rs).cuda()][:, torch.from_numpy(cs).cuda()].float().cpu().numpy()
    assert rel_fro(ys, formats.float64_to_bf16_rne(mx.gemm_mx_ref(rx, rw))) <= 1e-3


@pytest.mark.parametrize("which", ["mxfp4", "nvfp4_rowwise_rne", "nvfp4_2d", "nvfp4_fused_rne"])
def test_tile_ring_wait_bound_reports_timeout(which):
    """Failure detection without a GPU fault for the TMA-ring quantizers: the
    test hook makes the next launch skip its first CTA's first tile load, the
    bounded wait runs out (about 2 s), the kernel drains what it issued and
    reports NVFP4_ERR_TIMEOUT, and the next launch on the same context is
    bit-exact again."""
    import time

    x = mx_edge_tensor(256, 512, 31)
    xf = f32(x)
    xg = x.cuda()

    def run():
        if which == "mxfp4":
            return B.nvfp4_quantize_mx(xg, B.NVFP4_Q_ROWWISE)[0]
        if which == "nvfp4_2d":
            return B.nvfp4_quantize(xg, B.NVFP4_Q_2D)
        if which == "nvfp4_fused_rne":
            return B.nvfp4_quantize(xg, B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, B.NVFP4_ROUND_RNE, rht=True, seed=4)
        return B.nvfp4_quantize(xg, B.NVFP4_Q_ROWWISE, B.NVFP4_ROUND_RNE)[0]

    assert B.nvfp4_get_status() == B.NVFP4_OK
    B.nvfp4_debug_stall_next_quantize(True)
    t0 = time.time()
    run()
    st = B.nvfp4_get_status()
    dt = time.time() - t0
    assert st == B.NVFP4_ERR_TIMEOUT
    assert 1.0 < dt < 30.0
    q = run()
    assert B.nvfp4_get_status() == B.NVFP4_OK
    if which == "mxfp4":
        assert_mx_equal(q, mx.quantize_mx(xf), what="after the timeout")
    elif which == "nvfp4_fused_rne":
        assert_q_equal(q[0], quant.quantize_1d(xf, "rne"), what="rowwise after the timeout")
        assert_q_equal(q[1], quant.quantize_transpose(xf, "rne", rht_seed=4), what="transposed after the timeout")
    elif which == "nvfp4_2d":
        r = quant.quantize_2d(xf)
        assert_q_equal(q[0], dict(codes=r["codes"], scales=r["scales"], amax=r["amax"], ts=r["ts"]), what="W")
        assert_q_equal(q[1], dict(codes=r["codes_t"], scales=r["scales_t"], amax=r["amax"], ts=r["ts"]), what="W^T")
    else:
        assert_q_equal(q, quant.quantize_1d(xf, "rne"), what="after the timeout")
