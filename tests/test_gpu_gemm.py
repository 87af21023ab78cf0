"""GPU parity of the block-scaled FP4 GEMM against the oracle's FP64 GEMM on
the dequantized operands.  One-hot probes pin the operand nibble order, the
row mapping and the scale-factor layout that the tensor cores consume."""

import numpy as np
import pytest
import torch

from nvfp4_bit_numerics_gb300 import binding as B
from oracle import formats, gemm, quant
from tests.gpu_util import ensure_lib, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_lib()


def make_q(codes_u4, scales_lin, ts):
    """Device QTensor from unpacked 4-bit codes [rows, K] and linear E4M3
    scale codes [rows, K/16] (the scales are put in the MMA layout by the
    oracle's layout definition)."""
    rows, K = codes_u4.shape
    q = B.QTensor(
        torch.from_numpy(formats.pack_nibbles(codes_u4)).cuda(),
        torch.from_numpy(quant.swizzle_scales(scales_lin)).cuda(),
        torch.zeros(1, dtype=torch.float32, device="cuda"),
        torch.tensor([ts], dtype=torch.float32, device="cuda"),
        rows, K, B.NVFP4_SCALES_MMA)
    return q


def ref_gemm(ac, asc, ta, bc, bsc, tb):
    return gemm.gemm_ref(formats.pack_nibbles(ac), asc, np.float32(ta), formats.pack_nibbles(bc), bsc,
                         np.float32(tb))


@pytest.mark.parametrize("N", [128, 256])
def test_one_hot_layout_probe(N):
    """A single nonzero in A (row i, element k) and in B (row j, element k)
    must land at D[i, j] only, scaled by exactly the block scales of
    (i, k/16) and (j, k/16); every other block carries a different scale."""
    M, K = 128, 512
    rng = np.random.default_rng(0)
    positions = [(0, 0, 0), (1, 1, 1), (37, 63, 200), (127, 64, N - 1), (64, 255, 128 % N), (33, 256, 7),
                 (96, 511, N // 2 + 3), (31, 300, 32), (32, 301, 31)]
    for (i, k, j) in positions:
        j = j % N
        ac = np.zeros((M, K), np.uint8)
        bc = np.zeros((N, K), np.uint8)
        ac[i, k] = 7        # +6
        bc[j, k] = 0xB      # -1.5
        asc = rng.integers(0x30, 0x40, size=(M, K // 16)).astype(np.uint8)
        bsc = rng.integers(0x40, 0x50, size=(N, K // 16)).astype(np.uint8)
        asc[i, k // 16] = 0x41  # 2.25
        bsc[j, k // 16] = 0x3C  # 1.5
        d = B.nvfp4_gemm(make_q(ac, asc, 1.0), make_q(bc, bsc, 1.0), out_dtype=torch.float32).cpu().numpy()
        nz = np.argwhere(d != 0)
        assert nz.tolist() == [[i, j]], ((i, k, j), nz[:5].tolist())
        assert d[i, j] == 6.0 * 2.25 * -1.5 * 1.5, ((i, k, j), d[i, j])


def test_tiny_exact_fp32():
    """K = 64 with unit scales: every FP32 partial sum is exact, so the FP32
    output equals the oracle bit for bit."""
    rng = np.random.default_rng(1)
    M, N, K = 128, 256, 64
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    one = lambda r: np.full((r, K // 16), 0x38, np.uint8)
    d = B.nvfp4_gemm(make_q(ac, one(M), 1.0), make_q(bc, one(N), 1.0), out_dtype=torch.float32).cpu().numpy()
    ref = ref_gemm(ac, one(M), 1.0, bc, one(N), 1.0)
    np.testing.assert_array_equal(d.astype(np.float64), ref)


GEMM_SHAPES = [(128, 256, 256), (256, 512, 1024), (384, 384, 320), (128, 128, 192), (512, 768, 2048),
               (256, 256, 64), (1024, 1280, 1536)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_random_gemm(M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    asc = rng.integers(0x20, 0x60, size=(M, K // 16)).astype(np.uint8)
    bsc = rng.integers(0x20, 0x60, size=(N, K // 16)).astype(np.uint8)
    ta, tb = 0.013, 0.37
    qa, qb = make_q(ac, asc, ta), make_q(bc, bsc, tb)
    ref = ref_gemm(ac, asc, ta, bc, bsc, tb)
    d32 = B.nvfp4_gemm(qa, qb, out_dtype=torch.float32).cpu().numpy()
    assert B.nvfp4_get_status() == B.NVFP4_OK
    assert rel_fro(d32, ref) <= 1e-5
    d16 = B.nvfp4_gemm(qa, qb).float().cpu().numpy()
    assert rel_fro(d16, formats.float64_to_bf16_rne(ref)) <= 1e-3
    assert rel_fro(d16, ref) <= 4e-3  # BF16 output rounding alone


def test_grouped_tile_order_covers_every_tile():
    """A GEMM whose B codes exceed 32 MB with N < M walks B in groups of 16
    block rows (20 block rows here: a group of 16 and a partial one of 4).
    The output, pre-filled with NaN, must be written everywhere, and sampled
    rows of both groups match the oracle."""
    M, N, K = 5120, 4096, 18432  # B codes: 4096 x 18432 / 2 = 36 MiB
    assert N * K // 2 > (32 << 20) and N < M
    rng = np.random.default_rng(31)
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    asc = rng.integers(0x28, 0x48, size=(M, K // 16)).astype(np.uint8)
    bsc = rng.integers(0x28, 0x48, size=(N, K // 16)).astype(np.uint8)
    ta, tb = 0.05, 0.02
    qa, qb = make_q(ac, asc, ta), make_q(bc, bsc, tb)
    d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.nvfp4_gemm(qa, qb, out=d)
    torch.cuda.synchronize()
    assert B.nvfp4_get_status() == B.NVFP4_OK
    assert not torch.isnan(d).any()
    rows = np.array([3, 700, 2047, 3000, 4095, 4100, 4700, 5119])  # block rows 0-15 and 16-19
    ref = ref_gemm(ac[rows], asc[rows], ta, bc, bsc, tb)
    got = d[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    assert rel_fro(got, formats.float64_to_bf16_rne(ref)) <= 1e-3


def test_strided_output():
    rng = np.random.default_rng(3)
    M, N, K = 128, 256, 256
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sc = lambda r: rng.integers(0x30, 0x40, size=(r, K // 16)).astype(np.uint8)
    asc, bsc = sc(M), sc(N)
    out = torch.full((M, N + 64), 7.0, dtype=torch.float32, device="cuda")
    B.nvfp4_gemm(make_q(ac, asc, 1.0), make_q(bc, bsc, 1.0), out=out[:, :N])
    o = out.cpu().numpy()
    assert np.all(o[:, N:] == 7.0)
    assert rel_fro(o[:, :N], ref_gemm(ac, asc, 1.0, bc, bsc, 1.0)) <= 1e-5


@pytest.mark.parametrize("pad", [0, 8, 136])
def test_strided_bf16_output_pair_kernel(pad):
    """BF16 output with a row stride on the CTA-pair kernel (M, N multiples
    of 256), whose epilogue writes 16-column boxes with bulk tensor stores:
    the padding columns stay untouched and every value matches."""
    rng = np.random.default_rng(5 + pad)
    M, N, K = 512, 768, 512
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sc = lambda r: rng.integers(0x30, 0x40, size=(r, K // 16)).astype(np.uint8)
    asc, bsc = sc(M), sc(N)
    out = torch.full((M, N + pad), 7.0, dtype=torch.bfloat16, device="cuda")
    B.nvfp4_gemm(make_q(ac, asc, 0.5), make_q(bc, bsc, 2.0), out=out[:, :N])
    assert B.nvfp4_get_status() == B.NVFP4_OK
    o = out.float().cpu().numpy()
    assert np.all(o[:, N:] == 7.0)
    ref = formats.float64_to_bf16_rne(ref_gemm(ac, asc, 0.5, bc, bsc, 2.0))
    assert rel_fro(o[:, :N], ref) <= 1e-3


@pytest.mark.parametrize("M,N,K", [(512, 768, 512), (128, 256, 320), (384, 384, 256)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_gemm_output_amax_equals_amax_of_output(M, N, K, out_dtype):
    """The epilogue's amax of D (both kernels, both output types) is exactly
    the amax pass over the stored output, and the output itself is the same
    as without it."""
    rng = np.random.default_rng(M + N + K)
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    asc = rng.integers(0x28, 0x48, size=(M, K // 16)).astype(np.uint8)
    bsc = rng.integers(0x28, 0x48, size=(N, K // 16)).astype(np.uint8)
    qa, qb = make_q(ac, asc, 0.75), make_q(bc, bsc, 1.5)
    d, amax = B.nvfp4_gemm_amax(qa, qb, out_dtype=out_dtype)
    plain = B.nvfp4_gemm(qa, qb, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert torch.equal(d, plain)
    want = float(d.float().abs().max().item())
    assert amax.item() == want
    if out_dtype == torch.bfloat16:
        assert B.nvfp4_amax(d, B.NVFP4_AMAX_PLAIN)[0].item() == want
    assert B.nvfp4_get_status() == B.NVFP4_OK


def test_gemm_repeatable():
    rng = np.random.default_rng(4)
    M, N, K = 256, 512, 768
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    asc = rng.integers(0x30, 0x40, size=(M, K // 16)).astype(np.uint8)
    bsc = rng.integers(0x30, 0x40, size=(N, K // 16)).astype(np.uint8)
    qa, qb = make_q(ac, asc, 1.0), make_q(bc, bsc, 1.0)
    a = B.nvfp4_gemm(qa, qb)
    b = B.nvfp4_gemm(qa, qb)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert B.nvfp4_get_status() == B.NVFP4_OK


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (128, 384, 512)])
def test_pipeline_wait_bound_reports_timeout(M, N, K):
    """Failure detection without a GPU fault: the test hook makes one launch
    skip its first stage's loads, so the pipeline waits run out (about 2 s),
    the kernel stops and reports NVFP4_ERR_TIMEOUT, and the next GEMM on the
    same context is correct.  (256x512: CTA-pair kernel; 128x384: 1-CTA.)"""
    import time

    rng = np.random.default_rng(9)
    ac = rng.integers(0, 16, (M, K)).astype(np.uint8)
    bc = rng.integers(0, 16, (N, K)).astype(np.uint8)
    asc = rng.integers(0x30, 0x40, size=(M, K // 16)).astype(np.uint8)
    bsc = rng.integers(0x30, 0x40, size=(N, K // 16)).astype(np.uint8)
    qa, qb = make_q(ac, asc, 1.0), make_q(bc, bsc, 1.0)
    assert B.nvfp4_get_status() == B.NVFP4_OK
    B.nvfp4_debug_stall_next_gemm(True)
    t0 = time.time()
    B.nvfp4_gemm(qa, qb)
    st = B.nvfp4_get_status()
    dt = time.time() - t0
    assert st == B.NVFP4_ERR_TIMEOUT
    assert 1.0 < dt < 30.0
    d = B.nvfp4_gemm(qa, qb, out_dtype=torch.float32).cpu().numpy()
    assert B.nvfp4_get_status() == B.NVFP4_OK
    assert rel_fro(d, ref_gemm(ac, asc, 1.0, bc, bsc, 1.0)) <= 1e-5


@pytest.mark.parametrize("K,N,w2d,rht", [(4096, 4096, True, False), (5120, 5120, False, True),
                                         (8192, 8192, False, False), (8192, 8192, False, True),
                                         (5120, 20480, True, False), (20480, 5120, True, False)])
def test_gemm_sweep_full_size_sampled(K, N, w2d, rht):
    """The GEMM shape sweep at full size (M = 16384, heavy-tailed X ~ t(3),
    W ~ N(0, 0.02)): X quantized 1x16, W with 16x16 blocks or 1x16, with or
    without the Hadamard transform along K on both operands; sampled rows of
    the output against the oracle."""
    from nvfp4_bit_numerics_gb300 import workloads
    from tests.gpu_util import assert_q_equal, f32

    x, w, _ = workloads.gemm_sweep(K, N)
    M = x.shape[0]
    xf, wf = f32(x), f32(w)
    seed = 4
    qx, _ = B.nvfp4_quantize(x.cuda(), B.NVFP4_Q_ROWWISE, rht=rht, seed=seed)
    if w2d:
        qw, _ = B.nvfp4_quantize(w.cuda(), B.NVFP4_Q_2D)
    else:
        qw, _ = B.nvfp4_quantize(w.cuda(), B.NVFP4_Q_ROWWISE, rht=rht, seed=seed)
    d = B.nvfp4_gemm(qx, qw)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(2).choice(M, 8, replace=False))
    ax = quant.amax_rht(xf, seed, axis=1) if rht else quant.tensor_amax(xf)
    rx = quant.quantize_1d(xf, "rne", rht_seed=seed if rht else None, amax=ax, row_ids=rows)
    assert_q_equal(qx, rx, rows=rows, what="X")
    if w2d:
        r2 = quant.quantize_2d(wf)
        rw = dict(codes=r2["codes"], scales=r2["scales"], amax=r2["amax"], ts=r2["ts"])
    else:
        rw = quant.quantize_1d(wf, "rne", rht_seed=seed if rht else None)
    assert_q_equal(qw, rw, what="W")
    ref = gemm.gemm_ref(rx["codes"], rx["scales"], rx["ts"], rw["codes"], rw["scales"], rw["ts"])
    got = d[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    assert rel_fro(got, formats.float64_to_bf16_rne(ref)) <= 1e-3
    if rht:
        # the transform cancels: the product is close to the unquantized X W^T
        exact = xf[rows].astype(np.float64) @ wf.astype(np.float64).T
        assert rel_fro(got, exact) < 0.15


@pytest.mark.parametrize("shapes", [((256, 512, 768), (512, 256, 1024)), ((1024, 256, 512), (256, 512, 256)),
                                    ((384, 256, 256), (256, 256, 512))])
def test_gemm2_equals_two_gemms(shapes):
    """nvfp4_gemm2 gives each product bit-identical to its own nvfp4_gemm, in
    one launch when all four operands have rows % 256 == 0 (the CTA-pair
    kernel's two-problem schedule) and in two otherwise (the last case)."""
    (m0, k0, n0), (m1, k1, n1) = shapes
    g = torch.Generator().manual_seed(17)
    ops = []
    for m, k in ((m0, k0), (n0, k0), (m1, k1), (n1, k1)):
        x = (torch.randn((m, k), generator=g)).to(torch.bfloat16).cuda()
        ops.append(B.nvfp4_quantize(x, B.NVFP4_Q_ROWWISE, B.NVFP4_ROUND_RNE)[0])
    a0, b0, a1, b1 = ops
    # outputs pre-filled with NaN: a tile the schedule skipped would show
    d0 = torch.full((m0, n0), float("nan"), dtype=torch.bfloat16, device="cuda")
    d1 = torch.full((m1, n1), float("nan"), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    n_before = B.nvfp4_kernel_launch_count()
    d0, d1 = B.nvfp4_gemm2(a0, b0, a1, b1, out0=d0, out1=d1)
    torch.cuda.synchronize()
    launches = B.nvfp4_kernel_launch_count() - n_before
    assert B.nvfp4_get_status() == B.NVFP4_OK
    pair = all(r % 256 == 0 for r in (m0, n0, m1, n1))
    assert launches == (1 if pair else 2)
    assert torch.equal(d0, B.nvfp4_gemm(a0, b0))
    assert torch.equal(d1, B.nvfp4_gemm(a1, b1))

