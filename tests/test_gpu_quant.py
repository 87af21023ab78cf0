"""GPU parity of the quantize kernels against the oracle: amax, tensor scale,
block scales and packed codes must match bit for bit."""

import numpy as np
import pytest
import torch

from nvfp4_bit_numerics_gb300 import binding as B
from nvfp4_bit_numerics_gb300 import workloads
from oracle import quant
from tests.gpu_util import assert_q_equal, ensure_lib, f32, outlier_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_lib()


SHAPES = [(64, 64), (128, 256), (192, 320), (512, 1024)]


@pytest.mark.parametrize("shape", SHAPES)
def test_amax_variants(shape):
    x = outlier_tensor(*shape, seed=1)
    xg = x.cuda()
    a = B.nvfp4_amax(xg, B.NVFP4_AMAX_PLAIN | B.NVFP4_AMAX_RHT_ROWS | B.NVFP4_AMAX_RHT_COLS, rht_seed=77)
    got = a.cpu().numpy()
    xf = f32(x)
    assert got[0] == quant.tensor_amax(xf)
    assert got[1] == quant.amax_rht(xf, 77, axis=1)
    assert got[2] == quant.amax_rht(xf, 77, axis=0)
    # each variant alone, too
    for flag, slot in ((1, 0), (2, 1), (4, 2)):
        b = B.nvfp4_amax(xg, flag, rht_seed=77)
        assert b.cpu().numpy()[slot] == got[slot]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("rounding", ["rne", "sr"])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("layout", [B.NVFP4_SCALES_MMA, B.NVFP4_SCALES_LINEAR])
def test_rowwise(shape, rounding, rht, layout):
    if layout == B.NVFP4_SCALES_MMA and shape[0] % 128:
        pytest.skip("MMA layout needs rows % 128")
    x = outlier_tensor(*shape, seed=2)
    seed = 0x1234567890ABCDEF
    rnd = B.NVFP4_ROUND_SR if rounding == "sr" else B.NVFP4_ROUND_RNE
    out, _ = B.nvfp4_quantize(x.cuda(), B.NVFP4_Q_ROWWISE, rnd, rht=rht, seed=seed, sr_stream=5, layout=layout)
    ref = quant.quantize_1d(f32(x), rounding, seed=seed, stream_id=5, rht_seed=seed if rht else None)
    assert_q_equal(out, ref, what="rowwise %s rht=%s" % (rounding, rht))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("rounding", ["rne", "sr"])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("layout", [B.NVFP4_SCALES_MMA, B.NVFP4_SCALES_LINEAR])
def test_transpose(shape, rounding, rht, layout):
    if layout == B.NVFP4_SCALES_MMA and shape[1] % 128:
        pytest.skip("MMA layout needs the transposed rows % 128")
    x = outlier_tensor(*shape, seed=3)
    seed = 42
    rnd = B.NVFP4_ROUND_SR if rounding == "sr" else B.NVFP4_ROUND_RNE
    out, _ = B.nvfp4_quantize(x.cuda(), B.NVFP4_Q_TRANSPOSE, rnd, rht=rht, seed=seed, sr_stream=1, layout=layout)
    ref = quant.quantize_transpose(f32(x), rounding, seed=seed, stream_id=1, rht_seed=seed if rht else None)
    assert_q_equal(out, ref, what="transpose %s rht=%s" % (rounding, rht))


@pytest.mark.parametrize("shape", [(128, 256), (256, 384), (512, 1024)])
@pytest.mark.parametrize("rounding", ["rne", "sr"])
def test_fused_rowwise_and_transpose(shape, rounding):
    x = outlier_tensor(*shape, seed=4)
    seed = 9
    rnd = B.NVFP4_ROUND_SR if rounding == "sr" else B.NVFP4_ROUND_RNE
    out, out_t = B.nvfp4_quantize(x.cuda(), B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, rnd, rht=True, seed=seed, sr_stream=0,
                                  sr_stream_t=1)
    xf = f32(x)
    ref = quant.quantize_1d(xf, rounding, seed=seed, stream_id=0)
    ref_t = quant.quantize_transpose(xf, rounding, seed=seed, stream_id=1, rht_seed=seed)
    assert_q_equal(out, ref, what="fused rowwise")
    assert_q_equal(out_t, ref_t, what="fused transpose")


@pytest.mark.parametrize("shape", [(64, 128), (192, 256), (320, 192)])
@pytest.mark.parametrize("rounding", ["rne", "sr"])
def test_fused_ragged_tiles_linear_layout(shape, rounding):
    """Token counts that end in a half tile (rows % 128 == 64), linear scale
    layout on both outputs."""
    x = outlier_tensor(*shape, seed=14)
    seed = 21
    rnd = B.NVFP4_ROUND_SR if rounding == "sr" else B.NVFP4_ROUND_RNE
    out, out_t = B.nvfp4_quantize(x.cuda(), B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, rnd, rht=True, seed=seed, sr_stream=4,
                                  sr_stream_t=6, layout=B.NVFP4_SCALES_LINEAR)
    xf = f32(x)
    assert_q_equal(out, quant.quantize_1d(xf, rounding, seed=seed, stream_id=4), what="ragged rowwise")
    assert_q_equal(out_t, quant.quantize_transpose(xf, rounding, seed=seed, stream_id=6, rht_seed=seed),
                   what="ragged transpose")


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (512, 1024), (384, 128), (128, 192), (64, 64)])
def test_quant_2d(shape):
    w = outlier_tensor(*shape, seed=5, sigma=0.02)
    layout = B.NVFP4_SCALES_MMA if shape[0] % 128 == 0 and shape[1] % 128 == 0 else B.NVFP4_SCALES_LINEAR
    out, out_t = B.nvfp4_quantize(w.cuda(), B.NVFP4_Q_2D, layout=layout)
    ref = quant.quantize_2d(f32(w))
    assert_q_equal(out, dict(codes=ref["codes"], scales=ref["scales"], amax=ref["amax"], ts=ref["ts"]), what="W")
    assert_q_equal(out_t, dict(codes=ref["codes_t"], scales=ref["scales_t"], amax=ref["amax"], ts=ref["ts"]),
                   what="W^T")


def test_edge_values_and_ties():
    """Exact E2M1 midpoints after scaling, subnormal bf16 inputs, +-0, the
    largest bf16 values: the hardware conversions must agree with the
    format definitions the oracle implements."""
    rng = np.random.default_rng(6)
    rows, cols = 128, 512
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    # blocks whose max is 6 * 2^k make enc a power of two: midpoints stay exact
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0, 0.1, -0.1, 0.0, -0.0, 6.0, 3.0])
    for r in range(0, 32):
        blk = x[r, :16]
        blk[:] = mids * 2.0 ** (r - 16)
        blk[14] = 6.0 * 2.0 ** (r - 16)
    x[40, :64] = np.float32(1e-39)  # bf16 subnormals
    x[41, :16] = -np.float32(2.0 ** -133)
    x[42, :16] = 0.0
    x[43, 16:32] = -0.0
    x[44, :8] = 3.0e38
    x[44, 8:16] = -3.0e38
    xb = workloads.to_bf16(x)
    xf = f32(xb)
    for rnd, name in ((B.NVFP4_ROUND_RNE, "rne"), (B.NVFP4_ROUND_SR, "sr")):
        out, _ = B.nvfp4_quantize(xb.cuda(), B.NVFP4_Q_ROWWISE, rnd, seed=3, sr_stream=2)
        ref = quant.quantize_1d(xf, name, seed=3, stream_id=2)
        assert_q_equal(out, ref, what="edge " + name)


def test_subnormal_only_blocks_of_a_tiny_tensor():
    """Blocks that hold nothing but BF16 subnormals, in a tensor whose max is
    so small that those blocks get a nonzero E4M3 scale: every block max (the
    BF16-packed maxima of the rowwise blocks, the float maxima of the
    transposed blocks, the sums taken for the transformed blocks) must see the
    subnormals, not flush them.  Their enc overflows to inf, so their codes
    saturate at +-6 on both sides."""
    rng = np.random.default_rng(12)
    rows, cols = 128, 256
    x = (rng.standard_normal((rows, cols)) * 1e-34).astype(np.float32)
    x[0, 0] = 1e-33
    i = np.arange(16)
    x[3, 16:32] = np.float32(2.0 ** -129) * (1 + i % 3)      # rowwise blocks
    x[5, 32:48] = -np.float32(2.0 ** -130) * (1 + i % 5)
    x[16:32, 64] = np.float32(2.0 ** -129) * (1 + i % 4)     # a transposed block
    x[32:48, 100] = 0.0                                      # transformed: all 16 outputs +-2^-127
    x[40, 100] = np.float32(2.0 ** -125)
    xb = workloads.to_bf16(x)
    xf = f32(xb)
    assert np.all(np.abs(xf[3, 16:32]) < 2.0 ** -126) and np.all(xf[3, 16:32] != 0)
    ref = quant.quantize_1d(xf, "rne")
    for rht in (False, True):
        ref_t = quant.quantize_transpose(xf, "rne", rht_seed=5 if rht else None)
        out, out_t = B.nvfp4_quantize(xb.cuda(), B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, B.NVFP4_ROUND_RNE, rht=rht, seed=5)
        assert_q_equal(out, ref, what="fused rowwise rht=%s" % rht)
        assert_q_equal(out_t, ref_t, what="fused transpose rht=%s" % rht)
        out_t, _ = B.nvfp4_quantize(xb.cuda(), B.NVFP4_Q_TRANSPOSE, B.NVFP4_ROUND_RNE, rht=rht, seed=5)
        assert_q_equal(out_t, ref_t, what="transpose rht=%s" % rht)
    out, _ = B.nvfp4_quantize(xb.cuda(), B.NVFP4_Q_ROWWISE, B.NVFP4_ROUND_RNE)
    assert_q_equal(out, ref, what="rowwise")
    for blk in ((3, 1), (5, 2)):
        assert ref["scales"][blk] != 0


def test_zero_tensor():
    """amax = 0: s_enc = ts = 1 and every scale is 0.  The rowwise codes are
    +0; the Hadamard sign flips give signed zeros in the transposed output,
    whose codes (0x0 or 0x8) must match the oracle's."""
    x = torch.zeros(128, 256, dtype=torch.bfloat16)
    out, out_t = B.nvfp4_quantize(x.cuda(), B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, rht=True, seed=1)
    torch.cuda.synchronize()
    for q in (out, out_t):
        assert q.tensor_scale.item() == 1.0 and q.amax.item() == 0.0
        assert int(q.scales.count_nonzero()) == 0
    assert int(out.codes.count_nonzero()) == 0
    assert_q_equal(out_t, quant.quantize_transpose(f32(x), "rne", rht_seed=1), what="zero transpose")
    assert B.nvfp4_get_status() == B.NVFP4_OK


def test_empty_tensor_amax():
    """An empty tensor (no rows) has amax 0 in every slot (the slots are
    zeroed and nothing is launched), and the status stays clean."""
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    out = torch.full((3,), 5.0, dtype=torch.float32, device="cuda")
    B.nvfp4_amax(x, B.NVFP4_AMAX_PLAIN | B.NVFP4_AMAX_RHT_ROWS | B.NVFP4_AMAX_RHT_COLS, rht_seed=1, out=out)
    torch.cuda.synchronize()
    assert out.tolist() == [0.0, 0.0, 0.0]
    assert B.nvfp4_get_status() == B.NVFP4_OK


def test_nonfinite_sets_status():
    x = torch.randn(128, 256).to(torch.bfloat16)
    x[7, 9] = float("inf")
    B.nvfp4_get_status()  # clear
    B.nvfp4_quantize(x.cuda(), B.NVFP4_Q_ROWWISE)
    assert B.nvfp4_get_status() == B.NVFP4_ERR_NONFINITE
    assert B.nvfp4_get_status() == B.NVFP4_OK  # read clears
    x[7, 9] = float("nan")
    B.nvfp4_amax(x.cuda(), B.NVFP4_AMAX_PLAIN)
    assert B.nvfp4_get_status() == B.NVFP4_ERR_NONFINITE


def test_deterministic_and_padding_untouched():
    """Same seed -> same bits; MMA scale buffers are fully written."""
    x = outlier_tensor(256, 512, seed=7).cuda()
    a, _ = B.nvfp4_quantize(x, B.NVFP4_Q_ROWWISE, B.NVFP4_ROUND_SR, seed=11)
    b = B.empty_qtensor(256, 512)
    b.codes.fill_(0xAA)
    b.scales.fill_(0xAA)
    B.nvfp4_quantize(x, B.NVFP4_Q_ROWWISE, B.NVFP4_ROUND_SR, seed=11, out=b)
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)


@pytest.mark.parametrize("rows,cols", [(8192, 5120), (8192, 20480)])
def test_full_size_quant_sweep_sampled(rows, cols):
    """The quantize-only sweep at full size: the amaxes over the whole tensor
    exactly, and the codes/scales of sampled rows (rowwise SR with the
    transform along the row) and sampled transposed rows (RHT + RNE)."""
    a, b = workloads.quant_sweep()
    x = a if cols == 5120 else b
    xf = f32(x)
    xg = x.cuda()
    seed = 2024
    amax = B.nvfp4_amax(xg, 7, rht_seed=seed).cpu().numpy()
    ref_amax = [quant.tensor_amax(xf), quant.amax_rht(xf, seed, axis=1), quant.amax_rht(xf, seed, axis=0)]
    for i in range(3):
        assert amax[i] == ref_amax[i], (i, amax[i], ref_amax[i])
    rng = np.random.default_rng(0)
    rows_s = np.sort(rng.choice(rows, 24, replace=False))
    cols_s = np.sort(rng.choice(cols, 24, replace=False))
    out, _ = B.nvfp4_quantize(xg, B.NVFP4_Q_ROWWISE, B.NVFP4_ROUND_SR, rht=True, seed=seed, sr_stream=3)
    ref = quant.quantize_1d(xf, "sr", seed=seed, stream_id=3, rht_seed=seed, amax=ref_amax[1], row_ids=rows_s)
    assert_q_equal(out, ref, rows=rows_s, what="full rowwise")
    o2, o2t = B.nvfp4_quantize(xg, B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, B.NVFP4_ROUND_RNE, rht=True, seed=seed)
    ref_t = quant.quantize_transpose(xf, "rne", rht_seed=seed, amax=ref_amax[2], col_ids=cols_s)
    assert_q_equal(o2t, ref_t, rows=cols_s, what="full transpose")
    ref_r = quant.quantize_1d(xf, "rne", amax=ref_amax[0], row_ids=rows_s)
    assert_q_equal(o2, ref_r, rows=rows_s, what="full fused rowwise")
    w2, w2t = B.nvfp4_quantize(xg, B.NVFP4_Q_2D)
    # rows 0..1023 hold whole 16x16 blocks; the scale uses the full tensor's amax
    ref2 = quant.quantize_2d(xf[:1024, :], amax=ref_amax[0])
    assert np.array_equal(w2.codes[:1024].cpu().numpy(), ref2["codes"])
    assert np.array_equal(w2t.codes[:, :512].cpu().numpy(), ref2["codes_t"])
