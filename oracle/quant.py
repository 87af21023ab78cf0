"""NVFP4 quantization: tensor scale, block scales, element codes.
TEST INFRASTRUCTURE ONLY.

Pretraining Large Language Models with NVFP4, Resumo técnico §2 (Formato
NVFP4: "Bloco Menor", "Fatores de Escala Precisos", "Escala em Dois Níveis"):
blocks of 16 elements, an E4M3 scale per block, and an FP32 scale per tensor,
so that the largest element of each block (1 of 16, i.e. 6.25%) lands at the
top of the E2M1 range with near-FP8 precision.  §2 item 3 ("Escala
Bidimensional"): weights use 16x16 blocks so that the weight used forward and
its transpose used backward quantize identically.  §2 item 4: gradients are
rounded stochastically, everything else round-to-nearest-even.

Reading of the two-level scale (the pages give no formula; this is the
plainest scheme in which the tensor's largest value maps to E2M1 6 times E4M3
448, and each block's largest value maps to E2M1 6 times its block scale).
All arithmetic is IEEE float32 with round-to-nearest-even, in this order:

  1. amax    = max |x| over the tensor being quantized (after the Hadamard
               transform where one applies)
  2. s_enc   = 2688 / amax              (2688 = 6 * 448; s_enc = 1 if amax == 0)
  3. ts      = 1 / s_enc                (the stored FP32 per-tensor decode scale)
  4. per block b:  sd = amax_b / 6;  E = e4m3_rne_sat(sd * s_enc)
  5. enc     = s_enc / E                (0 when E == 0)
  6. v_i     = x_i * enc
  7. code_i  = E2M1 rounding of v_i     (RNE, or stochastic for gradients)

Decoding: x_i ~ e2m1(code_i) * e4m3(E) * ts.  A non-finite amax is an error
(the GPU path reports it; the oracle raises).
"""

import numpy as np

from . import formats
from .philox import sr_uniform16
from .rht import rht_along_axis, rht_signs

F32 = np.float32


def tensor_amax(x):
    x = np.asarray(x, dtype=np.float32)
    if x.size == 0:
        return F32(0.0)
    return F32(np.max(np.abs(x)))


def tensor_scales(amax):
    """Step 2-3: (s_enc, ts) as float32 from a float32 amax."""
    amax = F32(amax)
    if not np.isfinite(amax):
        raise FloatingPointError("non-finite amax")
    if amax == 0:
        return F32(1.0), F32(1.0)
    s_enc = F32(F32(2688.0) / amax)
    ts = F32(F32(1.0) / s_enc)
    return s_enc, ts


def block_scale_codes(amax_b, s_enc):
    """Step 4-5 for an array of block amaxes: (E codes uint8, enc float32)."""
    amax_b = np.asarray(amax_b, dtype=np.float32)
    sd = (amax_b / F32(6.0)).astype(np.float32)
    E = formats.e4m3_encode_rne_sat((sd * s_enc).astype(np.float32))
    Ef = formats.e4m3_to_float32(E)
    # float32 IEEE results throughout: for a tensor whose amax lies near the
    # bottom of the float range s_enc / E can round to +inf, as a float32
    # division does (numpy would only warn about it)
    with np.errstate(divide="ignore", over="ignore"):
        enc = np.where(E == 0, F32(0.0), (s_enc / np.where(E == 0, F32(1.0), Ef)).astype(np.float32))
    return E, enc.astype(np.float32)


def _encode(v, rounding, seed, stream_id, elem_index):
    if rounding == "rne":
        return formats.e2m1_encode_rne(v)
    if rounding == "sr":
        u = sr_uniform16(seed, stream_id, elem_index)
        return formats.e2m1_encode_sr(v, u)
    raise ValueError(rounding)


def quantize_rows(x, amax, rounding="rne", seed=0, stream_id=0, row_ids=None, n_cols_total=None):
    """1x16 blocks along the last axis of a 2D float32 array.

    ``row_ids`` (optional) are the rows' indices in the full tensor, so that
    stochastic rounding draws the same bits as for the whole tensor; the
    element index is row * n_cols + col in the quantized (output) layout.
    Returns (codes uint8 [R, C] unpacked, E uint8 [R, C/16]).
    """
    x = np.asarray(x, dtype=np.float32)
    R, C = x.shape
    assert C % 16 == 0
    s_enc, _ = tensor_scales(amax)
    xb = x.reshape(R, C // 16, 16)
    amax_b = np.max(np.abs(xb), axis=2) if R * C else np.zeros((R, C // 16), np.float32)
    E, enc = block_scale_codes(amax_b, s_enc)
    v = (xb * enc[:, :, None]).astype(np.float32).reshape(R, C)
    if row_ids is None:
        row_ids = np.arange(R)
    ncol = C if n_cols_total is None else n_cols_total
    elem = (np.asarray(row_ids, dtype=np.uint64)[:, None] * np.uint64(ncol)
            + np.arange(C, dtype=np.uint64)[None, :])
    codes = _encode(v, rounding, seed, stream_id, elem) if R * C else np.zeros((R, C), np.uint8)
    return codes.astype(np.uint8), E


def quantize_1d(x, rounding="rne", seed=0, stream_id=0, rht_seed=None, amax=None, row_ids=None):
    """Quantize a [R, C] tensor with 1x16 blocks along C (the reduction dim).

    With ``rht_seed`` the 16x16 random Hadamard transform is first applied to
    every 16-chunk along C.  ``amax`` is the whole tensor's amax (after the
    transform); when ``row_ids`` selects a subset of rows it must be given.
    Returns dict(codes [R, C/2] packed, scales [R, C/16] E4M3, amax, ts).
    """
    x = np.asarray(x, dtype=np.float32)
    if row_ids is not None:
        assert amax is not None
        x = x[np.asarray(row_ids)]
    return _quantize_selected(x, rounding, seed, stream_id, rht_seed, amax, row_ids)


def _quantize_selected(x, rounding, seed, stream_id, rht_seed, amax, row_ids):
    """quantize_1d on rows already taken from the full tensor (row_ids)."""
    if rht_seed is not None:
        x = rht_along_axis(x, rht_signs(rht_seed), axis=1)
    if amax is None:
        amax = tensor_amax(x)
    codes, E = quantize_rows(x, amax, rounding, seed, stream_id, row_ids)
    _, ts = tensor_scales(amax)
    return dict(codes=formats.pack_nibbles(codes), scales=E, amax=F32(amax), ts=ts)


def quantize_transpose(x, rounding="rne", seed=0, stream_id=0, rht_seed=None, amax=None, col_ids=None):
    """Quantize x^T for a GEMM that reduces over x's rows (tokens).

    x is [M, C]; the result is the [C, M] tensor x^T, optionally transformed
    by the random Hadamard transform along M in 16-token chunks, quantized
    with 1x16 blocks along M.  ``col_ids`` selects output rows (input
    columns).  Same return dict as ``quantize_1d``.
    """
    x = np.asarray(x, dtype=np.float32)
    if col_ids is None:
        return quantize_1d(np.ascontiguousarray(x.T), rounding, seed, stream_id, rht_seed, amax)
    assert amax is not None
    xt = np.ascontiguousarray(x[:, np.asarray(col_ids)].T)
    return _quantize_selected(xt, rounding, seed, stream_id, rht_seed, amax, col_ids)


def quantize_2d(w, amax=None):
    """16x16 block quantization of a weight W [N, K] (RNE).

    One E4M3 scale per 16x16 block.  The codes of W (K-major, for the forward
    GEMM) and of W^T (N-major, for the data-gradient GEMM) are the same
    elements transposed.  Reading: the GEMM consumes one scale per 16
    contiguous elements, so the block scale is replicated into the 16 row
    slots of W's [N, K/16] scale tensor and of W^T's [K, N/16] one.
    Returns dict(codes [N, K/2], scales [N, K/16], codes_t [K, N/2],
    scales_t [K, N/16], scales_2d [N/16, K/16], amax, ts).
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert N % 16 == 0 and K % 16 == 0
    if amax is None:
        amax = tensor_amax(w)
    s_enc, ts = tensor_scales(amax)
    blocks = w.reshape(N // 16, 16, K // 16, 16)
    amax_b = np.max(np.abs(blocks), axis=(1, 3)) if w.size else np.zeros((N // 16, K // 16), np.float32)
    E, enc = block_scale_codes(amax_b, s_enc)
    v = (blocks * enc[:, None, :, None]).astype(np.float32).reshape(N, K)
    codes = formats.e2m1_encode_rne(v)
    return dict(
        codes=formats.pack_nibbles(codes),
        scales=np.repeat(E, 16, axis=0),
        codes_t=formats.pack_nibbles(np.ascontiguousarray(codes.T)),
        scales_t=np.repeat(np.ascontiguousarray(E.T), 16, axis=0),
        scales_2d=E,
        amax=F32(amax),
        ts=ts,
    )


def amax_rht(x, rht_seed, axis, chunk_elems=1 << 21):
    """amax of the tensor after the 16-chunk Hadamard transform along ``axis``
    (processed in slices of whole 16-chunks to bound memory)."""
    x = np.asarray(x, dtype=np.float32)
    signs = rht_signs(rht_seed)
    other = 1 - axis
    n = x.shape[other]
    step = max(1, chunk_elems // max(1, x.shape[axis]))
    best = F32(0.0)
    for s in range(0, n, step):
        part = x[s:s + step] if other == 0 else x[:, s:s + step]
        if part.size:
            best = max(best, F32(np.max(np.abs(rht_along_axis(part, signs, axis)))))
    return F32(best)


def dequantize(q, rows=None):
    """float64 values of a 1x16-scaled tensor dict (codes, scales, ts)."""
    codes, scales = q["codes"], q["scales"]
    if rows is not None:
        codes, scales = codes[rows], scales[rows]
    vals = formats.e2m1_decode(formats.unpack_nibbles(codes))
    sc = np.repeat(formats.e4m3_decode(scales), 16, axis=-1)
    return vals * sc * np.float64(q["ts"])


# ---------------------------------------------------------------------------
# Scale-factor layout consumed by the block-scaled tensor-core MMA
# ---------------------------------------------------------------------------


def swizzled_scale_bytes(rows, cols16):
    return ((rows + 127) // 128) * ((cols16 + 3) // 4) * 512


def swizzle_scales(E):
    """Linear [R, C/16] E4M3 scales -> the MMA's blocked layout (bytes).

    The block-scaled MMA reads scales in tiles of 128 rows x 4 scale columns
    (512 bytes); tiles are stored row-tile-major (all column tiles of rows
    0..127 first).  Inside a tile, row r and scale column c sit at byte
    (r % 32) * 16 + (r // 32) * 4 + c, so that 32 rows x 16 bytes form one
    tensor-memory copy.  Rows are padded to 128 and columns to 4 with zeros.
    (A hardware convention, not from the pages.)
    """
    E = np.asarray(E, dtype=np.uint8)
    R, C = E.shape
    Rp, Cp = (R + 127) // 128 * 128, (C + 3) // 4 * 4
    pad = np.zeros((Rp, Cp), np.uint8)
    pad[:R, :C] = E
    # [rt, r32-group g, r%32, ct, c%4] -> [rt, ct, r%32, g, c%4]
    t = pad.reshape(Rp // 128, 4, 32, Cp // 4, 4).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(t).reshape(-1)


def unswizzle_scales(buf, R, C):
    Rp, Cp = (R + 127) // 128 * 128, (C + 3) // 4 * 4
    t = np.asarray(buf, dtype=np.uint8).reshape(Rp // 128, Cp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(t).reshape(Rp, Cp)[:R, :C]
