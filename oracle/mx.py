"""MXFP4: E2M1 elements in blocks of 32 with power-of-two (UE8M0) scales.
TEST INFRASTRUCTURE ONLY.

Pretraining Large Language Models with NVFP4, Resumo técnico §1 ("Limitações
de Formatos Existentes") and §2 ("Fatores de Escala Precisos"): the
microscaling format the method is compared with, MXFP4, scales blocks of 32
elements by powers of two (UE8M0), which can waste dynamic range and saturate
large values; §3 ("Validação de NVFP4 vs. MXFP4") compares the two.  The pages
give no formula; the reading is the OCP Microscaling Formats v1.0 one for an
E2M1 element type (largest element exponent 2, since 6 = 1.5 * 2^2):

  1. amax_b = max |x| over the block of 32 consecutive elements along the
              reduction (last) dimension
  2. E      = floor(log2(amax_b)) - 2 + 127, clamped to [0, 254]; E = 0 for
              amax_b = 0                       (the UE8M0 code; 255 is NaN)
  3. v_i    = x_i * 2^(127 - E)                (one float32 multiply, RNE;
              2^(127 - E) is a float32, subnormal at E = 254)
  4. code_i = E2M1 round-to-nearest-even of v_i, saturating at +-6

so the block's largest value lands in [4, 8) and anything above 6 saturates.
There is no per-tensor scale.  Decoding: x_i ~ e2m1(code_i) * 2^(E - 127).
"""

import numpy as np

from . import formats

F32 = np.float32
BLOCK = 32


def e8m0_decode(codes):
    """Value of each UE8M0 code as float64: 2^(c - 127), NaN for 0xFF."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, c - 127))


def floor_log2(a):
    """floor(log2(a)) of positive float32 values, exactly (frexp gives
    a = m 2^e with m in [0.5, 1), so floor(log2 a) = e - 1; subnormals
    included)."""
    _, e = np.frexp(np.asarray(a, dtype=np.float64))
    return e.astype(np.int64) - 1


def block_scale_codes(amax_b):
    """UE8M0 codes of float32 block amaxes (step 2 above)."""
    a = np.asarray(amax_b, dtype=F32)
    code = np.where(a > 0, floor_log2(np.where(a > 0, a, F32(1))) - 2 + 127, 0)
    return np.clip(code, 0, 254).astype(np.uint8)


def scale_multiplier(codes):
    """The float32 2^(127 - E) of each code (exact: 2^-127 is a float32
    subnormal, 2^127 a normal)."""
    return np.ldexp(np.float64(1.0), 127 - np.asarray(codes, dtype=np.int64)).astype(F32)


def quantize_mx(x):
    """MXFP4 rowwise: x float32 [rows, cols], cols % 32 == 0.
    Returns dict(codes=[rows, cols/2] packed, scales=[rows, cols/32] UE8M0)."""
    x = np.asarray(x, dtype=F32)
    rows, cols = x.shape
    assert cols % BLOCK == 0
    xb = x.reshape(rows, cols // BLOCK, BLOCK)
    amax_b = np.max(np.abs(xb), axis=-1)
    E = block_scale_codes(amax_b)
    v = (xb * scale_multiplier(E)[..., None]).astype(F32)  # one float32 rounding
    codes = formats.e2m1_encode_rne(v.reshape(rows, cols))
    return dict(codes=formats.pack_nibbles(codes), scales=E)


def dequantize_mx(q):
    vals = formats.e2m1_decode(formats.unpack_nibbles(q["codes"]))
    return vals * np.repeat(e8m0_decode(q["scales"]), BLOCK, axis=-1)


def gemm_mx_ref(a, b):
    """D = A B^T in float64 on dequantized MXFP4 operands A [M, K], B [N, K]
    (the same definition as the NVFP4 GEMM, with UE8M0 scales per 32)."""
    return dequantize_mx(a) @ dequantize_mx(b).T
