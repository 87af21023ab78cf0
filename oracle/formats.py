"""E2M1 and E4M3 number formats, and 4-bit packing.  TEST INFRASTRUCTURE ONLY.

Pretraining Large Language Models with NVFP4, Resumo técnico §2 (Formato
NVFP4): elements are 4-bit floats in blocks of 16, each block has an E4M3
scale, and the tensor has a second, FP32 scale.  The pages name the formats
but not their bits; the bit layouts below are the OCP ones:

* E2M1 (OCP Microscaling Formats v1.0, FP4 element): 1 sign bit, 2 exponent
  bits (bias 1), 1 mantissa bit, no inf/NaN.  Magnitudes {0, .5, 1, 1.5, 2, 3,
  4, 6}.
* E4M3 "FN" (OCP 8-bit Floating Point): 1 sign, 4 exponent bits (bias 7), 3
  mantissa bits, subnormals, max 448, no inf, NaN = S.1111.111.  Block scales
  are non-negative and saturate to 448.
"""

import numpy as np

# ---------------------------------------------------------------------------
# E2M1
# ---------------------------------------------------------------------------


def e2m1_decode(codes):
    """Value of each 4-bit code (uint8 array, low nibble used), as float64.

    code = s·8 + e·2 + m; value = (-1)^s · (e == 0 ? 0.5·m : 2^(e-1)·(1 + m/2)).
    """
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e.astype(np.int64) - 1))
    return np.where(s == 1, -mag, mag)


def e2m1_magnitudes():
    """The eight non-negative E2M1 values, in code order 0..7."""
    return e2m1_decode(np.arange(8, dtype=np.uint8))


def e2m1_encode_rne(v):
    """Round float32 values to E2M1 codes, round-to-nearest-even, saturating.

    Round-to-nearest-even is the deterministic rounding the method keeps for
    weights and activations (Resumo técnico §2, item 4, which names it as the
    rounding that stochastic rounding replaces for gradients).

    Worked binade by binade: the E2M1 spacing is 0.5 on [0, 2), 1 on [2, 4)
    and 2 on [4, 8); within a binade the value is spacing·rint(|v|/spacing),
    and rint's ties-to-even integer is the even-mantissa neighbour.  Anything
    that rounds above 6 saturates to 6.  The sign is kept, so a negative value
    that rounds to zero gives code 0x8.  |v|/spacing is exact (power of two).
    """
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    spacing = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    q = np.rint(a / spacing) * spacing
    q = np.minimum(q, 6.0)
    # value -> code: magnitudes are strictly increasing in the code
    mags = e2m1_magnitudes()
    mag_code = np.searchsorted(mags, q).astype(np.uint8)
    assert np.all(mags[mag_code] == q)
    sign = np.signbit(v).astype(np.uint8)
    return (sign << 3) | mag_code


def e2m1_sr_bracket(a):
    """For |v| in [0, 6): the grid neighbours lo <= |v| < hi as code indices.

    Returns (lo_code, lo, hi) with lo, hi float64 grid values.
    """
    mags = e2m1_magnitudes()
    lo_code = np.searchsorted(mags, a, side="right") - 1
    lo_code = np.clip(lo_code, 0, 6)
    return lo_code.astype(np.uint8), mags[lo_code], mags[lo_code + 1]


def e2m1_encode_sr(v, u16):
    """Stochastic rounding of float32 values to E2M1 codes.

    Resumo técnico §2, item 4 (stochastic rounding on gradients only) and
    O essencial §5 (round up or down with a probability): the value rounds to
    its upper grid neighbour with probability equal to its fractional distance
    from the lower one, so the rounding is unbiased.

    Reading (the pages give no bit budget): the probability is realised with a
    16-bit uniform u per element, rounding up iff u < frac·2^16, so that
    P(up) = ceil(frac·2^16)/2^16.  frac = (|v| - lo)/(hi - lo) is exact in
    float32 (the subtraction is exact by Sterbenz's lemma or because lo is 0,
    and hi - lo is a power of two).  |v| >= 6 saturates to 6.  Sign is kept.
    """
    v = np.asarray(v, dtype=np.float32)
    u16 = np.asarray(u16, dtype=np.uint32)
    a32 = np.abs(v)
    sat = a32 >= np.float32(6.0)
    a_in = np.where(sat, np.float32(0.0), a32)
    lo_code, lo, hi = e2m1_sr_bracket(a_in.astype(np.float64))
    step = (hi - lo).astype(np.float32)
    frac = (a_in - lo.astype(np.float32)) * (np.float32(1.0) / step)
    up = u16.astype(np.float32) < frac * np.float32(65536.0)
    mag_code = np.where(sat, np.uint8(7), lo_code + up.astype(np.uint8)).astype(np.uint8)
    sign = np.signbit(v).astype(np.uint8)
    return (sign << 3) | mag_code


def pack_nibbles(codes):
    """Pack 4-bit codes two per byte along the last axis.

    Byte j holds element 2j in bits 0-3 and element 2j+1 in bits 4-7 (the
    little-endian sub-byte order; the pages do not fix one).
    """
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_nibbles(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# ---------------------------------------------------------------------------
# E4M3 (OCP "FN" variant)
# ---------------------------------------------------------------------------


def e4m3_decode(codes):
    """Value of each E4M3 code as float64 (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8)
    s = (c >> 7) & 1
    e = ((c >> 3) & 0xF).astype(np.int64)
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


E4M3_MAX = 448.0


def e4m3_encode_rne_sat(x):
    """Non-negative float32 -> E4M3 code, round-to-nearest-even, saturating at 448.

    Nearest of the 127 finite non-negative E4M3 values (codes 0..126 are
    increasing in value); on a tie the code with the even mantissa wins.
    Values above 448 give 448 (0x7E).  Input must be finite and >= 0.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    assert np.all(x >= 0) and np.all(np.isfinite(x))
    table = e4m3_decode(np.arange(127, dtype=np.uint8))
    hi = np.clip(np.searchsorted(table, x, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_hi = np.abs(table[hi] - x)
    d_lo = np.abs(x - table[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    code = np.where(x >= E4M3_MAX, np.uint8(0x7E), code)
    return code


def e4m3_to_float32(codes):
    return e4m3_decode(codes).astype(np.float32)


# ---------------------------------------------------------------------------
# BF16 helpers (inputs are BF16; the oracle holds them as float32 values)
# ---------------------------------------------------------------------------


def bf16_bits_to_float32(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def float64_to_bf16_rne(x):
    """Round float64 values to BF16 (RNE), returned as float64 values.

    Goes through float32 only when that is exact for the final result: the
    rounding is done on the float64 value directly with the BF16 spacing.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    m, e = np.frexp(x[nz])  # x = m·2^e, 0.5 <= |m| < 1
    # BF16 keeps 8 significant bits; min normal exponent -126 (frexp e = -125)
    e = np.maximum(e, -125)
    scale = np.ldexp(1.0, e - 8)
    out[nz] = np.rint(x[nz] / scale) * scale
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out
