// device_common.cuh -- NVFP4 device primitives for sm_103a.
//
// Number formats, the two-level scale, the 16-point Hadamard transform and
// Philox4x32-10, as used by the quantize kernels.  Method: "Pretraining Large
// Language Models with NVFP4" (gist.science summary), Resumo técnico §2
// Metodologia (NVFP4 format, two-level scaling, random Hadamard transform,
// 2D weight blocks, stochastic rounding).  Bit layouts: OCP Microscaling
// Formats v1.0 (E2M1) and OCP 8-bit Floating Point (E4M3).
//
// Every float operation of the scale chain is an explicit IEEE
// round-to-nearest-even intrinsic (__fmul_rn, __fdiv_rn, __fadd_rn), so the
// results do not depend on FMA contraction or fast-math flags.
#pragma once

#include <cstdint>
#include <cuda_fp8.h>

namespace nvfp4 {

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// ---------------------------------------------------------------------------
// BF16 unpacking: a 16-byte vector holds 8 bf16 values
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4& q, float* v) {
  v[0] = bf16lo(q.x); v[1] = bf16hi(q.x);
  v[2] = bf16lo(q.y); v[3] = bf16hi(q.y);
  v[4] = bf16lo(q.z); v[5] = bf16hi(q.z);
  v[6] = bf16lo(q.w); v[7] = bf16hi(q.w);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// |x| as ordered unsigned bits: for non-negative floats (and NaN above inf)
// integer order equals float order, so max over bits is an exact amax.
__device__ __forceinline__ uint32_t abs_bits(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

// ---------------------------------------------------------------------------
// E4M3 block scale
// ---------------------------------------------------------------------------
// float -> E4M3 code, round-to-nearest-even, saturating to 448 (x >= 0).
__device__ __forceinline__ uint32_t e4m3_rn_satfinite(float x) {
  return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// E4M3 code -> float, exact: bias 7, 3 mantissa bits, subnormal step 2^-9.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : __uint_as_float(0x3B000000u /*2^-9*/) * (float)m;
}

// Per-tensor encode scale s_enc = 2688 / amax (6 * 448), 1 for amax == 0.
__device__ __forceinline__ float tensor_encode_scale(float amax) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(2688.0f, amax);
}
__device__ __forceinline__ float tensor_decode_scale(float s_enc) { return __fdiv_rn(1.0f, s_enc); }

// fl(a / 6) for a >= 0.  From 2^-120 up: q = fl(a * fl(1/6)), then one
// correction with the exact remainder r = fma(-q, 6, a) and q' = fma(r,
// fl(1/6), q) -- the remainder-correction step of FMA-based division
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990) applied to the
// constant divisor 6.  q' equals the correctly rounded quotient for every
// float in [2^-120, inf) (checked exhaustively against a double-precision
// division); below, where a / 6 nears the subnormal range, the IEEE division
// itself.
__device__ __forceinline__ float div6_rn(float a) {
  if (a < 0x1p-120f) return __fdiv_rn(a, 6.0f);
  const float r6 = 1.0f / 6.0f;
  const float q = __fmul_rn(a, r6);
  return __fmaf_rn(__fmaf_rn(-q, 6.0f, a), r6, q);
}

// Block scale from the block amax: E = e4m3(fl(fl(amax_b / 6) * s_enc)),
// enc = fl(s_enc / e4m3(E)) or 0 when E == 0.
__device__ __forceinline__ void block_scale(float amax_b, float s_enc, uint32_t& E, float& enc) {
  E = e4m3_rn_satfinite(__fmul_rn(div6_rn(amax_b), s_enc));
  enc = E ? __fdiv_rn(s_enc, e4m3_value(E)) : 0.0f;
}

// enc of every E4M3 code for one tensor (128 entries; codes 0 and 0x7F,
// which never occurs under satfinite, hold 0); the thread with index i in
// [0, 128) fills entry i, other indices do nothing.
__device__ __forceinline__ void fill_enc_table(float* tab, float s_enc, int i) {
  if (i >= 0 && i < 128) tab[i] = (i == 0 || i == 0x7F) ? 0.0f : __fdiv_rn(s_enc, e4m3_value((uint32_t)i));
}

// block_scale with enc taken from the tensor's table.
__device__ __forceinline__ void block_scale_tab(float amax_b, float s_enc, const float* tab, uint32_t& E,
                                                float& enc) {
  E = e4m3_rn_satfinite(__fmul_rn(div6_rn(amax_b), s_enc));
  enc = tab[E];
}

// ---------------------------------------------------------------------------
// E2M1 element codes (s.ee.m; magnitudes 0 .5 1 1.5 2 3 4 6)
// ---------------------------------------------------------------------------
// Eight values -> four bytes; element 2j in bits 0-3 of byte j.  cvt packs its
// first source operand into the high nibble.  RNE, saturating at +-6, sign
// kept for values that round to zero.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float* v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// ---------------------------------------------------------------------------
// Packed float pairs: two IEEE float32 values in one 64-bit register pair,
// operated on by the paired instructions (add/sub/mul/fma .rn.f32x2), which
// round each half exactly as the scalar instruction would.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo_bits, uint32_t hi_bits) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo_bits), "r"(hi_bits));
  return r;
}
__device__ __forceinline__ float f2_lo(uint64_t p) { return __uint_as_float((uint32_t)p); }
__device__ __forceinline__ float f2_hi(uint64_t p) { return __uint_as_float((uint32_t)(p >> 32)); }
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// a * b + c in one rounding per half
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// The two BF16 values of a 32-bit word as a float pair (element 0 low).
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t w) { return f2_pack(w << 16, w & 0xFFFF0000u); }

// max(|a|, |b|) of each BF16 half (the sign of the result is not used).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Stochastic rounding of 16 values to E2M1 codes (8 bytes).  The rule: with
// lo the lower grid neighbour of |s| (grid 0 .5 1 1.5 2 3 4 6) and step the
// grid spacing there, frac = (|s| - lo) / step, and |s| rounds up iff
// u < frac * 2^16 (u the element's 16-bit uniform); the sign is kept and
// values above 6 give 6.  The caller passes nu = 2^22 - 1 - 64 u.
// y = RU(|s| * 2^-126) maps the grid onto float bit patterns: .5, 1, 1.5,
// 2, 3, 4, 6 become 1, 2, 3, 4, 5, 6, 7 times 2^22 (the grid below 1 lands in
// the subnormals, whose spacing is uniform like the grid's there), so in
// every binade the lower 22 bits of y are m = ceil(frac * 2^22), exact above
// 1 and rounded up by RU below.  For an integer n, n < x <=> n < ceil(x), so
// 64 u < frac * 2^22 <=> 64 u < m <=> m + nu >= 2^22: adding nu carries into
// bit 22 exactly when the value rounds up, and clearing the lower 22 bits
// leaves the lower or the upper neighbour (a carry out of the mantissa steps
// the exponent, the next grid point as well).  Scaling back by 2^126 is
// exact; the saturating conversion turns results above 6 into 6.  Non-finite
// inputs (which the amax pass reports) give unspecified codes.
__device__ __forceinline__ float mul_ru_2m126(float a) {
  float y;
  asm("mul.rp.f32 %0, %1, 0f00800000;" : "=f"(y) : "f"(a));
  return y;
}
__device__ __forceinline__ uint2 sr_codes16(const float* s, const uint32_t* nu) {
  const uint64_t k126 = f2_pack(0x7E800000u, 0x7E800000u);
  float z[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float a = s[2 * j], b = s[2 * j + 1];
    const uint32_t ra = (__float_as_uint(mul_ru_2m126(fabsf(a))) + nu[2 * j]) & 0xFFC00000u;
    const uint32_t rb = (__float_as_uint(mul_ru_2m126(fabsf(b))) + nu[2 * j + 1]) & 0xFFC00000u;
    const uint64_t zz = f2_mul(f2_pack(ra, rb), k126);
    z[2 * j] = __uint_as_float((uint32_t)zz | (__float_as_uint(a) & 0x80000000u));
    z[2 * j + 1] = __uint_as_float((uint32_t)(zz >> 32) | (__float_as_uint(b) & 0x80000000u));
  }
  return make_uint2(e2m1x8_rn(z), e2m1x8_rn(z + 8));
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of
// (c0,c1,c2,c3) -> (hi(M1 c2)^c1^k0, lo(M1 c2), hi(M0 c0)^c3^k1, lo(M0 c0)),
// the key bumped by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
struct u32x4 {
  uint32_t x, y, z, w;
};

// With the key schedule computed inline (for calls made once per thread).
__device__ __forceinline__ u32x4 philox4x32_10_seed(u32x4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)c.x * 0xD2511F53u, p1 = (uint64_t)c.z * 0xCD9E8D57u;
    c = u32x4{(uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1, (uint32_t)p0};
  }
  return c;
}

// The ten round keys of a 64-bit seed (round r uses lo32(seed) + r W0 and
// hi32(seed) + r W1), computed on the host and passed as a __grid_constant__
// kernel parameter, so that each key is a constant-bank operand of its XOR
// instead of an add repeated in every call.
struct PhiloxKey {
  uint32_t k[20];
};
inline PhiloxKey philox_key(uint64_t seed) {
  PhiloxKey key;
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    key.k[2 * r] = k0;
    key.k[2 * r + 1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return key;
}

__device__ __forceinline__ u32x4 philox4x32_10(u32x4 c, const PhiloxKey& key) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)c.x * 0xD2511F53u, p1 = (uint64_t)c.z * 0xCD9E8D57u;
    c = u32x4{(uint32_t)(p1 >> 32) ^ c.y ^ key.k[2 * r], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ key.k[2 * r + 1],
              (uint32_t)p0};
  }
  return c;
}

// The stochastic-rounding inputs nu = 2^22 - 1 - 64 u of 16 consecutive
// elements starting at e0 (e0 % 8 == 0): their uniforms u come from two
// Philox calls with counters (e0/8, e0/8 + 1), low half of each word first.
__device__ __forceinline__ void sr_nu16(const PhiloxKey& key, uint32_t stream, uint64_t e0, uint32_t* nu) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint64_t g = (e0 >> 3) + h;
    const u32x4 w = philox4x32_10(u32x4{(uint32_t)g, (uint32_t)(g >> 32), stream, 0u}, key);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      nu[8 * h + 2 * j] = 0x3FFFFFu - ((ws[j] & 0xFFFFu) << 6);
      nu[8 * h + 2 * j + 1] = 0x3FFFFFu - ((ws[j] >> 16) << 6);
    }
  }
}

// Hadamard sign mask: bit j set -> sign s_j = -1.  Word 0 of
// Philox(seed, (0, 0, 2, 0)), low 16 bits.
constexpr uint32_t kRhtStream = 2;
__device__ __forceinline__ uint32_t rht_sign_mask(uint64_t seed) {
  return philox4x32_10_seed(u32x4{0u, 0u, kRhtStream, 0u}, (uint32_t)seed, (uint32_t)(seed >> 32)).x & 0xFFFFu;
}

// NaN-propagating maximum of three floats (a NaN anywhere makes the result
// NaN, so it keeps the non-finite detection of a bit-pattern max).
__device__ __forceinline__ float fmax_nan3(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Sign flips of Q on packed BF16 words of row (token) j: both halves of a
// word belong to row j, so one XOR flips both.
__device__ __forceinline__ uint32_t rht_sign_word(uint32_t sign_mask, int j) {
  return ((sign_mask >> j) & 1u) * 0x80008000u;
}

// Q = 1/4 H16 diag(s) on 16 values in registers: sign flips (exact), the
// in-place butterfly with strides 1, 2, 4, 8 (which sums the products
// H[i][j] s_j x_j as a pairwise tree in index order), then * 0.25.  A zero
// has no sign in Q x, so exact-zero outputs are made +0 (adding +0 does
// that and leaves every other value unchanged); the butterfly and other
// summation orders differ only in the sign of exact zeros.
__device__ __forceinline__ void rht16_unsigned(float* v);
__device__ __forceinline__ void rht16(float* v, uint32_t sign_mask) {
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(__float_as_uint(v[j]) ^ (((sign_mask >> j) & 1u) << 31));
  rht16_unsigned(v);
}

// rht16 for values whose signs were already flipped (rht_sign_word).
__device__ __forceinline__ void rht16_unsigned(float* v) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
  // v * 0.25 + 0 in one rounding: equal to the product rounded and then
  // +0 added except where v / 4 underflows to zero (|v| <= 2^-148), which
  // sums of BF16 values (multiples of 2^-133) never reach.
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmaf_rn(v[j], 0.25f, 0.0f);
}

// ---------------------------------------------------------------------------
// One 1x16 block: amax_b, scale, 16 codes -> (8 code bytes as uint2, E)
// ---------------------------------------------------------------------------
// enc_tab: the tensor's table of fill_enc_table.
template <bool kSR>
__device__ __forceinline__ uint2 quantize16(const float* v, float s_enc, const float* enc_tab, uint32_t& E,
                                            const PhiloxKey& key, uint32_t stream, uint64_t e0) {
  // block amax as a float max of |v| (the absolute value is an operand
  // modifier); equal to the bit-pattern max for finite values, and the
  // tensor's amax pass already reports non-finite input
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  float enc;
  block_scale_tab(m, s_enc, enc_tab, E, enc);
  float s[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) s[i] = __fmul_rn(v[i], enc);
  if constexpr (kSR) {
    uint32_t nu[16];
    sr_nu16(key, stream, e0, nu);
    return sr_codes16(s, nu);
  }
  return make_uint2(e2m1x8_rn(s), e2m1x8_rn(s + 8));
}

// The same block with round-to-nearest-even and enc computed by its division
// (the value fill_enc_table stores), for kernels without a table.
__device__ __forceinline__ uint2 quantize16_rne(const float* v, float s_enc, uint32_t& E) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  float enc;
  block_scale(m, s_enc, E, enc);
  float s[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) s[i] = __fmul_rn(v[i], enc);
  uint2 out;
  out.x = e2m1x8_rn(s);
  out.y = e2m1x8_rn(s + 8);
  return out;
}

// Byte offset of scale (row r, block kb) in the MMA scale layout of a tensor
// with n_kb = cols/16 blocks per row (n_kb % 4 == 0): 512-byte tiles of 128
// rows x 4 blocks, row-tile major; (r%32)*16 + ((r/32)%4)*4 + kb%4 inside.
__device__ __forceinline__ int64_t sf_mma_offset(int64_t r, int64_t kb, int64_t n_kb) {
  return ((r >> 7) * (n_kb >> 2) + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

__device__ __forceinline__ int64_t sf_offset(int layout, int64_t r, int64_t kb, int64_t n_kb) {
  return layout ? sf_mma_offset(r, kb, n_kb) : r * n_kb + kb;
}

}  // namespace nvfp4
