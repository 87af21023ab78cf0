// mx_kernels.cu -- MXFP4 quantization for sm_103a: E2M1 elements in blocks of
// 32 along the reduction dimension, each block with one UE8M0 (power-of-two)
// scale and no per-tensor scale.
//
// Method: "Pretraining Large Language Models with NVFP4" (gist.science
// summary), Resumo técnico §1 ("Limitações de Formatos Existentes") and §2
// ("Fatores de Escala Precisos"): MXFP4 is the microscaling format NVFP4 is
// measured against -- 32-element blocks, power-of-two scales.  The scale rule
// is the OCP Microscaling Formats v1.0 one for an E2M1 element type (largest
// element exponent 2):
//   E    = floor(log2(amax_b)) - 2 + 127, clamped at 0 (0 for an all-zero block)
//   v_i  = x_i * 2^(127 - E)   (one float32 multiply)
//   code = E2M1 round-to-nearest-even of v_i, saturating at +-6.
// For a finite BF16 amax_b, floor(log2(amax_b)) + 127 is the exponent field of
// its bits, 0 for zeros and subnormals (whose E clamps to 0 as well), and E is
// at most 252, so 2^(127 - E) is a normal float32 built from the bits
// (254 - E) << 23.  The multiply by a power of two is exact unless the product
// falls below 2^-126, where it is far below the first rounding threshold
// (0.25) of E2M1.
//
// The kernel is bound by HBM bandwidth: 2 bytes read per element, 0.5 + 1/16
// bytes written per element and output (codes and MMA-layout scale words).
// It runs on the TMA tile ring of tile_ring.cuh (128 x 64 BF16 tiles in a
// 3-slot shared-memory ring): threads 0-127 encode one 64-element row chunk
// each (rowwise output), threads 128-255 a column pair over 32 rows each
// (transposed output), so every thread writes whole code runs and scale
// words while the next tiles are already in flight.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "tile_ring.cuh"

namespace nvfp4 {
namespace {

constexpr int kCtasPerSm = 3;

struct MxOut {
  uint8_t* codes;
  uint8_t* scales;
  int layout;
};

struct MxParams {
  int64_t rows, cols;
  MxOut orow, ot;
  uint32_t* status;
  int debug_stall;  // failure-detection test hook (tile_ring)
};

// UE8M0 code of a block whose max |x| has the BF16 bits `amax16` (sign clear,
// finite), and the float32 multiplier 2^(127 - E).
__device__ __forceinline__ uint32_t mx_scale(uint32_t amax16, float& mult) {
  const int e = (int)((amax16 >> 7) & 0xFFu) - 2;
  const uint32_t E = e > 0 ? (uint32_t)e : 0u;
  mult = __uint_as_float((254u - E) << 23);
  return E;
}

// a *= m, b *= m: two IEEE round-to-nearest float32 multiplies in one packed
// instruction.
__device__ __forceinline__ void mul2_rn(float& a, float& b, float m) {
  asm("{\n\t.reg .b64 x, y;\n\t"
      "mov.b64 x, {%0, %1};\n\t"
      "mov.b64 y, {%2, %2};\n\t"
      "mul.rn.f32x2 x, x, y;\n\t"
      "mov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a), "+f"(b)
      : "f"(m));
}

// 32 values -> 16 bytes of codes (element 2j in the low nibble of byte j).
__device__ __forceinline__ uint4 mx_encode32(float* v, float mult) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) mul2_rn(v[i], v[i + 1], mult);
  return make_uint4(e2m1x8_rn(v), e2m1x8_rn(v + 8), e2m1x8_rn(v + 16), e2m1x8_rn(v + 24));
}

// Scale word of the 64-element chunk `chunk` of row r: in the MMA layout the
// word of the NVFP4 tile layout for that chunk, holding (E0, E1, 0, 0) -- the
// bytes a block-scaled MMA with two scales per 64 elements reads; in the
// linear layout the two bytes at [r, 2 chunk] of the [rows, cols/32] matrix.
__device__ __forceinline__ void mx_store_scales(const MxOut& o, int64_t r, int64_t chunk, int64_t cols,
                                                uint32_t E0, uint32_t E1) {
  if (o.layout == NVFP4_SCALES_MMA)
    *reinterpret_cast<uint32_t*>(o.scales + sf_mma_offset(r, 4 * chunk, cols >> 4)) = E0 | (E1 << 8);
  else
    *reinterpret_cast<uint16_t*>(o.scales + r * (cols >> 5) + 2 * chunk) = (uint16_t)(E0 | (E1 << 8));
}

// Shared-memory offsets.  A tile is 128 rows of 128 bytes with the 128-byte
// swizzle: 16-byte chunk j of row r is stored at chunk j ^ (r % 8).  Each
// consumer thread keeps its role for the whole kernel, so the eight offsets
// it reads from are computed once; every load is then the tile base plus a
// precomputed offset plus a constant.
//
// Rowwise thread r: off[j] = byte offset of chunk j (elements 8j .. 8j+7) of
// row r.
__device__ __forceinline__ void row_offsets(int r, uint32_t* off) {
#pragma unroll
  for (int j = 0; j < 8; ++j) off[j] = ring_chunk(r, j);
}

// Transposed thread u (0..127): the column pair (2 cp, 2 cp + 1) over the 32
// rows 32 rb .. 32 rb + 31, where rb % 2 = u % 2 (so the two 32-row blocks of
// a 64-element scale word sit in neighbouring lanes).  The odd lane reads its
// rows in the order i ^ 4, so that in every step the warp's two row sets fall
// on different swizzle chunks (no bank conflicts): row i of its block is at
// off[(i % 8) ^ order] + 1024 (i / 8) with order = 4 (u % 2).
struct ColRole {
  int rb, cp;
  uint32_t rot;  // 16 for the odd lane: rotates its code words back to row order
};
__device__ __forceinline__ ColRole col_role(int u, uint32_t* off) {
  ColRole c;
  const int rb_lo = u & 1, order = rb_lo << 2;
  c.rb = ((u >> 6) << 1) | rb_lo;
  c.cp = ((u >> 1) & 15) | (((u >> 5) & 1) << 4);
  c.rot = (uint32_t)order << 2;
  const int cq = c.cp >> 2, cw = (c.cp & 3) * 4;  // chunk and byte of column 2 cp
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int ko = k ^ order;  // row within the 8-row group = its swizzle phase
    off[k] = (uint32_t)((32 * c.rb + ko) * 128 + (((cq ^ ko) & 7) << 4) + cw);
  }
  return c;
}

// Eight BF16 values (the low or high halves of eight words) -> one word of
// E2M1 codes, scaled by mult.
template <bool kHigh>
__device__ __forceinline__ uint32_t encode8_halves(const uint32_t* w, float mult) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = kHigh ? bf16hi(w[i]) : bf16lo(w[i]);
#pragma unroll
  for (int i = 0; i < 8; i += 2) mul2_rn(v[i], v[i + 1], mult);
  return e2m1x8_rn(v);
}

// Rowwise output: row r (< valid) of the tile, 64 elements from column c0.
__device__ __forceinline__ void encode_row(uint32_t tile, const uint32_t* off, int64_t gr, int64_t c0,
                                           int64_t cols, const MxOut& o) {
  uint32_t E[2];
  uint4 out[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    uint4 w[4];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i] = lds128(tile + off[4 * b + i]);
      m = __vmaxu2(m, __vmaxu2(__vmaxu2(w[i].x & 0x7FFF7FFFu, w[i].y & 0x7FFF7FFFu),
                               __vmaxu2(w[i].z & 0x7FFF7FFFu, w[i].w & 0x7FFF7FFFu)));
    }
    float mult;
    E[b] = mx_scale(max(m & 0xFFFFu, m >> 16), mult);
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack8(w[i], v + 8 * i);
    out[b] = mx_encode32(v, mult);
  }
  uint4* cp = reinterpret_cast<uint4*>(o.codes + gr * (cols >> 1) + (c0 >> 1));
  cp[0] = out[0];
  cp[1] = out[1];
  mx_store_scales(o, gr, c0 >> 6, cols, E[0], E[1]);
}

// Transposed output of one thread (see ColRole): rows gr = c0 + 2 cp and
// gr + 1 of x^T, columns gm = m0 + 32 rb .. gm + 31, one 32-bit word (both
// columns) read per row.
__device__ __forceinline__ void encode_cols(uint32_t tile, const uint32_t* off, const ColRole& c,
                                            int64_t m0, int64_t c0, int64_t rows, const MxOut& o) {
  uint32_t w[32];
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    w[i] = lds32(tile + off[i & 7] + 1024 * (i >> 3));
    m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
  }
  float ma, mb;
  const uint32_t Ea = mx_scale(m & 0xFFFFu, ma), Eb = mx_scale(m >> 16, mb);
  uint32_t ca[4], cb[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ca[k] = encode8_halves<false>(w + 8 * k, ma);
    cb[k] = encode8_halves<true>(w + 8 * k, mb);
    ca[k] = __funnelshift_l(ca[k], ca[k], c.rot);
    cb[k] = __funnelshift_l(cb[k], cb[k], c.rot);
  }
  const int64_t gr = c0 + 2 * c.cp, gm = m0 + 32 * c.rb;
  *reinterpret_cast<uint4*>(o.codes + gr * (rows >> 1) + (gm >> 1)) = make_uint4(ca[0], ca[1], ca[2], ca[3]);
  *reinterpret_cast<uint4*>(o.codes + (gr + 1) * (rows >> 1) + (gm >> 1)) = make_uint4(cb[0], cb[1], cb[2], cb[3]);
  // even lane: column 2cp's word (own Ea, partner's Ea); odd lane: column
  // 2cp+1's word (partner's Eb, own Eb)
  const bool odd = c.rb & 1;
  const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, odd ? Ea : Eb, 1);
  if (odd)
    mx_store_scales(o, gr + 1, gm >> 6, rows, other, Eb);
  else
    mx_store_scales(o, gr, gm >> 6, rows, Ea, other);
}

template <bool kRow, bool kT>
__global__ void __launch_bounds__(kRingThreads, kCtasPerSm) mx_quant_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                            MxParams p) {
  extern __shared__ uint8_t smem_raw[];
  const int t = threadIdx.x;
  // consumers: threads 0-127 rowwise, 128-255 transposed; their offsets
  // into a tile are fixed for the whole kernel
  uint32_t off[8];
  ColRole col{};
  if (t < 128) row_offsets(t, off);
  else if (t < 256) col = col_role(t - 128, off);
  tile_ring(&xmap, p.rows, p.cols, p.status, p.debug_stall, smem_raw, [&](uint32_t tile, int64_t m0, int64_t c0, int valid) {
    if (t < 128) {
      if (kRow && t < valid) encode_row(tile, off, m0 + t, c0, p.cols, p.orow);
    } else if (kT) {
      if (64 * (col.rb >> 1) < valid) encode_cols(tile, off, col, m0, c0, p.rows, p.ot);  // warp-uniform
    }
  });
}

template <bool kRow, bool kT>
cudaError_t launch(const CUtensorMap& map, const MxParams& p, unsigned grid, cudaStream_t s) {
  static std::atomic<bool> attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(mx_quant_kernel<kRow, kT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  mx_quant_kernel<kRow, kT><<<grid, kRingThreads, kRingSmemBytes, s>>>(map, p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_mx(const void* x, int64_t rows, int64_t cols, const nvfp4_tensor* out_row,
                            const nvfp4_tensor* out_t, cudaStream_t s) {
  MxParams p{};
  p.rows = rows;
  p.cols = cols;
  if (out_row) p.orow = MxOut{out_row->codes, out_row->scales, out_row->scale_layout};
  if (out_t) p.ot = MxOut{out_t->codes, out_t->scales, out_t->scale_layout};
  p.status = device_status_ptr();
  const int64_t tiles = ring_tiles(rows, cols);
  if (tiles >= kRingMaxTiles) return cudaErrorInvalidValue;
  if (tiles == 0) return cudaSuccess;
  CUtensorMap map;
  if (!make_ring_map(&map, x, rows, cols)) return cudaErrorInvalidValue;
  const unsigned grid = ring_grid(tiles, kCtasPerSm);
  // the one-shot test flag is taken only by a call that launches
  p.debug_stall = take_ring_debug_stall();
  if (out_row && out_t) return launch<true, true>(map, p, grid, s);
  if (out_t) return launch<false, true>(map, p, grid, s);
  return launch<true, false>(map, p, grid, s);
}

}  // namespace nvfp4
