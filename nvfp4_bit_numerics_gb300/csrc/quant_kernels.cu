// quant_kernels.cu -- the NVFP4 quantization kernels for sm_103a: global
// amax, 1x16 rowwise quantization (round-to-nearest-even on the TMA tile ring
// of tile_ring.cuh, stochastic rounding with per-thread loads), the 128x64
// tile kernels that write the rowwise and/or the transposed (token-major,
// Hadamard-transformed) operand from one read (round-to-nearest-even on the
// tile ring, stochastic rounding with register-staged tiles), and the 16x16 2D
// weight quantization (on the tile ring) that writes W and W^T.
//
// Method: "Pretraining Large Language Models with NVFP4" (gist.science
// summary), Resumo técnico §2 Metodologia: two-level NVFP4 scaling ("Escala
// em Dois Níveis"), random Hadamard transform on the Wgrad inputs (item 2),
// 2D 16x16 weight scaling (item 3), stochastic rounding of gradients (item 4).
//
// The kernels read BF16 with 16-byte vector loads or TMA tiles, keep their
// working set in registers or a small shared-memory tile, and write packed
// codes with 8- or 16-byte stores.  The plain amax and the RNE passes are
// bound by HBM bandwidth; the passes that transform (Hadamard) or round
// stochastically (Philox and the rounding itself per element) are bound by
// instruction throughput, which is what their arithmetic is arranged to
// minimise.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "tile_ring.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
// The kernels index their work units (tiles, 16-row chunks, 64-element row
// groups) with 32-bit integers; the launchers refuse tensors with 2^31 units
// or more (over 2^42 elements).
constexpr int64_t kMaxUnits = int64_t(1) << 31;

int sm_count() { return device_sm_count(); }

int grid_for(int64_t units, int per_sm) {
  const int64_t cap = (int64_t)sm_count() * per_sm;
  const int64_t need = (units + kThreads - 1) / kThreads;
  return (int)(need < cap ? (need > 0 ? need : 1) : cap);
}

__device__ __forceinline__ void warp_amax_to_global(uint32_t m, uint32_t* out, uint32_t* status) {
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31) == 0 && m) {
    atomicMax(out, m);
    if (m >= 0x7F800000u) raise_status(status, kStatusNonFinite);
  }
}

// ---------------------------------------------------------------------------
// amax kernels.  out[] holds float bits; the caller zeroes it first.
// ---------------------------------------------------------------------------

// max |x| over n_vec 16-byte vectors, in the bf16 bit domain (two halves per
// word compared with a SIMD max), converted to float bits at the end.
__global__ void __launch_bounds__(kThreads) amax_plain_kernel(const uint4* __restrict__ x, int64_t n_vec,
                                                              uint32_t* out, uint32_t* status) {
  uint32_t m2 = 0;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  for (; i + 3 * stride < n_vec; i += 4 * stride) {
    uint4 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) q[u] = ldg_nc_v4(x + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      m2 = __vmaxu2(__vmaxu2(m2, q[u].x & 0x7FFF7FFFu),
                    __vmaxu2(__vmaxu2(q[u].y & 0x7FFF7FFFu, q[u].z & 0x7FFF7FFFu), q[u].w & 0x7FFF7FFFu));
  }
  for (; i < n_vec; i += stride) {
    const uint4 q = ldg_nc_v4(x + i);
    m2 = __vmaxu2(__vmaxu2(m2, q.x & 0x7FFF7FFFu),
                  __vmaxu2(__vmaxu2(q.y & 0x7FFF7FFFu, q.z & 0x7FFF7FFFu), q.w & 0x7FFF7FFFu));
  }
  const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16) << 16;
  warp_amax_to_global(m, out, status);
}

// Plain amax and amax of the 16-point transform along the contiguous
// dimension: one thread per 16-element chunk of a row.
__global__ void __launch_bounds__(kThreads) amax_rht_rows_kernel(const uint4* __restrict__ x, int64_t n_chunks,
                                                                 uint64_t seed, uint32_t* out_plain,
                                                                 uint32_t* out_rht, uint32_t* status) {
  const uint32_t smask = rht_sign_mask(seed);
  uint32_t mp = 0, mr = 0;
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n_chunks; i += (int64_t)gridDim.x * kThreads) {
    float v[16];
    unpack8(ldg_nc_v4(x + 2 * i), v);
    unpack8(ldg_nc_v4(x + 2 * i + 1), v + 8);
#pragma unroll
    for (int j = 0; j < 16; ++j) mp = max(mp, abs_bits(v[j]));
    rht16(v, smask);
#pragma unroll
    for (int j = 0; j < 16; ++j) mr = max(mr, abs_bits(v[j]));
  }
  if (out_plain) warp_amax_to_global(mp, out_plain, status);
  warp_amax_to_global(mr, out_rht, status);
}

// Plain amax and amax of the 16-point transform along the rows (tokens):
// one thread per (16-row block, 8-column group); a warp reads 512
// contiguous bytes of each of the 16 rows.
__global__ void __launch_bounds__(kThreads, 2) amax_rht_cols_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                 int64_t cols, uint64_t seed, uint32_t* out_plain,
                                                                 uint32_t* out_rht, uint32_t* status) {
  const uint32_t smask = rht_sign_mask(seed);
  const int64_t groups = cols >> 3;
  // unit counts are below 2^32 (the launcher checks), so the index math is
  // 32-bit: a 64-bit division is a long subroutine
  const uint32_t units = (uint32_t)((rows >> 4) * groups), groups32 = (uint32_t)groups;
  uint32_t mp2 = 0;  // max |x| of both BF16 halves, on the bit patterns
  float mr = 0.0f;
  for (uint32_t u = blockIdx.x * kThreads + threadIdx.x; u < units; u += gridDim.x * kThreads) {
    const uint32_t rb = u / groups32, cg = u - rb * groups32;
    const uint16_t* p = x + (rb * 16) * cols + cg * 8;
    uint4 q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = ldg_nc_v4(p + i * cols);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      mp2 = __vmaxu2(__vmaxu2(mp2, q[i].x & 0x7FFF7FFFu),
                     __vmaxu2(__vmaxu2(q[i].y & 0x7FFF7FFFu, q[i].z & 0x7FFF7FFFu), q[i].w & 0x7FFF7FFFu));
      const uint32_t sw = rht_sign_word(smask, i);  // row i of the chunk
      q[i].x ^= sw; q[i].y ^= sw; q[i].z ^= sw; q[i].w ^= sw;
    }
    // the two columns of each 32-bit word as float pairs through the first
    // three butterfly stages; the last stage only feeds the maximum:
    // max(|fl(a + b)|, |fl(a - b)|) = fl(|a| + |b|) (rounding is monotonic)
#pragma unroll
    for (int c2 = 0; c2 < 4; ++c2) {
      uint64_t pp[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pp[i] = f2_from_bf16x2(c2 == 0 ? q[i].x : c2 == 1 ? q[i].y : c2 == 2 ? q[i].z : q[i].w);
#pragma unroll
      for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if ((i & h) == 0) {
            const uint64_t a = pp[i], b = pp[i + h];
            pp[i] = f2_add(a, b);
            pp[i + h] = f2_sub(a, b);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint64_t a = pp[i], b = pp[i + 8];
        mr = fmax_nan3(mr, __fadd_rn(fabsf(f2_lo(a)), fabsf(f2_lo(b))), __fadd_rn(fabsf(f2_hi(a)), fabsf(f2_hi(b))));
      }
    }
  }
  // the transform's * 1/4, applied once: fl(max |v| / 4) = max fl(|v| / 4)
  mr = __fmul_rn(mr, 0.25f);
  if (out_plain) warp_amax_to_global(max(mp2 & 0xFFFFu, mp2 >> 16) << 16, out_plain, status);
  warp_amax_to_global(__float_as_uint(mr), out_rht, status);
}

// ---------------------------------------------------------------------------
// Shared per-tensor prologue: s_enc from the amax; block 0 stores ts and
// flags a non-finite amax.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float tensor_prologue(const float* amax, float* ts_out, uint32_t* status) {
  const float a = *amax;
  const float s_enc = tensor_encode_scale(a);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (ts_out) *ts_out = tensor_decode_scale(s_enc);
    if (!(abs_bits(a) < 0x7F800000u)) raise_status(status, kStatusNonFinite);
  }
  return s_enc;
}

// ---------------------------------------------------------------------------
// 1x16 rowwise quantization with stochastic rounding: one thread per 64
// elements (4 independent blocks) of a row, read with 16-byte global loads.
// ---------------------------------------------------------------------------
template <bool kSR, bool kRHT>
__global__ void __launch_bounds__(kThreads) quant_rowwise_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                 int64_t cols, const float* amax, uint8_t* codes,
                                                                 uint8_t* scales, int layout, float* ts_out,
                                                                 uint64_t seed, const __grid_constant__ PhiloxKey key,
                                                                 uint32_t stream, uint32_t* status) {
  const float s_enc = tensor_prologue(amax, ts_out, status);
  __shared__ float enc_tab[128];
  fill_enc_table(enc_tab, s_enc, threadIdx.x);
  __syncthreads();
  const uint32_t smask = kRHT ? rht_sign_mask(seed) : 0u;
  const int64_t gpr = cols >> 6;  // 64-element groups per row
  const uint32_t units = (uint32_t)(rows * gpr), gpr32 = (uint32_t)gpr;  // < 2^32 (launcher)
  const int64_t n_kb = cols >> 4;
  for (uint32_t u = blockIdx.x * kThreads + threadIdx.x; u < units; u += gridDim.x * kThreads) {
    const int64_t r = u / gpr32, g = u - (uint32_t)r * gpr32;
    const int64_t c0 = g * 64;
    const uint16_t* p = x + r * cols + c0;
    uint4 q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = ldg_nc_v4(p + 8 * i);
    uint32_t cw[8];
    uint32_t sc = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float v[16];
      unpack8(q[2 * b], v);
      unpack8(q[2 * b + 1], v + 8);
      if constexpr (kRHT) rht16(v, smask);
      uint32_t E;
      const uint2 o = quantize16<kSR>(v, s_enc, enc_tab, E, key, stream, (uint64_t)(r * cols + c0 + 16 * b));
      cw[2 * b] = o.x;
      cw[2 * b + 1] = o.y;
      sc |= E << (8 * b);
    }
    uint4* cp = reinterpret_cast<uint4*>(codes + r * (cols >> 1) + (c0 >> 1));
    cp[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    cp[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    *reinterpret_cast<uint32_t*>(scales + sf_offset(layout, r, c0 >> 4, n_kb)) = sc;
  }
}

// ---------------------------------------------------------------------------
// 1x16 rowwise round-to-nearest-even quantization on the TMA tile ring
// (tile_ring.cuh): 128 x 64 tiles stream into a shared-memory ring while the
// 8 consumer warps encode; thread t takes row t/2 of the tile, elements
// 32 (t%2) .. +31 (2 blocks: 16 code bytes, two scale bytes), with the 16-point
// transform along each 16-chunk when asked.  The row reads of 8 threads (4
// rows x 2 halves) fall on 8 different swizzle chunks, free of bank
// conflicts.  Used for the rowwise RNE kinds, which are bound by HBM; the
// stochastic-rounding kinds, bound by instruction throughput, keep
// quant_rowwise_kernel, whose threads hold 4 independent blocks each.
// ---------------------------------------------------------------------------
template <bool kRHT>
__global__ void __launch_bounds__(kRingThreads, 3)
    quant_rowwise_ring_kernel(const __grid_constant__ CUtensorMap xmap, int64_t rows, int64_t cols,
                              const float* amax, uint8_t* codes, uint8_t* scales, int layout, float* ts_out,
                              uint64_t seed, uint32_t* status, int debug_stall) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float enc_tab[128];
  const int t = threadIdx.x;
  const float s_enc = tensor_prologue(amax, ts_out, status);
  fill_enc_table(enc_tab, s_enc, t);
  const uint32_t smask = kRHT ? rht_sign_mask(seed) : 0u;
  const int r = t >> 1, hh = t & 1;
  uint32_t roff[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) roff[i] = ring_chunk(r, 4 * hh + i);
  const PhiloxKey no_key{};  // round-to-nearest-even draws no random numbers
  tile_ring(&xmap, rows, cols, status, debug_stall, smem_raw, [&](uint32_t tile, int64_t m0, int64_t c0, int valid) {
    if (r >= valid) return;
    const int64_t gr = m0 + r, gc = c0 + 32 * hh;
    uint32_t cw[4], sc = 0;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      float v[16];
      unpack8(lds128(tile + roff[2 * b]), v);
      unpack8(lds128(tile + roff[2 * b + 1]), v + 8);
      if constexpr (kRHT) rht16(v, smask);
      uint32_t E;
      const uint2 o = quantize16<false>(v, s_enc, enc_tab, E, no_key, 0, 0);
      cw[2 * b] = o.x;
      cw[2 * b + 1] = o.y;
      sc |= E << (8 * b);
    }
    *reinterpret_cast<uint4*>(codes + gr * (cols >> 1) + (gc >> 1)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    *reinterpret_cast<uint16_t*>(scales + sf_offset(layout, gr, gc >> 4, cols >> 4)) = (uint16_t)sc;
  });
}

// The 16-point transform Q = 1/4 H16 diag(s) on 16 pairs at once (two
// independent vectors, one per half): the butterfly with strides 1, 2, 4, 8,
// then * 0.25 + 0 in one rounding (as rht16_unsigned; the signs are applied
// to the BF16 words before).  Also returns each half's block amax
// max_i |(Q x)_i|, exact.
__device__ __forceinline__ void rht16_pairs(uint64_t* p, float& ma, float& mb) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const uint64_t a = p[i], b = p[i + h];
        p[i] = f2_add(a, b);
        p[i + h] = f2_sub(a, b);
      }
    }
  }
  // last stage (stride 8); max(|fl(a + b)|, |fl(a - b)|) = fl(|a| + |b|)
  // (rounding is monotonic), so the block amax of each half is a quarter of
  // the largest fl(|a| + |b|) over the 8 butterflies
  float ta[8], tb[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t a = p[i], b = p[i + 8];
    ta[i] = __fadd_rn(fabsf(f2_lo(a)), fabsf(f2_lo(b)));
    tb[i] = __fadd_rn(fabsf(f2_hi(a)), fabsf(f2_hi(b)));
    p[i] = f2_add(a, b);
    p[i + 8] = f2_sub(a, b);
  }
  ma = __fmul_rn(fmax3(fmax3(ta[0], ta[1], ta[2]), fmax3(ta[3], ta[4], ta[5]), fmaxf(ta[6], ta[7])), 0.25f);
  mb = __fmul_rn(fmax3(fmax3(tb[0], tb[1], tb[2]), fmax3(tb[3], tb[4], tb[5]), fmaxf(tb[6], tb[7])), 0.25f);
  const uint64_t quarter = f2_pack(0x3E800000u, 0x3E800000u), zero = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) p[i] = f2_fma(p[i], quarter, zero);
}

// One 1x16 block given as 8 BF16 words (elements 2j, 2j+1 in word j): amax
// (a max over the BF16 magnitudes, exact), scale, 16 codes (8 bytes), the
// values scaled as float pairs.  Same results as quantize16.
template <bool kSR>
__device__ __forceinline__ uint2 quantize16_words(const uint32_t* w, float s_enc, const float* enc_tab, uint32_t& E,
                                                  const PhiloxKey& key, uint32_t stream, uint64_t e0) {
  const uint32_t m2 = bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(w[0], w[1]), bf16x2_absmax(w[2], w[3])),
                                    bf16x2_absmax(bf16x2_absmax(w[4], w[5]), bf16x2_absmax(w[6], w[7])));
  const float m = fmaxf(fabsf(bf16lo(m2)), fabsf(bf16hi(m2)));
  float enc;
  block_scale_tab(m, s_enc, enc_tab, E, enc);
  const uint64_t enc2 = f2_pack(__float_as_uint(enc), __float_as_uint(enc));
  float s[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint64_t q = f2_mul(f2_from_bf16x2(w[j]), enc2);
    s[2 * j] = f2_lo(q);
    s[2 * j + 1] = f2_hi(q);
  }
  if constexpr (kSR) {
    uint32_t nu[16];
    sr_nu16(key, stream, e0, nu);
    return sr_codes16(s, nu);
  }
  return make_uint2(e2m1x8_rn(s), e2m1x8_rn(s + 8));
}

// ---------------------------------------------------------------------------
// Tile kernel: one read of x [rows, cols] BF16 per 128x64 tile, staged in
// shared memory, then
//  - rowwise:    1x16 blocks along cols of x       -> out_row [rows, cols]
//  - transposed: 1x16 blocks along rows of x (after the optional 16-point
//                transform along rows)             -> out_t   [cols, rows]
// Persistent over tiles; the next tile's global loads are issued before the
// current tile is encoded.  Thread t: rowwise, row t/2 and two 16-element
// blocks; transposed, the column pair 2(t%32), 2(t%32)+1 over the 16 rows
// 16(t/32)..16(t/32)+15 (one 32-bit shared-memory word per row), the two
// columns carried as float pairs through the transform and the scaling.
// Launched for the stochastic-rounding kinds, which are bound by instruction
// issue (Philox draws and the rounding itself): 3 CTAs of 8 warps per SM keep
// more warps to issue from than the ring kernel below, and measured faster.
// ---------------------------------------------------------------------------
struct TileOut {
  uint8_t* codes;
  uint8_t* scales;
  const float* amax;
  float* ts;
  int layout;
  uint32_t stream;
};

constexpr int kTile = 64;       // column width of the tile kernel
constexpr int kTileRows = 128;  // rows (tokens) per tile of the tile kernel
constexpr int kTilePitch = 72;  // uint16 per smem row: 144 B, conflict-free 16 B row reads

template <bool kRow, bool kT, bool kRHT, bool kSR>
__global__ void __launch_bounds__(kThreads, 3) quant_tile_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                              int64_t cols, TileOut orow, TileOut ot,
                                                              uint64_t seed, const __grid_constant__ PhiloxKey key,
                                                              uint32_t* status) {
  __shared__ __align__(16) uint16_t tile[kTileRows * kTilePitch];
  const int t = threadIdx.x;
  const int64_t tiles_c = cols / kTile;
  const int64_t n_tiles = ((rows + kTileRows - 1) / kTileRows) * tiles_c;  // rows % 64 == 0

  float s_row = 1.0f, s_t = 1.0f;
  if constexpr (kRow) s_row = tensor_prologue(orow.amax, orow.ts, status);
  if constexpr (kT) s_t = tensor_prologue(ot.amax, ot.ts, status);
  // enc tables (rowwise tensor, transposed tensor); the first tile's
  // __syncthreads orders them before use
  __shared__ float enc_tab[2][128];
  if constexpr (kRow) fill_enc_table(enc_tab[0], s_row, t);
  if constexpr (kT) fill_enc_table(enc_tab[1], s_t, t - 128);
  const uint32_t smask = kRHT ? rht_sign_mask(seed) : 0u;

  const uint32_t tiles_c32 = (uint32_t)tiles_c;  // tile counts < 2^32 (launcher): 32-bit index math
  uint4 q[4];
  auto load_tile = [&](uint32_t tl) {
    const uint32_t tm = tl / tiles_c32, tc = tl - tm * tiles_c32;
    const int64_t m0 = (int64_t)tm * kTileRows, c0 = (int64_t)tc * kTile;
    const int valid = rows - m0 < kTileRows ? (int)(rows - m0) : kTileRows;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int v = t + k * kThreads;
      q[k] = (v >> 3) < valid ? ldg_nc_v4(x + (m0 + (v >> 3)) * cols + c0 + (v & 7) * 8) : make_uint4(0, 0, 0, 0);
    }
  };
  if (blockIdx.x < (uint32_t)n_tiles) load_tile(blockIdx.x);
  for (uint32_t tl = blockIdx.x; tl < (uint32_t)n_tiles; tl += gridDim.x) {
    const uint32_t tm = tl / tiles_c32, tc = tl - tm * tiles_c32;
    const int64_t m0 = (int64_t)tm * kTileRows, c0 = (int64_t)tc * kTile;
    const int valid = rows - m0 < kTileRows ? (int)(rows - m0) : kTileRows;  // 64 or 128
    __syncthreads();  // the previous tile's readers are done
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int v = t + k * kThreads;
      *reinterpret_cast<uint4*>(&tile[(v >> 3) * kTilePitch + (v & 7) * 8]) = q[k];
    }
    __syncthreads();
    if (tl + gridDim.x < (uint32_t)n_tiles) load_tile(tl + gridDim.x);

    if (kRow && (t >> 1) < valid) {
      const int r = t >> 1, hb = (t & 1) * 2;  // row, first of two blocks
      const int64_t gr = m0 + r, gc = c0 + hb * 16;
      uint32_t cw[4], sc = 0;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint4* sp = reinterpret_cast<const uint4*>(&tile[r * kTilePitch + (hb + b) * 16]);
        const uint4 w0 = sp[0], w1 = sp[1];
        const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t E;
        const uint2 o =
            quantize16_words<kSR>(wv, s_row, enc_tab[0], E, key, orow.stream, (uint64_t)(gr * cols + gc + 16 * b));
        cw[2 * b] = o.x;
        cw[2 * b + 1] = o.y;
        sc |= E << (8 * b);
      }
      *reinterpret_cast<uint4*>(orow.codes + gr * (cols >> 1) + (gc >> 1)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      *reinterpret_cast<uint16_t*>(orow.scales + sf_offset(orow.layout, gr, gc >> 4, cols >> 4)) = (uint16_t)sc;
    }
    if (kT && 16 * (t >> 5) < valid) {
      const int pc = (t & 31) * 2, ch = t >> 5;
      uint64_t p[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        uint32_t w = *reinterpret_cast<const uint32_t*>(&tile[(16 * ch + i) * kTilePitch + pc]);
        if constexpr (kRHT) w ^= rht_sign_word(smask, i);  // both columns are in row i
        p[i] = f2_from_bf16x2(w);
      }
      const int64_t gm = m0 + 16 * ch;  // column of the transposed tensor
      // the block of each column: amax and scale, then both columns scaled
      // as pairs
      float ma = 0.0f, mb = 0.0f;
      if constexpr (kRHT) {
        rht16_pairs(p, ma, mb);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          ma = fmaxf(ma, fabsf(f2_lo(p[i])));
          mb = fmaxf(mb, fabsf(f2_hi(p[i])));
        }
      }
      uint32_t Ea, Eb;
      float enca, encb;
      block_scale_tab(ma, s_t, enc_tab[1], Ea, enca);
      block_scale_tab(mb, s_t, enc_tab[1], Eb, encb);
      const uint64_t enc2 = f2_pack(__float_as_uint(enca), __float_as_uint(encb));
      float sa[16], sb[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint64_t v = f2_mul(p[i], enc2);
        sa[i] = f2_lo(v);
        sb[i] = f2_hi(v);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float* s = h ? sb : sa;
        const int64_t gr = c0 + pc + h;  // row of the transposed tensor
        uint2 o;
        if constexpr (kSR) {
          uint32_t nu[16];
          sr_nu16(key, ot.stream, (uint64_t)(gr * rows + gm), nu);
          o = sr_codes16(s, nu);
        } else {
          o = make_uint2(e2m1x8_rn(s), e2m1x8_rn(s + 8));
        }
        *reinterpret_cast<uint2*>(ot.codes + gr * (rows >> 1) + (gm >> 1)) = o;
        ot.scales[sf_offset(ot.layout, gr, gm >> 4, rows >> 4)] = (uint8_t)(h ? Eb : Ea);
      }
    }
  }
}

// Barrier of the 256 consumer threads of the ring kernels (named barrier 1;
// the producer warp does not take part).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// ---------------------------------------------------------------------------
// The same fused quantization with round-to-nearest-even on the TMA tile
// ring (tile_ring.cuh), for the kinds that are bound by memory traffic: each
// 128 x 64 tile is read once into the shared-memory ring; thread t has the
// roles of quant_tile_kernel (rowwise, row t/2 and elements 32 (t%2) .. +31:
// 8 threads of a quarter warp read 8 different swizzle chunks; transposed,
// the column pair 2(t%32), 2(t%32)+1 over rows 16(t/32) .. +15: a warp reads
// one whole 128-byte row).  The transposed codes and scales of a tile are
// collected in shared memory (double-buffered) and stored as whole 64-byte
// row segments and 4-byte scale words; the rowwise scales of a row go out as
// one word.  The stochastic-rounding kinds, bound by instruction issue, keep
// quant_tile_kernel: on this ring they ran slower at 2 CTAs per SM (16
// encoding warps) and at 3 (72 registers, with spills).
// ---------------------------------------------------------------------------
constexpr int kTileRingCtas = 3;  // CTAs per SM: up to 72 registers a thread, 3-slot rings

template <bool kRow, bool kT, bool kRHT>
__global__ void __launch_bounds__(kRingThreads, kTileRingCtas)
    quant_tile_ring_kernel(const __grid_constant__ CUtensorMap xmap, int64_t rows, int64_t cols, TileOut orow,
                      TileOut ot, uint64_t seed, uint32_t* status,
                      int debug_stall) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float enc_tab[2][128];
  __shared__ __align__(16) uint2 tbuf[2][8 * 64];  // [buffer][token chunk * 64 + swizzled transposed row]
  __shared__ __align__(4) uint8_t tE[2][64 * 8];   // [buffer][transposed row * 8 + token chunk]
  int buf = 0;
  const int t = threadIdx.x;
  const PhiloxKey key{};  // round-to-nearest-even draws no random numbers
  float s_row = 1.0f, s_t = 1.0f;
  if constexpr (kRow) s_row = tensor_prologue(orow.amax, orow.ts, status);
  if constexpr (kT) s_t = tensor_prologue(ot.amax, ot.ts, status);
  if constexpr (kRow) fill_enc_table(enc_tab[0], s_row, t);
  if constexpr (kT) fill_enc_table(enc_tab[1], s_t, t - 128);
  // sign mask of the transform in both halves: row i's flip is bit 15 and
  // bit 31 of (P << (15 - i)), the sign bits of the two BF16 values of a word
  const uint32_t P = kRHT ? rht_sign_mask(seed) * 0x00010001u : 0u;
  // rowwise role
  const int r = t >> 1, hh = t & 1;
  uint32_t roff[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) roff[i] = ring_chunk(r, 4 * hh + i);
  // transposed role: rows 16 ch + i; the 16-byte chunk of the column pair
  // sits at j ^ i (i % 8) in row 16 ch + i
  const int pc = (t & 31) * 2, ch = t >> 5;
  const uint32_t t_base = (uint32_t)(16 * ch * 128 + (pc & 7) * 2), j16 = (uint32_t)((pc >> 3) << 4);
  tile_ring(&xmap, rows, cols, status, debug_stall, smem_raw, [&](uint32_t tile, int64_t m0, int64_t c0, int valid) {
    if (kRow && r < valid) {
      const int64_t gr = m0 + r, gc = c0 + 32 * hh;
      uint32_t cw[4], sc = 0;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint4 w0 = lds128(tile + roff[2 * b]), w1 = lds128(tile + roff[2 * b + 1]);
        const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t E;
        const uint2 o =
            quantize16_words<false>(wv, s_row, enc_tab[0], E, key, 0, 0);
        cw[2 * b] = o.x;
        cw[2 * b + 1] = o.y;
        sc |= E << (8 * b);
      }
      *reinterpret_cast<uint4*>(orow.codes + gr * (cols >> 1) + (gc >> 1)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      // the row's 4 scales of this tile (threads 2r, 2r + 1) as one word
      const uint32_t sc4 = sc | (__shfl_down_sync(0xFFFFFFFFu, sc, 1) << 16);
      if (hh == 0)
        *reinterpret_cast<uint32_t*>(orow.scales + sf_offset(orow.layout, gr, c0 >> 4, cols >> 4)) = sc4;
    }
    if (kT) {
      // the transposed codes and scales of this tile go through shared
      // memory (double-buffered), so that the stores to global memory are
      // whole 64-byte row segments and 4-byte scale words
      uint2* tb = tbuf[buf];
      uint8_t* te = tE[buf];
      if (16 * ch < valid) {
        uint64_t p[16];
        uint32_t rowp[8];  // tile + row base + swizzled chunk for rows i and i + 8
#pragma unroll
        for (int i = 0; i < 8; ++i) rowp[i] = (tile + t_base) + (j16 ^ (uint32_t)(i << 4));
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t w = lds32(rowp[i & 7] + (uint32_t)(i * 128));
          if constexpr (kRHT) w ^= (P << (15 - i)) & 0x80008000u;  // both columns are in row i
          p[i] = f2_from_bf16x2(w);
        }
        // the block of each column: amax and scale, then both columns scaled
        // as pairs
        float ma = 0.0f, mb = 0.0f;
        if constexpr (kRHT) {
          rht16_pairs(p, ma, mb);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            ma = fmaxf(ma, fabsf(f2_lo(p[i])));
            mb = fmaxf(mb, fabsf(f2_hi(p[i])));
          }
        }
        uint32_t Ea, Eb;
        float enca, encb;
        block_scale_tab(ma, s_t, enc_tab[1], Ea, enca);
        block_scale_tab(mb, s_t, enc_tab[1], Eb, encb);
        const uint64_t enc2 = f2_pack(__float_as_uint(enca), __float_as_uint(encb));
        float sa[16], sb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t v = f2_mul(p[i], enc2);
          sa[i] = f2_lo(v);
          sb[i] = f2_hi(v);
        }
        const uint2 o[2] = {make_uint2(e2m1x8_rn(sa), e2m1x8_rn(sa + 8)), make_uint2(e2m1x8_rn(sb), e2m1x8_rn(sb + 8))};
        // transposed rows pc, pc + 1 of token chunk ch: 16 bytes at row
        // position pc ^ 2 ch of chunk ch's 64-row column
        *reinterpret_cast<uint4*>(tb + ch * 64 + (pc ^ (2 * ch))) = make_uint4(o[0].x, o[0].y, o[1].x, o[1].y);
        te[pc * 8 + ch] = (uint8_t)Ea;
        te[(pc + 1) * 8 + ch] = (uint8_t)Eb;
      }
      consumer_sync();
      {  // thread t: transposed row k = t / 4, token chunks 2q, 2q + 1
        const int k = t >> 2, q = t & 3;
        if (32 * q < valid) {
          const uint2 a = tb[(2 * q) * 64 + (k ^ (4 * q))], b = tb[(2 * q + 1) * 64 + (k ^ (4 * q + 2))];
          *reinterpret_cast<uint4*>(ot.codes + (c0 + k) * (rows >> 1) + (m0 >> 1) + 16 * q) =
              make_uint4(a.x, a.y, b.x, b.y);
        }
      }
      if (t < 128) {  // scale word g (4 token chunks) of transposed row k
        const int k = t >> 1, g = t & 1;
        if (64 * g < valid)
          *reinterpret_cast<uint32_t*>(ot.scales + sf_offset(ot.layout, c0 + k, (m0 >> 4) + 4 * g, rows >> 4)) =
              *reinterpret_cast<const uint32_t*>(te + k * 8 + 4 * g);
      }
      buf ^= 1;
    }
  });
}

// ---------------------------------------------------------------------------
// 2D weight quantization on the TMA tile ring (tile_ring.cuh): 128 x 64 tiles
// (8 x 4 blocks of 16 x 16) stream into a shared-memory ring while the 8
// consumer warps encode them.
//  - block pass: the 8 threads (consecutive lanes) of block (br, bc) hold
//    rows p and p + 8 of it; the block amax is a max over BF16 pairs, then a
//    shuffle over the 8; each thread encodes its two rows (W codes, K-major,
//    8 bytes per row).
//  - scales: one 32-bit word per row of W (its 4 blocks of the tile) and two
//    per row of W^T (its 8 blocks), from the tile's 32 block scales.
//  - column pass: thread (cp, brr) encodes the 16 x 2 slice (columns 2 cp,
//    2 cp + 1 of block row brr) with the block's scale, reading one 32-bit
//    word per row (a warp reads one whole 128-byte row: no bank conflicts);
//    encoding an element twice gives the same code, so W^T is exactly W
//    transposed.  The W^T codes of the tile (64 rows of 64 bytes) are
//    collected in shared memory, swizzled so that neither the 16-byte writes
//    nor the 8-byte reads conflict, and written after the next tile's
//    barrier as one 16-byte store per thread, whole sectors per row.
// Block scales and W^T codes are double-buffered, so one barrier of the 256
// consumer threads per tile orders everything.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kRingThreads, 3)
    quant_2d_ring_kernel(const __grid_constant__ CUtensorMap wmap, int64_t rows, int64_t cols, const float* amax,
                         TileOut ow, TileOut owt, int has_t, uint32_t* status, int debug_stall) {
  extern __shared__ uint8_t smem_raw[];
  // double-buffered per-tile state: block scales and the W^T codes, stored
  // after the next tile's barrier (one barrier per tile)
  __shared__ float s_enc[2][8][4];
  __shared__ uint32_t s_E[2][8][4];
  __shared__ __align__(16) uint2 tbuf[2][8 * 64];  // [buffer][block row * 64 + swizzled W^T row]
  const int t = threadIdx.x;
  const float s_tensor = tensor_prologue(amax, ow.ts, status);
  if (has_t && blockIdx.x == 0 && t == 0) *owt.ts = tensor_decode_scale(s_tensor);
  // block pass role
  const int blk = t >> 3, p = t & 7, br = blk >> 2, bc = blk & 3;
  uint32_t roff[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    roff[2 * h] = ring_chunk(16 * br + p + 8 * h, 2 * bc);
    roff[2 * h + 1] = ring_chunk(16 * br + p + 8 * h, 2 * bc + 1);
  }
  // column pass role: column pair (2 cp, 2 cp + 1), block row brr; its 16-byte
  // chunk of row 16 brr + i sits at (cp / 4) ^ (i % 8)
  const int cp = t & 31, brr = t >> 5;
  const uint32_t t_base = (uint32_t)(16 * brr * 128 + (cp & 3) * 4), j16 = (uint32_t)((cp >> 2) << 4);
  const int64_t n_kb_w = cols >> 4, n_kb_t = rows >> 4;
  int buf = 0;
  bool pending = false;  // tbuf[buf ^ 1] holds the previous tile's W^T codes
  int64_t pm0 = 0, pc0 = 0;
  int pvalid = 0;
  // thread t: W^T row t / 4 of tile (m0, c0), 16 bytes (block rows 2q, 2q + 1)
  auto write_t = [&](int b, int64_t m0, int64_t c0, int valid) {
    const int k = t >> 2, q = t & 3;
    if (32 * q < valid) {
      const uint2 lo = tbuf[b][(2 * q) * 64 + (k ^ (4 * q))], hi = tbuf[b][(2 * q + 1) * 64 + (k ^ (4 * q + 2))];
      *reinterpret_cast<uint4*>(owt.codes + (c0 + k) * (rows >> 1) + (m0 >> 1) + 16 * q) =
          make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
  };
  tile_ring(&wmap, rows, cols, status, debug_stall, smem_raw, [&](uint32_t tile, int64_t m0, int64_t c0, int valid) {
    // ---- block pass: amax, scale, W codes
    const bool row_ok = 16 * br < valid;
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 q = lds128(tile + roff[j]);
      w[4 * j] = q.x;
      w[4 * j + 1] = q.y;
      w[4 * j + 2] = q.z;
      w[4 * j + 3] = q.w;
    }
    uint32_t m2 = bf16x2_absmax(w[0], w[1]);
#pragma unroll
    for (int j = 2; j < 16; ++j) m2 = bf16x2_absmax(m2, w[j]);
    float m = fmaxf(fabsf(bf16lo(m2)), fabsf(bf16hi(m2)));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
    uint32_t E;
    float enc;
    block_scale(m, s_tensor, E, enc);
    if (p == 0) {
      s_E[buf][br][bc] = E;
      s_enc[buf][br][bc] = enc;
    }
    if (row_ok) {
      const uint64_t enc2 = f2_pack(__float_as_uint(enc), __float_as_uint(enc));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float sv[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint64_t v = f2_mul(f2_from_bf16x2(w[8 * h + j]), enc2);
          sv[2 * j] = f2_lo(v);
          sv[2 * j + 1] = f2_hi(v);
        }
        const int64_t gr = m0 + 16 * br + p + 8 * h, gc = c0 + 16 * bc;
        *reinterpret_cast<uint2*>(ow.codes + gr * (cols >> 1) + (gc >> 1)) =
            make_uint2(e2m1x8_rn(sv), e2m1x8_rn(sv + 8));
      }
    }
    consumer_sync();
    if (has_t && pending) write_t(buf ^ 1, pm0, pc0, pvalid);
    // ---- scales: W rows (4 blocks of the tile per word), W^T rows (4 block
    // rows per word)
    if (t < 128) {
      if (t < valid) {
        const int b = t >> 4;
        const uint32_t w4 =
            s_E[buf][b][0] | (s_E[buf][b][1] << 8) | (s_E[buf][b][2] << 16) | (s_E[buf][b][3] << 24);
        *reinterpret_cast<uint32_t*>(ow.scales + sf_offset(ow.layout, m0 + t, c0 >> 4, n_kb_w)) = w4;
      }
    } else if (has_t) {
      const int u = t - 128, k = u >> 1, g = u & 1;
      if (64 * g < valid) {
        const int b = k >> 4;
        const uint32_t w4 = s_E[buf][4 * g][b] | (s_E[buf][4 * g + 1][b] << 8) | (s_E[buf][4 * g + 2][b] << 16) |
                            (s_E[buf][4 * g + 3][b] << 24);
        *reinterpret_cast<uint32_t*>(owt.scales + sf_offset(owt.layout, c0 + k, (m0 >> 4) + 4 * g, n_kb_t)) = w4;
      }
    }
    if (has_t) {
      // ---- column pass: W^T codes of this block row (encoding an element
      // twice gives the same code, so W^T is exactly W transposed)
      if (16 * brr < valid) {
        const float e = s_enc[buf][brr][cp >> 3];
        const uint64_t e2 = f2_pack(__float_as_uint(e), __float_as_uint(e));
        uint32_t rowp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rowp[i] = (tile + t_base) + (j16 ^ (uint32_t)(i << 4));
        float va[16], vb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t v = f2_mul(f2_from_bf16x2(lds32(rowp[i & 7] + (uint32_t)(i * 128))), e2);
          va[i] = f2_lo(v);
          vb[i] = f2_hi(v);
        }
        *reinterpret_cast<uint4*>(&tbuf[buf][brr * 64 + ((2 * cp) ^ (2 * brr))]) =
            make_uint4(e2m1x8_rn(va), e2m1x8_rn(va + 8), e2m1x8_rn(vb), e2m1x8_rn(vb + 8));
      }
      pending = true;
      pm0 = m0;
      pc0 = c0;
      pvalid = valid;
    }
    buf ^= 1;
  });
  if (has_t && pending) write_t(buf ^ 1, pm0, pc0, pvalid);  // after the ring's closing barrier
}

}  // namespace

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
cudaError_t launch_amax(const void* x, int64_t rows, int64_t cols, float* plain, float* rht_rows, float* rht_cols,
                        uint64_t rht_seed, cudaStream_t s) {
  uint32_t* status = device_status_ptr();
  uint32_t* o_plain = reinterpret_cast<uint32_t*>(plain);
  uint32_t* o_rows = reinterpret_cast<uint32_t*>(rht_rows);
  uint32_t* o_cols = reinterpret_cast<uint32_t*>(rht_cols);
  for (uint32_t* o : {o_plain, o_rows, o_cols}) {
    if (!o) continue;
    const cudaError_t e = cudaMemsetAsync(o, 0, 4, s);
    if (e != cudaSuccess) return e;
  }
  const int64_t n = rows * cols;
  if (n == 0) return cudaSuccess;
  if ((rows / 16) * (cols / 8) >= kMaxUnits) return cudaErrorInvalidValue;
  // the plain amax rides along with the first transform pass that runs
  if (o_cols) {
    const int64_t units = (rows / 16) * (cols / 8);
    amax_rht_cols_kernel<<<grid_for(units, 4), kThreads, 0, s>>>(static_cast<const uint16_t*>(x), rows, cols,
                                                                 rht_seed, o_plain, o_cols, status);
    count_launch();
    o_plain = nullptr;
  }
  if (o_rows) {
    const int64_t units = n / 16;
    amax_rht_rows_kernel<<<grid_for(units, 8), kThreads, 0, s>>>(static_cast<const uint4*>(x), units, rht_seed,
                                                                 o_plain, o_rows, status);
    count_launch();
    o_plain = nullptr;
  }
  if (o_plain) {
    const int64_t nv = n / 8;
    amax_plain_kernel<<<grid_for(nv / 4 + 1, 8), kThreads, 0, s>>>(static_cast<const uint4*>(x), nv, o_plain,
                                                                   status);
    count_launch();
  }
  return cudaGetLastError();
}

namespace {

template <bool kRHT>
cudaError_t launch_rowwise_ring(const void* x, int64_t rows, int64_t cols, const nvfp4_tensor& out,
                                const float* amax, uint64_t seed, cudaStream_t s) {
  const int64_t tiles = ring_tiles(rows, cols);
  if (tiles >= kRingMaxTiles) return cudaErrorInvalidValue;
  CUtensorMap map;
  if (!make_ring_map(&map, x, rows, cols)) return cudaErrorInvalidValue;
  auto kern = quant_rowwise_ring_kernel<kRHT>;
  static std::atomic<bool> attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  kern<<<ring_grid(tiles, 3), kRingThreads, kRingSmemBytes, s>>>(map, rows, cols, amax, out.codes, out.scales,
                                                                  out.scale_layout, out.tensor_scale, seed,
                                                                  device_status_ptr(), take_ring_debug_stall());
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_rowwise(const void* x, int64_t rows, int64_t cols, const nvfp4_tensor& out,
                                 const float* amax, bool rht, bool sr, uint64_t seed, uint32_t stream_id,
                                 cudaStream_t s) {
  if (!sr) return rht ? launch_rowwise_ring<true>(x, rows, cols, out, amax, seed, s)
                      : launch_rowwise_ring<false>(x, rows, cols, out, amax, seed, s);
  const int64_t units = rows * (cols / 64);
  if (units >= kMaxUnits) return cudaErrorInvalidValue;
  const int grid = grid_for(units, 8);
  const PhiloxKey key = philox_key(seed);
  auto args = [&](auto kern) {
    kern<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), rows, cols, amax, out.codes, out.scales,
                                   out.scale_layout, out.tensor_scale, seed, key, stream_id, device_status_ptr());
  };
  if (rht) args(quant_rowwise_kernel<true, true>);
  else args(quant_rowwise_kernel<true, false>);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_quant_tile(const void* x, int64_t rows, int64_t cols, const nvfp4_tensor* out_row,
                              const float* amax_row, const nvfp4_tensor* out_t, const float* amax_t, bool rht_t,
                              bool sr, uint64_t seed, uint32_t stream_row, uint32_t stream_t, cudaStream_t s) {
  TileOut orow{}, ot{};
  if (out_row) orow = TileOut{out_row->codes, out_row->scales, amax_row, out_row->tensor_scale, out_row->scale_layout,
                              stream_row};
  if (out_t) ot = TileOut{out_t->codes, out_t->scales, amax_t, out_t->tensor_scale, out_t->scale_layout, stream_t};
  const bool row = out_row != nullptr, tr = out_t != nullptr;
  uint32_t* status = device_status_ptr();
  if (!sr) {  // round-to-nearest-even: the ring kernel
    const int64_t tiles = ring_tiles(rows, cols);
    if (tiles >= kRingMaxTiles) return cudaErrorInvalidValue;
    CUtensorMap map;
    if (!make_ring_map(&map, x, rows, cols)) return cudaErrorInvalidValue;
    int dev = 0;
    cudaGetDevice(&dev);
    auto run = [&](auto kern, std::atomic<bool>* attr_set) -> cudaError_t {
      if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
      }
      kern<<<ring_grid(tiles, kTileRingCtas), kRingThreads, kRingSmemBytes, s>>>(map, rows, cols, orow, ot, seed,
                                                                                  status, take_ring_debug_stall());
      count_launch();
      return cudaGetLastError();
    };
#define NVFP4_RING(R, T, H)                                \
  do {                                                     \
    static std::atomic<bool> attr_set[64] = {};           \
    return run(quant_tile_ring_kernel<R, T, H>, attr_set); \
  } while (0)
    if (row && tr) {
      if (rht_t) NVFP4_RING(true, true, true);
      NVFP4_RING(true, true, false);
    }
    if (tr) {
      if (rht_t) NVFP4_RING(false, true, true);
      NVFP4_RING(false, true, false);
    }
    NVFP4_RING(true, false, false);
#undef NVFP4_RING
  }
  // stochastic rounding: the register-staged tile kernel
  const int64_t tiles = ((rows + kTileRows - 1) / kTileRows) * (cols / kTile);
  if (tiles >= kMaxUnits) return cudaErrorInvalidValue;
  const int64_t cap = (int64_t)sm_count() * 8;
  const dim3 grid((unsigned)(tiles < cap ? (tiles > 0 ? tiles : 1) : cap));
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  const PhiloxKey key = philox_key(seed);
#define NVFP4_TILE(R, T, H) \
  quant_tile_kernel<R, T, H, true><<<grid, kThreads, 0, s>>>(xp, rows, cols, orow, ot, seed, key, status)
  if (row && tr) {
    if (rht_t) NVFP4_TILE(true, true, true);
    else NVFP4_TILE(true, true, false);
  } else if (tr) {
    if (rht_t) NVFP4_TILE(false, true, true);
    else NVFP4_TILE(false, true, false);
  } else {
    NVFP4_TILE(true, false, false);
  }
#undef NVFP4_TILE
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_quant_2d(const void* w, int64_t rows, int64_t cols, const nvfp4_tensor& out,
                            const nvfp4_tensor* out_t, const float* amax, cudaStream_t s) {
  TileOut ow{out.codes, out.scales, amax, out.tensor_scale, out.scale_layout, 0};
  TileOut owt{};
  if (out_t) owt = TileOut{out_t->codes, out_t->scales, amax, out_t->tensor_scale, out_t->scale_layout, 0};
  const int64_t tiles = ring_tiles(rows, cols);
  if (tiles >= kRingMaxTiles) return cudaErrorInvalidValue;
  CUtensorMap map;
  if (!make_ring_map(&map, w, rows, cols)) return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(quant_2d_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  quant_2d_ring_kernel<<<ring_grid(tiles, 3), kRingThreads, kRingSmemBytes, s>>>(
      map, rows, cols, amax, ow, owt, out_t ? 1 : 0, device_status_ptr(), take_ring_debug_stall());
  count_launch();
  return cudaGetLastError();
}

}  // namespace nvfp4
