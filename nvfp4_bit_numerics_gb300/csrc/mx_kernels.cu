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
// The kernel is bound by HBM bandwidth: 2 bytes read per element, 0.5 + 1/32
// bytes written per element and output.  One read of a 128 x 64 tile, staged
// in shared memory, feeds the rowwise output (threads 0-127, one 64-element
// row chunk each) and the transposed output (threads 128-255, one 64-row
// column chunk each), so every thread writes whole 32-byte code runs and one
// whole scale word.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerTile = 128;
constexpr int kColsPerTile = 64;
constexpr int kPitch = 72;  // uint16 per shared-memory row: 144 B, conflict-free 16-byte row reads
constexpr int64_t kMaxTiles = int64_t(1) << 31;

struct MxOut {
  uint8_t* codes;
  uint8_t* scales;
  int layout;
};

// UE8M0 code of a block whose max |x| has the BF16 bits `amax16` (sign clear,
// finite), and the float32 multiplier 2^(127 - E).
__device__ __forceinline__ uint32_t mx_scale(uint32_t amax16, float& mult) {
  const int e = (int)((amax16 >> 7) & 0xFFu) - 2;
  const uint32_t E = e > 0 ? (uint32_t)e : 0u;
  mult = __uint_as_float((254u - E) << 23);
  return E;
}

// 32 values -> 16 bytes of codes (element 2j in the low nibble of byte j).
__device__ __forceinline__ uint4 mx_encode32(const float* v, float mult) {
  float s[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) s[i] = __fmul_rn(v[i], mult);
  return make_uint4(e2m1x8_rn(s), e2m1x8_rn(s + 8), e2m1x8_rn(s + 16), e2m1x8_rn(s + 24));
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

template <bool kRow, bool kT>
__global__ void __launch_bounds__(kThreads, 4) mx_quant_tile_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                    int64_t cols, MxOut orow, MxOut ot) {
  __shared__ __align__(16) uint16_t tile[kRowsPerTile * kPitch];
  const int t = threadIdx.x;
  const uint32_t tiles_c = (uint32_t)(cols / kColsPerTile);
  const uint32_t n_tiles = (uint32_t)((rows + kRowsPerTile - 1) / kRowsPerTile) * tiles_c;  // < 2^31 (launcher)
  for (uint32_t tl = blockIdx.x; tl < n_tiles; tl += gridDim.x) {
    const uint32_t tm = tl / tiles_c, tc = tl - tm * tiles_c;
    const int64_t m0 = (int64_t)tm * kRowsPerTile, c0 = (int64_t)tc * kColsPerTile;
    const int valid = rows - m0 < kRowsPerTile ? (int)(rows - m0) : kRowsPerTile;  // 64 or 128
    uint4 q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int v = t + k * kThreads;  // row v/8, 8-element piece v%8
      q[k] = (v >> 3) < valid ? ldg_nc_v4(x + (m0 + (v >> 3)) * cols + c0 + (v & 7) * 8) : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();  // the previous tile's readers are done
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int v = t + k * kThreads;
      *reinterpret_cast<uint4*>(&tile[(v >> 3) * kPitch + (v & 7) * 8]) = q[k];
    }
    __syncthreads();

    if (t < 128) {
      if (kRow && t < valid) {
        const int64_t gr = m0 + t;
        uint32_t E[2];
        uint4 o[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint4* sp = reinterpret_cast<const uint4*>(&tile[t * kPitch + 32 * b]);
          uint4 w[4];
          uint32_t m = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            w[i] = sp[i];
            m = __vmaxu2(m, __vmaxu2(__vmaxu2(w[i].x & 0x7FFF7FFFu, w[i].y & 0x7FFF7FFFu),
                                     __vmaxu2(w[i].z & 0x7FFF7FFFu, w[i].w & 0x7FFF7FFFu)));
          }
          float mult;
          E[b] = mx_scale(max(m & 0xFFFFu, m >> 16), mult);
          float v[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) unpack8(w[i], v + 8 * i);
          o[b] = mx_encode32(v, mult);
        }
        uint4* cp = reinterpret_cast<uint4*>(orow.codes + gr * (cols >> 1) + (c0 >> 1));
        cp[0] = o[0];
        cp[1] = o[1];
        mx_store_scales(orow, gr, c0 >> 6, cols, E[0], E[1]);
      }
    } else if (kT) {
      const int u = t - 128, c = u & 63, h = u >> 6;  // tile column, 64-row half
      if (64 * h < valid) {
        const int64_t gr = c0 + c, gm = m0 + 64 * h;  // row and first column of the transposed tensor
        uint32_t E[2];
        uint4 o[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float v[32];
          uint32_t m = 0;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint32_t w = tile[(64 * h + 32 * b + i) * kPitch + c];
            m = max(m, w & 0x7FFFu);
            v[i] = __uint_as_float(w << 16);
          }
          float mult;
          E[b] = mx_scale(m, mult);
          o[b] = mx_encode32(v, mult);
        }
        uint4* cp = reinterpret_cast<uint4*>(ot.codes + gr * (rows >> 1) + (gm >> 1));
        cp[0] = o[0];
        cp[1] = o[1];
        mx_store_scales(ot, gr, gm >> 6, rows, E[0], E[1]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_quant_mx(const void* x, int64_t rows, int64_t cols, const nvfp4_tensor* out_row,
                            const nvfp4_tensor* out_t, cudaStream_t s) {
  MxOut orow{}, ot{};
  if (out_row) orow = MxOut{out_row->codes, out_row->scales, out_row->scale_layout};
  if (out_t) ot = MxOut{out_t->codes, out_t->scales, out_t->scale_layout};
  const int64_t tiles = ((rows + kRowsPerTile - 1) / kRowsPerTile) * (cols / kColsPerTile);
  if (tiles >= kMaxTiles) return cudaErrorInvalidValue;
  if (tiles == 0) return cudaSuccess;
  const int64_t cap = (int64_t)device_sm_count() * 4;
  const unsigned grid = (unsigned)(tiles < cap ? tiles : cap);
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  if (out_row && out_t) mx_quant_tile_kernel<true, true><<<grid, kThreads, 0, s>>>(xp, rows, cols, orow, ot);
  else if (out_t) mx_quant_tile_kernel<false, true><<<grid, kThreads, 0, s>>>(xp, rows, cols, orow, ot);
  else mx_quant_tile_kernel<true, false><<<grid, kThreads, 0, s>>>(xp, rows, cols, orow, ot);
  count_launch();
  return cudaGetLastError();
}

}  // namespace nvfp4
