// tile_ring.cuh -- a persistent TMA pipeline over the 128 x 64 BF16 tiles of
// a row-major [rows, cols] tensor, shared by the quantization kernels that
// read each tile once and write rowwise and/or transposed outputs from it.
//
// One producer warp streams this CTA's tiles (16 KB each, 128-byte swizzle:
// 16-byte chunk j of row r stored at chunk j ^ (r % 8)) into a 3-slot
// shared-memory ring with cp.async.bulk.tensor; 8 consumer warps wait for a
// tile, hand it to the kernel's consumer, and release the slot.  Every wait
// is bounded (device_async.cuh); on a timeout the consumers stop, the
// producer stops issuing, waits (bounded) for the loads it issued, and the
// kernel returns with NVFP4_ERR_TIMEOUT in the status word.  Rows past the
// end of the tensor read as zeros (rows % 64 == 0, so the last tile holds 64
// or 128 valid rows).
#pragma once

#include <cuda.h>

#include <cstdint>

#include "device_async.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kRingConsumerWarps = 8;
constexpr int kRingThreads = 32 * (kRingConsumerWarps + 1);  // + the producer warp
constexpr int kRingTileRows = 128;
constexpr int kRingTileCols = 64;
constexpr int kRingTileBytes = kRingTileRows * kRingTileCols * 2;
constexpr int kRingStages = 3;
constexpr int kRingSmemBytes = kRingStages * kRingTileBytes + 1024;  // + alignment of the ring to 1024 B
constexpr int64_t kRingMaxTiles = int64_t(1) << 31;

// Number of tiles of a [rows, cols] tensor (rows % 64 == 0, cols % 64 == 0).
__host__ __device__ inline int64_t ring_tiles(int64_t rows, int64_t cols) {
  return ((rows + kRingTileRows - 1) / kRingTileRows) * (cols / kRingTileCols);
}

// Byte offset of the 16-byte chunk j (elements 8j .. 8j+7) of tile row r.
__device__ __forceinline__ uint32_t ring_chunk(int r, int j) { return (uint32_t)(r * 128 + (((j ^ r) & 7) << 4)); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Runs the pipeline; consume(tile, m0, c0, valid) is called by every thread
// of the 8 consumer warps (threadIdx.x < 256) for each of this CTA's tiles in
// order: tile = shared-memory address of the swizzled tile, (m0, c0) its
// first row and column, valid its number of rows (64 or 128).  smem_raw is
// the kernel's dynamic shared memory (kRingSmemBytes).  Everything the
// consumers set up before the call is ordered before the first tile by the
// barrier below.
// With debug_stall set (a failure-detection test hook), CTA 0 never issues
// the load of its first tile: its consumers' wait for that tile runs into its
// bound, the kernel reports NVFP4_ERR_TIMEOUT and returns.
template <class Consume>
__device__ __forceinline__ void tile_ring(const CUtensorMap* xmap, int64_t rows, int64_t cols, uint32_t* status,
                                          int debug_stall, uint8_t* smem_raw, Consume&& consume) {
  __shared__ __align__(8) uint64_t bars[2 * kRingStages];  // full[s], empty[s]
  __shared__ int abort_flag;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms are 1024 B
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(kRingStages + s); };
  volatile int* abort = &abort_flag;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  if (t == 0) {
    for (int s = 0; s < kRingStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kRingConsumerWarps);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const uint32_t tiles_c = (uint32_t)(cols / kRingTileCols);
  const uint32_t n_tiles = (uint32_t)ring_tiles(rows, cols);  // < 2^31 (launchers)
  if (warp == kRingConsumerWarps) {
    if (lane == 0) {
      int n = 0;
      uint32_t issued = 0;  // bit s: the latest tile of slot s had its load issued
      for (uint32_t tl = blockIdx.x; tl < n_tiles; tl += gridDim.x, ++n) {
        const int s = n % kRingStages;
        if (n >= kRingStages && !mbar_wait(empty_bar(s), (uint32_t)((n / kRingStages) - 1) & 1u, abort, status))
          break;
        if (debug_stall && n == 0 && blockIdx.x == 0) {  // nothing issued or armed for this tile
          issued &= ~(1u << s);
          continue;
        }
        const uint32_t tm = tl / tiles_c, tc = tl - tm * tiles_c;
        mbar_arrive_expect_tx(full_bar(s), kRingTileBytes);
        tma_load_2d(ring + (uint32_t)s * kRingTileBytes, xmap, (int)(tc * kRingTileCols), (int)(tm * kRingTileRows),
                    full_bar(s));
        issued |= 1u << s;
      }
      // every load this CTA issued has landed before it exits: the last
      // kRingStages tiles' phases (the earlier ones were consumed), skipping a
      // tile whose load was never issued, each wait bounded and independent of
      // the abort flag
      volatile int never = 0;
      for (int k = n - kRingStages > 0 ? n - kRingStages : 0; k < n; ++k)
        if ((issued >> (k % kRingStages)) & 1u)
          mbar_wait(full_bar(k % kRingStages), (uint32_t)(k / kRingStages) & 1u, &never, status);
    }
  } else {
    int n = 0;
    for (uint32_t tl = blockIdx.x; tl < n_tiles; tl += gridDim.x, ++n) {
      const int s = n % kRingStages;
      if (!mbar_wait(full_bar(s), (uint32_t)(n / kRingStages) & 1u, abort, status)) break;
      const uint32_t tm = tl / tiles_c, tc = tl - tm * tiles_c;
      const int64_t m0 = (int64_t)tm * kRingTileRows, c0 = (int64_t)tc * kRingTileCols;
      const int valid = rows - m0 < kRingTileRows ? (int)(rows - m0) : kRingTileRows;
      consume(ring + (uint32_t)s * kRingTileBytes, m0, c0, valid);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
    }
  }
  __syncthreads();
}

// The failure-detection test flag of the next ring launch (taken once).
inline int take_ring_debug_stall() { return ring_debug_stall_flag().exchange(0); }

// 2D map over x [rows, cols] BF16 with the ring's box (64 columns x 128
// rows, 128-byte swizzle); rows past the end read as zeros.
inline bool make_ring_map(CUtensorMap* m, const void* x, int64_t rows, int64_t cols) {
  auto fn = tensor_map_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {kRingTileCols, kRingTileRows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Grid of a ring kernel: one CTA per tile up to ctas_per_sm per SM.
inline unsigned ring_grid(int64_t tiles, int ctas_per_sm) {
  const int64_t cap = (int64_t)device_sm_count() * ctas_per_sm;
  return (unsigned)(tiles < cap ? (tiles > 0 ? tiles : 1) : cap);
}

}  // namespace
}  // namespace nvfp4
