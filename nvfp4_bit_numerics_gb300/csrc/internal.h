// internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "nvfp4.h"

namespace nvfp4 {

// Bits of the per-device status word.
constexpr uint32_t kStatusNonFinite = 1u << 4;
constexpr uint32_t kStatusTimeout = 1u << 5;

// Per-device status word (a __device__ variable of api.cu), as a device
// address usable by kernels of every translation unit.  Sets cudaError on
// failure and returns nullptr.
uint32_t* device_status_ptr();

// Host-side count of kernels launched by the library (for the bench's
// launch accounting).
extern std::atomic<uint64_t> g_launches;
inline void count_launch(uint64_t n = 1) { g_launches.fetch_add(n, std::memory_order_relaxed); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled of the driver, resolved once (nullptr if the driver
// does not provide it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encode_fn();

// Number of SMs of the current device (cached per device; 152 if the query
// fails).
int device_sm_count();

// Quantize launchers (quant_kernels.cu).  Arguments are already validated.
// Each non-null output is zeroed and then receives its amax: max|x|, max|Qx|
// with Q along the contiguous dimension, max|Qx| with Q along rows.
cudaError_t launch_amax(const void* x, int64_t rows, int64_t cols, float* plain, float* rht_rows, float* rht_cols,
                        uint64_t rht_seed, cudaStream_t s);
cudaError_t launch_quant_rowwise(const void* x, int64_t rows, int64_t cols, const nvfp4_tensor& out,
                                 const float* amax, bool rht, bool sr, uint64_t seed, uint32_t stream_id,
                                 cudaStream_t s);
cudaError_t launch_quant_tile(const void* x, int64_t rows, int64_t cols, const nvfp4_tensor* out_row,
                              const float* amax_row, const nvfp4_tensor* out_t, const float* amax_t,
                              bool rht_t, bool sr, uint64_t seed, uint32_t stream_row, uint32_t stream_t,
                              cudaStream_t s);
cudaError_t launch_quant_2d(const void* w, int64_t rows, int64_t cols, const nvfp4_tensor& out,
                            const nvfp4_tensor* out_t, const float* amax, cudaStream_t s);

// MXFP4 quantization (mx_kernels.cu): x [rows, cols] BF16 -> out_row
// [rows, cols] and/or out_t [cols, rows], 1x32 blocks, UE8M0 scales, RNE.
// Arguments are already validated (rows % 64 == 0, cols % 64 == 0).
cudaError_t launch_quant_mx(const void* x, int64_t rows, int64_t cols, const nvfp4_tensor* out_row,
                            const nvfp4_tensor* out_t, cudaStream_t s);

// Failure-detection test hook: the next GEMM launch never issues its first
// stage's loads, so its bounded waits run out (gemm_kernel.cu).
void set_gemm_debug_stall(int on);

// The same for the next TMA-ring quantize launch (tile_ring.cuh): CTA 0 never
// loads its first tile.  The flag lives in api.cu.
std::atomic<int>& ring_debug_stall_flag();

// GEMM launcher (gemm_kernel.cu).  Arguments are already validated.  With
// amax_out set (a zeroed device float), the epilogue also takes the max |D|
// over the BF16 (or FP32) output into it.  With yq set (BF16 output, M and N
// multiples of 256), the epilogue also quantizes the BF16 output into yq
// (1x16 RNE, MMA scale layout, tensor amax read from yq->amax); d may then be
// nullptr (no BF16 store).
nvfp4_status launch_gemm(const nvfp4_tensor& a, const nvfp4_tensor& b, void* d, int32_t d_dtype, int64_t ldd,
                         cudaStream_t s, float* amax_out = nullptr, const nvfp4_tensor* yq = nullptr);
// Two BF16-output GEMMs (d_i = a_i b_i^T) in one launch of the CTA-pair
// kernel when both take it and share the operand format, so that the second
// one's tiles fill the first one's last round; otherwise two launches.
nvfp4_status launch_gemm2(const nvfp4_tensor& a0, const nvfp4_tensor& b0, void* d0, int64_t ldd0,
                          const nvfp4_tensor& a1, const nvfp4_tensor& b1, void* d1, int64_t ldd1, cudaStream_t s);

}  // namespace nvfp4
