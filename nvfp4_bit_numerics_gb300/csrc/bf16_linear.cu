// bf16_linear.cu -- the linear layers the method keeps in BF16.
//
// Method: "Pretraining Large Language Models with NVFP4" (gist.science
// summary), Resumo técnico §2, item 1 ("Precisão Mista Seletiva"): the
// sensitive linear layers -- the last ones of the network, about 15% -- stay
// in BF16 while the rest trains in NVFP4.  Such a layer runs the same three
// GEMMs without quantization: Y = X W^T, dX = dY W, dW = dY^T X, BF16 in and
// out with FP32 accumulation.  These are plain dense GEMMs, so they go to
// cuBLAS (cublasGemmEx, CUBLAS_COMPUTE_32F).
//
// Row-major [r, c] buffers are column-major [c, r] matrices to cuBLAS, so
// each product is issued as its transpose:
//   Y^T  [N, M] = W   X^T   -> (op T on w [K, N]) x (x [K, M])
//   dX^T [K, M] = W^T dY^T  -> (w [K, N]) x (dy [N, M])
//   dW^T [K, N] = X^T dY    -> (x [K, M]) x (op T on dy [N, M])
// (the bracketed shapes are the column-major views of the row-major inputs).
#include <cublas_v2.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace nvfp4 {
namespace {

// One cuBLAS handle per device, created on first use.  The mutex is held
// while a call binds the handle to its stream and enqueues its GEMMs.
std::mutex g_blas_mutex;
cublasHandle_t g_blas[64] = {nullptr};

cublasHandle_t blas_handle() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!g_blas[dev]) {
    cublasHandle_t h = nullptr;
    if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return nullptr;
    g_blas[dev] = h;
  }
  return g_blas[dev];
}

// C (col-major m x n, ldc) = op(A) op(B), BF16 operands, FP32 accumulation.
bool gemm_bf16(cublasHandle_t h, cublasOperation_t ta, cublasOperation_t tb, int64_t m, int64_t n, int64_t k,
               const void* a, int64_t lda, const void* b, int64_t ldb, void* c, int64_t ldc) {
  const float one = 1.0f, zero = 0.0f;
  return cublasGemmEx(h, ta, tb, (int)m, (int)n, (int)k, &one, a, CUDA_R_16BF, (int)lda, b, CUDA_R_16BF, (int)ldb,
                      &zero, c, CUDA_R_16BF, (int)ldc, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) ==
         CUBLAS_STATUS_SUCCESS;
}

nvfp4_status check_bf16(int64_t M, int64_t K, int64_t N) {
  if (M <= 0 || K <= 0 || N <= 0 || K % 8 || N % 8) return NVFP4_ERR_SHAPE;
  if (M > (1 << 30) || K > (1 << 30) || N > (1 << 30)) return NVFP4_ERR_SHAPE;
  return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

nvfp4_status nvfp4_linear_bf16_fwd(const void* x, const void* w, int64_t M, int64_t K, int64_t N, void* y,
                                   nvfp4_stream stream) {
  const nvfp4_status st = check_bf16(M, K, N);
  if (st != NVFP4_OK) return st;
  if (!x || !w || !y) return NVFP4_ERR_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return NVFP4_ERR_ALIGN;
  std::lock_guard<std::mutex> lock(g_blas_mutex);
  cublasHandle_t h = blas_handle();
  if (!h || cublasSetStream(h, static_cast<cudaStream_t>(stream)) != CUBLAS_STATUS_SUCCESS) return NVFP4_ERR_CUDA;
  return gemm_bf16(h, CUBLAS_OP_T, CUBLAS_OP_N, N, M, K, w, K, x, K, y, N) ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status nvfp4_linear_bf16_bwd(const void* dy, const void* x, const void* w, int64_t M, int64_t K, int64_t N,
                                   void* dx, void* dw, nvfp4_stream stream) {
  const nvfp4_status st = check_bf16(M, K, N);
  if (st != NVFP4_OK) return st;
  if (!dy || !x || !w || !dx || !dw) return NVFP4_ERR_ARG;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(w) || !aligned16(dx) || !aligned16(dw)) return NVFP4_ERR_ALIGN;
  std::lock_guard<std::mutex> lock(g_blas_mutex);
  cublasHandle_t h = blas_handle();
  if (!h || cublasSetStream(h, static_cast<cudaStream_t>(stream)) != CUBLAS_STATUS_SUCCESS) return NVFP4_ERR_CUDA;
  if (!gemm_bf16(h, CUBLAS_OP_N, CUBLAS_OP_N, K, M, N, w, K, dy, N, dx, K)) return NVFP4_ERR_CUDA;
  return gemm_bf16(h, CUBLAS_OP_N, CUBLAS_OP_T, K, N, M, x, K, dy, N, dw, K) ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // extern "C"
