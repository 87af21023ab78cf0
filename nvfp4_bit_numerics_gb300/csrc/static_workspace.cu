// static_workspace.cu -- nvfp4_linear_fwd for callers that cannot allocate.
//
// nvfp4_linear_fwd needs a caller-provided device workspace for the quantized
// operands.  Some callers cannot allocate one: a plugin that lives inside a
// host framework whose allocator owns all of the GPU's memory and forbids
// direct cudaMalloc, or a service whose device-memory budget is fixed at
// start-up.  nvfp4_linear_fwd_noalloc gives them the same forward pass with
// the workspace taken from a fixed array that belongs to this library.
//
// The array (kStaticWorkspaceBytes) is a file-scope __device__ variable, so
// every GPU that loads the library holds it until the process exits.  Every
// call shares it and it keeps the last call's contents; nothing in it needs
// to start at zero (the forward pass writes each byte it reads, and zeroes its
// amax slots itself).  Two calls whose work overlaps on the GPU race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;  // 32 MiB; stated in include/nvfp4.h

static __device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];

// Device address of g_static_workspace per device, looked up once with that
// device current.  In host code the array's name is only a host-side
// stand-in, never a device address.  A reset of the device's primary context
// would move the array; calls after one are not supported (stated in
// include/nvfp4.h).
void* g_workspace_addr[64] = {nullptr};
std::mutex g_workspace_mutex;

nvfp4_status static_workspace_addr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_workspace_mutex);
  if (!g_workspace_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return NVFP4_ERR_CUDA;
    g_workspace_addr[dev] = p;
  }
  *out = g_workspace_addr[dev];
  return NVFP4_OK;
}

}  // namespace

extern "C" {

nvfp4_status nvfp4_linear_fwd_noalloc(const void* x_dev, const void* w_dev, int64_t M, int64_t K, int64_t N,
                                      uint64_t seed, void* y_dev, nvfp4_stream stream) {
  // sizes beyond the array are rejected before anything is launched
  const size_t need = nvfp4_linear_workspace_bytes(M, K, N);
  if (need == 0) return NVFP4_ERR_SHAPE;
  if (need > kStaticWorkspaceBytes) return NVFP4_ERR_WORKSPACE;
  void* ws = nullptr;
  const nvfp4_status st = static_workspace_addr(&ws);
  if (st != NVFP4_OK) return st;
  return nvfp4_linear_fwd(x_dev, w_dev, M, K, N, seed, y_dev, ws, kStaticWorkspaceBytes, stream);
}

}  // extern "C"
