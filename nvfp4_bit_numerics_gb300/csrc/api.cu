// api.cu -- the C ABI declared in include/nvfp4.h: argument validation, the
// per-device status word, the linear-layer workspace layout and the Fprop /
// Dgrad / Wgrad orchestration.
//
// Method: "Pretraining Large Language Models with NVFP4" (gist.science
// summary), Resumo técnico §2 Metodologia.  One layer step enqueues, on the
// caller's stream:
//   fwd: amax(X) and amax(Hadamard(X^T)) in one read;
//        X -> {X rowwise RNE, X^T Hadamard RNE} in one read;
//        meanwhile, on the library's side stream of the device (forked from
//        and joined back into the caller's stream with events; on the
//        caller's stream itself while it is being captured): amax(W),
//        W -> {W, W^T} with 16x16 blocks (item 3);
//        Y = X W^T on the tensor cores.
//   bwd: amax(dY) and amax(Hadamard(dY^T)) in one read;
//        dY -> {dY rowwise SR, dY^T Hadamard SR} in one read (items 2, 4);
//        dX = dY W and dW = dY^T X on the tensor cores.
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace nvfp4 {

std::atomic<uint64_t> g_launches{0};

namespace {

__device__ uint32_t g_status_word;

std::atomic<uint32_t*> g_status_ptr[64] = {};

// Random stream ids of one layer step (Philox key = the step's seed).
constexpr uint32_t kStreamDy = 0;   // stochastic rounding of dY (Dgrad operand)
constexpr uint32_t kStreamDyT = 1;  // stochastic rounding of dY^T (Wgrad operand)

nvfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

// Codes and scales set and aligned, a known scale layout and format; an
// NVFP4 tensor also needs its tensor scale.
bool valid_tensor(const nvfp4_tensor* t) {
  if (!t || !t->codes || !t->scales || !aligned16(t->codes) || !aligned16(t->scales)) return false;
  if (t->scale_layout != NVFP4_SCALES_LINEAR && t->scale_layout != NVFP4_SCALES_MMA) return false;
  if (t->format == NVFP4_FORMAT_NVFP4) return t->tensor_scale != nullptr;
  return t->format == NVFP4_FORMAT_MXFP4;
}

bool layout_ok(const nvfp4_tensor* t) {
  if (t->scale_layout == NVFP4_SCALES_MMA) return t->rows % 128 == 0 && t->cols % 64 == 0;
  return true;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

std::atomic<int>& ring_debug_stall_flag() {
  static std::atomic<int> flag{0};
  return flag;
}

int device_sm_count() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 152;
  }
  return cached[dev];
}

uint32_t* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_status_ptr[dev];
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_ARG: return "invalid argument";
    case NVFP4_ERR_SHAPE: return "invalid shape";
    case NVFP4_ERR_ALIGN: return "misaligned pointer or pitch";
    case NVFP4_ERR_NONFINITE: return "non-finite amax";
    case NVFP4_ERR_TIMEOUT: return "device pipeline wait timed out";
    case NVFP4_ERR_CUDA: return "CUDA runtime error";
    case NVFP4_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

uint64_t nvfp4_kernel_launch_count(void) { return g_launches.load(); }

void nvfp4_debug_stall_next_gemm(int32_t on) { set_gemm_debug_stall(on); }

void nvfp4_debug_stall_next_quantize(int32_t on) { ring_debug_stall_flag().store(on ? 1 : 0); }

nvfp4_status nvfp4_get_status(nvfp4_stream stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return NVFP4_ERR_CUDA;
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_status_word, sizeof(w)) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (w) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  if (w & kStatusTimeout) return NVFP4_ERR_TIMEOUT;
  if (w & kStatusNonFinite) return NVFP4_ERR_NONFINITE;
  return NVFP4_OK;
}

size_t nvfp4_scale_bytes(int64_t rows, int64_t cols, int32_t layout) {
  if (rows < 0 || cols < 0) return 0;
  const int64_t nkb = cols / 16;
  if (layout == NVFP4_SCALES_MMA) return (size_t)(((rows + 127) / 128) * ((nkb + 3) / 4) * 512);
  return (size_t)(rows * nkb);
}

nvfp4_status nvfp4_amax(const void* x, int64_t rows, int64_t cols, int32_t flags, uint64_t rht_seed,
                        float* amax_dev, nvfp4_stream stream) {
  if (!amax_dev || (flags & ~7) || !flags) return NVFP4_ERR_ARG;
  if (rows < 0 || cols < 0 || cols % 16) return NVFP4_ERR_SHAPE;
  if ((flags & NVFP4_AMAX_RHT_COLS) && rows % 16) return NVFP4_ERR_SHAPE;
  if (rows * cols > 0 && (!x || !aligned16(x))) return x ? NVFP4_ERR_ALIGN : NVFP4_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(amax_dev) & 3u) != 0) return NVFP4_ERR_ALIGN;
  return from_cuda(launch_amax(x, rows, cols, (flags & NVFP4_AMAX_PLAIN) ? amax_dev : nullptr,
                               (flags & NVFP4_AMAX_RHT_ROWS) ? amax_dev + 1 : nullptr,
                               (flags & NVFP4_AMAX_RHT_COLS) ? amax_dev + 2 : nullptr, rht_seed,
                               static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, const nvfp4_quant_cfg* cfg,
                            const nvfp4_tensor* out, const nvfp4_tensor* out_t, nvfp4_stream stream) {
  if (!cfg || !x) return NVFP4_ERR_ARG;
  if (cfg->kind < NVFP4_Q_ROWWISE || cfg->kind > NVFP4_Q_2D) return NVFP4_ERR_ARG;
  if (cfg->rounding != NVFP4_ROUND_RNE && cfg->rounding != NVFP4_ROUND_SR) return NVFP4_ERR_ARG;
  if (rows <= 0 || cols <= 0 || rows % 64 || cols % 64) return NVFP4_ERR_SHAPE;
  if (!aligned16(x)) return NVFP4_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool sr = cfg->rounding == NVFP4_ROUND_SR;
  const bool rht = cfg->rht != 0;
  const nvfp4_tensor* o_row = nullptr;
  const nvfp4_tensor* o_t = nullptr;
  switch (cfg->kind) {
    case NVFP4_Q_ROWWISE: o_row = out; break;
    case NVFP4_Q_TRANSPOSE: o_t = out; break;
    case NVFP4_Q_ROWWISE_AND_TRANSPOSE: o_row = out; o_t = out_t; break;
    case NVFP4_Q_2D: o_row = out; o_t = out_t; break;
  }
  if (!o_row && !o_t) return NVFP4_ERR_ARG;
  if (cfg->kind == NVFP4_Q_ROWWISE_AND_TRANSPOSE && !o_t) return NVFP4_ERR_ARG;
  for (const nvfp4_tensor* t : {o_row, o_t}) {
    if (!t) continue;
    if (!valid_tensor(t) || !t->amax || t->format != NVFP4_FORMAT_NVFP4) return NVFP4_ERR_ARG;
    if (!layout_ok(t)) return NVFP4_ERR_SHAPE;
  }
  if (o_row && (o_row->rows != rows || o_row->cols != cols)) return NVFP4_ERR_SHAPE;
  if (o_t && (o_t->rows != cols || o_t->cols != rows)) return NVFP4_ERR_SHAPE;

  cudaError_t e = cudaSuccess;
  if (cfg->kind == NVFP4_Q_2D) {
    if (cfg->compute_amax) {
      e = launch_amax(x, rows, cols, o_row->amax, nullptr, nullptr, 0, s);
      // the W^T output shares W's amax
      if (e == cudaSuccess && o_t && o_t->amax != o_row->amax)
        e = cudaMemcpyAsync(o_t->amax, o_row->amax, sizeof(float), cudaMemcpyDeviceToDevice, s);
      if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    }
    return from_cuda(launch_quant_2d(x, rows, cols, *o_row, o_t, o_row->amax, s));
  }

  if (cfg->compute_amax) {
    float* a_row = o_row ? o_row->amax : nullptr;
    float* a_t = o_t ? o_t->amax : nullptr;
    if (cfg->kind == NVFP4_Q_ROWWISE) {
      e = rht ? launch_amax(x, rows, cols, nullptr, a_row, nullptr, cfg->seed, s)
              : launch_amax(x, rows, cols, a_row, nullptr, nullptr, 0, s);
    } else if (rht) {
      // one read gives max|x| (rowwise output) and max|Q x| along rows
      e = launch_amax(x, rows, cols, a_row, nullptr, a_t, cfg->seed, s);
    } else {
      e = launch_amax(x, rows, cols, a_t, nullptr, nullptr, 0, s);
      if (e == cudaSuccess && a_row && a_row != a_t)
        e = cudaMemcpyAsync(a_row, a_t, sizeof(float), cudaMemcpyDeviceToDevice, s);
    }
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  if (cfg->kind == NVFP4_Q_ROWWISE)
    return from_cuda(launch_quant_rowwise(x, rows, cols, *o_row, o_row->amax, rht, sr, cfg->seed, cfg->sr_stream, s));
  // `out` takes sr_stream; the transposed output of the fused kind takes sr_stream_t
  const uint32_t stream_t = cfg->kind == NVFP4_Q_TRANSPOSE ? cfg->sr_stream : cfg->sr_stream_t;
  return from_cuda(launch_quant_tile(x, rows, cols, o_row, o_row ? o_row->amax : nullptr, o_t, o_t->amax, rht, sr,
                                     cfg->seed, cfg->sr_stream, stream_t, s));
}

size_t nvfp4_mx_scale_bytes(int64_t rows, int64_t cols, int32_t layout) {
  if (rows < 0 || cols < 0) return 0;
  // the MMA layout pads each pair of 32-element scales to a 4-byte word
  if (layout == NVFP4_SCALES_MMA) return nvfp4_scale_bytes(rows, cols, layout);
  return (size_t)(rows * (cols / 32));
}

nvfp4_status nvfp4_quantize_mx(const void* x, int64_t rows, int64_t cols, int32_t kind, const nvfp4_tensor* out,
                               const nvfp4_tensor* out_t, nvfp4_stream stream) {
  if (!x) return NVFP4_ERR_ARG;
  const nvfp4_tensor* o_row = nullptr;
  const nvfp4_tensor* o_t = nullptr;
  switch (kind) {
    case NVFP4_Q_ROWWISE: o_row = out; break;
    case NVFP4_Q_TRANSPOSE: o_t = out; break;
    case NVFP4_Q_ROWWISE_AND_TRANSPOSE:
      o_row = out;
      o_t = out_t;
      if (!o_t) return NVFP4_ERR_ARG;
      break;
    default: return NVFP4_ERR_ARG;
  }
  if (!o_row && !o_t) return NVFP4_ERR_ARG;
  if (rows <= 0 || cols <= 0 || rows % 64 || cols % 64) return NVFP4_ERR_SHAPE;
  if (!aligned16(x)) return NVFP4_ERR_ALIGN;
  for (const nvfp4_tensor* t : {o_row, o_t}) {
    if (!t) continue;
    if (!valid_tensor(t) || t->format != NVFP4_FORMAT_MXFP4) return NVFP4_ERR_ARG;
    if (!layout_ok(t)) return NVFP4_ERR_SHAPE;
  }
  if (o_row && (o_row->rows != rows || o_row->cols != cols)) return NVFP4_ERR_SHAPE;
  if (o_t && (o_t->rows != cols || o_t->cols != rows)) return NVFP4_ERR_SHAPE;
  return from_cuda(launch_quant_mx(x, rows, cols, o_row, o_t, static_cast<cudaStream_t>(stream)));
}

namespace {

// Argument checks shared by the GEMM entry points (nothing launched).
nvfp4_status check_gemm(const nvfp4_tensor* a, const nvfp4_tensor* b, const void* d, int32_t d_dtype,
                        int64_t ldd) {
  if (!valid_tensor(a) || !valid_tensor(b) || !d) return NVFP4_ERR_ARG;
  if (a->format != b->format) return NVFP4_ERR_ARG;
  if (d_dtype != NVFP4_OUT_BF16 && d_dtype != NVFP4_OUT_F32) return NVFP4_ERR_ARG;
  if (a->scale_layout != NVFP4_SCALES_MMA || b->scale_layout != NVFP4_SCALES_MMA) return NVFP4_ERR_ARG;
  const int64_t M = a->rows, N = b->rows, K = a->cols;
  if (M <= 0 || N <= 0 || K <= 0 || b->cols != K) return NVFP4_ERR_SHAPE;
  if (M % 128 || N % 128 || K % 64 || ldd < N) return NVFP4_ERR_SHAPE;
  if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return NVFP4_ERR_SHAPE;
  const int64_t esz = d_dtype == NVFP4_OUT_F32 ? 4 : 2;
  if (!aligned16(d) || (ldd * esz) % 16) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

}  // namespace

nvfp4_status nvfp4_gemm(const nvfp4_tensor* a, const nvfp4_tensor* b, void* d, int32_t d_dtype, int64_t ldd,
                        nvfp4_stream stream) {
  const nvfp4_status st = check_gemm(a, b, d, d_dtype, ldd);
  if (st != NVFP4_OK) return st;
  return launch_gemm(*a, *b, d, d_dtype, ldd, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_gemm2(const nvfp4_tensor* a0, const nvfp4_tensor* b0, void* d0, int64_t ldd0,
                         const nvfp4_tensor* a1, const nvfp4_tensor* b1, void* d1, int64_t ldd1,
                         nvfp4_stream stream) {
  nvfp4_status st = check_gemm(a0, b0, d0, NVFP4_OUT_BF16, ldd0);
  if (st != NVFP4_OK) return st;
  st = check_gemm(a1, b1, d1, NVFP4_OUT_BF16, ldd1);
  if (st != NVFP4_OK) return st;
  // the outputs' byte ranges (rows - 1 strides plus one row of BF16) must
  // not intersect: the two products' tiles run concurrently
  const uintptr_t p0 = reinterpret_cast<uintptr_t>(d0), p1 = reinterpret_cast<uintptr_t>(d1);
  const uintptr_t e0 = p0 + (uintptr_t)((a0->rows - 1) * ldd0 + b0->rows) * 2u;
  const uintptr_t e1 = p1 + (uintptr_t)((a1->rows - 1) * ldd1 + b1->rows) * 2u;
  if (p0 < e1 && p1 < e0) return NVFP4_ERR_ARG;
  return launch_gemm2(*a0, *b0, d0, ldd0, *a1, *b1, d1, ldd1, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_gemm_amax(const nvfp4_tensor* a, const nvfp4_tensor* b, void* d, int32_t d_dtype, int64_t ldd,
                             float* amax_dev, nvfp4_stream stream) {
  if (!amax_dev) return NVFP4_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(amax_dev) & 3u) != 0) return NVFP4_ERR_ALIGN;
  const nvfp4_status st = check_gemm(a, b, d, d_dtype, ldd);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(amax_dev, 0, sizeof(float), s) != cudaSuccess) return NVFP4_ERR_CUDA;
  return launch_gemm(*a, *b, d, d_dtype, ldd, s, amax_dev);
}

nvfp4_status nvfp4_gemm_quant(const nvfp4_tensor* a, const nvfp4_tensor* b, const nvfp4_tensor* y_q, void* d,
                              int64_t ldd, float* amax_dev, nvfp4_stream stream) {
  if (!y_q || !valid_tensor(y_q) || !y_q->amax || y_q->format != NVFP4_FORMAT_NVFP4) return NVFP4_ERR_ARG;
  if (y_q->scale_layout != NVFP4_SCALES_MMA) return NVFP4_ERR_ARG;
  if (amax_dev && amax_dev == y_q->amax) return NVFP4_ERR_ARG;  // the output amax would clear the input one
  // the GEMM checks, with the code buffer standing in for an absent BF16 output
  const nvfp4_status st = check_gemm(a, b, d ? d : y_q->codes, NVFP4_OUT_BF16, d ? ldd : b->rows);
  if (st != NVFP4_OK) return st;
  if (a->format != NVFP4_FORMAT_NVFP4) return NVFP4_ERR_ARG;
  if (a->rows % 256 || b->rows % 256) return NVFP4_ERR_SHAPE;
  if (y_q->rows != a->rows || y_q->cols != b->rows) return NVFP4_ERR_SHAPE;
  if (amax_dev && (reinterpret_cast<uintptr_t>(amax_dev) & 3u) != 0) return NVFP4_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (amax_dev && cudaMemsetAsync(amax_dev, 0, sizeof(float), s) != cudaSuccess) return NVFP4_ERR_CUDA;
  return launch_gemm(*a, *b, d, NVFP4_OUT_BF16, ldd, s, amax_dev, y_q);
}

// ---------------------------------------------------------------------------
// Linear layer
// ---------------------------------------------------------------------------
// Workspace: a 256-byte header of FP32 scalars, then six NVFP4 tensors, each
// region 256-byte aligned.  Header floats:
//   [0] amax X      [2] amax Q(X^T)   [3] amax W (shared by W and W^T)
//   [4] amax dY     [6] amax Q(dY^T)
//   [8..13] tensor scales of xq, wq, wtq, xtq, dyq, dytq
namespace {

struct WsLayout {
  size_t off_codes[6], off_scales[6], total;
  int64_t rows[6], cols[6];
};

WsLayout ws_layout(int64_t M, int64_t K, int64_t N) {
  WsLayout L{};
  const int64_t r[6] = {M, N, K, K, M, N};
  const int64_t c[6] = {K, K, N, M, N, M};
  size_t off = 256;
  for (int i = 0; i < 6; ++i) {
    L.rows[i] = r[i];
    L.cols[i] = c[i];
    L.off_codes[i] = off;
    off = align256(off + (size_t)(r[i] * c[i] / 2));
    L.off_scales[i] = off;
    off = align256(off + nvfp4_scale_bytes(r[i], c[i], NVFP4_SCALES_MMA));
  }
  L.total = off;
  return L;
}

void fill_views(uint8_t* ws, int64_t M, int64_t K, int64_t N, nvfp4_linear_views* v) {
  const WsLayout L = ws_layout(M, K, N);
  float* hdr = reinterpret_cast<float*>(ws);
  float* amax_of[6] = {hdr + 0, hdr + 3, hdr + 3, hdr + 2, hdr + 4, hdr + 6};
  nvfp4_tensor* t[6] = {&v->xq, &v->wq, &v->wtq, &v->xtq, &v->dyq, &v->dytq};
  for (int i = 0; i < 6; ++i) {
    t[i]->codes = ws + L.off_codes[i];
    t[i]->scales = ws + L.off_scales[i];
    t[i]->amax = amax_of[i];
    t[i]->tensor_scale = hdr + 8 + i;
    t[i]->rows = L.rows[i];
    t[i]->cols = L.cols[i];
    t[i]->scale_layout = NVFP4_SCALES_MMA;
    t[i]->format = NVFP4_FORMAT_NVFP4;
  }
}

// Per-device side stream and fork/join events of nvfp4_linear_fwd, created
// on first use.  The mutex is held while a call enqueues its fork, its side
// work and its join, so calls from several host threads do not interleave
// them (an event wait captures the event's state when it is enqueued).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mutex;
SideStream g_side[64];

cudaError_t side_stream(SideStream** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  SideStream& ss = g_side[dev];
  if (!ss.s) {
    if ((e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &ss;
  return cudaSuccess;
}

nvfp4_status check_linear(int64_t M, int64_t K, int64_t N, void* ws, size_t ws_bytes) {
  if (!ws) return NVFP4_ERR_ARG;
  if (M <= 0 || K <= 0 || N <= 0 || M % 128 || K % 128 || N % 128) return NVFP4_ERR_SHAPE;
  if (!aligned16(ws)) return NVFP4_ERR_ALIGN;
  if (ws_bytes < ws_layout(M, K, N).total) return NVFP4_ERR_WORKSPACE;
  return NVFP4_OK;
}

}  // namespace

size_t nvfp4_linear_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  if (M <= 0 || K <= 0 || N <= 0) return 0;
  return ws_layout(M, K, N).total;
}

nvfp4_status nvfp4_linear_get_views(void* ws, int64_t M, int64_t K, int64_t N, nvfp4_linear_views* views) {
  if (!ws || !views) return NVFP4_ERR_ARG;
  if (M <= 0 || K <= 0 || N <= 0 || M % 128 || K % 128 || N % 128) return NVFP4_ERR_SHAPE;
  fill_views(static_cast<uint8_t*>(ws), M, K, N, views);
  return NVFP4_OK;
}

nvfp4_status nvfp4_linear_fwd(const void* x, const void* w, int64_t M, int64_t K, int64_t N, uint64_t seed, void* y,
                              void* ws, size_t ws_bytes, nvfp4_stream stream) {
  nvfp4_status st = check_linear(M, K, N, ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  if (!x || !w || !y) return NVFP4_ERR_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return NVFP4_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  nvfp4_linear_views v;
  fill_views(static_cast<uint8_t*>(ws), M, K, N, &v);
  // W's quantization (HBM-bound) overlaps X's (partly ALU-bound).  Under
  // stream capture nothing is forked: a stream that joins a capture stays in
  // it until the capture ends, and the side stream is shared by every caller
  // on the device, so all of the layer is enqueued on the caller's stream.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();
    cap = cudaStreamCaptureStatusActive;
  }
  const bool fork = cap == cudaStreamCaptureStatusNone;
  std::unique_lock<std::mutex> lock(g_side_mutex, std::defer_lock);
  SideStream* ss = nullptr;
  cudaError_t e = cudaSuccess;
  if (fork) {
    lock.lock();
    e = side_stream(&ss);
    if (e == cudaSuccess) e = cudaEventRecord(ss->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->s, ss->fork, 0);
  }
  cudaStream_t sw = fork ? (ss ? ss->s : s) : s;
  if (e == cudaSuccess) e = launch_amax(w, N, K, v.wq.amax, nullptr, nullptr, 0, sw);
  if (e == cudaSuccess) e = launch_quant_2d(w, N, K, v.wq, &v.wtq, v.wq.amax, sw);
  if (e == cudaSuccess) e = launch_amax(x, M, K, v.xq.amax, nullptr, v.xtq.amax, seed, s);
  if (e == cudaSuccess)
    e = launch_quant_tile(x, M, K, &v.xq, v.xq.amax, &v.xtq, v.xtq.amax, true, false, seed, 0, 0, s);
  if (ss) {
    // join even after an error above, so the caller's stream never runs
    // ahead of side work that was enqueued
    const cudaError_t ej = cudaEventRecord(ss->join, ss->s);
    const cudaError_t ew = ej == cudaSuccess ? cudaStreamWaitEvent(s, ss->join, 0) : ej;
    if (e == cudaSuccess) e = ew;
  }
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  return launch_gemm(v.xq, v.wq, y, NVFP4_OUT_BF16, N, s);
}

nvfp4_status nvfp4_linear_bwd(const void* dy, int64_t M, int64_t K, int64_t N, uint64_t seed, void* dx, void* dw,
                              void* ws, size_t ws_bytes, nvfp4_stream stream) {
  nvfp4_status st = check_linear(M, K, N, ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  if (!dy || !dx || !dw) return NVFP4_ERR_ARG;
  if (!aligned16(dy) || !aligned16(dx) || !aligned16(dw)) return NVFP4_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  nvfp4_linear_views v;
  fill_views(static_cast<uint8_t*>(ws), M, K, N, &v);
  cudaError_t e = launch_amax(dy, M, N, v.dyq.amax, nullptr, v.dytq.amax, seed, s);
  if (e == cudaSuccess)
    e = launch_quant_tile(dy, M, N, &v.dyq, v.dyq.amax, &v.dytq, v.dytq.amax, true, true, seed, kStreamDy,
                          kStreamDyT, s);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  // Dgrad and Wgrad are independent: one launch for both when the CTA-pair
  // kernel takes both
  return launch_gemm2(v.dyq, v.wtq, dx, K, v.dytq, v.xtq, dw, K, s);
}

}  // extern "C"
