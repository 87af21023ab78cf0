// gemm_kernel.cu -- block-scaled FP4 (NVFP4) GEMM on the sm_103a tensor cores.
//
//   D[M, N] = ts_a * ts_b * sum_k e2m1(A[m,k]) e4m3(SA[m,k/16]) e2m1(B[n,k]) e4m3(SB[n,k/16])
//
// and, for MXFP4 operands (Params::mx; Resumo técnico §1, the 32-element,
// power-of-two-scaled format NVFP4 is compared with),
//
//   D[M, N] = sum_k e2m1(A[m,k]) 2^(SA[m,k/32]-127) e2m1(B[n,k]) 2^(SB[n,k/32]-127)
//
// with tcgen05.mma.kind::mxf4.block_scale.scale_vec::2X and UE8M0 scales.  The
// MXFP4 scales arrive in the same 512-byte tiles as the NVFP4 ones, each
// 4-byte word holding the two scales of a 64-element K chunk in bytes 0 and 1
// (the bytes the 2X MMA reads with scale-factor id 0), so everything but the
// MMA instruction and its descriptor is shared.
//
// The GEMMs of "Pretraining Large Language Models with NVFP4" (gist.science
// summary), Resumo técnico §3 ("Suporte de Hardware": Blackwell tensor cores
// take NVFP4 natively) -- Fprop, Dgrad and Wgrad of a linear layer, each a
// product of two K-major NVFP4 operands with FP32 accumulation.
//
// Two kernels.  For M and N multiples of 256, nvfp4_gemm_pair_kernel (CTA
// pairs, 256 x 256 tiles, tcgen05.mma.cta_group::2, scale tiles loaded with
// each operand stage and copied into tensor memory by tcgen05.cp from the
// MMA warp; described before it below).  It runs one GEMM, or two
// independent ones of the same operand format over one tile schedule (the
// Dgrad and Wgrad of a layer: the second GEMM's tiles fill the rounds the
// first leaves part-empty).  Otherwise the single-CTA kernel, whose design
// is:
// (one CTA per SM, persistent over 128 x BN output tiles)
//   warp 0      TMA producer: 2D tiled loads of the packed codes (128-byte
//               rows, 128B swizzle) and 1D bulk loads of the scale tiles,
//               into a ring of shared-memory stages guarded by mbarriers.
//   warp 1      owns the tensor memory; one lane waits one barrier per stage
//               (`sf_ready`, raised by the staging warps after the stage's
//               operands and scales landed), issues
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X with
//               the FP32 accumulator in tensor memory, then tcgen05.commit
//               frees the stage.
//   warps 2-5   scale staging: each warp (one per tensor-memory lane
//               quadrant) copies the stage's scale tiles from shared memory
//               into that stage's own tensor-memory scale columns with
//               tcgen05.st, so the tensor pipe runs MMAs only.
//   warps 6-13  epilogue: tcgen05.ld of the accumulator (each warp reads its
//               lane quadrant, half of the columns) with scaling by
//               ts_a * ts_b and BF16 rounding chunk by chunk, release of the
//               accumulator to the MMA warp, then the stores, overlapping the
//               next tile's main loop.
// Every mbarrier wait is bounded (%globaltimer); on expiry the kernel records
// NVFP4_ERR_TIMEOUT in the status word, drains its own copies and MMAs,
// frees tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <atomic>
#include <type_traits>

#include "device_async.cuh"
#include "device_common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kBM = 128;          // rows of A per tile (MMA M)
constexpr int kBKBytes = 128;     // bytes of K per stage per row = 256 FP4 values
constexpr int kMmaK = 64;         // FP4 values per MMA
constexpr int kKPerStage = 256;   // FP4 values per stage
constexpr int kNumThreads = 448;  // 14 warps
constexpr int kEpiWarps = 8;
constexpr int kSfWarps = 4;
constexpr int kFirstEpiWarp = 6;

template <int BN>
struct Cfg {
  static constexpr int kABytes = kBM * kBKBytes;
  static constexpr int kBBytes = BN * kBKBytes;
  static constexpr int kSfaBytes = (kBM / 128) * 4 * 512;
  static constexpr int kSfbBytes = (BN / 128) * 4 * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kStagesSmem = (220 * 1024) / kStageBytes > 8 ? 8 : (220 * 1024) / kStageBytes;
  static constexpr int kStagesTmem = (512 - BN) / (16 + 4 * (BN / 32));
  static constexpr int kStages = kStagesSmem < kStagesTmem ? kStagesSmem : kStagesTmem;
  static constexpr int kSfStageCols = 16 + 4 * (BN / 32);
  static constexpr int kSfaCol = BN;
  static constexpr int kSfbCol = BN + 16;
  static constexpr int kTmemCols = 512;
  static constexpr int kEpiCols = BN / 2;        // accumulator columns per epilogue warp
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes = kStages * kStageBytes + kBarBytes + 1024;
};

struct Params {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* ts_a;
  const float* ts_b;
  void* d;
  int64_t ldd;
  int d_f32;
  int M, N, K;
  int sf_tiles_k;  // 4-scale tiles per 128-row scale tile row = K / 64
  int n_fastest;   // tile order: 0 = walk M, 1 = walk N, >= 2 = walk N in groups of that many block rows
  int debug_stall; // failure-detection test: the first stage's loads are never issued
  int tma_store;   // pair kernel: BF16 output written by bulk tensor stores
  uint32_t* amax_out;  // if set: max |D| over the stored output, as float bits (atomicMax)
  int mx;              // operands are MXFP4 (UE8M0 scales per 32, no tensor scales)
  // pair kernel: the BF16 output quantized to NVFP4 (1x16, RNE) in the
  // epilogue, with the tensor amax given by the caller (q_codes != nullptr)
  uint8_t* q_codes;
  uint8_t* q_scales;
  const float* q_amax;
  float* q_ts;
  uint32_t* status;
};

// Tile index -> (m block, n block).  Consecutive tiles (which run at the same
// time on neighbouring SMs) walk the dimension whose operand is the smaller,
// so that operand stays resident in L2 while the larger one streams once.
// n_fastest >= 2 (the walked B operand too large to stay in L2 across waves
// of tiles): groups of n_fastest block rows, m fastest inside a group, so that
// the tiles in flight together touch fewer B slabs.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int n_fastest, int& mb, int& nb) {
  if (n_fastest >= 2) {
    const int G = n_fastest, per = G * num_n;
    const int g = tile / per, idx = tile - g * per;
    const int m_first = g * G;
    const int gl = num_m - m_first < G ? num_m - m_first : G;
    mb = m_first + idx % gl;
    nb = idx / gl;
  } else if (n_fastest) {
    nb = tile % num_n;
    mb = tile / num_n;
  } else {
    mb = tile % num_m;
    nb = tile / num_m;
  }
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128 B,
// 8-row swizzle atoms 1024 B apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1), K-major,
// UE4M3 scales, N >> 3 at bit 17, M >> 4 at bit 24, dense K = 64.
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same for MXFP4 operands: bit 23 selects UE8M0 scales.
__host__ __device__ constexpr uint32_t idesc_block_scaled(int M, int N, bool mx) {
  return idesc_mxf4nvf4(M, N) | (mx ? (1u << 23) : 0u);
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                       uint32_t accumulate, bool mx) {
  if (mx)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
  else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Output amax for the consumer of D (the next layer's quantization): the
// largest |value| as stored.  BF16: max over the magnitude bit patterns of
// packed pairs; FP32: max over the magnitude bits (NaN, whose bits exceed
// inf's, propagates).  One atomic per warp; non-negative float bits order
// like the floats.
template <int kWords>
__device__ __forceinline__ void amax_bf16_words(const uint32_t* packed, uint32_t* amax_out) {
  uint32_t m2 = 0;
#pragma unroll
  for (int i = 0; i < kWords; ++i) m2 = __vmaxu2(m2, packed[i] & 0x7FFF7FFFu);
  const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max(m2 & 0xFFFFu, m2 >> 16) << 16);
  if ((threadIdx.x & 31) == 0 && m) atomicMax(amax_out, m);
}
__device__ __forceinline__ void amax_bits_to_global(uint32_t m, uint32_t* amax_out) {
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31) == 0 && m) atomicMax(amax_out, m);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int BN>
__global__ void __launch_bounds__(kNumThreads, 1)
    nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                      Params p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bar_base = base + C::kStages * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + C::kStages * C::kStageBytes);
  // barrier slots: full[S], empty[S], tmem_full, tmem_empty, mma_done
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::kStages + s); };
  auto sf_bar = [&](int s) { return bar_base + 8u * (2 * C::kStages + s); };
  auto sf_full_bar = [&](int s) { return bar_base + 8u * (3 * C::kStages + s); };
  const uint32_t tmem_full = bar_base + 8u * (4 * C::kStages);
  const uint32_t tmem_empty = tmem_full + 8u;
  const uint32_t mma_done = tmem_full + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4 * C::kStages + 3);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = p.M / kBM, num_n = p.N / BN;
  const int n_tiles = num_m * num_n;
  const int k_stages = (p.K + kKPerStage - 1) / kKPerStage;
  const int last_nk = ((p.K - 1) % kKPerStage) / kMmaK + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sf_bar(s), kSfWarps);
      mbar_init(sf_full_bar(s), 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, kEpiWarps);
    mbar_init(mma_done, 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_phase = 0;  // per-stage bits, for the drain
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, num_m, num_n, p.n_fastest, mb, nb);
        for (int ks = 0; ks < k_stages; ++ks) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort, p.status)) { ok = false; break; }
          if (p.debug_stall && tile == (int)blockIdx.x && ks == 0) {
            // nothing is issued or armed for this stage: the consumers' bounded
            // waits run out and the kernel reports NVFP4_ERR_TIMEOUT
            if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
            continue;
          }
          const int nk = (ks == k_stages - 1) ? last_nk : 4;
          const uint32_t sf_bytes = (uint32_t)nk * 512u;
          const uint32_t sa = base + stage * C::kStageBytes;
          // scale tiles first, on their own barrier: their staging into
          // tensor memory overlaps the transfer of the operand tiles
          mbar_arrive_expect_tx(sf_full_bar(stage), sf_bytes * (1 + BN / 128));
          const uint32_t sfa_s = sa + C::kABytes + C::kBBytes;
          bulk_load(sfa_s, p.sfa + ((int64_t)mb * p.sf_tiles_k + ks * 4) * 512, sf_bytes, sf_full_bar(stage));
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            bulk_load(sfa_s + C::kSfaBytes + h * 2048,
                      p.sfb + ((int64_t)(nb * (BN / 128) + h) * p.sf_tiles_k + ks * 4) * 512, sf_bytes,
                      sf_full_bar(stage));
          mbar_arrive_expect_tx(full_bar(stage), C::kABytes + C::kBBytes);
          tma_load_2d(sa, &tmap_a, ks * kBKBytes, mb * kBM, full_bar(stage));
          tma_load_2d(sa + C::kABytes, &tmap_b, ks * kBKBytes, nb * BN, full_bar(stage));
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // drain: every issued stage's copies have landed before the CTA exits
      for (int s = 0; s < C::kStages; ++s)
        if (issued & (1u << s)) {
          volatile int never = 0;
          mbar_wait(sf_full_bar(s), (issued_phase >> s) & 1u, &never, p.status);
          mbar_wait(full_bar(s), (issued_phase >> s) & 1u, &never, p.status);
        }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ----------------------------
    // The loop is instantiated once per operand format, so the MMA issue path
    // carries no format test (a per-MMA branch slowed it by a quarter).
    auto issue = [&](auto mx_tag) {
      constexpr bool kMX = decltype(mx_tag)::value;
      const uint32_t idesc = idesc_block_scaled(kBM, BN, kMX);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(tmem_empty, acc_phase ^ 1u, abort, p.status)) break;
        tc_fence_after();
        for (int ks = 0; ks < k_stages; ++ks) {
          // sf_ready also covers `full`: the staging warps wait for it first
          if (!mbar_wait(sf_bar(stage), phase, abort, p.status)) { ok = false; break; }
          tc_fence_after();
          const int nk = (ks == k_stages - 1) ? last_nk : 4;
          const uint32_t sa = base + stage * C::kStageBytes;
          uint64_t da = desc_sw128(sa), db = desc_sw128(sa + C::kABytes);
          uint32_t sfa = tmem + (uint32_t)(stage * C::kSfStageCols + C::kSfaCol);
          uint32_t sfb = tmem + (uint32_t)(stage * C::kSfStageCols + C::kSfbCol);
          for (int j = 0; j < nk; ++j) {
            tc_mma(tmem, da, db, idesc, sfa, sfb, (ks | j) != 0, kMX);
            da += 2;  // +32 bytes along K inside the 128-byte swizzle atom
            db += 2;
            sfa += 4;
            sfb += BN / 32;
          }
          tc_commit(empty_bar(stage));
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tmem_full);
        acc_phase ^= 1u;
      }
    };
    if (lane == 0) {
      if (p.mx) issue(std::true_type{});
      else issue(std::false_type{});
      // all MMAs and copies issued by this thread have finished
      tc_commit(mma_done);
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, p.status);
    }
  } else if (warp < kFirstEpiWarp) {
    // ------------- scale factors: shared memory -> tensor memory -------------
    // The MMA reads the scales of row r from tensor-memory lane r, column
    // r/32 of the tile's 4 columns (replicated over the lane quadrants): lane
    // i, column c of a scale tile holds the c-th word of the 512-byte tile's
    // 16-byte row i.  Each stage has its own scale columns, so a stage's
    // columns are rewritten only after its previous MMAs completed (the
    // producer refills a stage, scale tiles first, only after the MMA commit
    // freed it, so `sf_full` of a stage also means its columns are free).
    const int q = warp & 3;
    int stage = 0;
    uint32_t phase = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
      bool ok = true;
      for (int ks = 0; ks < k_stages; ++ks) {
        int ready = 0;
        if (lane == 0)
          ready = (mbar_wait(sf_full_bar(stage), phase, abort, p.status) &&
                   mbar_wait(full_bar(stage), phase, abort, p.status)) ? 1 : 0;
        ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
        if (!ready) { ok = false; break; }
        const uint8_t* sfa_s = base_ptr + stage * C::kStageBytes + C::kABytes + C::kBBytes;
        const uint8_t* sfb_s = sfa_s + C::kSfaBytes;
        uint32_t r[C::kSfStageCols];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 w = *reinterpret_cast<const uint4*>(sfa_s + 512 * j + 16 * lane);
          r[4 * j] = w.x; r[4 * j + 1] = w.y; r[4 * j + 2] = w.z; r[4 * j + 3] = w.w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int h = 0; h < BN / 128; ++h) {
            const uint4 w = *reinterpret_cast<const uint4*>(sfb_s + 2048 * h + 512 * j + 16 * lane);
            const int o = 16 + (BN / 32) * j + 4 * h;
            r[o] = w.x; r[o + 1] = w.y; r[o + 2] = w.z; r[o + 3] = w.w;
          }
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(C::kSfaCol + stage * C::kSfStageCols);
#pragma unroll
        for (int c = 0; c < C::kSfStageCols / 16; ++c) tmem_st16(taddr + 16 * c, r + 16 * c);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sf_bar(stage));
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;
    const int half = (warp - kFirstEpiWarp) >> 2;
    const float alpha = p.mx ? 1.0f : __fmul_rn(*p.ts_a, *p.ts_b);
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
      int mb, nb;
        tile_coords(tile, num_m, num_n, p.n_fastest, mb, nb);
      // one lane waits, the warp follows its verdict (tcgen05.ld is warp-wide)
      int ready = 0;
      if (lane == 0) ready = mbar_wait(tmem_full, acc_phase, abort, p.status) ? 1 : 0;
      ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
      if (!ready) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(half * C::kEpiCols);
      const int64_t row = (int64_t)mb * kBM + 32 * q + lane;
      const int64_t col0 = (int64_t)nb * BN + half * C::kEpiCols;
      uint32_t packed[C::kEpiCols / 2];
      uint32_t m32 = 0;  // FP32 output: max magnitude bits
#pragma unroll
      for (int c = 0; c < C::kEpiCols / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(taddr + 32 * c, v);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (!p.d_f32) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[16 * c + i] = pack_bf16x2(__fmul_rn(alpha, __uint_as_float(v[2 * i])),
                                             __fmul_rn(alpha, __uint_as_float(v[2 * i + 1])));
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(p.d) + row * p.ldd + col0 + 32 * c);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 o = make_uint4(__float_as_uint(__fmul_rn(alpha, __uint_as_float(v[4 * i]))),
                                       __float_as_uint(__fmul_rn(alpha, __uint_as_float(v[4 * i + 1]))),
                                       __float_as_uint(__fmul_rn(alpha, __uint_as_float(v[4 * i + 2]))),
                                       __float_as_uint(__fmul_rn(alpha, __uint_as_float(v[4 * i + 3]))));
            dst[i] = o;
            m32 = max(m32, max(max(o.x & 0x7FFFFFFFu, o.y & 0x7FFFFFFFu), max(o.z & 0x7FFFFFFFu, o.w & 0x7FFFFFFFu)));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);
      acc_phase ^= 1u;
      if (!p.d_f32) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.d) + row * p.ldd + col0);
#pragma unroll
        for (int c = 0; c < C::kEpiCols / 8; ++c)
          dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        if (p.amax_out) amax_bf16_words<C::kEpiCols / 2>(packed, p.amax_out);
      } else if (p.amax_out) {
        amax_bits_to_global(m32, p.amax_out);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols) : "memory");
  }
}


// ---------------------------------------------------------------------------
// CTA-pair kernel: 256 x 256 output tiles, tcgen05.mma.cta_group::2.
// The two CTAs of a cluster each hold 128 rows of A and 128 of the 256 rows of
// B in shared memory (same offsets); one MMA issued by the even CTA computes
// all 256 x 256, each CTA's tensor memory receiving its own 128 rows.  Per SM
// this halves the MMA instructions and cuts the operand bytes per flop by a
// third relative to the single-CTA kernel.
//   warp 0      producer (both CTAs): waits its own `empty` barrier, then
//               loads the stage: its A and B halves (2D tiles, 128-byte
//               swizzle) and the stage's scale tiles (this CTA's 128 A rows,
//               all 256 B rows) as 2D tiles of 8-byte words; every copy
//               signals the even CTA's `full` barrier, which the even CTA's
//               producer armed for both CTAs' bytes.
//   warp 1      even CTA: the MMA warp.  The whole warp runs the loop in step
//               (so descriptors and addresses stay warp-uniform; a stage's
//               barrier is one test by all lanes, lane 0 waiting only when it
//               is not complete yet) and one lane, elected once, issues, per
//               stage: 12 tcgen05.cp.32x128b.warpx4
//               copies of the scale tiles from shared memory into the stage's
//               tensor-memory scale region (replicated into the four lane
//               quadrants, the layout the MMA reads), the 4 MMAs
//               (tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale), and a
//               commit that frees the stage in both CTAs.  Copies and MMAs
//               issued by one thread execute in order, so the copies of a
//               stage land before its MMAs read them.
//   warps 2-9   epilogue (both CTAs) for the CTA's 128 rows; each lane
//               reads its row's 128 accumulator columns with one wait and
//               the warp releases the accumulator at once (a remote arrive
//               on the even CTA for the odd CTA), then
//               write BF16 output as 32-row x 16-column boxes staged in a
//               1 KB shared-memory buffer per warp and sent with bulk tensor
//               stores.  Optionally each lane also takes the max |D| of its
//               values (amax_out) and quantizes its row's 128 BF16 values to
//               NVFP4 1x16 blocks with a given tensor amax (q_codes), writing
//               the codes and MMA-layout scales itself.
// Persistent: pair q of P walks its tiles in order, all three roles
// computing the same sequence.  One GEMM: tiles q, q + P, ...  Two GEMMs
// (kTwo; the second one's maps and parameters in g1): the PairSched order
// below, in which the pairs that the first GEMM's last round leaves idle start
// on the second one early.  The per-tile work is the same in both modes, so a
// GEMM gives the same bits either way.
// ---------------------------------------------------------------------------
constexpr int kPairBN = 256;
constexpr int kPairABytes = 128 * kBKBytes;  // per CTA
constexpr int kPairBBytes = 128 * kBKBytes;  // per CTA (half of B)
constexpr int kPairSfaBytes = 4 * 512;      // this CTA's 128 A rows, 4 MMAs
constexpr int kPairSfbBytes = 2 * 4 * 512;  // all 256 B rows, 4 MMAs
constexpr int kPairStageBytes = kPairABytes + kPairBBytes + kPairSfaBytes + kPairSfbBytes;  // 38 KB
constexpr int kPairSfCols = 16 + 4 * (kPairBN / 32);  // tensor-memory scale columns per stage
constexpr int kPairStages = 5;                        // shared-memory stages = tensor-memory scale regions
static_assert(kPairBN + kPairStages * kPairSfCols <= 512, "accumulator + scale regions exceed tensor memory");
static_assert(kPairStageBytes % 1024 == 0, "stages must keep the 1024-byte alignment of the swizzled tiles");
constexpr int kPairEpiWarps = 8;
constexpr int kPairFirstEpiWarp = 2;
constexpr int kPairEpiBufBytes = 1024;  // per epilogue warp: 32 rows x 16 BF16
constexpr int kPairBarBytes = 512;
constexpr int kPairSmemBytes = kPairStages * kPairStageBytes + kPairEpiWarps * kPairEpiBufBytes + kPairBarBytes + 1024;
static_assert(kPairSmemBytes <= 232448, "pair kernel shared memory exceeds the 227 KB opt-in limit");
constexpr int kPairThreads = 32 * (kPairFirstEpiWarp + kPairEpiWarps);
constexpr uint64_t kDrainNs = 50000;  // after an abort: time for loads already issued to land

// One GEMM of a pair-kernel launch: its operand, scale and output maps and
// its parameters.  A launch runs one GEMM, or two of the same operand format
// (the Dgrad and Wgrad of a layer) over one tile schedule.
struct alignas(64) PairProblem {
  CUtensorMap a, b, sfa, sfb, d;
  Params p;
};

// Tile schedule of a launch over P CTA pairs: the n0 tiles of problem 0 go
// round-robin (pair q takes q, q + P, ...; the first rem0 = n0 % P pairs take
// one more, "long" pairs), then the n1 tiles of problem 1: k1 head rounds over
// the S = P - rem0 short pairs only (they start on problem 1 one problem-0 tile
// earlier), then round-robin over all pairs.  Every tile of each problem goes
// to exactly one pair; consecutive tiles still run at the same time on
// neighbouring pairs (the L2 reuse the tile order is chosen for).
struct PairSched {
  int n0, n1, P, rem0, k1;
};

// The i-th tile of `pair` (false once the pair has no more tiles).
__device__ __forceinline__ bool pair_tile(const PairSched& sc, int pair, int i, int& prob, int& tile) {
  const int c0 = (sc.n0 - pair + sc.P - 1) / sc.P;  // this pair's problem-0 tiles
  if (i < c0) {
    prob = 0;
    tile = pair + i * sc.P;
    return true;
  }
  const int i1 = i - c0, S = sc.P - sc.rem0;
  int j;
  if (pair >= sc.rem0 && i1 < sc.k1)
    j = i1 * S + (pair - sc.rem0);
  else
    j = S * sc.k1 + (pair >= sc.rem0 ? i1 - sc.k1 : i1) * sc.P + pair;
  if (j >= sc.n1) return false;
  prob = 1;
  tile = j;
  return true;
}

// The tile sequence of a pair: pair_tile for two problems; for one, plain
// round-robin over n_tiles with the tile index as the only loop variable.
template <bool kTwo>
struct TileIter {
  const PairSched& sc;
  int pair, it = 0, prob = 0, tile = 0;
  bool ok;
  __device__ __forceinline__ TileIter(const PairSched& s, int pr, int, int) : sc(s), pair(pr) {
    ok = pair_tile(sc, pair, 0, prob, tile);
  }
  __device__ __forceinline__ void next() { ok = pair_tile(sc, pair, ++it, prob, tile); }
};
template <>
struct TileIter<false> {
  int prob = 0, tile, n, step;
  bool ok;
  __device__ __forceinline__ TileIter(const PairSched&, int pr, int n_tiles, int num_pairs)
      : tile(pr), n(n_tiles), step(num_pairs) {
    ok = tile < n;
  }
  __device__ __forceinline__ void next() {
    tile += step;
    ok = tile < n;
  }
};

__device__ __forceinline__ uint32_t map_to_cta(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on the even CTA's copy of a barrier.  The arrivals that use it
// follow a completed tensor-memory access (tcgen05.wait::ld) and a
// tcgen05.fence::before_thread_sync, which order that access before the
// arrive; there is no ordinary memory to release, so the odd CTA uses the
// relaxed cluster-scope arrive and the even CTA its local arrive.
__device__ __forceinline__ void mbar_arrive_leader(uint32_t local_addr, uint32_t rank) {
  if (rank == 0) {
    mbar_arrive(local_addr);
  } else {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(0));
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(r) : "memory");
  }
}

// Bulk tensor store of a shared-memory box, tracked in the issuing thread's
// bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t accumulate, bool mx) {
  if (mx)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
  else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}

// Shared-memory descriptor of one 512-byte scale tile for tcgen05.cp: 32 rows
// of 16 bytes, no swizzle, core matrices of 8 rows x 16 bytes 128 bytes apart
// (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t desc_sf_tile(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(128 >> 4) << 32) |
         ((uint64_t)1 << 46);
}

// Copy a 32-row x 16-byte tile from this CTA's shared memory into tensor-memory
// lanes 0-31 at column `taddr`, replicated into all four lane quadrants, in both
// CTAs of the pair (each CTA from its own shared memory).
__device__ __forceinline__ void tc_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tc_commit_pair_multicast(uint32_t bar) {
  const uint16_t mask = 3;
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(mask)
               : "memory");
}

__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// One lane of a converged warp is elected to issue.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

template <bool kTwo>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    nvfp4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                           const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                           const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ Params p,
                           const __grid_constant__ PairProblem g1, const PairSched sched) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t epi_base = base + kPairStages * kPairStageBytes;
  const uint32_t bar_base = epi_base + kPairEpiWarps * kPairEpiBufBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + (bar_base - base));
  // barrier slots: full[S], empty[S], tmem_full, tmem_empty, mma_done
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (kPairStages + s); };
  const uint32_t tmem_full = bar_base + 8u * (2 * kPairStages);
  const uint32_t tmem_empty = tmem_full + 8u;
  const uint32_t mma_done = tmem_full + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kPairStages + 3);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = p.M / 256, num_n = p.N / kPairBN;
  const int n_tiles = num_m * num_n;
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
  const int k_stages = (p.K + kKPerStage - 1) / kKPerStage;
  const int last_nk = ((p.K - 1) % kKPerStage) / kMmaK + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, 2 * kPairEpiWarps);
    mbar_init(mma_done, 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_sfa)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_sfb)) : "memory");
    if constexpr (kTwo) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&g1.a)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&g1.b)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&g1.sfa)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&g1.sfb)) : "memory");
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (TileIter<kTwo> ti(sched, pair, n_tiles, num_pairs); ti.ok; ti.next()) {
        const int tile = ti.tile;
        // the tile's problem: problem 0 in the kernel's own parameters, 1 in g1
        const bool second = kTwo && ti.prob;
        const CUtensorMap* map_a = second ? &g1.a : &tmap_a;
        const CUtensorMap* map_b = second ? &g1.b : &tmap_b;
        const CUtensorMap* map_sfa = second ? &g1.sfa : &tmap_sfa;
        const CUtensorMap* map_sfb = second ? &g1.sfb : &tmap_sfb;
        int mb, nb, t_stages = k_stages;
        if constexpr (kTwo) {
          const Params& gp = second ? g1.p : p;
          tile_coords(tile, gp.M / 256, gp.N / kPairBN, gp.n_fastest, mb, nb);
          t_stages = (gp.K + kKPerStage - 1) / kKPerStage;
        } else {
          tile_coords(tile, num_m, num_n, p.n_fastest, mb, nb);
        }
        bool ok = true;
        for (int ks = 0; ks < t_stages; ++ks) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort, p.status)) { ok = false; break; }
          if (p.debug_stall && tile == pair && !second && ks == 0) {
            // nothing is issued or armed for this stage: the MMA warp's
            // bounded wait runs out and the kernel reports NVFP4_ERR_TIMEOUT
            if (++stage == kPairStages) { stage = 0; phase ^= 1u; }
            continue;
          }
          const uint32_t sa = base + stage * kPairStageBytes;
          const uint32_t leader_full = map_to_cta(full_bar(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2u * kPairStageBytes);
          tma_load_2d_pair(sa, map_a, ks * kBKBytes, mb * 256 + (int)rank * 128, leader_full);
          tma_load_2d_pair(sa + kPairABytes, map_b, ks * kBKBytes, nb * kPairBN + (int)rank * 128, leader_full);
          // scale tiles as 8-byte words: 4 tiles (2 KB) of this CTA's A rows,
          // 4 tiles of each of the two 128-row halves of B
          tma_load_2d_pair(sa + kPairABytes + kPairBBytes, map_sfa, ks * 256, 2 * mb + (int)rank, leader_full);
          tma_load_2d_pair(sa + kPairABytes + kPairBBytes + kPairSfaBytes, map_sfb, ks * 256, 2 * nb,
                           leader_full);
          if (++stage == kPairStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // after an abort, loads already issued may still be in flight: give
      // them time to land before the CTA can exit
      if (*abort) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < kDrainNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA warp (even CTA) --------------------
    // lane 0 waits, the warp follows its verdict (uniform by construction)
    auto warp_wait = [&](uint32_t bar, uint32_t parity) {
      int r = 0;
      if (lane == 0) r = mbar_wait(bar, parity, abort, p.status) ? 1 : 0;
      return __shfl_sync(0xFFFFFFFFu, r, 0) != 0;
    };
    // per stage: every lane tests the barrier (one instruction, the same
    // answer for all); only when it is not complete yet does lane 0 wait
    auto stage_wait = [&](uint32_t bar, uint32_t parity) {
      if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
      return warp_wait(bar, parity);
    };
    // one instantiation per operand format: the issue path carries no
    // format test
    auto issue = [&](auto mx_tag) {
      constexpr bool kMX = decltype(mx_tag)::value;
      const uint32_t idesc = idesc_block_scaled(256, kPairBN, kMX);
      const uint32_t tmem_u = __shfl_sync(0xFFFFFFFFu, tmem, 0);
      // the lane that issues every copy, MMA and commit of this warp
      const bool leader = elect_one();
      // descriptors of stage 0; stage s adds s * kPairStageBytes
      const uint64_t da0 = desc_sw128(base), db0 = desc_sw128(base + kPairABytes);
      const uint64_t dsf0 = desc_sf_tile(base + kPairABytes + kPairBBytes);
      constexpr uint64_t kStageDesc = kPairStageBytes >> 4;
      constexpr uint64_t kTileDesc = 512 >> 4;
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (TileIter<kTwo> ti(sched, pair, n_tiles, num_pairs); ok && ti.ok; ti.next()) {
        int k_stages_t = k_stages, last_nk_t = last_nk;
        if constexpr (kTwo) {
          const Params& gp = ti.prob ? g1.p : p;
          k_stages_t = (gp.K + kKPerStage - 1) / kKPerStage;
          last_nk_t = ((gp.K - 1) % kKPerStage) / kMmaK + 1;
        }
        if (!warp_wait(tmem_empty, acc_phase ^ 1u)) break;
        tc_fence_after();
        for (int ks = 0; ks < k_stages_t; ++ks) {
          if (!stage_wait(full_bar(stage), phase)) { ok = false; break; }
          tc_fence_after();
          const uint64_t soff = (uint64_t)stage * kStageDesc;
          const uint64_t da = da0 + soff, db = db0 + soff, dsf = dsf0 + soff;
          const uint32_t sfa = tmem_u + (uint32_t)(kPairBN + stage * kPairSfCols), sfb = sfa + 16;
          if (leader) {
            // scale tiles: A tile j -> columns 4j; B tile (j, h) -> 16 + 8j + 4h
#pragma unroll
            for (int j = 0; j < 4; ++j) tc_cp_sf_pair(sfa + 4 * j, dsf + j * kTileDesc);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int j = 0; j < 4; ++j) tc_cp_sf_pair(sfb + 8 * j + 4 * h, dsf + (4 + 4 * h + j) * kTileDesc);
            if (ks != k_stages_t - 1 || last_nk_t == 4) {
              tc_mma_pair(tmem_u, da, db, idesc, sfa, sfb, ks != 0, kMX);
              tc_mma_pair(tmem_u, da + 2, db + 2, idesc, sfa + 4, sfb + 8, 1u, kMX);
              tc_mma_pair(tmem_u, da + 4, db + 4, idesc, sfa + 8, sfb + 16, 1u, kMX);
              tc_mma_pair(tmem_u, da + 6, db + 6, idesc, sfa + 12, sfb + 24, 1u, kMX);
            } else {
              // +32 bytes along K per MMA inside the 128-byte swizzle atom
              for (int j = 0; j < last_nk_t; ++j)
                tc_mma_pair(tmem_u, da + 2 * j, db + 2 * j, idesc, sfa + 4 * j, sfb + 8 * j, (ks | j) != 0, kMX);
            }
            tc_commit_pair_multicast(empty_bar(stage));
          }
          if (++stage == kPairStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (leader) tc_commit_pair_multicast(tmem_full);
        __syncwarp();
        acc_phase ^= 1u;
      }
    };
    if (rank == 0) {
      if (p.mx) issue(std::true_type{});
      else issue(std::false_type{});
      // every copy and MMA issued by this warp has finished
      if (elect_one()) tc_commit_pair(mma_done);
      __syncwarp();
      if (lane == 0) {
        volatile int never = 0;
        mbar_wait(mma_done, 0, &never, p.status);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;
    const int half = (warp - kPairFirstEpiWarp) >> 2;
    constexpr int kCols = kPairBN / 2;
    const float alpha = p.mx ? 1.0f : __fmul_rn(*p.ts_a, *p.ts_b);
    float q_senc = 1.0f;  // quantized output: the encode scale of its tensor amax
    if (p.q_codes) {
      const float a = *p.q_amax;
      q_senc = tensor_encode_scale(a);
      if (blockIdx.x == 0 && warp == kPairFirstEpiWarp && lane == 0) {
        *p.q_ts = tensor_decode_scale(q_senc);
        if (!(abs_bits(a) < 0x7F800000u)) raise_status(p.status, kStatusNonFinite);
      }
    }
    if constexpr (kTwo) {  // the second problem's quantized output: its tensor scale
      if (g1.p.q_codes && blockIdx.x == 0 && warp == kPairFirstEpiWarp && lane == 0) {
        const float a = *g1.p.q_amax;
        *g1.p.q_ts = tensor_decode_scale(tensor_encode_scale(a));
        if (!(abs_bits(a) < 0x7F800000u)) raise_status(p.status, kStatusNonFinite);
      }
    }
    uint32_t acc_phase = 0;
    for (TileIter<kTwo> ti(sched, pair, n_tiles, num_pairs); ti.ok; ti.next()) {
      const int tile = ti.tile;
      // the tile's problem (with two problems, its scales and output are read
      // per tile)
      const bool second = kTwo && ti.prob;
      const Params& tpp = second ? g1.p : p;
      const CUtensorMap* map_d = second ? &g1.d : &tmap_d;
      float alpha_t = alpha, q_senc_t = q_senc;
      if (second) {
        alpha_t = g1.p.mx ? 1.0f : __fmul_rn(*g1.p.ts_a, *g1.p.ts_b);
        q_senc_t = g1.p.q_codes ? tensor_encode_scale(*g1.p.q_amax) : 1.0f;
      }
      int mb, nb;
      if constexpr (kTwo) tile_coords(tile, tpp.M / 256, tpp.N / kPairBN, tpp.n_fastest, mb, nb);
      else tile_coords(tile, num_m, num_n, p.n_fastest, mb, nb);
      int ready = 0;
      if (lane == 0) ready = mbar_wait(tmem_full, acc_phase, abort, p.status) ? 1 : 0;
      ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
      if (!ready) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(half * kCols);
      const int64_t row = (int64_t)mb * 256 + (int64_t)rank * 128 + 32 * q + lane;
      const int64_t col0 = (int64_t)nb * kPairBN + half * kCols;
      // all 128 accumulator columns of this lane's row into registers with one
      // wait; the accumulator goes back to the MMA warp at once, and the next
      // tile's MMAs run while this tile is scaled, rounded and stored
      uint32_t v[kCols];
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) tmem_ld32(taddr + 32 * c, v + 32 * c);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_leader(tmem_empty, rank);
      acc_phase ^= 1u;
      if (tpp.d_f32) {
        uint32_t m32 = 0;  // max magnitude bits
        uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(tpp.d) + row * tpp.ldd + col0);
#pragma unroll
        for (int i = 0; i < kCols / 4; ++i) {
          const uint4 o = make_uint4(__float_as_uint(__fmul_rn(alpha_t, __uint_as_float(v[4 * i]))),
                                     __float_as_uint(__fmul_rn(alpha_t, __uint_as_float(v[4 * i + 1]))),
                                     __float_as_uint(__fmul_rn(alpha_t, __uint_as_float(v[4 * i + 2]))),
                                     __float_as_uint(__fmul_rn(alpha_t, __uint_as_float(v[4 * i + 3]))));
          dst[i] = o;
          m32 = max(m32, max(max(o.x & 0x7FFFFFFFu, o.y & 0x7FFFFFFFu), max(o.z & 0x7FFFFFFFu, o.w & 0x7FFFFFFFu)));
        }
        if (tpp.amax_out) amax_bits_to_global(m32, tpp.amax_out);
      } else {
        // 16-column chunks, each one 1x16 block of the row: scaled and
        // rounded to BF16, then (as asked) folded into the output amax,
        // quantized to NVFP4, and sent through this warp's 1 KB buffer (32
        // rows of 32 B, 32-byte swizzle: 16-byte half h of row r at h ^ bit 2
        // of r) with one bulk tensor store; the buffer is rewritten once the
        // previous store has read it
        const uint32_t buf = epi_base + (uint32_t)(warp - kPairFirstEpiWarp) * kPairEpiBufBytes;
        const uint32_t sw = (uint32_t)((lane >> 2) & 1);
        uint32_t m2 = 0;               // max BF16 magnitude bits of both halves
        uint32_t sc[2] = {0u, 0u};     // quantized output: 8 block scales
        uint32_t qw[4] = {0u, 0u, 0u, 0u};
        uint4* cdst = tpp.q_codes ? reinterpret_cast<uint4*>(tpp.q_codes + row * (tpp.N >> 1) + (col0 >> 1)) : nullptr;
#pragma unroll
        for (int j = 0; j < kCols / 16; ++j) {
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            pk[i] = pack_bf16x2(__fmul_rn(alpha_t, __uint_as_float(v[16 * j + 2 * i])),
                                __fmul_rn(alpha_t, __uint_as_float(v[16 * j + 2 * i + 1])));
          if (tpp.amax_out) {
#pragma unroll
            for (int i = 0; i < 8; ++i) m2 = __vmaxu2(m2, pk[i] & 0x7FFF7FFFu);
          }
          if (tpp.q_codes) {
            // as the rowwise RNE quantizer would quantize the stored BF16 output
            float f[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              f[2 * i] = bf16lo(pk[i]);
              f[2 * i + 1] = bf16hi(pk[i]);
            }
            uint32_t E;
            const uint2 o = quantize16_rne(f, q_senc_t, E);
            sc[j >> 2] |= E << (8 * (j & 3));
            qw[2 * (j & 1)] = o.x;
            qw[2 * (j & 1) + 1] = o.y;
            if (j & 1) cdst[j >> 1] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
          }
          if (tpp.tma_store) {
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t a = buf + (uint32_t)lane * 32u + (((uint32_t)h ^ sw) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pk[4 * h]), "r"(pk[4 * h + 1]),
                           "r"(pk[4 * h + 2]), "r"(pk[4 * h + 3])
                           : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tma_store_2d(map_d, (int)col0 + 16 * j, (int)(row - lane), buf);
          }
        }
        if (tpp.amax_out) amax_bits_to_global(max(m2 & 0xFFFFu, m2 >> 16) << 16, tpp.amax_out);
        if (tpp.q_codes) {
          const int64_t n_kb = tpp.N >> 4, kb0 = col0 >> 4;
          *reinterpret_cast<uint32_t*>(tpp.q_scales + sf_mma_offset(row, kb0, n_kb)) = sc[0];
          *reinterpret_cast<uint32_t*>(tpp.q_scales + sf_mma_offset(row, kb0 + 4, n_kb)) = sc[1];
        }
      }
    }
    // the output is in global memory (and the buffers free) before exit
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }

  // Both CTAs stay until every MMA (which reads both CTAs' shared memory) is
  // done and both epilogues have read their accumulators.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
std::atomic<int> g_debug_stall{0};

// 2D map over packed codes: inner dimension = row bytes, box = 128 B x box_rows.
bool make_code_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
  auto fn = tensor_map_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)kBKBytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D map over a BF16 [rows, cols] output with row stride ld elements; box =
// 16 columns x 32 rows, 32-byte swizzle (the epilogue's staging layout).
bool make_out_map(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows, uint64_t ld) {
  auto fn = tensor_map_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D map over an MMA-layout scale tensor as 8-byte words: one row per 128
// tensor rows (tiles_k 512-byte tiles = tiles_k * 64 words), box = 4 tiles
// (256 words, 2 KB) x box_rows rows.
bool make_sf_map(CUtensorMap* m, const void* base, uint64_t tiles_k, uint64_t row_tiles, uint32_t box_rows) {
  auto fn = tensor_map_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {tiles_k * 64, row_tiles};
  cuuint64_t strides[1] = {tiles_k * 512};
  cuuint32_t box[2] = {256, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() { return device_sm_count(); }

template <int BN>
nvfp4_status run(const nvfp4_tensor& a, const nvfp4_tensor& b, void* d, int32_t d_dtype, int64_t ldd,
                 float* amax_out, cudaStream_t s) {
  using C = Cfg<BN>;
  static std::atomic<bool> attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(nvfp4_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
      return NVFP4_ERR_CUDA;
    attr_set[dev] = true;
  }
  CUtensorMap ma, mb;
  const int64_t K = a.cols;
  if (!make_code_map(&ma, a.codes, (uint64_t)K / 2, (uint64_t)a.rows, kBM) ||
      !make_code_map(&mb, b.codes, (uint64_t)K / 2, (uint64_t)b.rows, BN))
    return NVFP4_ERR_CUDA;
  Params p;
  p.sfa = a.scales;
  p.sfb = b.scales;
  p.ts_a = a.tensor_scale;
  p.ts_b = b.tensor_scale;
  p.d = d;
  p.ldd = ldd;
  p.d_f32 = d_dtype == NVFP4_OUT_F32;
  p.M = (int)a.rows;
  p.N = (int)b.rows;
  p.K = (int)K;
  p.sf_tiles_k = (int)(K / 64);
  p.n_fastest = p.N < p.M;
  p.debug_stall = g_debug_stall.exchange(0);
  p.status = device_status_ptr();
  p.amax_out = reinterpret_cast<uint32_t*>(amax_out);
  p.mx = a.format == NVFP4_FORMAT_MXFP4;
  p.q_codes = nullptr;
  p.q_scales = nullptr;
  p.q_amax = nullptr;
  p.q_ts = nullptr;
  p.tma_store = 0;
  const int tiles = (p.M / kBM) * (p.N / BN);
  const int grid = tiles < sm_count() ? tiles : sm_count();
  nvfp4_gemm_kernel<BN><<<grid, kNumThreads, C::kSmemBytes, s>>>(ma, mb, p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}


// The maps and parameters of one GEMM of the pair kernel.
nvfp4_status make_pair_problem(PairProblem& g, const nvfp4_tensor& a, const nvfp4_tensor& b, void* d,
                               int32_t d_dtype, int64_t ldd, float* amax_out, const nvfp4_tensor* yq,
                               int debug_stall) {
  const int64_t K = a.cols;
  if (!make_code_map(&g.a, a.codes, (uint64_t)K / 2, (uint64_t)a.rows, 128) ||
      !make_code_map(&g.b, b.codes, (uint64_t)K / 2, (uint64_t)b.rows, 128) ||
      !make_sf_map(&g.sfa, a.scales, (uint64_t)K / 64, (uint64_t)a.rows / 128, 1) ||
      !make_sf_map(&g.sfb, b.scales, (uint64_t)K / 64, (uint64_t)b.rows / 128, 2))
    return NVFP4_ERR_CUDA;
  Params& p = g.p;
  p.sfa = a.scales;
  p.sfb = b.scales;
  p.ts_a = a.tensor_scale;
  p.ts_b = b.tensor_scale;
  p.d = d;
  p.ldd = ldd;
  p.d_f32 = d_dtype == NVFP4_OUT_F32;
  p.M = (int)a.rows;
  p.N = (int)b.rows;
  p.K = (int)K;
  p.sf_tiles_k = (int)(K / 64);
  // walk N when B is the smaller operand; when its packed codes exceed 32 MB
  // they do not stay in L2 from one wave of tiles to the next (the Dgrad B,
  // W^T, at 5120 x 20480: 52 MB), so walk it in groups of 16 block rows
  // (measured: Dgrad 2.5 % faster; no change where B stays in L2)
  p.n_fastest = p.N < p.M ? ((int64_t)p.N * p.K / 2 > (int64_t(32) << 20) ? 16 : 1) : 0;
  p.debug_stall = debug_stall;
  p.status = device_status_ptr();
  p.amax_out = reinterpret_cast<uint32_t*>(amax_out);
  p.mx = a.format == NVFP4_FORMAT_MXFP4;
  p.q_codes = yq ? yq->codes : nullptr;
  p.q_scales = yq ? yq->scales : nullptr;
  p.q_amax = yq ? yq->amax : nullptr;
  p.q_ts = yq ? yq->tensor_scale : nullptr;
  // BF16 output goes through bulk tensor stores (the API guarantees the
  // 16-byte aligned base and row stride they need); FP32 through plain
  // stores; no BF16 output (quantized output only) stores nothing
  g.d = g.a;  // unused for FP32 or no BF16 output
  p.tma_store = !p.d_f32 && d != nullptr;
  if (p.tma_store && !make_out_map(&g.d, d, (uint64_t)p.N, (uint64_t)p.M, (uint64_t)ldd)) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

// The schedule of n0 tiles of k-length c0 and n1 tiles of k-length c1 over
// P pairs (pair_tile): the number of head rounds k1 that gives the shortest
// longest pair, found by counting every pair's stages.
// The search is linear in the tile count per candidate; a layer calls this
// with the same shapes every step, so the last answer is kept per thread.
PairSched make_sched(int n0, int c0, int n1, int c1, int P) {
  PairSched best{n0, n1, P, n1 ? n0 % P : 0, 0};
  if (!n1 || best.rem0 == 0) return best;
  thread_local int last_key[5] = {-1, -1, -1, -1, -1};
  thread_local PairSched last{};
  if (last_key[0] == n0 && last_key[1] == c0 && last_key[2] == n1 && last_key[3] == c1 && last_key[4] == P)
    return last;
  int64_t best_span = -1;
  for (int k1 = 0; k1 <= c0 / (c1 > 0 ? c1 : 1) + 1; ++k1) {
    PairSched sc{n0, n1, P, n0 % P, k1};
    int64_t span = 0;
    for (int pr = 0; pr < P; ++pr) {
      int64_t load = 0;
      const int cnt0 = (n0 - pr + P - 1) / P;
      load += (int64_t)cnt0 * c0;
      const int S = P - sc.rem0;
      for (int i1 = 0;; ++i1) {
        int j;
        if (pr >= sc.rem0 && i1 < k1) j = i1 * S + (pr - sc.rem0);
        else j = S * k1 + (pr >= sc.rem0 ? i1 - k1 : i1) * P + pr;
        if (j >= n1) break;
        load += c1;
      }
      span = load > span ? load : span;
    }
    if (best_span < 0 || span < best_span) {
      best_span = span;
      best = sc;
    }
  }
  last = best;
  last_key[0] = n0;
  last_key[1] = c0;
  last_key[2] = n1;
  last_key[3] = c1;
  last_key[4] = P;
  return best;
}

template <bool kTwo>
nvfp4_status launch_pair(const PairProblem& g0, const PairProblem& g1, const PairSched& sc, cudaStream_t s) {
  static std::atomic<bool> attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(nvfp4_gemm_pair_kernel<kTwo>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPairSmemBytes) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    attr_set[dev] = true;
  }
  nvfp4_gemm_pair_kernel<kTwo><<<2 * sc.P, kPairThreads, kPairSmemBytes, s>>>(g0.a, g0.b, g0.sfa, g0.sfb, g0.d, g0.p,
                                                                               g1, sc);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

int pair_tiles(const nvfp4_tensor& a, const nvfp4_tensor& b) { return (int)((a.rows / 256) * (b.rows / kPairBN)); }
int pair_stages(const nvfp4_tensor& a) { return (int)((a.cols + kKPerStage - 1) / kKPerStage); }

nvfp4_status run_pair(const nvfp4_tensor& a, const nvfp4_tensor& b, void* d, int32_t d_dtype, int64_t ldd,
                      float* amax_out, const nvfp4_tensor* yq, cudaStream_t s) {
  PairProblem g0{}, g1{};
  const nvfp4_status st = make_pair_problem(g0, a, b, d, d_dtype, ldd, amax_out, yq, g_debug_stall.exchange(0));
  if (st != NVFP4_OK) return st;
  const int tiles = pair_tiles(a, b);
  const int pairs_max = sm_count() / 2;
  const int P = tiles < pairs_max ? tiles : pairs_max;
  return launch_pair<false>(g0, g1, PairSched{tiles, 0, P, 0, 0}, s);
}

// Two BF16-output GEMMs of the same operand format over one tile schedule
// (the problem with the longer K first, so that the pairs left short by its
// last round start on the other one).
nvfp4_status run_pair2(const nvfp4_tensor& a0, const nvfp4_tensor& b0, void* d0, int64_t ldd0,
                       const nvfp4_tensor& a1, const nvfp4_tensor& b1, void* d1, int64_t ldd1, cudaStream_t s) {
  const bool swap = a1.cols > a0.cols;
  const nvfp4_tensor &A0 = swap ? a1 : a0, &B0 = swap ? b1 : b0, &A1 = swap ? a0 : a1, &B1 = swap ? b0 : b1;
  void* D0 = swap ? d1 : d0;
  void* D1 = swap ? d0 : d1;
  const int64_t L0 = swap ? ldd1 : ldd0, L1 = swap ? ldd0 : ldd1;
  PairProblem g0{}, g1{};
  nvfp4_status st = make_pair_problem(g0, A0, B0, D0, NVFP4_OUT_BF16, L0, nullptr, nullptr, g_debug_stall.exchange(0));
  if (st != NVFP4_OK) return st;
  st = make_pair_problem(g1, A1, B1, D1, NVFP4_OUT_BF16, L1, nullptr, nullptr, 0);
  if (st != NVFP4_OK) return st;
  const int n0 = pair_tiles(A0, B0), n1 = pair_tiles(A1, B1);
  const int pairs_max = sm_count() / 2;
  const int P = n0 + n1 < pairs_max ? n0 + n1 : pairs_max;
  return launch_pair<true>(g0, g1, make_sched(n0, pair_stages(A0), n1, pair_stages(A1), P), s);
}

}  // namespace

void set_gemm_debug_stall(int on) { g_debug_stall.store(on ? 1 : 0); }

nvfp4_status launch_gemm2(const nvfp4_tensor& a0, const nvfp4_tensor& b0, void* d0, int64_t ldd0,
                          const nvfp4_tensor& a1, const nvfp4_tensor& b1, void* d1, int64_t ldd1, cudaStream_t s) {
  const bool pair0 = a0.rows % 256 == 0 && b0.rows % 256 == 0, pair1 = a1.rows % 256 == 0 && b1.rows % 256 == 0;
  if (pair0 && pair1 && a0.format == a1.format) return run_pair2(a0, b0, d0, ldd0, a1, b1, d1, ldd1, s);
  const nvfp4_status st = launch_gemm(a0, b0, d0, NVFP4_OUT_BF16, ldd0, s);
  if (st != NVFP4_OK) return st;
  return launch_gemm(a1, b1, d1, NVFP4_OUT_BF16, ldd1, s);
}

nvfp4_status launch_gemm(const nvfp4_tensor& a, const nvfp4_tensor& b, void* d, int32_t d_dtype, int64_t ldd,
                         cudaStream_t s, float* amax_out, const nvfp4_tensor* yq) {
  if (a.rows % 256 == 0 && b.rows % 256 == 0) return run_pair(a, b, d, d_dtype, ldd, amax_out, yq, s);
  if (yq) return NVFP4_ERR_SHAPE;  // the quantized output is produced by the CTA-pair kernel only
  if (b.rows % 256 == 0) return run<256>(a, b, d, d_dtype, ldd, amax_out, s);
  return run<128>(a, b, d, d_dtype, ldd, amax_out, s);
}

}  // namespace nvfp4
