// nvfp4_oracle.cpp -- plain C++17 CPU oracle of the NVFP4 linear-layer path.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
// and its Python binding) includes, links or calls this file; it shares no
// code with the CUDA kernels.  Only the test suite, the smoke check and the
// CPU-baseline leg of the benchmark load it (through oracle/cxx.py).
//
// What it computes -- the same definitions as the numpy oracle next to it,
// written out again element by element:
//   * "Pretraining Large Language Models with NVFP4" (gist.science summary),
//     Resumo técnico §2, "Formato NVFP4" (16-element blocks, an E4M3 scale
//     per block, an FP32 scale per tensor: "Bloco Menor", "Fatores de Escala
//     Precisos", "Escala em Dois Níveis") and "Técnicas de Treinamento
//     Integradas" items 2 (random Hadamard transform on the Wgrad inputs),
//     3 (16x16 weight blocks) and 4 (stochastic rounding of gradients,
//     round-to-nearest-even elsewhere); §3 "Suporte de Hardware" (the GEMM
//     takes block-scaled FP4 operands and accumulates in high precision);
//   * OCP Microscaling Formats v1.0 (E2M1) and OCP 8-bit Floating Point
//     (E4M3 "FN") for the bit layouts the pages only name;
//   * Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2,
//     3" (SC'11), for Philox4x32-10.
// The readings where the pages are silent (the op order of the two-level
// scale, 16-bit uniforms for stochastic rounding, the Philox counter layout,
// the Sylvester Hadamard matrix and its summation order, low-nibble-first
// packing) are the ones the numpy oracle states in its docstrings.
//
// Arithmetic: IEEE binary32 with round-to-nearest-even for every operation
// marked float, binary64 for the GEMM sums.  Build with -ffp-contract=off and
// without fast-math, so no multiply-add is fused and nothing flushes to zero.
// Work is split over rows with std::thread; every output element is computed
// by one thread in a fixed order, so results do not depend on the count.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Row-parallel loop: body(r0, r1) over [0, n) split into `threads` ranges.
// ---------------------------------------------------------------------------
template <class F>
void parallel_rows(int64_t n, int threads, F&& body) {
  if (threads <= 0) threads = (int)std::max(1u, std::thread::hardware_concurrency());
  if (threads > n) threads = (int)std::max<int64_t>(1, n);
  if (threads <= 1) {
    body(int64_t(0), n);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t per = (n + threads - 1) / threads;
  for (int t = 0; t < threads; ++t) {
    const int64_t a = t * per, b = std::min(n, a + per);
    if (a >= b) break;
    pool.emplace_back([&body, a, b] { body(a, b); });
  }
  for (auto& th : pool) th.join();
}

// ---------------------------------------------------------------------------
// E2M1: code = s*8 + e*2 + m; magnitude (e == 0) ? m/2 : 2^(e-1) (1 + m/2).
// ---------------------------------------------------------------------------
double e2m1_magnitude(int code7) {
  const int e = (code7 >> 1) & 3, m = code7 & 1;
  return e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
}

double e2m1_value(uint8_t code) {
  const double mag = e2m1_magnitude(code & 7);
  return (code & 8) ? -mag : mag;
}

// Round to the nearest of the eight magnitudes; on a tie the one whose
// mantissa bit is 0 wins; 6 and above saturate to 6.  The sign bit of v is
// kept (a negative value that rounds to zero is code 8).
uint8_t e2m1_rne(float v) {
  const double a = std::fabs((double)v);
  int best = 7;
  if (a < 6.0) {
    double best_d = INFINITY;
    for (int c = 0; c < 8; ++c) {
      const double d = std::fabs(a - e2m1_magnitude(c));
      if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
        best = c;
        best_d = d;
      }
    }
  }
  return (uint8_t)((std::signbit(v) ? 8 : 0) | best);
}

// Stochastic rounding with a 16-bit uniform u: lo <= |v| < hi the grid
// neighbours, frac = (|v| - lo) * (1 / (hi - lo)) in float32 (both steps
// exact), round up iff float(u) < frac * 65536.  |v| >= 6 gives 6.
uint8_t e2m1_sr(float v, uint32_t u) {
  const float a = std::fabs(v);
  int code = 7;
  if (!(a >= 6.0f)) {
    int lo = 0;
    for (int c = 1; c < 7; ++c)
      if ((double)a >= e2m1_magnitude(c)) lo = c;
    const float flo = (float)e2m1_magnitude(lo), fhi = (float)e2m1_magnitude(lo + 1);
    const float step = fhi - flo;
    const float frac = (a - flo) * (1.0f / step);
    const float thresh = frac * 65536.0f;
    code = ((float)u < thresh) ? lo + 1 : lo;
  }
  return (uint8_t)((std::signbit(v) ? 8 : 0) | code);
}

// ---------------------------------------------------------------------------
// E4M3 (OCP "FN"): bias 7, 3 mantissa bits, subnormal step 2^-9, max 448,
// S.1111.111 is NaN.
// ---------------------------------------------------------------------------
double e4m3_value(uint8_t code) {
  const int e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return (code & 0x80) ? -mag : mag;
}

// Non-negative finite float -> nearest of codes 0..126 (increasing values),
// ties to the even code; 448 and above saturate to 0x7E.
uint8_t e4m3_rne_sat(float x) {
  const double a = (double)x;
  if (a >= 448.0) return 0x7E;
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c < 127; ++c) {
    const double d = std::fabs(a - e4m3_value((uint8_t)c));
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)best;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (SC'11 §4.2, constants of its Table 2).
// ---------------------------------------------------------------------------
const uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u, kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;

void philox(const uint32_t in[4], uint32_t k0, uint32_t k1, uint32_t out[4]) {
  uint32_t c0 = in[0], c1 = in[1], c2 = in[2], c3 = in[3];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint64_t p0 = (uint64_t)kM0 * c0, p1 = (uint64_t)kM1 * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n1 = (uint32_t)p1;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    const uint32_t n3 = (uint32_t)p0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// 16-bit uniform of element e: counter (lo32(e/8), hi32(e/8), stream, 0),
// word (e%8)/2, low half for even e.
uint32_t sr_uniform(uint64_t seed, uint32_t stream, uint64_t e) {
  const uint64_t g = e >> 3;
  const uint32_t in[4] = {(uint32_t)g, (uint32_t)(g >> 32), stream, 0u};
  uint32_t w[4];
  philox(in, (uint32_t)seed, (uint32_t)(seed >> 32), w);
  const uint32_t word = w[(e & 7) >> 1];
  return (e & 1) ? (word >> 16) : (word & 0xFFFFu);
}

// ---------------------------------------------------------------------------
// 16x16 random Hadamard transform: signs s_j = -1 where bit j of word 0 of
// Philox(seed, (0, 0, 2, 0)) is set; y_i = 1/4 sum_j H[i][j] s_j x_j with
// H[i][j] = (-1)^popcount(i & j), the 16 exact terms summed as a float32
// pairwise tree in index order, then * 0.25 and + 0 (an exact zero is +0).
// ---------------------------------------------------------------------------
const uint32_t kRhtStream = 2;

void rht_signs(uint64_t seed, float s[16]) {
  const uint32_t in[4] = {0u, 0u, kRhtStream, 0u};
  uint32_t w[4];
  philox(in, (uint32_t)seed, (uint32_t)(seed >> 32), w);
  for (int j = 0; j < 16; ++j) s[j] = ((w[0] >> j) & 1u) ? -1.0f : 1.0f;
}

int hadamard(int i, int j) {
  int p = 0;
  for (int b = i & j; b; b >>= 1) p ^= b & 1;
  return p ? -1 : 1;
}

void rht16(const float x[16], const float s[16], float y[16]) {
  for (int i = 0; i < 16; ++i) {
    float t[16];
    for (int j = 0; j < 16; ++j) t[j] = (float)hadamard(i, j) * s[j] * x[j];  // exact sign flips
    for (int width = 16; width > 1; width /= 2)
      for (int k = 0; k < width / 2; ++k) t[k] = t[2 * k] + t[2 * k + 1];
    const float q = t[0] * 0.25f;
    y[i] = q + 0.0f;
  }
}

// ---------------------------------------------------------------------------
// Two-level scale (all float32): s_enc = 2688 / amax (1 if amax == 0),
// ts = 1 / s_enc; per block E = e4m3(fl(amax_b / 6) * s_enc),
// enc = s_enc / e4m3(E) (0 if E == 0); v_i = x_i * enc.
// ---------------------------------------------------------------------------
bool tensor_scales(float amax, float* s_enc, float* ts) {
  if (!std::isfinite(amax)) return false;
  if (amax == 0.0f) {
    *s_enc = 1.0f;
    *ts = 1.0f;
    return true;
  }
  *s_enc = 2688.0f / amax;
  *ts = 1.0f / *s_enc;
  return true;
}

void block_scale(float amax_b, float s_enc, uint8_t* E, float* enc) {
  const float sd = amax_b / 6.0f;
  const float prod = sd * s_enc;
  *E = e4m3_rne_sat(prod);
  *enc = (*E == 0) ? 0.0f : s_enc / (float)e4m3_value(*E);
}

// One row of C values (C % 16 == 0): block scales and codes.  Element j of
// the row has index base + j in the quantized tensor (stochastic rounding).
void quantize_row(const float* v, int64_t C, float s_enc, int sr, uint64_t seed, uint32_t stream, uint64_t base,
                  uint8_t* codes_packed, uint8_t* scales) {
  for (int64_t b = 0; b < C / 16; ++b) {
    float amax_b = 0.0f;
    for (int j = 0; j < 16; ++j) amax_b = std::max(amax_b, std::fabs(v[16 * b + j]));
    uint8_t E;
    float enc;
    block_scale(amax_b, s_enc, &E, &enc);
    scales[b] = E;
    for (int j = 0; j < 16; ++j) {
      const int64_t col = 16 * b + j;
      const float x = v[col] * enc;
      const uint8_t c = sr ? e2m1_sr(x, sr_uniform(seed, stream, base + (uint64_t)col)) : e2m1_rne(x);
      if (col & 1) codes_packed[col >> 1] |= (uint8_t)(c << 4);
      else codes_packed[col >> 1] = c;
    }
  }
}

}  // namespace

extern "C" {

// --- formats and generator, one value at a time ---------------------------
uint8_t ox_e2m1_encode_rne(float v) { return e2m1_rne(v); }
uint8_t ox_e2m1_encode_sr(float v, uint32_t u16) { return e2m1_sr(v, u16); }
double ox_e2m1_decode(uint8_t c) { return e2m1_value(c); }
uint8_t ox_e4m3_encode_rne_sat(float x) { return e4m3_rne_sat(x); }
double ox_e4m3_decode(uint8_t c) { return e4m3_value(c); }
void ox_philox4x32_10(const uint32_t* ctr, uint32_t k0, uint32_t k1, uint32_t* out) { philox(ctr, k0, k1, out); }
uint32_t ox_sr_uniform16(uint64_t seed, uint32_t stream, uint64_t e) { return sr_uniform(seed, stream, e); }
void ox_rht_signs(uint64_t seed, float* s) { rht_signs(seed, s); }
void ox_rht16(const float* x, const float* s, float* y) { rht16(x, s, y); }

// The same over arrays of n values.
void ox_e2m1_encode_rne_n(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e2m1_rne(v[i]);
}
void ox_e2m1_encode_sr_n(const float* v, const uint32_t* u16, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e2m1_sr(v[i], u16[i]);
}
void ox_e4m3_encode_rne_sat_n(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_rne_sat(x[i]);
}
void ox_sr_uniform16_n(uint64_t seed, uint32_t stream, const uint64_t* e, int64_t n, uint32_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = sr_uniform(seed, stream, e[i]);
}

// --- amax ------------------------------------------------------------------
// max |x| over the [rows, cols] float32 tensor (NaN if a value is NaN).
float ox_amax(const float* x, int64_t rows, int64_t cols, int threads) {
  std::vector<float> part((size_t)std::max<int64_t>(rows, 1), 0.0f);
  parallel_rows(rows, threads, [&](int64_t r0, int64_t r1) {
    for (int64_t r = r0; r < r1; ++r) {
      float m = 0.0f;
      for (int64_t c = 0; c < cols; ++c) {
        const float a = std::fabs(x[r * cols + c]);
        if (std::isnan(a)) { m = NAN; break; }
        m = std::max(m, a);
      }
      part[(size_t)r] = m;
    }
  });
  float m = 0.0f;
  for (int64_t r = 0; r < rows; ++r) {
    if (std::isnan(part[(size_t)r])) return NAN;
    m = std::max(m, part[(size_t)r]);
  }
  return m;
}

// max |Q x| with Q applied to consecutive 16-chunks along `axis` (0: down
// the rows, i.e. 16 consecutive rows of one column; 1: along a row).
float ox_amax_rht(const float* x, int64_t rows, int64_t cols, int axis, uint64_t seed, int threads) {
  float s[16];
  rht_signs(seed, s);
  const int64_t units = axis == 0 ? cols : rows;  // lines the chunks run along
  std::vector<float> part((size_t)std::max<int64_t>(units, 1), 0.0f);
  parallel_rows(units, threads, [&](int64_t u0, int64_t u1) {
    for (int64_t u = u0; u < u1; ++u) {
      const int64_t len = axis == 0 ? rows : cols;
      float m = 0.0f;
      for (int64_t k = 0; k < len; k += 16) {
        float v[16], y[16];
        for (int j = 0; j < 16; ++j) v[j] = axis == 0 ? x[(k + j) * cols + u] : x[u * cols + k + j];
        rht16(v, s, y);
        for (int j = 0; j < 16; ++j) m = std::isnan(y[j]) || std::isnan(m) ? NAN : std::max(m, std::fabs(y[j]));
      }
      part[(size_t)u] = m;
    }
  });
  float m = 0.0f;
  for (int64_t u = 0; u < units; ++u) {
    if (std::isnan(part[(size_t)u])) return NAN;
    m = std::max(m, part[(size_t)u]);
  }
  return m;
}

// --- quantization -----------------------------------------------------------
// Rows `row_ids[i]` (i < n_rows) of the [R, C] tensor x (transposed first
// when `transpose`: the quantized tensor is then x^T [C, R]), optionally
// transformed by the Hadamard transform along the blocked dimension, then
// quantized with 1x16 blocks along it.  Output row i has codes at
// codes[i * Cq / 2] and scales at scales[i * Cq / 16], Cq the blocked length.
// `amax` is the whole quantized tensor's amax (after the transform).
// Stochastic rounding draws element (row_id * Cq + col)'s uniform.
// Returns 0, or 1 for a non-finite amax.
int ox_quantize_rows(const float* x, int64_t R, int64_t C, int transpose, const int64_t* row_ids, int64_t n_rows,
                     float amax, int sr, uint64_t seed, uint32_t stream, int rht, uint64_t rht_seed,
                     uint8_t* codes, uint8_t* scales, float* ts_out, int threads) {
  float s_enc, ts;
  if (!tensor_scales(amax, &s_enc, &ts)) return 1;
  *ts_out = ts;
  const int64_t Cq = transpose ? R : C;
  float sg[16];
  rht_signs(rht_seed, sg);
  parallel_rows(n_rows, threads, [&](int64_t i0, int64_t i1) {
    std::vector<float> row((size_t)Cq);
    for (int64_t i = i0; i < i1; ++i) {
      const int64_t r = row_ids[i];
      for (int64_t c = 0; c < Cq; ++c) row[(size_t)c] = transpose ? x[c * C + r] : x[r * C + c];
      if (rht)
        for (int64_t k = 0; k < Cq; k += 16) {
          float y[16];
          rht16(&row[(size_t)k], sg, y);
          std::memcpy(&row[(size_t)k], y, sizeof(y));
        }
      quantize_row(row.data(), Cq, s_enc, sr, seed, stream, (uint64_t)r * (uint64_t)Cq, codes + i * (Cq / 2),
                   scales + i * (Cq / 16));
    }
  });
  return 0;
}

// 16x16 blocks of a weight W [N, K]: one scale per block (the same chain,
// amax_b over the 256 values), codes of W [N, K/2] and of W^T [K, N/2], the
// block scale replicated into the 16 rows of W's [N, K/16] and W^T's
// [K, N/16] scale tensors.  Returns 0, or 1 for a non-finite amax.
int ox_quantize_2d(const float* w, int64_t N, int64_t K, float amax, uint8_t* codes, uint8_t* scales,
                   uint8_t* codes_t, uint8_t* scales_t, float* ts_out, int threads) {
  float s_enc, ts;
  if (!tensor_scales(amax, &s_enc, &ts)) return 1;
  *ts_out = ts;
  std::memset(codes, 0, (size_t)(N * K / 2));
  std::memset(codes_t, 0, (size_t)(N * K / 2));
  parallel_rows(N / 16, threads, [&](int64_t b0, int64_t b1) {
    for (int64_t bn = b0; bn < b1; ++bn)
      for (int64_t bk = 0; bk < K / 16; ++bk) {
        float amax_b = 0.0f;
        for (int i = 0; i < 16; ++i)
          for (int j = 0; j < 16; ++j) amax_b = std::max(amax_b, std::fabs(w[(16 * bn + i) * K + 16 * bk + j]));
        uint8_t E;
        float enc;
        block_scale(amax_b, s_enc, &E, &enc);
        for (int i = 0; i < 16; ++i) {
          scales[(16 * bn + i) * (K / 16) + bk] = E;
          scales_t[(16 * bk + i) * (N / 16) + bn] = E;
          for (int j = 0; j < 16; ++j) {
            const int64_t n = 16 * bn + i, k = 16 * bk + j;
            const uint8_t c = e2m1_rne(w[n * K + k] * enc);
            codes[n * (K / 2) + k / 2] |= (uint8_t)((k & 1) ? c << 4 : c);
            codes_t[k * (N / 2) + n / 2] |= (uint8_t)((n & 1) ? c << 4 : c);
          }
        }
      }
  });
  return 0;
}

// --- GEMM on dequantized operands -------------------------------------------
// D[i, j] = ts_a * ts_b * sum_k deqA[row_ids[i], k] deqB[j, k] for K-major
// NVFP4 A [*, K] and B [N, K] (packed codes, [rows, K/16] scales): each
// decoded value and product is exact in float64, the sum runs in k order in
// float64, and the sum is then scaled.  d is [n_rows, N].
void ox_gemm(const uint8_t* a_codes, const uint8_t* a_scales, float ts_a, const uint8_t* b_codes,
             const uint8_t* b_scales, float ts_b, int64_t N, int64_t K, const int64_t* row_ids, int64_t n_rows,
             double* d, int threads) {
  // decode B once (N x K doubles)
  std::vector<double> bd((size_t)(N * K));
  parallel_rows(N, threads, [&](int64_t j0, int64_t j1) {
    for (int64_t j = j0; j < j1; ++j)
      for (int64_t k = 0; k < K; ++k) {
        const uint8_t byte = b_codes[j * (K / 2) + k / 2];
        const uint8_t c = (k & 1) ? (byte >> 4) : (byte & 15);
        bd[(size_t)(j * K + k)] = e2m1_value(c) * e4m3_value(b_scales[j * (K / 16) + k / 16]);
      }
  });
  const double scale = (double)ts_a * (double)ts_b;
  parallel_rows(n_rows, threads, [&](int64_t i0, int64_t i1) {
    std::vector<double> ad((size_t)K);
    for (int64_t i = i0; i < i1; ++i) {
      const int64_t r = row_ids[i];
      for (int64_t k = 0; k < K; ++k) {
        const uint8_t byte = a_codes[r * (K / 2) + k / 2];
        const uint8_t c = (k & 1) ? (byte >> 4) : (byte & 15);
        ad[(size_t)k] = e2m1_value(c) * e4m3_value(a_scales[r * (K / 16) + k / 16]);
      }
      for (int64_t j = 0; j < N; ++j) {
        const double* b = &bd[(size_t)(j * K)];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += ad[(size_t)k] * b[k];
        d[i * N + j] = acc * scale;
      }
    }
  });
}

}  // extern "C"
