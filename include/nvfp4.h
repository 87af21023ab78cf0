/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 linear-layer library.
 *
 * The library quantizes BF16 tensors to NVFP4 and multiplies them on the
 * block-scaled FP4 tensor cores, for the three GEMMs of one linear layer:
 * Fprop (Y = X W^T), Dgrad (dX = dY W) and Wgrad (dW = dY^T X).  The method is
 * the one of "Pretraining Large Language Models with NVFP4" (gist.science
 * summary), Resumo técnico §2 Metodologia:
 *   - NVFP4 format: E2M1 elements in blocks of 16, an E4M3 scale per block and
 *     an FP32 scale per tensor ("Formato NVFP4", "Escala em Dois Níveis");
 *   - 16x16 random Hadamard transform on both Wgrad inputs (item 2);
 *   - 2D 16x16 weight blocks, so W and W^T quantize identically (item 3);
 *   - stochastic rounding on gradients, round-to-nearest-even elsewhere
 *     (item 4);
 *   - FP32-accumulated GEMMs on tensor cores that take NVFP4 natively
 *     (Resumo técnico §3, "Suporte de Hardware").
 * It also quantizes to and multiplies MXFP4, the format the method is
 * compared with (Resumo técnico §1, "Limitações de Formatos Existentes":
 * 32-element blocks with power-of-two scales).
 *
 * Conventions shared by every entry point
 *   - All pointers named *_dev or held in nvfp4_tensor are DEVICE pointers on
 *     the current CUDA device; BF16 buffers are row-major.  The caller owns
 *     every buffer; the library allocates no device memory on these calls.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Nothing synchronises except nvfp4_get_status.
 *   - Argument, shape and alignment errors are returned synchronously, before
 *     anything is launched.  Errors found on the device (a non-finite amax, a
 *     pipeline wait that exceeded its bound) are OR-ed into a per-device
 *     status word that nvfp4_get_status reads and clears.
 *   - Device pointers must be 16-byte aligned.
 *   - Results are a pure function of the inputs and `seed`: stochastic
 *     rounding and the Hadamard signs come from Philox4x32-10 (Salmon et al.,
 *     SC'11) keyed by the 64-bit seed, with the counter derived from the
 *     element's index in the quantized tensor.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_ARG = 1,        /* null pointer or invalid enum value */
  NVFP4_ERR_SHAPE = 2,      /* a dimension breaks the size rules of the call */
  NVFP4_ERR_ALIGN = 3,      /* a device pointer or row pitch is not 16-byte aligned */
  NVFP4_ERR_NONFINITE = 4,  /* device: a tensor amax was inf or NaN */
  NVFP4_ERR_TIMEOUT = 5,    /* device: a GEMM pipeline wait exceeded its bound */
  NVFP4_ERR_CUDA = 6,       /* a CUDA runtime call failed */
  NVFP4_ERR_WORKSPACE = 7   /* workspace smaller than nvfp4_linear_workspace_bytes */
} nvfp4_status;

typedef void* nvfp4_stream; /* cudaStream_t */

/* Layout of a block-scale tensor of a [rows, cols] quantized tensor. */
enum {
  NVFP4_SCALES_LINEAR = 0, /* row-major [rows, cols/16] E4M3 bytes */
  NVFP4_SCALES_MMA = 1     /* tiles of 128 rows x 4 scales (512 B), row-tile
                              major; inside a tile row r, scale c is at byte
                              (r%32)*16 + (r/32)*4 + c.  This is the layout the
                              block-scaled tensor-core MMA consumes.  Requires
                              rows % 128 == 0 and cols % 64 == 0. */
};
/* For an MXFP4 tensor the same two names mean:
 *   NVFP4_SCALES_LINEAR  row-major [rows, cols/32] UE8M0 bytes;
 *   NVFP4_SCALES_MMA     the tile layout above with one 4-byte word per 64
 *                        elements of a row: bytes (E0, E1, 0, 0), E0 the
 *                        scale of elements 0-31 and E1 of 32-63 -- the bytes
 *                        a block-scaled MMA with two scales per 64 elements
 *                        reads.  Same size as the NVFP4 MMA layout. */

/* Element format of an nvfp4_tensor (its `format` field). */
enum {
  NVFP4_FORMAT_NVFP4 = 0, /* E2M1, E4M3 scale per 16 elements, FP32 tensor scale */
  NVFP4_FORMAT_MXFP4 = 1  /* E2M1, UE8M0 scale per 32 elements (value 2^(E-127),
                             code 255 unused), no tensor scale */
};

/*
 * A quantized NVFP4 tensor of logical shape [rows, cols]; cols is the
 * dimension the 1x16 blocks run along (the GEMM reduction dimension).
 *   codes         device, [rows, cols/2] bytes; byte j of a row holds element
 *                 2j in bits 0-3 and element 2j+1 in bits 4-7; each element is
 *                 an E2M1 code s.ee.m (value (-1)^s * {0,.5,1,1.5,2,3,4,6}).
 *   scales        device, E4M3 block scales in `scale_layout`;
 *                 nvfp4_scale_bytes() gives the size.
 *   amax          device, 1 float: max |x| of the tensor being quantized
 *                 (after the Hadamard transform where one applies).  An input
 *                 of nvfp4_quantize unless its cfg asks to compute it.
 *   tensor_scale  device, 1 float: the FP32 per-tensor decode scale
 *                 ts = 1 / (2688 / amax) (1 when amax == 0), written by
 *                 nvfp4_quantize; value = e2m1(code) * e4m3(scale) * ts.
 *   format        NVFP4_FORMAT_*; zero (NVFP4) in a zero-initialised struct.
 *                 An MXFP4 tensor has UE8M0 scales per 32 elements and no
 *                 amax or tensor scale (both may be NULL):
 *                 value = e2m1(code) * 2^(scale - 127).
 */
typedef struct {
  uint8_t* codes;
  uint8_t* scales;
  float* amax;
  float* tensor_scale;
  int64_t rows;
  int64_t cols;
  int32_t scale_layout;
  int32_t format;
} nvfp4_tensor;

/* What nvfp4_quantize produces. */
enum {
  /* out = x [rows, cols] quantized with 1x16 blocks along cols. */
  NVFP4_Q_ROWWISE = 0,
  /* out = x^T [cols, rows], 1x16 blocks along rows (the token dimension of a
     Wgrad operand). */
  NVFP4_Q_TRANSPOSE = 1,
  /* both outputs from one read of x: out = ROWWISE (never transformed),
     out_t = TRANSPOSE (transformed when cfg.rht). */
  NVFP4_Q_ROWWISE_AND_TRANSPOSE = 2,
  /* weights: one scale per 16x16 block.  out = W [rows, cols]; out_t
     (optional, may be NULL) = W^T [cols, rows].  The two hold the same codes
     transposed and the same block scales, replicated into every row of the
     block.  Always round-to-nearest-even, never transformed. */
  NVFP4_Q_2D = 3
};

enum { NVFP4_ROUND_RNE = 0, NVFP4_ROUND_SR = 1 };

/*
 * Options of nvfp4_quantize.
 *   kind          NVFP4_Q_*.
 *   rounding      NVFP4_ROUND_RNE or NVFP4_ROUND_SR, for every output of the
 *                 call (2D is always RNE).
 *   rht           nonzero: apply the 16x16 random Hadamard transform
 *                 Q = 1/4 * H16 * diag(s) to each 16-chunk along the blocked
 *                 dimension before quantizing -- along cols for ROWWISE, along
 *                 rows (tokens) for the transposed output.
 *   compute_amax  nonzero: first compute out->amax (and out_t->amax) from x;
 *                 zero: use the values already there (from nvfp4_amax).
 *   seed          Philox key: stochastic rounding and the Hadamard signs
 *                 (signs = bits of word 0 of Philox(seed, (0, 0, 2, 0))).
 *   sr_stream     Philox stream id of `out`'s stochastic rounding.
 *   sr_stream_t   Philox stream id of `out_t`'s stochastic rounding.
 */
typedef struct {
  int32_t kind;
  int32_t rounding;
  int32_t rht;
  int32_t compute_amax;
  uint64_t seed;
  uint32_t sr_stream;
  uint32_t sr_stream_t;
} nvfp4_quant_cfg;

/* nvfp4_amax variants (bit flags), each writing its own slot of amax_dev. */
enum {
  NVFP4_AMAX_PLAIN = 1,    /* amax_dev[0] = max |x| */
  NVFP4_AMAX_RHT_ROWS = 2, /* amax_dev[1] = max |Q x| with Q along cols (16-chunks of a row) */
  NVFP4_AMAX_RHT_COLS = 4  /* amax_dev[2] = max |Q x| with Q along rows (16-row chunks of a column) */
};

/*
 * nvfp4_amax -- global amax of a BF16 tensor, the input of the FP32
 * per-tensor scale (Resumo técnico §2, "Escala em Dois Níveis").
 *   x_dev       BF16 [rows, cols], row-major.
 *   flags       OR of NVFP4_AMAX_*; every requested slot of amax_dev (3
 *               floats) is overwritten.  A non-finite amax also sets
 *               NVFP4_ERR_NONFINITE in the device status word.
 *   rht_seed    seed of the Hadamard signs for the RHT variants.
 * Sizes: cols % 16 == 0; RHT_COLS also needs rows % 16 == 0.  rows*cols may
 * be 0 (the amax is then 0).
 */
nvfp4_status nvfp4_amax(const void* x_dev, int64_t rows, int64_t cols, int32_t flags,
                        uint64_t rht_seed, float* amax_dev, nvfp4_stream stream);

/*
 * nvfp4_quantize -- BF16 -> NVFP4 (Resumo técnico §2: "Formato NVFP4" and
 * items 2-4).  Two-level scaling, all in IEEE float32:
 *   s_enc = 2688 / amax;  ts = 1 / s_enc;
 *   per block: E = e4m3_rne_satfinite((amax_b / 6) * s_enc);
 *              enc = s_enc / e4m3(E)  (0 if E == 0);
 *              code_i = e2m1_round(x_i * enc)   (RNE or stochastic).
 * Stochastic rounding of element e (its row-major index in the quantized
 * tensor): u = 16 bits of Philox(seed, (lo32(e/8), hi32(e/8), stream, 0)),
 * word (e%8)/2, low half for even e; round up iff u < frac * 65536.
 *   x_dev   BF16 [rows, cols].
 *   out     see nvfp4_quant_cfg.kind for its shape; must match.
 *   out_t   transposed output for the kinds that have one, else ignored.
 * Sizes: rows % 64 == 0 and cols % 64 == 0 (rows, cols > 0); an MMA scale
 * layout also needs its tensor's rows % 128 == 0.  Outputs must have format
 * NVFP4_FORMAT_NVFP4 (MXFP4 outputs: nvfp4_quantize_mx).
 */
nvfp4_status nvfp4_quantize(const void* x_dev, int64_t rows, int64_t cols,
                            const nvfp4_quant_cfg* cfg, const nvfp4_tensor* out,
                            const nvfp4_tensor* out_t, nvfp4_stream stream);

/* Bytes of the block-scale tensor of a [rows, cols] NVFP4 tensor. */
size_t nvfp4_scale_bytes(int64_t rows, int64_t cols, int32_t scale_layout);

/*
 * nvfp4_quantize_mx -- BF16 -> MXFP4 (Resumo técnico §1, "Limitações de
 * Formatos Existentes", and §2, "Fatores de Escala Precisos": the format
 * NVFP4 is compared with).  Scale rule of OCP Microscaling Formats v1.0 for
 * E2M1, per block of 32 consecutive elements along the blocked dimension:
 *   E = floor(log2(max |x|)) - 2 + 127, clamped to >= 0 (0 for a zero block);
 *   code_i = e2m1_rne_satfinite(x_i * 2^(127 - E))  (one float32 multiply).
 * The block's largest value lands in [4, 8); values above 6 saturate.
 *   x_dev   BF16 [rows, cols]; finite values (the codes written for a block
 *           holding inf or NaN are unspecified; nothing is flagged).
 *   kind    NVFP4_Q_ROWWISE (out = x, blocks along cols), NVFP4_Q_TRANSPOSE
 *           (out = x^T [cols, rows], blocks along rows) or
 *           NVFP4_Q_ROWWISE_AND_TRANSPOSE (out = x, out_t = x^T, one read).
 *   out, out_t  format NVFP4_FORMAT_MXFP4, codes and scales set; amax and
 *           tensor_scale are ignored.
 * Sizes: rows % 64 == 0 and cols % 64 == 0 (rows, cols > 0); an MMA scale
 * layout also needs its tensor's rows % 128 == 0.
 */
nvfp4_status nvfp4_quantize_mx(const void* x_dev, int64_t rows, int64_t cols, int32_t kind,
                               const nvfp4_tensor* out, const nvfp4_tensor* out_t,
                               nvfp4_stream stream);

/* Bytes of the block-scale tensor of a [rows, cols] MXFP4 tensor. */
size_t nvfp4_mx_scale_bytes(int64_t rows, int64_t cols, int32_t scale_layout);

enum { NVFP4_OUT_BF16 = 0, NVFP4_OUT_F32 = 1 };

/*
 * nvfp4_gemm -- block-scaled FP4 GEMM on the tensor cores (Resumo técnico §3,
 * "Suporte de Hardware"): D[M, N] = ts_a * ts_b * sum_k A[m, k] B[n, k] with
 * every operand element decoded as e2m1(code) * e4m3(block scale), FP32
 * accumulation, output rounded to BF16 (or stored as FP32).
 *   a        [M, K] NVFP4, scales in NVFP4_SCALES_MMA layout.
 *   b        [N, K] NVFP4, scales in NVFP4_SCALES_MMA layout.
 *   d_dev    [M, ldd] BF16 or FP32 (d_dtype = NVFP4_OUT_*), row-major.
 * With both operands in NVFP4_FORMAT_MXFP4 the same call multiplies MXFP4:
 * elements decode as e2m1(code) * 2^(scale - 127) with one scale per 32, and
 * there is no tensor scale.  Mixed formats are rejected (NVFP4_ERR_ARG).
 * Sizes: M % 128 == 0, N % 128 == 0, K % 64 == 0, ldd >= N, and ldd times the
 * element size a multiple of 16 bytes.  M, N or K == 0 is rejected.
 */
nvfp4_status nvfp4_gemm(const nvfp4_tensor* a, const nvfp4_tensor* b, void* d_dev, int32_t d_dtype,
                        int64_t ldd, nvfp4_stream stream);

/*
 * nvfp4_gemm2 -- two independent GEMMs of nvfp4_gemm, d0 = a0 b0^T and
 * d1 = a1 b1^T (BF16 outputs), in one launch: the layer's Dgrad and Wgrad
 * (Resumo técnico §2, "Técnicas de Treinamento Integradas", items 2-4, and
 * §3, "Suporte de Hardware").  When both products take the CTA-pair kernel
 * (all of a0, b0, a1, b1 with rows % 256 == 0) and share the operand format,
 * their 256 x 256 tiles run over one persistent tile schedule in which the
 * CTA pairs that the first product's last round leaves idle start on the
 * second; each output is bit-identical to its nvfp4_gemm.  Otherwise the two
 * products are launched one after the other.
 *   a0, b0, d0_dev, ldd0 and a1, b1, d1_dev, ldd1: as a, b, d_dev, ldd of
 *            nvfp4_gemm with d_dtype NVFP4_OUT_BF16, each pair checked the same
 *            way.  d0 and d1 must not overlap (NVFP4_ERR_ARG if their byte
 *            ranges intersect).
 */
nvfp4_status nvfp4_gemm2(const nvfp4_tensor* a0, const nvfp4_tensor* b0, void* d0_dev, int64_t ldd0,
                         const nvfp4_tensor* a1, const nvfp4_tensor* b1, void* d1_dev, int64_t ldd1,
                         nvfp4_stream stream);

/*
 * nvfp4_gemm_amax -- nvfp4_gemm that also yields the amax its output's
 * consumer needs: the global amax that sets the per-tensor scale of the next
 * quantization (Resumo técnico §2, two-level scaling), taken in the epilogue
 * instead of by a separate read of D.
 *   amax_dev  one float in device memory, 4-byte aligned; zeroed on `stream`
 *             first, then it receives max |D| over the stored values (after
 *             BF16 rounding for BF16 output; +inf or NaN if D holds one).
 *             Pass it to nvfp4_quantize of D with compute_amax = 0 as the
 *             output tensor's amax.
 * Other arguments, sizes and errors as nvfp4_gemm.
 */
nvfp4_status nvfp4_gemm_amax(const nvfp4_tensor* a, const nvfp4_tensor* b, void* d_dev, int32_t d_dtype,
                             int64_t ldd, float* amax_dev, nvfp4_stream stream);

/*
 * nvfp4_gemm_quant -- nvfp4_gemm whose epilogue also writes its output
 * already quantized for the next layer's Fprop: D is rounded to BF16 and each
 * row's 1x16 blocks are quantized to NVFP4 with round-to-nearest-even, exactly
 * as nvfp4_quantize(ROWWISE, RNE, no transform, compute_amax = 0) of that BF16
 * D would quantize it, so the BF16 D need not be written and read back.  The
 * pages fix no policy for the tensor amax of a tensor quantized where it is
 * produced; the caller supplies it (for instance the previous step's
 * nvfp4_gemm_amax of the same layer, a delayed amax).
 *   y_q       [M, N] NVFP4, NVFP4_SCALES_MMA; its amax (device, 1 float) is
 *             read; its codes, scales and tensor_scale are written.  A
 *             non-finite amax sets NVFP4_ERR_NONFINITE in the status word.
 *   d_dev     BF16 [M, ldd] output as in nvfp4_gemm, or NULL for none.
 *   amax_dev  NULL, or one float that receives max |D| (as nvfp4_gemm_amax);
 *             must not be y_q->amax.
 * Operands: NVFP4 (not MXFP4).  Sizes: M % 256 == 0, N % 256 == 0 (the
 * CTA-pair kernel), K % 64 == 0; other rules as nvfp4_gemm.
 */
nvfp4_status nvfp4_gemm_quant(const nvfp4_tensor* a, const nvfp4_tensor* b, const nvfp4_tensor* y_q,
                              void* d_dev, int64_t ldd, float* amax_dev, nvfp4_stream stream);

/*
 * One NVFP4 linear layer Y = X W^T, X [M, K] tokens x in-features, W [N, K]:
 * the three GEMMs of a training step -- Fprop, Dgrad and Wgrad -- with the
 * quantization recipe of "Pretraining Large Language Models with NVFP4"
 * (gist.science summary), Resumo técnico §2, "Técnicas de Treinamento
 * Integradas": item 2 (random Hadamard transform on both Wgrad inputs, along
 * the token dimension the Wgrad GEMM reduces over), item 3 (16x16 weight
 * blocks, so the W of Fprop and the W^T of Dgrad are one quantization) and
 * item 4 (stochastic rounding of the gradient dY, round-to-nearest-even for X
 * and W), on the two-level NVFP4 format of the same section ("Formato NVFP4",
 * "Escala em Dois Níveis": each operand's FP32 scale comes from the amax of
 * the tensor actually quantized, after the transform where one applies).
 *
 * nvfp4_linear_fwd: amax of X, of the Hadamard-transformed X^T and of W;
 *   X -> rowwise RNE (Fprop operand) and X^T -> Hadamard + RNE (saved Wgrad
 *   operand) in one read; W -> 16x16 blocks giving W (Fprop) and W^T (saved
 *   Dgrad operand); then Y = X W^T (BF16).
 * nvfp4_linear_bwd: amax of dY and of the transformed dY^T; dY -> rowwise SR
 *   (Philox stream 0) and dY^T -> Hadamard + SR (stream 1) in one read; then
 *   dX = dY W and dW = dY^T X (BF16) from the saved operands, both in one
 *   GEMM launch when M, K and N are multiples of 256 (as nvfp4_gemm2).  The
 *   Hadamard signs come from `seed` (stream 2) and must be the same seed as
 *   fwd's, so the transform cancels in dW.
 *   x_dev, w_dev, dy_dev, y_dev, dx_dev, dw_dev: BF16 row-major.
 *   ws_dev   workspace of nvfp4_linear_workspace_bytes(M, K, N) bytes; fwd
 *            writes the saved operands there and bwd reads them, so the same
 *            workspace must be passed to both, untouched in between.
 * Sizes: M, K, N positive multiples of 128.
 * Streams: everything is ordered on `stream`.  Outside stream capture, fwd
 * runs W's amax and 2D quantization on a side stream that the library
 * creates once per device, forked from `stream` and joined back into it with
 * events before the GEMM (so it overlaps X's quantization); calls from several
 * host threads are serialised while they enqueue.  While `stream` is being
 * captured into a graph, fwd enqueues all of its work on `stream` itself.
 * Make the first call on a device outside capture (it creates the side
 * stream and sets kernel attributes).
 */
size_t nvfp4_linear_workspace_bytes(int64_t M, int64_t K, int64_t N);
nvfp4_status nvfp4_linear_fwd(const void* x_dev, const void* w_dev, int64_t M, int64_t K, int64_t N,
                              uint64_t seed, void* y_dev, void* ws_dev, size_t ws_bytes,
                              nvfp4_stream stream);
nvfp4_status nvfp4_linear_bwd(const void* dy_dev, int64_t M, int64_t K, int64_t N, uint64_t seed,
                              void* dx_dev, void* dw_dev, void* ws_dev, size_t ws_bytes,
                              nvfp4_stream stream);

/* Views of the quantized operands inside a linear-layer workspace. */
typedef struct {
  nvfp4_tensor xq;   /* X   [M, K] rowwise RNE       (Fprop A) */
  nvfp4_tensor wq;   /* W   [N, K] 16x16 RNE         (Fprop B) */
  nvfp4_tensor wtq;  /* W^T [K, N] 16x16 RNE         (Dgrad B) */
  nvfp4_tensor xtq;  /* X^T [K, M] Hadamard + RNE    (Wgrad B) */
  nvfp4_tensor dyq;  /* dY  [M, N] rowwise SR        (Dgrad A) */
  nvfp4_tensor dytq; /* dY^T[N, M] Hadamard + SR     (Wgrad A) */
} nvfp4_linear_views;

nvfp4_status nvfp4_linear_get_views(void* ws_dev, int64_t M, int64_t K, int64_t N,
                                    nvfp4_linear_views* views);

/*
 * nvfp4_linear_fwd_noalloc -- nvfp4_linear_fwd without a caller workspace.
 * The paper has no counterpart; this is a convenience of the library.
 *
 * Some callers cannot allocate device memory of their own: a plugin inside a
 * host framework whose allocator owns all of the GPU's memory and forbids
 * direct cudaMalloc, or a service whose device-memory budget is fixed at
 * start-up.  This entry point computes the same Y = X W^T as
 * nvfp4_linear_fwd (same kernels, same results) but takes its workspace from
 * a 32 MiB array that the library itself holds in device memory, on every GPU
 * that loads the library, until the process exits.  It allocates nothing.
 *   x_dev, w_dev, y_dev  as in nvfp4_linear_fwd (the caller still owns them).
 * Limits: nvfp4_linear_workspace_bytes(M, K, N) must be at most 32 MiB
 * (33554432 bytes), e.g. M = K = N = 2048; larger layers return
 * NVFP4_ERR_WORKSPACE before anything is launched.  Other size rules as
 * nvfp4_linear_fwd.
 * The first call on a device looks up the array's device address (with that
 * device current) and keeps it for the rest of the process; make that first
 * call before any stream capture.  A cudaDeviceReset (or any other reset of
 * the device's primary context) reloads the library's device code at a new
 * address, so this entry point must not be called on that device after such
 * a reset in the same process.  Every
 * call shares the one array and leaves its contents behind; nothing in it has
 * to start at zero.  Calls whose work overlaps on the GPU (other streams, or
 * other host threads) race on the array: serialise them.  The quantized
 * operands left in the array are not a valid input for nvfp4_linear_bwd.
 */
nvfp4_status nvfp4_linear_fwd_noalloc(const void* x_dev, const void* w_dev, int64_t M, int64_t K, int64_t N,
                                      uint64_t seed, void* y_dev, nvfp4_stream stream);

/*
 * The linear layers the method keeps in BF16 (Resumo técnico §2, item 1,
 * "Precisão Mista Seletiva": the sensitive layers -- the last ones of the
 * network, about 15% -- stay in BF16 while the rest trains in NVFP4): the
 * same layer step without quantization, BF16 in and out, FP32 accumulation,
 * on cuBLAS.
 *   nvfp4_linear_bf16_fwd: Y = X W^T.
 *   nvfp4_linear_bf16_bwd: dX = dY W and dW = dY^T X.
 *   x_dev [M, K], w_dev [N, K], dy_dev [M, N], y_dev [M, N], dx_dev [M, K],
 *   dw_dev [N, K]: BF16, row-major, contiguous.
 * Sizes: M, K, N positive, K and N multiples of 8 (16-byte rows).
 * Streams: enqueued on `stream`.  The first call on a device creates the
 * library's cuBLAS handle for it (cuBLAS allocates its own workspace then);
 * make it outside stream capture.  Calls from several host threads are
 * serialised while they enqueue.  A cuBLAS failure returns NVFP4_ERR_CUDA.
 */
nvfp4_status nvfp4_linear_bf16_fwd(const void* x_dev, const void* w_dev, int64_t M, int64_t K, int64_t N,
                                   void* y_dev, nvfp4_stream stream);
nvfp4_status nvfp4_linear_bf16_bwd(const void* dy_dev, const void* x_dev, const void* w_dev, int64_t M,
                                   int64_t K, int64_t N, void* dx_dev, void* dw_dev, nvfp4_stream stream);

/*
 * nvfp4_get_status -- synchronises `stream`, then returns and clears the
 * current device's status word (NVFP4_OK if no device-side error was seen
 * since the last call); NVFP4_ERR_CUDA if the synchronisation failed.
 */
nvfp4_status nvfp4_get_status(nvfp4_stream stream);
const char* nvfp4_status_string(nvfp4_status status);

/* Number of kernels this library launched since load (host-side count). */
uint64_t nvfp4_kernel_launch_count(void);

/*
 * nvfp4_debug_stall_next_gemm -- failure-detection test hook (no counterpart
 * in the paper).  With on != 0, the next nvfp4_gemm launch never issues the
 * loads of its first pipeline stage, so every pipeline wait of that launch
 * runs into its bound (about 2 s): the kernel stops its roles, frees its
 * tensor memory and returns, nvfp4_get_status then reports
 * NVFP4_ERR_TIMEOUT, and the CUDA context stays usable.  The output of that
 * launch is unspecified.  The flag applies to one launch only.
 */
void nvfp4_debug_stall_next_gemm(int32_t on);

/*
 * nvfp4_debug_stall_next_quantize -- the same test hook for the quantize
 * kernels fed by a TMA tile pipeline (nvfp4_quantize_mx, and nvfp4_quantize
 * of every round-to-nearest-even kind and of NVFP4_Q_2D).  With on != 0, the
 * next such launch never loads the first tile of its first CTA; that CTA's
 * wait for it
 * runs into its bound (about 2 s), the kernel stops, waits (bounded) for the
 * loads it did issue and returns; nvfp4_get_status then reports
 * NVFP4_ERR_TIMEOUT and the CUDA context stays usable.  The output of that
 * launch is unspecified.  The flag applies to one launch only.
 */
void nvfp4_debug_stall_next_quantize(int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H */
