/*
 * fos.h -- Four Over Six NVFP4 quantization and block-scaled FP4 GEMM for
 * NVIDIA B300 (sm_103a).  Plain C ABI: device pointers, sizes, an options
 * struct and a CUDA stream.
 *
 * What the library computes (cited by page title and section):
 *   - "FP4" (Ultralytics glossary), "FP4 Nasıl Çalışır": FP4 is E2M1 with the
 *     value grid {0, ±0.5, ±1, ±1.5, ±2, ±3, ±4, ±6}; NVFP4 groups 16 values
 *     under one E4M3 block scale and adds an FP32 per-tensor scale.
 *   - "Four Over Six" (Transformers docs), first section: each 16-value block
 *     is scaled so that its largest magnitude lands on 4 or on 6, whichever
 *     gives the lower quantization error; options: random Hadamard transform,
 *     2D block scaling, transposed inputs, stochastic rounding.
 *   - "FP4", "FP4 ile Çıkarım ve Eğitim": FP4 matrix products accumulate at
 *     higher precision (fos_gemm accumulates in FP32 in tensor memory).
 *
 * Exact definition (identical bit for bit to the CPU reference used by the
 * tests):
 *   y      = x, or 0.25*H16*diag(s)*x per 16-block along the blocking
 *            dimension when the RHT is on (H16 Sylvester Hadamard, butterflies
 *            of stride 1,2,4,8; s_j = 1-2*bit_j of word 0 of
 *            Philox4x32-10(counter (0,0,0,1), key = hadamard_seed)).
 *   s_t    = amax / 2688 (= 6*448), amax = max|y| over the tensor.
 *   t_M    = M*s_t rounded to FP32, for M in {6, 4}, once per tensor.
 *   per block (16 values, or a 16x16 tile): a = max|y|;
 *   sf_M   = E4M3_rne_satfinite(a / t_M), the quotient correctly rounded to
 *            FP32 (the block maximum mapped to M);  eff_M = float(sf_M) * s_t;
 *   q      = y * min(1/eff_M, FLT_MAX);  code = E2M1(q) (RNE, or stochastic:
 *            round up iff ((w >> 8) * 2^-24) < p, w = word (i mod 4) of
 *            Philox4x32-10(counter (lo32(i/4), hi32(i/4), 0, 0), key = sr_seed),
 *            i = r*cols + c the source index of the element);
 *   E_M    = (sum (q - g)^2) * eff_M^2 with g the code's value (sum over a
 *            16-block: two FMA chains over even/odd positions then one add;
 *            over a 2D tile: per source row as above, then a pairwise tree),
 *            or sum y^2 when sf_M == 0;
 *   keep 4 iff E_4 < E_6 (ties keep 6).
 *
 * All pointers named "device" are device pointers owned by the caller.  The
 * library allocates no device memory and keeps no global state besides
 * cached driver entry points; every call enqueues asynchronous work on
 * `stream` and returns without synchronizing.  A call that fails argument
 * validation returns FOS_ERR_INVALID_ARG (or FOS_ERR_UNSUPPORTED) and
 * enqueues nothing.  FOS_ERR_CUDA means a launch failed; the CUDA error is
 * left for cudaGetLastError().
 */
#ifndef FOS_H
#define FOS_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FOS_ABI_VERSION 2

typedef enum fos_status {
  FOS_OK = 0,
  FOS_ERR_INVALID_ARG = 1,
  FOS_ERR_UNSUPPORTED = 2,
  FOS_ERR_CUDA = 3,
  FOS_ERR_TIMEOUT = 4 /* written to a device status word by a kernel whose bounded wait ran out */
} fos_status;

typedef enum fos_scale_rule {
  FOS_SCALE_4OVER6 = 0, /* the adaptive rule: keep the candidate with lower error */
  FOS_SCALE_6 = 1,      /* plain NVFP4: block max mapped to 6 */
  FOS_SCALE_4 = 2       /* block max mapped to 4 (baseline for tests) */
} fos_scale_rule;

typedef enum fos_rounding { FOS_ROUND_RNE = 0, FOS_ROUND_STOCHASTIC = 1 } fos_rounding;

typedef enum fos_sf_layout {
  /* 128 rows x 4 scale columns per 512-byte tile, tiles row-major over
   * (row tile, column tile), (r, c) at (r%32)*16 + ((r%128)/32)*4 + c%4 inside
   * a tile; rows padded to 128 and scale columns to 4 with zero bytes.  This
   * is the layout the block-scaled tensor-core MMA reads (fos_gemm). */
  FOS_SF_SWIZZLED_128x4 = 0,
  FOS_SF_ROWMAJOR = 1 /* [rows][cols/16], no padding */
} fos_sf_layout;

typedef enum fos_dtype { FOS_DTYPE_F32 = 0, FOS_DTYPE_BF16 = 1 } fos_dtype;

typedef struct fos_quant_options {
  uint32_t struct_size;  /* sizeof(fos_quant_options) */
  int32_t scale_rule;    /* fos_scale_rule */
  int32_t rounding;      /* fos_rounding */
  int32_t block_2d;      /* 0: 1x16 blocks; 1: 16x16 tiles, one scale per tile */
  int32_t transpose;     /* 1: the output describes X^T (blocks run along X's rows) */
  int32_t hadamard;      /* 1: apply the random Hadamard transform first */
  int32_t sf_layout;     /* fos_sf_layout */
  int32_t one_launch;    /* 1: 1D blocks along rows without a supplied amax in one
                            cooperative launch (fos_quantize); 0: two launches */
  uint64_t sr_seed;      /* key of the stochastic-rounding Philox stream */
  uint64_t hadamard_seed;/* key of the RHT sign vector */
  const float* tensor_amax; /* optional device pointer: use this amax and skip the amax pass */
} fos_quant_options;

/* A quantized matrix: rows x cols logical values, blocks along cols. */
typedef struct fos_nvfp4_tensor {
  const uint8_t* codes;      /* device: rows x ld_codes bytes, 2 codes per byte, even column in the low nibble */
  const uint8_t* sf;         /* device: E4M3 block scales in sf_layout */
  const float* tensor_scale; /* device: 1 float, s_t */
  int64_t rows;
  int64_t cols;              /* multiple of 16 */
  int64_t ld_codes;          /* bytes between rows, >= cols/2 */
  int32_t sf_layout;
  int32_t reserved;
} fos_nvfp4_tensor;

/* Library and CUDA-side version; FOS_ABI_VERSION of the built library. */
int32_t fos_abi_version(void);
const char* fos_status_string(fos_status s);

/* Bytes of the scale buffer for an output of out_rows x out_cols values
 * (out_cols % 16 == 0).  INVALID_ARG on negative sizes or a bad layout. */
fos_status fos_sf_bytes(int64_t out_rows, int64_t out_cols, int32_t sf_layout, size_t* bytes);

/* Device scratch fos_quantize needs for these options (0 when
 * opt->tensor_amax is given). */
fos_status fos_quantize_workspace_size(int64_t rows, int64_t cols, const fos_quant_options* opt,
                                       size_t* bytes);

/*
 * fos_tensor_amax -- the tensor amax step: *amax_out = max|y| over the bf16
 * matrix X [rows, cols] (row stride ld_x elements), y = X or its RHT along
 * cols (transpose = 0) or along rows (transpose = 1).
 *   x: device, 16-byte aligned, ld_x % 8 == 0, cols % 16 == 0, and
 *      rows % 16 == 0 when hadamard && transpose.
 *   amax_out: device float.  workspace: device, >= fos_quantize_workspace_size().
 */
fos_status fos_tensor_amax(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int32_t hadamard,
                           int32_t transpose, uint64_t hadamard_seed, float* amax_out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/*
 * fos_quantize -- NVFP4 quantization with the Four Over Six block-scale rule.
 *   x         device bf16 [rows, cols], row stride ld_x elements; 16-byte
 *             aligned; ld_x % 8 == 0; cols % 16 == 0; rows % 16 == 0 when
 *             opt->transpose or opt->block_2d.  Values must be finite.
 *   Output orientation: R_out x C_out = rows x cols, or cols x rows when
 *   opt->transpose.  Blocks run along C_out.
 *   codes     device, R_out rows of ld_codes bytes (ld_codes >= C_out/2,
 *             ld_codes % 8 == 0, 8-byte aligned); two E2M1 codes per byte.
 *   sf        device, fos_sf_bytes(R_out, C_out, opt->sf_layout) bytes; pad
 *             bytes are written 0.  For 2D tiles the tile's scale is stored in
 *             each of its 16 rows.
 *   tensor_scale  device float, receives s_t.
 *   choice    optional device [R_out][C_out/16] bytes: 1 where the block kept
 *             the 4 candidate (NULL: not written).
 *   workspace device scratch of fos_quantize_workspace_size() bytes (may be
 *             NULL when opt->tensor_amax is given); its contents need no
 *             initialisation, and calls sharing one workspace must not
 *             overlap on the GPU.
 * The RHT output is not undone: codes describe the transformed values.
 * Without a supplied amax the call runs an amax pass, then the quantize pass as
 * its programmatic dependent (it reads the pass's partial maxima from the
 * workspace).  With opt->one_launch, 1D blocks along rows run both passes in
 * one cooperative launch instead (amax pass, grid barrier in the workspace --
 * its three words are cleared by a 12-byte cudaMemsetAsync on `stream` first
 * -- and a quantize pass that re-reads the input mostly from L2); the two
 * launches measure faster on B300.  A device wait that runs out (a copy or the
 * grid barrier taking over a second) leaves *tensor_scale = NaN: the outputs
 * are then not valid.
 */
fos_status fos_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                        const fos_quant_options* opt, uint8_t* codes, int64_t ld_codes, uint8_t* sf,
                        float* tensor_scale, uint8_t* choice, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/* One matrix of a batch (fos_quantize_batch): source and outputs as in
 * fos_quantize under the batch's options.  R_out x C_out is rows x cols, or
 * cols x rows when opt->transpose is set. */
typedef struct fos_quant_job {
  const void* x;        /* device bf16 [rows, cols], row stride ld_x elements */
  int64_t rows, cols, ld_x;
  uint8_t* codes;       /* device, R_out x ld_codes bytes */
  int64_t ld_codes;
  uint8_t* sf;          /* device, fos_sf_bytes(R_out, C_out, opt->sf_layout) bytes */
  float* tensor_scale;  /* device float: the job's s_t */
  uint8_t* choice;      /* optional device [R_out][C_out/16] bytes, or NULL */
} fos_quant_job;

/* Device scratch fos_quantize_batch needs for n_jobs jobs (8 KiB per job). */
fos_status fos_quantize_batch_workspace_size(int32_t n_jobs, size_t* bytes);

/*
 * fos_quantize_batch -- quantize n_jobs matrices (a layer's weight set, say)
 * with the same options, each with its own tensor amax; results identical to
 * one fos_quantize call per job.
 *   - 1D blocks along rows: the launches are chained so that each job's
 *     memory-bound amax pass runs beside the issue-bound quantization of the
 *     job before it: launch 0 takes job 0's block maxima, launch i+1
 *     quantizes job i while 2 extra warps per CTA take job i+1's block
 *     maxima, and the last launch quantizes the last job.  Order the jobs by
 *     size, smallest first, to overlap the most.
 *   - opt->transpose or opt->block_2d: one launch takes the amax passes of up
 *     to 32 jobs (the tensor maxima of fos_tensor_amax: of the values, or of
 *     their RHT along the blocks' direction), then one quantize launch per
 *     job follows, last job first (its input is the likeliest to be still in
 *     L2); more jobs repeat this per group of 32.
 * The quantize launches use programmatic dependent launch: each may start
 * (its input copies, and in the chained form the next job's maxima) while its
 * predecessor finishes, and waits for it before reading the maxima it needs.
 * Scale-pad clears, when a shape needs them, are enqueued before all of these.
 *   opt       shared options; tensor_amax is not supported here
 *             (FOS_ERR_UNSUPPORTED; use fos_quantize); one_launch does not
 *             apply and is ignored.
 *   workspace device scratch of fos_quantize_batch_workspace_size() bytes,
 *             4-byte aligned, no initialisation needed.
 * Validation covers every job (fos_quantize's checks) before anything is
 * enqueued.  The jobs' outputs must not overlap one another or any source.
 */
fos_status fos_quantize_batch(const fos_quant_job* jobs, int32_t n_jobs, const fos_quant_options* opt,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fos_quantize_noalloc -- fos_quantize for callers that cannot allocate
 * device memory (plugin hosts and inference runtimes that give an operator
 * only its inputs and outputs and forbid cudaMalloc after start-up).  The
 * pages have no counterpart; this is a library convenience.  Same arguments,
 * results and validation as fos_quantize, minus the workspace: the amax
 * pass's partial maxima go to a fixed 8448-byte array in device memory owned by
 * the library (held on every GPU that loads it until the process exits).
 *   - The first call on a device looks up the array's address; make it
 *     before any stream capture.
 *   - All calls share the array: calls that overlap on the GPU race on it.
 *     Nothing in it needs clearing between calls.
 *   - A call whose scratch need exceeds the array returns FOS_ERR_INVALID_ARG
 *     (with the current kernels every call that fos_quantize accepts fits).
 *   - Allocates nothing and calls no allocating routine.
 */
fos_status fos_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                const fos_quant_options* opt, uint8_t* codes, int64_t ld_codes, uint8_t* sf,
                                float* tensor_scale, uint8_t* choice, cudaStream_t stream);

/*
 * fos_dequantize -- x_hat = g * (float(sf) * s_t), each product rounded to FP32;
 * out_dtype FOS_DTYPE_F32, or FOS_DTYPE_BF16 (the FP32 value rounded to
 * nearest even).  out: device [q->rows][ld_out] elements.
 */
fos_status fos_dequantize(const fos_nvfp4_tensor* q, void* out, int32_t out_dtype, int64_t ld_out,
                          cudaStream_t stream);

/*
 * fos_gemm -- C = (s_tA * s_tB) * sum_k (gA*sfA)(gB*sfB), the NVFP4 linear-layer
 * contraction C[m][n] = A[m,:] . B[n,:] with A [M,K] and B [N,K] both
 * quantized along K.  Products and FP32 accumulation run on the tcgen05
 * tensor cores (block-scaled MMA, 16-value E4M3 scales); the result is
 * scaled once in FP32 and rounded to bf16.
 *   A, B      the same K, K % 64 == 0 (one MMA step); FOS_SF_SWIZZLED_128x4
 *             scales, 16-byte aligned; codes 16-byte aligned with
 *             ld_codes % 16 == 0.  M (= A->rows) is any size >= 0 (ragged
 *             tiles are clipped on store); N (= B->rows) % 8 == 0.
 *   C         device bf16 [M][ldc], ldc >= N, ldc % 8 == 0, 16-byte aligned.
 *   dev_status optional device int32: a kernel whose bounded pipeline wait
 *             runs out writes FOS_ERR_TIMEOUT there and leaves C incomplete.
 */
fos_status fos_gemm(const fos_nvfp4_tensor* A, const fos_nvfp4_tensor* B, void* C, int64_t ldc,
                    int32_t* dev_status, cudaStream_t stream);

/* ---- MXFP4 with the 4/6 choice ---- */

/* An MXFP4 matrix: rows x cols values, 32-value blocks along cols, one E8M0
 * scale byte per block and no tensor scale. */
typedef struct fos_mxfp4_tensor {
  const uint8_t* codes; /* device: rows x ld_codes bytes, 2 codes per byte, even column in the low nibble */
  const uint8_t* sf;    /* device: E8M0 block scales in sf_layout, cols/32 scale columns */
  int64_t rows;
  int64_t cols;         /* multiple of 32 */
  int64_t ld_codes;     /* bytes between rows, >= cols/2 */
  int32_t sf_layout;    /* fos_sf_layout over the cols/32 scale columns */
  int32_t reserved;
} fos_mxfp4_tensor;

/* Bytes of an MXFP4 scale buffer for rows x cols values (cols % 32 == 0):
 * rows * cols/32 row-major, or the 128x4 tiles of FOS_SF_SWIZZLED_128x4 over
 * cols/32 scale columns (one tile spans 128 rows x 128 values). */
fos_status fos_mxfp4_sf_bytes(int64_t rows, int64_t cols, int32_t sf_layout, size_t* bytes);

/*
 * fos_quantize_mxfp4 -- MXFP4 ("FP4" glossary page: 32 values under one 8-bit
 * power-of-two scale; E8M0 and the shared exponent as in the OCP
 * Microscaling specification) with the Four Over Six choice between two
 * power-of-two scales.  Per 32-value block along a row, with amax its largest
 * magnitude:
 *   X6 = floor(log2 amax) - 2 (the specification's exponent: maximum into
 *        [4, 8), values above 6 saturate), X4 = X6 + 1 (maximum below 4),
 *        both clamped to [-127, 127];
 *   codes_M = E2M1_rne_satfinite(y * 2^-X_M) (sign kept);
 *   S_M = sum (q - g)^2 over each 16-value half (even and odd FMA chains,
 *        then one add), the two halves added;
 *   keep 4 iff 4 * S_4 < S_6 (ties keep 6); scale byte = X + 127.
 * An all-zero block gets byte 0 and zero codes.  A block that holds a NaN or
 * an infinity gets the E8M0 NaN byte 0xFF, zero codes and choice 0: it
 * dequantizes to NaN (MXFP4 has no other way to carry it).  No tensor scale, no amax
 * pass: one launch.
 *   x         device bf16 [rows][ld_x], 16-byte aligned, ld_x % 8 == 0,
 *             cols % 32 == 0.
 *   sf_layout FOS_SF_ROWMAJOR ([rows][cols/32]) or FOS_SF_SWIZZLED_128x4
 *             (the layout fos_gemm_mxfp4 reads; pad bytes are written 0).
 *   codes     device [rows][ld_codes] bytes, ld_codes >= cols/2, % 4 == 0,
 *             4-byte aligned (16-byte aligned rows are stored 16 bytes at a time).
 *   scales    device, fos_mxfp4_sf_bytes(rows, cols, sf_layout) bytes;
 *             choice optional, [rows][cols/32], 1 where the block kept the
 *             4-candidate.
 *   scale_rule FOS_SCALE_4OVER6, or FOS_SCALE_6 / FOS_SCALE_4 to force one.
 */
fos_status fos_quantize_mxfp4(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int32_t scale_rule,
                              int32_t sf_layout, uint8_t* codes, int64_t ld_codes, uint8_t* scales,
                              uint8_t* choice, cudaStream_t stream);

/* fos_dequantize_mxfp4 -- x_hat = g * 2^(byte - 127), exact in FP32;
 * FOS_DTYPE_BF16 output is that value rounded to nearest even.
 * out: device [q->rows][ld_out] elements, ld_out >= q->cols. */
fos_status fos_dequantize_mxfp4(const fos_mxfp4_tensor* q, void* out, int32_t out_dtype, int64_t ld_out,
                                cudaStream_t stream);

/*
 * fos_gemm_mxfp4 -- C = sum_k (gA * 2^XA)(gB * 2^XB): the contraction of two
 * MXFP4 operands A [M,K] and B [N,K], both quantized along K, with FP32
 * accumulation on the tensor cores ("FP4", "FP4 ile Çıkarım ve Eğitim":
 * FP4 products accumulate at higher precision) and bf16 output.  The same
 * block-scaled MMA as fos_gemm with E8M0 scales; each 32-value scale serves
 * both 16-value halves of its block, so the product is exactly that of the
 * dequantized operands up to the FP32 accumulation.
 *   A, B      the same K, K % 64 == 0; FOS_SF_SWIZZLED_128x4 scales
 *             (fos_quantize_mxfp4), 16-byte aligned; codes 16-byte aligned
 *             with ld_codes % 16 == 0.  M any size >= 0; N % 8 == 0.
 *   C         device bf16 [M][ldc], ldc >= N, ldc % 8 == 0, 16-byte aligned.
 *   dev_status optional device int32, as for fos_gemm.
 */
fos_status fos_gemm_mxfp4(const fos_mxfp4_tensor* A, const fos_mxfp4_tensor* B, void* C, int64_t ldc,
                          int32_t* dev_status, cudaStream_t stream);

/* ---- quantized linear backward ---- */

/*
 * Options of fos_linear_backward.  The "Four Over Six" page ("Training")
 * states that its quantized linear layer has a backward pass; the FP4
 * glossary page ("FP4 ile Çıkarım ve Eğitim") describes the training recipe
 * this follows: random Hadamard transforms against outliers and stochastic
 * rounding for gradients.
 */
typedef struct fos_backward_options {
  uint32_t struct_size;   /* sizeof(fos_backward_options) */
  int32_t scale_rule;     /* fos_scale_rule of all four operands */
  int32_t grad_rounding;  /* fos_rounding of both copies of dY (stochastic in the training recipe) */
  int32_t wgrad_hadamard; /* 1: RHT along M on dY^T and X^T, one sign vector (their product is unchanged) */
  int32_t weight_2d;      /* 1: W^T with 16x16 tiles (the exact transpose of a 2D forward W) */
  int32_t reserved;       /* must be 0 */
  uint64_t sr_seed;       /* stochastic rounding key; both copies of dY use it (source index) */
  uint64_t hadamard_seed; /* RHT sign-vector key */
} fos_backward_options;

/* Device scratch of fos_linear_backward for M x N x K (see its layout). */
fos_status fos_linear_backward_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);

/*
 * fos_linear_backward_operands -- the four quantized operands as they lie in
 * a fos_linear_backward workspace (valid after a call on that workspace):
 *   ops[0] dY   [M, N] blocks along N   (dgrad A)
 *   ops[1] W^T  [K, N] blocks along N   (dgrad B)
 *   ops[2] dY^T [N, M] blocks along M   (wgrad A)
 *   ops[3] X^T  [K, M] blocks along M   (wgrad B)
 * Codes rows are padded to 16-byte strides; scales are FOS_SF_SWIZZLED_128x4.
 * The workspace holds, each section 256-byte aligned and in this order, the
 * codes then the scales of ops[0..3], the four tensor scales, and the
 * quantizer's scratch.
 */
fos_status fos_linear_backward_operands(int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                                        fos_nvfp4_tensor ops[4]);

/*
 * fos_linear_backward -- the NVFP4 backward of Y = X W^T (X [M,K], W [N,K],
 * dY [M,N], all bf16 row-major):
 *   dX = dY . W       [M, K]: dY quantized along N, W quantized along N
 *                     (transposed input), one fos_gemm;
 *   dW = dY^T . X     [N, K]: dY and X quantized along M (transposed input,
 *                     optional RHT), one fos_gemm.
 * Each quantization is exactly fos_quantize's; each product is fos_gemm's.
 * With both products and stochastic rounding, dY's two quantizations run as
 * one launch (one read of dY; each element's Philox word, the same in both, is
 * evaluated once).  Each GEMM is launched as a programmatic dependent of the
 * quantize launch before it (W^T's, X^T's): its CTAs load dY's operand, which
 * is complete, during that launch's tail, and wait for it before the other.
 *   M % 64 == 0, N % 64 == 0 (the contraction lengths), K % 16 == 0; all > 0.
 *   dy, x, w  device bf16, 16-byte aligned, ld % 8 == 0, ld >= the row length.
 *   dx, dw    device bf16 outputs [M][ld_dx], [N][ld_dw] (ld >= K, ld % 8 == 0,
 *             16-byte aligned); either may be NULL to skip that half (its
 *             operands are then not produced).
 *   dev_status optional device int32 for the GEMMs' FOS_ERR_TIMEOUT.  A
 *             quantizer that gives up leaves a NaN tensor scale, which makes
 *             the product that uses it NaN.
 * Everything is enqueued on `stream` in the order dgrad, wgrad.
 */
fos_status fos_linear_backward(const void* dy, int64_t ld_dy, const void* x, int64_t ld_x, const void* w,
                               int64_t ld_w, int64_t M, int64_t N, int64_t K, const fos_backward_options* opt,
                               void* dx, int64_t ld_dx, void* dw, int64_t ld_dw, void* workspace,
                               size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

/* ---- quantized linear forward ---- */

/* Device scratch of fos_linear_forward for X [M, K] (K % 64 == 0). */
fos_status fos_linear_forward_workspace_size(int64_t M, int64_t K, size_t* bytes);

/* X's quantized operand [M, K] as it lies in a fos_linear_forward workspace
 * (valid after a call on it): codes with 16-byte-padded rows, then
 * FOS_SF_SWIZZLED_128x4 scales, then s_t, then the quantizer's scratch, each
 * 256-byte aligned. */
fos_status fos_linear_forward_operand(int64_t M, int64_t K, void* workspace, size_t workspace_bytes,
                                      fos_nvfp4_tensor* xq);

/*
 * fos_linear_forward -- Y = X W^T for the quantized linear layer ("Four Over
 * Six": the layer quantizes its input, then contracts in NVFP4): X bf16
 * [M, K] is quantized with x_opt into the workspace (exactly fos_quantize),
 * then multiplied by the already quantized W [N, K] (exactly fos_gemm).
 * The GEMM is launched as a programmatic dependent of the quantizer: its CTAs
 * start during the quantizer's tail and load W's first stages, and wait for
 * the quantizer before touching X's operand.  W may come from work enqueued
 * before this call (that work completes before the quantizer starts, and the
 * quantizer writes only X's operand).  Quantize W once, offline, with the
 * same RHT seed along K as x_opt when x_opt->hadamard is set.
 *   x_opt     transpose must be 0 and sf_layout FOS_SF_SWIZZLED_128x4;
 *             block_2d, hadamard, stochastic rounding and a supplied
 *             tensor_amax (delayed scaling) are allowed.
 *   w         K-major NVFP4 operand, w->cols == K (see fos_gemm).
 *   y         device bf16 [M][ld_y], ld_y >= w->rows, ld_y % 8 == 0.
 */
fos_status fos_linear_forward(const void* x, int64_t ld_x, int64_t M, int64_t K, const fos_quant_options* x_opt,
                              const fos_nvfp4_tensor* w, void* y, int64_t ld_y, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

/*
 * fos_selftest_wait_limits -- runs the library's bounded device waits into
 * their limits on purpose and reports what the kernels recorded, so a caller
 * (or a test) can check failure detection without faulting or hanging a GPU.
 * The pages have no counterpart; this is a library self-test.
 *   1. fos_gemm's kernel on dummy 128x128x256 operands whose producer never
 *      fills a stage: every wait runs out after timeout_ns and the kernel
 *      writes FOS_ERR_TIMEOUT to result[0], frees its tensor memory and exits.
 *   2. The one-launch row quantizer on a 16 x 64 zero matrix with a grid
 *      barrier that waits for one CTA more than the launch has: the barrier
 *      gives up after timeout_ns, tensor_scale becomes NaN, and result[1]
 *      receives FOS_ERR_TIMEOUT.
 *   scratch     device, >= 128 KiB, 256-byte aligned (operands and outputs).
 *   timeout_ns  1 .. 1e9; result device int32[2], cleared first.
 * Enqueued on `stream`; reads nothing back.  The CUDA context stays usable.
 */
fos_status fos_selftest_wait_limits(void* scratch, size_t scratch_bytes, uint64_t timeout_ns, int32_t* result,
                                    cudaStream_t stream);

/*
 * fos_selftest_mma_rate -- a measurement, not a product path: the tensor-pipe
 * throughput of the GEMM's own MMA instruction on this GPU, the ceiling that
 * fos_gemm's achieved rate is compared with.  The pages have no counterpart.
 * min(grid, SM count) CTAs (one per SM) each issue iters x 4 MMAs of
 * kind::mxf4nvf4 with E4M3 scales per 16 values, M = 128, N = n_cols, K = 64,
 * back to back on zero operands held in shared memory (scales 1.0): no loads,
 * no stores.  Work done: 2 * 128 * n_cols * 64 * 4 * iters flops per CTA;
 * the caller times the launch on `stream` (CUDA events).
 *   n_cols      128 or 256.
 *   iters       1 .. 2^24.
 *   dev_status  optional device int32: FOS_ERR_TIMEOUT if the completion wait
 *               outlasted its limit (2 s); left untouched otherwise.
 * Returns FOS_ERR_INVALID_ARG on other arguments, FOS_ERR_CUDA if the launch fails.
 */
fos_status fos_selftest_mma_rate(int32_t n_cols, int64_t iters, int32_t grid, int32_t* dev_status,
                                 cudaStream_t stream);

/* ---- element codecs (the conversions the quantizer uses), for testing ---- */

/* codes[i] = E2M1 code (RNE, saturating, sign kept) of x[i]; one code per byte. */
fos_status fos_e2m1_encode(const float* x, int64_t n, uint8_t* codes, cudaStream_t stream);
/* out[i] = E4M3 byte (RNE, saturating to 448) of x[i]. */
fos_status fos_e4m3_encode(const float* x, int64_t n, uint8_t* out, cudaStream_t stream);
/* out[4*i .. 4*i+3] = Philox4x32-10(counter[4*i..], key = (lo32(key), hi32(key))). */
fos_status fos_philox4x32_10(const uint32_t* counters, int64_t n, uint64_t key, uint32_t* out,
                             cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FOS_H */
