// Internal launch interface between the C ABI (fos_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "fos.h"

namespace fos {

// Upper bound on the number of CTAs of the amax pass (= partial maxima the
// quantize kernels reduce in their prologue).
constexpr int kMaxAmaxPartials = 2048;
// The column amax pass (the RHT down columns): adjacent source columns per
// lane, and per warp task.
constexpr int kAmaxColCPL = 8;
constexpr int kAmaxColTask = 32 * kAmaxColCPL;
// The row amax pass: blocks per warp task (4 per lane in flight).
constexpr int kAmaxRowBlocks = 128;
// Workspace: the partial maxima, then (at kBarrierOffset) the words of the
// one-launch row quantizer: the grid barrier's arrival counter, a flag that a
// CTA which gave up on a wait raises, and the counter of CTAs that finished
// (the last one writes the tensor scale, or NaN if the flag is up).  The host
// clears the kBarrierWords words before each launch.
constexpr size_t kBarrierOffset = kMaxAmaxPartials * sizeof(float);
constexpr int kBarrierWords = 3;
constexpr size_t kQuantWorkspaceBytes = kBarrierOffset + 256;
static_assert(kBarrierOffset + kBarrierWords * sizeof(unsigned int) <= kQuantWorkspaceBytes, "workspace layout");

struct AmaxParams {
  const uint16_t* x;
  int64_t rows, cols, ld;
  uint32_t hk0, hk1;  // RHT seed words
  bool aligned32;
  float* partials;
  float* partials_plain;  // optional (RHT down columns only): also max |x| untransformed
};

// The amax passes of up to kAmaxBatchJobs jobs in one launch.
constexpr int kAmaxBatchJobs = 32;
struct AmaxBatch {
  AmaxParams job[kAmaxBatchJobs];
  int32_t n_jobs;
};

struct QuantParams {
  const uint16_t* x;
  int64_t rows, cols, ld;  // source matrix
  int64_t R, nb;           // output rows and scale columns
  uint8_t* codes;
  int64_t ld_codes;
  uint8_t* sf;
  int32_t sf_layout;
  uint8_t* choice;
  float* tensor_scale;
  const float* amax_src;   // tensor_amax (n_partials == 0) or the amax partials
  int32_t n_partials;
  uint32_t sr_k0, sr_k1, hk0, hk1;  // SR and RHT seed words
  bool aligned32;
  bool codes16;            // codes and ld_codes 16-byte aligned
  // one-launch row quantizer (amax pass, grid barrier, quantize pass)
  float* ws_partials;      // one partial maximum per CTA
  unsigned int* ws_barrier;
  unsigned int barrier_extra;  // arrivals beyond the grid the barrier waits for (0; 1 only in the self-test)
  uint64_t timeout_ns;         // limit of every device wait (copies, the grid barrier)
  // chained row quantizer: the next job of a batch, whose block maxima this
  // launch also takes (one partial per CTA into next_partials)
  const uint16_t* next_x;
  int64_t next_rows, next_cols, next_ld;
  float* next_partials;
};

// Default limit of a device wait: a copy or barrier that takes a second has failed.
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;

struct DequantParams {
  const uint8_t* codes;
  const uint8_t* sf;
  const float* tensor_scale;
  int64_t rows, cols, ld_codes, ld_out;
  int32_t sf_layout;
  void* out;
};

int amax_grid(int64_t n_warp_tasks, bool hadamard, bool transpose);
int quant_grid(int64_t n_warp_tasks, int kind);
cudaError_t launch_amax(const AmaxParams& p, bool hadamard, bool transpose, int grid, cudaStream_t s);
// The amax passes of b.n_jobs jobs (kernel chosen as launch_amax chooses) in
// one launch of *grid CTAs: one resident wave, at most kMaxAmaxPartials and
// at most (total_tasks + 7) / 8.  Each job gets *grid partial maxima.
cudaError_t launch_amax_batch(const AmaxBatch& b, bool hadamard, bool transpose, int64_t total_tasks, int* grid,
                              cudaStream_t s);

// From one read of x [rows, cols] (rows % 16 == 0, 16-byte aligned, ld % 8 == 0):
// out[0] = max |x| and out[1] = max |y| for y the RHT of x down its columns
// (blocks of 16 rows), each exactly what the separate amax passes give.
// workspace: kQuantWorkspaceBytes of device scratch.
// With n_partials, out is not written: *n_partials receives the partial count,
// the partial maxima of max |y| at workspace and those of max |x| at
// workspace + kMaxAmaxPartials / 2 floats.
cudaError_t amax_plain_and_rht_cols(const void* x, int64_t rows, int64_t cols, int64_t ld, uint64_t hadamard_seed,
                                    float* out, void* workspace, cudaStream_t s, int* n_partials = nullptr);
// kind: 0 rows (1D), 1 cols (1D transposed), 2 2D, 3 2D transposed
// pdl: the launch may overlap the stream's previous kernel, which must be one
// of this library's amax or row-quantize launches (the quantize kernel reads
// x before waiting for it, and the partial maxima after).
cudaError_t launch_quant(const QuantParams& p, int rule, int kind, bool rht, bool sr, int grid, cudaStream_t s,
                         bool pdl = false);
// Both stochastic-rounding quantizations of one source in one launch: pc
// transposed (the RHT down the columns when rht), pr along the rows (no RHT),
// each with its tensor amax supplied (n_partials 0) and the same seed; n_tasks
// = the transposed stochastic-rounding kernel's warp tasks.  The results equal
// the two separate launches'.  A plain launch (no programmatic dependence).
cudaError_t launch_quant_dual_sr(const QuantParams& pc, const QuantParams& pr, int rule, bool rht, int64_t n_tasks,
                                 cudaStream_t s);

// One matrix's quantize launch for fos_quantize's arguments: its parameters,
// with the tensor amax read from amax_src (one float, or n_partials partial
// maxima), its kernel kind (as launch_quant takes it) and its warp tasks.
struct QuantLaunch {
  QuantParams p;
  int kind;
  int64_t tasks;
};
QuantLaunch quant_launch(const void* x, int64_t rows, int64_t cols, int64_t ld_x, const fos_quant_options* opt,
                         uint8_t* codes, int64_t ld_codes, uint8_t* sf, float* tensor_scale, uint8_t* choice,
                         const float* amax_src, int n_partials);
// Clears the pad bytes of p's swizzled scale tiles, when its shape leaves any.
cudaError_t pad_scales(const QuantParams& p, cudaStream_t s);

// Rows (1D) quantized from partials of an earlier launch while 2 extra warps
// per CTA take the block maxima of the next job (p.next_*); grid = chained_grid().
cudaError_t launch_quant_rows_chained(const QuantParams& p, int rule, bool rht, bool sr, int grid, cudaStream_t s);
int chained_grid();
// Rows (1D) with the tensor amax computed in the same launch: a cooperative
// launch of as many CTAs as fit on the GPU at once.
cudaError_t launch_quant_rows_fused(const QuantParams& p, int rule, bool rht, bool sr, int64_t n_tasks,
                                    cudaStream_t s);
cudaError_t launch_sf_pad(uint8_t* sf, int64_t bytes, int64_t R, int64_t nb, cudaStream_t s);
cudaError_t launch_dequant(const DequantParams& p, bool bf16, cudaStream_t s);
// The GEMM kernel on tiny dummy operands in `scratch` with a producer that
// never fills a stage, so its waits run out after timeout_ns and it writes
// FOS_ERR_TIMEOUT to *status.
fos_status gemm_stall_selftest(void* scratch, size_t scratch_bytes, uint64_t timeout_ns, int32_t* status,
                               cudaStream_t s);
// fos_gemm launched with programmatic dependent launch for a stream whose
// previous kernel produces A (its codes, scales and tensor scale) and writes
// nothing B depends on: each CTA loads B's first stages before waiting for
// that kernel, then A.  Only for that pairing: B is read before the wait.
fos_status gemm_after_producer_of_a(const fos_nvfp4_tensor* A, const fos_nvfp4_tensor* B, void* C, int64_t ldc,
                                    int32_t* dev_status, cudaStream_t stream);
// The same with the roles exchanged: the previous kernel produces B and A is
// complete already (A's first stages are loaded before the wait).
fos_status gemm_after_producer_of_b(const fos_nvfp4_tensor* A, const fos_nvfp4_tensor* B, void* C, int64_t ldc,
                                    int32_t* dev_status, cudaStream_t stream);
// *out = FOS_ERR_TIMEOUT if *tensor_scale is NaN, else FOS_OK.
cudaError_t launch_nan_to_status(const float* tensor_scale, int32_t* out, cudaStream_t s);
cudaError_t launch_e2m1_encode(const float* x, int64_t n, uint8_t* out, cudaStream_t s);
cudaError_t launch_e4m3_encode(const float* x, int64_t n, uint8_t* out, cudaStream_t s);
cudaError_t launch_philox(const uint32_t* ctr, int64_t n, uint64_t key, uint32_t* out, cudaStream_t s);

}  // namespace fos
