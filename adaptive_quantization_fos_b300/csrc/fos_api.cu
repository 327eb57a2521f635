// C ABI of the Four Over Six NVFP4 library: argument validation and launches.
// No function here allocates device memory or synchronizes the stream.
#include <cuda_runtime.h>

#include <cstdint>

#include "fos.h"
#include "fos_internal.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

fos_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FOS_OK : FOS_ERR_CUDA; }

bool valid_options(const fos_quant_options* o) {
  if (!o || o->struct_size < sizeof(fos_quant_options)) return false;
  if (o->scale_rule < FOS_SCALE_4OVER6 || o->scale_rule > FOS_SCALE_4) return false;
  if (o->rounding != FOS_ROUND_RNE && o->rounding != FOS_ROUND_STOCHASTIC) return false;
  if ((o->block_2d | o->transpose | o->hadamard) & ~1) return false;
  if (o->sf_layout != FOS_SF_SWIZZLED_128x4 && o->sf_layout != FOS_SF_ROWMAJOR) return false;
  return (o->one_launch & ~1) == 0;
}

int64_t sf_bytes_of(int64_t R, int64_t nb, int32_t layout) {
  if (layout == FOS_SF_ROWMAJOR) return R * nb;
  return ((R + 127) / 128) * 128 * ((nb + 3) / 4) * 4;
}

// Shared checks of the source matrix.
bool valid_source(const void* x, int64_t rows, int64_t cols, int64_t ld_x, bool rows16) {
  if (rows < 0 || cols < 0 || cols % 16 != 0 || ld_x < cols || ld_x % 8 != 0) return false;
  if ((!x && rows * cols != 0) || !aligned(x, 16)) return false;
  if (rows16 && rows % 16 != 0) return false;
  return true;
}

__global__ void amax_final_kernel(const float* partials, int n, float* out) {
  __shared__ float s[256];
  float m = 0.0f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, partials[i]);
  s[threadIdx.x] = m;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) s[threadIdx.x] = fmaxf(s[threadIdx.x], s[threadIdx.x + o]);
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = s[0];
}

// The warp tasks of launch_amax(hadamard, transpose) over x [rows, cols]: the
// RHT down the columns runs the column kernel, everything else the row kernel.
int64_t amax_tasks(int64_t rows, int64_t cols, bool hadamard, bool transpose) {
  if (hadamard && transpose) return (rows / 16) * ((cols + fos::kAmaxColTask - 1) / fos::kAmaxColTask);
  return rows * ((cols / 16 + fos::kAmaxRowBlocks - 1) / fos::kAmaxRowBlocks);
}

int amax_tasks_grid(int64_t rows, int64_t cols, bool hadamard, bool transpose) {
  return fos::amax_grid(amax_tasks(rows, cols, hadamard, transpose), hadamard, transpose);
}

// The checks fos_quantize makes of one matrix's source and outputs (less the
// workspace's).
bool valid_matrix(const void* x, int64_t rows, int64_t cols, int64_t ld_x, const fos_quant_options* opt,
                  const uint8_t* codes, int64_t ld_codes, const uint8_t* sf, const float* tensor_scale) {
  const bool tr = opt->transpose != 0;
  if (!valid_source(x, rows, cols, ld_x, tr || opt->block_2d)) return false;
  const int64_t R = tr ? cols : rows, C = tr ? rows : cols;
  const bool empty = R == 0 || C == 0;
  if ((!empty && (!codes || !sf)) || !tensor_scale) return false;
  return ld_codes >= C / 2 && ld_codes % 8 == 0 && aligned(codes, 8) && aligned(sf, 4);
}


}  // namespace

namespace fos {
QuantLaunch quant_launch(const void* x, int64_t rows, int64_t cols, int64_t ld_x, const fos_quant_options* opt,
                         uint8_t* codes, int64_t ld_codes, uint8_t* sf, float* tensor_scale, uint8_t* choice,
                         const float* amax_src, int n_partials) {
  const bool tr = opt->transpose != 0, two_d = opt->block_2d != 0, sr = opt->rounding == FOS_ROUND_STOCHASTIC;
  const int64_t R = tr ? cols : rows, C = tr ? rows : cols, nb = C / 16;
  QuantLaunch q{};
  QuantParams& p = q.p;
  p.x = static_cast<const uint16_t*>(x);
  p.rows = rows;
  p.cols = cols;
  p.ld = ld_x;
  p.R = R;
  p.nb = nb;
  p.codes = codes;
  p.ld_codes = ld_codes;
  p.sf = sf;
  p.sf_layout = opt->sf_layout;
  p.choice = choice;
  p.tensor_scale = tensor_scale;
  p.amax_src = amax_src;
  p.n_partials = n_partials;
  p.sr_k0 = (uint32_t)opt->sr_seed;
  p.sr_k1 = (uint32_t)(opt->sr_seed >> 32);
  p.hk0 = (uint32_t)opt->hadamard_seed;
  p.hk1 = (uint32_t)(opt->hadamard_seed >> 32);
  p.aligned32 = aligned(x, 32) && ld_x % 16 == 0;
  p.codes16 = aligned(codes, 16) && ld_codes % 16 == 0;
  p.timeout_ns = fos::kWaitTimeoutNs;
  if (two_d) {
    q.kind = tr ? 3 : 2;
    // warp tasks of 16 source rows x 4 tiles (stochastic rounding, not
    // transposed) or 2
    const int tpt = (!tr && sr) ? 4 : 2;
    q.tasks = (rows / 16) * ((cols / 16 + tpt - 1) / tpt);
  } else if (tr) {
    q.kind = 1;
    // warp tasks of 64 source rows x 128 (RNE) or 64 (stochastic) source columns
    const int64_t w = sr ? 64 : 128;
    q.tasks = ((rows / 16 + 3) / 4) * ((cols + w - 1) / w);
  } else {
    q.kind = 0;
    q.tasks = R * ((nb + 127) / 128);
  }
  return q;
}

cudaError_t pad_scales(const QuantParams& p, cudaStream_t s) {
  if (p.sf_layout != FOS_SF_SWIZZLED_128x4 || (p.R % 128 == 0 && p.nb % 4 == 0)) return cudaSuccess;
  return launch_sf_pad(p.sf, sf_bytes_of(p.R, p.nb, p.sf_layout), p.R, p.nb, s);
}

cudaError_t amax_plain_and_rht_cols(const void* x, int64_t rows, int64_t cols, int64_t ld, uint64_t hadamard_seed,
                                    float* out, void* workspace, cudaStream_t s, int* n_partials) {
  AmaxParams a{};
  a.x = static_cast<const uint16_t*>(x);
  a.rows = rows;
  a.cols = cols;
  a.ld = ld;
  a.hk0 = (uint32_t)hadamard_seed;
  a.hk1 = (uint32_t)(hadamard_seed >> 32);
  a.aligned32 = aligned(x, 32) && ld % 16 == 0;
  // the two partial arrays share the workspace's partial-maxima region
  a.partials = static_cast<float*>(workspace);
  a.partials_plain = a.partials + kMaxAmaxPartials / 2;
  int g = amax_tasks_grid(rows, cols, true, true);
  if (g > kMaxAmaxPartials / 2) g = kMaxAmaxPartials / 2;
  cudaError_t e = launch_amax(a, true, true, g, s);
  if (e != cudaSuccess) return e;
  if (n_partials) {  // the caller's quantize launches reduce the partials themselves
    *n_partials = g;
    return cudaSuccess;
  }
  amax_final_kernel<<<1, 256, 0, s>>>(a.partials_plain, g, out);
  amax_final_kernel<<<1, 256, 0, s>>>(a.partials, g, out + 1);
  return cudaGetLastError();
}
}  // namespace fos

extern "C" {

int32_t fos_abi_version(void) { return FOS_ABI_VERSION; }

const char* fos_status_string(fos_status s) {
  switch (s) {
    case FOS_OK: return "ok";
    case FOS_ERR_INVALID_ARG: return "invalid argument";
    case FOS_ERR_UNSUPPORTED: return "unsupported";
    case FOS_ERR_CUDA: return "CUDA launch error";
    case FOS_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

fos_status fos_sf_bytes(int64_t out_rows, int64_t out_cols, int32_t sf_layout, size_t* bytes) {
  if (!bytes || out_rows < 0 || out_cols < 0 || out_cols % 16 != 0) return FOS_ERR_INVALID_ARG;
  if (sf_layout != FOS_SF_SWIZZLED_128x4 && sf_layout != FOS_SF_ROWMAJOR) return FOS_ERR_INVALID_ARG;
  *bytes = (size_t)sf_bytes_of(out_rows, out_cols / 16, sf_layout);
  return FOS_OK;
}

fos_status fos_quantize_workspace_size(int64_t rows, int64_t cols, const fos_quant_options* opt, size_t* bytes) {
  if (!bytes || rows < 0 || cols < 0 || !valid_options(opt)) return FOS_ERR_INVALID_ARG;
  *bytes = opt->tensor_amax ? 0 : fos::kQuantWorkspaceBytes;
  return FOS_OK;
}

fos_status fos_tensor_amax(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int32_t hadamard,
                           int32_t transpose, uint64_t hadamard_seed, float* amax_out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  if (!valid_source(x, rows, cols, ld_x, hadamard && transpose) || !amax_out) return FOS_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < fos::kQuantWorkspaceBytes || !aligned(workspace, 4)) return FOS_ERR_INVALID_ARG;
  fos::AmaxParams a{};
  a.x = static_cast<const uint16_t*>(x);
  a.rows = rows;
  a.cols = cols;
  a.ld = ld_x;
  a.hk0 = (uint32_t)hadamard_seed;
  a.hk1 = (uint32_t)(hadamard_seed >> 32);
  a.aligned32 = aligned(x, 32) && ld_x % 16 == 0;
  a.partials = static_cast<float*>(workspace);
  const int g = amax_tasks_grid(rows, cols, hadamard != 0, transpose != 0);
  cudaError_t e = fos::launch_amax(a, hadamard != 0, transpose != 0, g, stream);
  if (e != cudaSuccess) return FOS_ERR_CUDA;
  amax_final_kernel<<<1, 256, 0, stream>>>(a.partials, g, amax_out);
  return cuda_status(cudaGetLastError());
}

fos_status fos_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x, const fos_quant_options* opt,
                        uint8_t* codes, int64_t ld_codes, uint8_t* sf, float* tensor_scale, uint8_t* choice,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!valid_options(opt)) return FOS_ERR_INVALID_ARG;
  if (!valid_matrix(x, rows, cols, ld_x, opt, codes, ld_codes, sf, tensor_scale)) return FOS_ERR_INVALID_ARG;
  if (!opt->tensor_amax &&
      (!workspace || workspace_bytes < fos::kQuantWorkspaceBytes || !aligned(workspace, 4)))
    return FOS_ERR_INVALID_ARG;
  const bool tr = opt->transpose != 0, two_d = opt->block_2d != 0, rht = opt->hadamard != 0;
  const bool sr = opt->rounding == FOS_ROUND_STOCHASTIC;

  // 1D blocks along rows without a supplied amax: both passes in one launch
  // only on request (two launches measure faster)
  const bool fused = opt->one_launch && !tr && !two_d && !opt->tensor_amax;
  int n_partials = 0;
  if (!opt->tensor_amax && !fused) {
    fos::AmaxParams a{};
    a.x = static_cast<const uint16_t*>(x);
    a.rows = rows;
    a.cols = cols;
    a.ld = ld_x;
    a.hk0 = (uint32_t)opt->hadamard_seed;
    a.hk1 = (uint32_t)(opt->hadamard_seed >> 32);
    a.aligned32 = aligned(x, 32) && ld_x % 16 == 0;
    a.partials = static_cast<float*>(workspace);
    n_partials = amax_tasks_grid(rows, cols, rht, tr);
    if (fos::launch_amax(a, rht, tr, n_partials, stream) != cudaSuccess) return FOS_ERR_CUDA;
  }

  fos::QuantLaunch q = fos::quant_launch(x, rows, cols, ld_x, opt, codes, ld_codes, sf, tensor_scale, choice,
                               opt->tensor_amax ? opt->tensor_amax : static_cast<const float*>(workspace),
                               n_partials);
  if (fused) {
    q.p.ws_partials = static_cast<float*>(workspace);
    q.p.ws_barrier = reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) + fos::kBarrierOffset);
    if (fos::launch_quant_rows_fused(q.p, opt->scale_rule, rht, sr, q.tasks, stream) != cudaSuccess)
      return FOS_ERR_CUDA;
  } else {
    const int grid = fos::quant_grid(q.tasks, q.kind);
    // after this call's own amax launch, the quantize launch may overlap its
    // tail; after the caller's work (a supplied amax), it may not: that work
    // may still be writing x
    if (fos::launch_quant(q.p, opt->scale_rule, q.kind, rht, sr, grid, stream, n_partials > 0) != cudaSuccess)
      return FOS_ERR_CUDA;
  }
  if (fos::pad_scales(q.p, stream) != cudaSuccess) return FOS_ERR_CUDA;
  return FOS_OK;
}

fos_status fos_quantize_batch_workspace_size(int32_t n_jobs, size_t* bytes) {
  if (!bytes || n_jobs < 0) return FOS_ERR_INVALID_ARG;
  *bytes = (size_t)n_jobs * fos::kBarrierOffset;  // one slot of partial maxima per job
  return FOS_OK;
}

fos_status fos_quantize_batch(const fos_quant_job* jobs, int32_t n_jobs, const fos_quant_options* opt,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!valid_options(opt) || n_jobs < 0 || (n_jobs > 0 && !jobs)) return FOS_ERR_INVALID_ARG;
  if (opt->tensor_amax) return FOS_ERR_UNSUPPORTED;
  if (n_jobs == 0) return FOS_OK;
  if (!workspace || workspace_bytes < (size_t)n_jobs * fos::kBarrierOffset || !aligned(workspace, 4))
    return FOS_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_jobs; ++i) {
    const fos_quant_job& j = jobs[i];
    if (!valid_matrix(j.x, j.rows, j.cols, j.ld_x, opt, j.codes, j.ld_codes, j.sf, j.tensor_scale))
      return FOS_ERR_INVALID_ARG;
  }
  const bool tr = opt->transpose != 0, two_d = opt->block_2d != 0, rht = opt->hadamard != 0;
  const bool sr = opt->rounding == FOS_ROUND_STOCHASTIC;
  auto slot = [&](int32_t i) {
    return reinterpret_cast<float*>(static_cast<char*>(workspace) + (size_t)i * fos::kBarrierOffset);
  };
  auto amax_of = [&](const fos_quant_job& j, float* partials) {
    fos::AmaxParams a{};
    a.x = static_cast<const uint16_t*>(j.x);
    a.rows = j.rows;
    a.cols = j.cols;
    a.ld = j.ld_x;
    a.hk0 = (uint32_t)opt->hadamard_seed;
    a.hk1 = (uint32_t)(opt->hadamard_seed >> 32);
    a.aligned32 = aligned(j.x, 32) && j.ld_x % 16 == 0;
    a.partials = partials;
    return a;
  };
  // The scale pads first (bytes no quantize launch writes), so that the
  // quantize launches follow one another directly: each may then start while
  // its predecessor finishes (programmatic dependent launch).
  for (int32_t i = 0; i < n_jobs; ++i) {
    const fos_quant_job& j = jobs[i];
    const int64_t R = tr ? j.cols : j.rows, nb = (tr ? j.rows : j.cols) / 16;
    if (opt->sf_layout == FOS_SF_SWIZZLED_128x4 && (R % 128 != 0 || nb % 4 != 0)) {
      if (fos::launch_sf_pad(j.sf, sf_bytes_of(R, nb, opt->sf_layout), R, nb, stream) != cudaSuccess)
        return FOS_ERR_CUDA;
    }
  }

  if (tr || two_d) {
    // Transposed or 2D jobs: the amax passes of up to kAmaxBatchJobs jobs in
    // one launch, then one quantize launch per job, back to back.
    for (int32_t g0 = 0; g0 < n_jobs; g0 += fos::kAmaxBatchJobs) {
      fos::AmaxBatch b{};
      b.n_jobs = n_jobs - g0 < fos::kAmaxBatchJobs ? n_jobs - g0 : fos::kAmaxBatchJobs;
      int64_t total = 0;
      for (int32_t k = 0; k < b.n_jobs; ++k) {
        const fos_quant_job& j = jobs[g0 + k];
        b.job[k] = amax_of(j, slot(g0 + k));
        total += amax_tasks(j.rows, j.cols, rht, tr);
      }
      int grid = 0;
      if (fos::launch_amax_batch(b, rht, tr, total, &grid, stream) != cudaSuccess) return FOS_ERR_CUDA;
      // the quantize launches of this group (each job's grid partial maxima),
      // last job first: the amax launch read the jobs in order, so the last
      // one's input is the most likely to be still in L2; the next group's
      // amax launch follows them as a plain launch
      for (int32_t k = b.n_jobs - 1; k >= 0; --k) {
        const fos_quant_job& j = jobs[g0 + k];
        const fos::QuantLaunch q = fos::quant_launch(j.x, j.rows, j.cols, j.ld_x, opt, j.codes, j.ld_codes, j.sf,
                                           j.tensor_scale, j.choice, slot(g0 + k), grid);
        if (fos::launch_quant(q.p, opt->scale_rule, q.kind, rht, sr, fos::quant_grid(q.tasks, q.kind), stream,
                              true) != cudaSuccess)
          return FOS_ERR_CUDA;
      }
    }
    return FOS_OK;
  }

  // Blocks along rows: job 0's block maxima in an amax launch of their own,
  // then launch i quantizes job i while taking job i+1's.
  int n_part = amax_tasks_grid(jobs[0].rows, jobs[0].cols, rht, false);
  if (fos::launch_amax(amax_of(jobs[0], slot(0)), rht, false, n_part, stream) != cudaSuccess) return FOS_ERR_CUDA;
  for (int32_t i = 0; i < n_jobs; ++i) {
    const fos_quant_job& j = jobs[i];
    fos::QuantLaunch q = fos::quant_launch(j.x, j.rows, j.cols, j.ld_x, opt, j.codes, j.ld_codes, j.sf, j.tensor_scale,
                                 j.choice, slot(i), n_part);
    if (i + 1 < n_jobs) {
      const fos_quant_job& nx = jobs[i + 1];
      q.p.next_x = static_cast<const uint16_t*>(nx.x);
      q.p.next_rows = nx.rows;
      q.p.next_cols = nx.cols;
      q.p.next_ld = nx.ld_x;
      q.p.next_partials = slot(i + 1);
      const int g = fos::chained_grid();
      if (fos::launch_quant_rows_chained(q.p, opt->scale_rule, rht, sr, g, stream) != cudaSuccess)
        return FOS_ERR_CUDA;
      n_part = g;
    } else {
      if (fos::launch_quant(q.p, opt->scale_rule, 0, rht, sr, fos::quant_grid(q.tasks, 0), stream, true) !=
          cudaSuccess)
        return FOS_ERR_CUDA;
    }
  }
  return FOS_OK;
}

fos_status fos_dequantize(const fos_nvfp4_tensor* q, void* out, int32_t out_dtype, int64_t ld_out,
                          cudaStream_t stream) {
  if (!q || !out || !q->codes || !q->sf || !q->tensor_scale) return FOS_ERR_INVALID_ARG;
  if (q->rows < 0 || q->cols < 0 || q->cols % 16 != 0 || q->ld_codes < q->cols / 2 || q->ld_codes % 8 != 0)
    return FOS_ERR_INVALID_ARG;
  if (q->sf_layout != FOS_SF_SWIZZLED_128x4 && q->sf_layout != FOS_SF_ROWMAJOR) return FOS_ERR_INVALID_ARG;
  if (out_dtype != FOS_DTYPE_F32 && out_dtype != FOS_DTYPE_BF16) return FOS_ERR_INVALID_ARG;
  if (ld_out < q->cols || !aligned(out, 16) || !aligned(q->codes, 8)) return FOS_ERR_INVALID_ARG;
  if ((out_dtype == FOS_DTYPE_F32 && ld_out % 4 != 0) || (out_dtype == FOS_DTYPE_BF16 && ld_out % 8 != 0))
    return FOS_ERR_INVALID_ARG;
  fos::DequantParams p{};
  p.codes = q->codes;
  p.sf = q->sf;
  p.tensor_scale = q->tensor_scale;
  p.rows = q->rows;
  p.cols = q->cols;
  p.ld_codes = q->ld_codes;
  p.ld_out = ld_out;
  p.sf_layout = q->sf_layout;
  p.out = out;
  return cuda_status(fos::launch_dequant(p, out_dtype == FOS_DTYPE_BF16, stream));
}

fos_status fos_selftest_wait_limits(void* scratch, size_t scratch_bytes, uint64_t timeout_ns, int32_t* result,
                                    cudaStream_t stream) {
  constexpr size_t kNeed = 1 << 17;
  if (!scratch || scratch_bytes < kNeed || !aligned(scratch, 256) || !result || !aligned(result, 4))
    return FOS_ERR_INVALID_ARG;
  if (timeout_ns == 0 || timeout_ns > fos::kWaitTimeoutNs) return FOS_ERR_INVALID_ARG;
  if (cudaMemsetAsync(result, 0, 2 * sizeof(int32_t), stream) != cudaSuccess) return FOS_ERR_CUDA;
  // 1. the GEMM with a producer that never fills a stage
  constexpr size_t kGemmPart = 80 << 10;
  fos_status st = fos::gemm_stall_selftest(scratch, kGemmPart, timeout_ns, result, stream);
  if (st != FOS_OK) return st;
  // 2. the one-launch quantizer on a 16 x 64 zero matrix with a grid barrier
  //    that waits for one CTA more than the launch has
  char* b = static_cast<char*>(scratch) + kGemmPart;
  uint16_t* x = reinterpret_cast<uint16_t*>(b);             // 2 KB
  uint8_t* codes = reinterpret_cast<uint8_t*>(b + 4096);    // 512 B
  uint8_t* sf = reinterpret_cast<uint8_t*>(b + 8192);       // 512 B
  float* ts = reinterpret_cast<float*>(b + 12288);
  void* ws = b + 16384;                                     // kQuantWorkspaceBytes
  static_assert(kGemmPart + 16384 + fos::kQuantWorkspaceBytes <= kNeed, "self-test scratch layout");
  if (cudaMemsetAsync(b, 0, 16384, stream) != cudaSuccess) return FOS_ERR_CUDA;
  fos::QuantParams p{};
  p.x = x;
  p.rows = 16;
  p.cols = 64;
  p.ld = 64;
  p.R = 16;
  p.nb = 4;
  p.codes = codes;
  p.ld_codes = 32;
  p.sf = sf;
  p.sf_layout = FOS_SF_SWIZZLED_128x4;
  p.tensor_scale = ts;
  p.aligned32 = true;
  p.codes16 = true;
  p.ws_partials = static_cast<float*>(ws);
  p.ws_barrier = reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + fos::kBarrierOffset);
  p.barrier_extra = 1;
  p.timeout_ns = timeout_ns;
  if (fos::launch_quant_rows_fused(p, FOS_SCALE_4OVER6, false, false, 16, stream) != cudaSuccess) return FOS_ERR_CUDA;
  return cuda_status(fos::launch_nan_to_status(ts, result + 1, stream));
}

fos_status fos_e2m1_encode(const float* x, int64_t n, uint8_t* codes, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!x || !codes))) return FOS_ERR_INVALID_ARG;
  if (n == 0) return FOS_OK;
  return cuda_status(fos::launch_e2m1_encode(x, n, codes, stream));
}

fos_status fos_e4m3_encode(const float* x, int64_t n, uint8_t* out, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!x || !out))) return FOS_ERR_INVALID_ARG;
  if (n == 0) return FOS_OK;
  return cuda_status(fos::launch_e4m3_encode(x, n, out, stream));
}

fos_status fos_philox4x32_10(const uint32_t* counters, int64_t n, uint64_t key, uint32_t* out, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!counters || !out))) return FOS_ERR_INVALID_ARG;
  if (n == 0) return FOS_OK;
  return cuda_status(fos::launch_philox(counters, n, key, out, stream));
}

}  // extern "C"
