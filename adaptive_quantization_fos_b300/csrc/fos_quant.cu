// NVFP4 Four Over Six quantization kernels for sm_103a.
//
// Kernels (all HBM-streaming; no tensor cores -- the work is per-element
// arithmetic, not a contraction):
//   amax_rows    max|y| of X (RHT along rows optional) -> one partial per CTA
//   amax_cols    max|y| with the RHT running down columns (transposed input)
//   quant_rows   1D blocks along rows: a warp task is a 2048-value row
//                segment from the warp's bulk-copy ring; lane l owns blocks
//                l, l+32, l+64, l+96 (plain, one-launch and chained forms)
//   quant_cols   1D blocks down columns (transposed output): a warp task is
//                64 rows x 128 (RNE) or 64 (SR) columns from a bulk-copy
//                ring; a lane owns 4 or 2 adjacent columns
//   quant_2d     16x16 tiles: 16 lanes own the 16 source rows of a tile
//   sf_pad_zero  zero the padding bytes of the swizzled scale layout
//   dequant      x_hat = g * (sf * s_t)
// Each quantize kernel reduces the amax partials itself in its prologue, so
// the amax pass needs no atomics, no memset and no extra finalize launch.
#include <cuda_runtime.h>

#include <atomic>
#include <cfloat>
#include <cstdint>

#include "fos_device.cuh"
#include "fos_internal.h"

namespace fos {

// ------------------------------------------------------------------ amax

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// CTA-wide max; every thread returns the result.
__device__ __forceinline__ float block_max(float v, float* s_red) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float u = lane < (int)(blockDim.x >> 5) ? s_red[lane] : 0.0f;
    u = warp_max(u);
    if (lane == 0) s_red[32] = u;
  }
  __syncthreads();
  float r = s_red[32];
  __syncthreads();
  return r;
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of
// the stream (launched with programmatic stream serialization) be scheduled
// once every CTA of this grid has executed it or exited; wait blocks until
// the grids this one depends on have completed and their writes are visible.
// Both are no-ops for a grid launched without that attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Named barrier 1 over the CTA's first n threads.
__device__ __forceinline__ void bar_sync_first(int n) { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }

// Max of non-negative floats (or NaN) through their bit patterns: every
// non-negative float orders like its bits, and NaN (0x7FC00000) lies above
// them all, so a NaN partial -- a pass that gave up on a wait -- survives the
// reduction instead of being dropped as fmaxf would drop it.
__device__ __forceinline__ float max_nan(float a, float b) {
  return __uint_as_float(max(__float_as_uint(a), __float_as_uint(b)));
}

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// NaN-preserving max over the first NW warps of the CTA only (named barrier
// 1), for kernels whose other warps have gone their own way.
template <int NW>
__device__ __forceinline__ float group_max(float v, float* s_red) {
  v = warp_max_nan(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_red[warp] = v;
  bar_sync_first(32 * NW);
  if (warp == 0) {
    float u = lane < NW ? s_red[lane] : 0.0f;
    u = warp_max_nan(u);
    if (lane == 0) s_red[32] = u;
  }
  bar_sync_first(32 * NW);
  const float r = s_red[32];
  bar_sync_first(32 * NW);
  return r;
}

__device__ __forceinline__ void load_block16(const uint16_t* p, bool aligned32, uint32_t (&w)[8]) {
  if (aligned32)
    ldg256(p, w);
  else
    ldg128x2(p, w);
}

// max|y| of 16 bf16 values held as 8 words (no transform): integer max of the
// magnitude bit patterns, which orders non-negative bf16 like their values.
__device__ __forceinline__ float absmax16_bits(const uint32_t (&w)[8]) {
  uint32_t m = w[0] & 0x7FFF7FFFu;
#pragma unroll
  for (int k = 1; k < 8; ++k) m = max_u16x2(m, w[k] & 0x7FFF7FFFu);
  return fmaxf(bf16lo(m), bf16hi(m));
}

// words -> 16 floats, flipping signs with the RHT sign mask first (exact).
__device__ __forceinline__ void unpack16(const uint32_t (&w)[8], uint32_t mask, float (&y)[16]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint32_t s = (((mask >> (2 * k)) & 1u) << 15) | (((mask >> (2 * k + 1)) & 1u) << 31);
    uint32_t v = w[k] ^ s;
    y[2 * k] = bf16lo(v);
    y[2 * k + 1] = bf16hi(v);
  }
}

// RHT butterflies (stride 1, 2, 4, 8) and the 1/4 scaling; signs already applied.
__device__ __forceinline__ void hadamard16(float (&v)[16]) { rht16(v, 0u); }

// The amax passes take the block maxima of the transform without its 1/4:
// rounding is monotone, so max_j |fl(w_j / 4)| = fl(max_j |w_j| / 4), and the
// scaling is applied once to a thread's running maximum (unscaled_to_amax).
__device__ __forceinline__ float unscaled_to_amax(float m) { return __fmul_rn(m, 0.25f); }

// max |y_j| of 16 floats with the three-input maximum of magnitudes
// (sm_100+): 7 instructions instead of 15.  Inputs are finite.
__device__ __forceinline__ float max3abs(float a, float b, float c) {
  float d;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float absmax16(const float (&y)[16]) {
  const float m0 = max3abs(y[0], y[1], y[2]), m1 = max3abs(y[3], y[4], y[5]), m2 = max3abs(y[6], y[7], y[8]);
  const float m3 = max3abs(y[9], y[10], y[11]), m4 = max3abs(y[12], y[13], y[14]);
  return fmaxf(max3abs(m0, m1, m2), max3abs(m3, m4, y[15]));
}

// A warp task is a row segment of up to kAmaxRowBlocks blocks (4 KB): each
// lane has its blocks' four 32-byte loads in flight before it reduces them.
// The thread's maximum over warp tasks gw, gw + nwarps, ... of p (with RHT:
// of the transform along the rows, its 1/4 applied).
template <bool RHT>
__device__ __forceinline__ float amax_rows_share(const AmaxParams& p, int64_t gw, int64_t nwarps) {
  const int lane = threadIdx.x & 31;
  const uint32_t rht_mask = RHT ? rht_sign_mask(p.hk0, p.hk1) : 0u;
  const int64_t nb = p.cols >> 4;
  const int64_t wpr = (nb + kAmaxRowBlocks - 1) / kAmaxRowBlocks;
  const int64_t n_tasks = p.rows * wpr;
  float m = 0.0f;
  for (int64_t t = gw; t < n_tasks; t += nwarps) {
    const int64_t r = t / wpr, c0 = (t - r * wpr) * kAmaxRowBlocks;
    const int nblk = nb - c0 < kAmaxRowBlocks ? (int)(nb - c0) : kAmaxRowBlocks;
    const uint16_t* src = p.x + r * p.ld + (c0 + lane) * 16;
    uint32_t w[kAmaxRowBlocks / 32][8];
#pragma unroll
    for (int j = 0; j < kAmaxRowBlocks / 32; ++j)
      if (lane + 32 * j < nblk) load_block16(src + 512 * j, p.aligned32, w[j]);
#pragma unroll
    for (int j = 0; j < kAmaxRowBlocks / 32; ++j) {
      if (lane + 32 * j >= nblk) break;
      if (!RHT) {
        m = fmaxf(m, absmax16_bits(w[j]));
      } else {
        float y[16];
        unpack16(w[j], rht_mask, y);
        butterflies16(y);  // 1/4 applied to the maximum below
        m = fmaxf(m, absmax16(y));
      }
    }
  }
  return RHT ? unscaled_to_amax(m) : m;
}

template <bool RHT>
__global__ void __launch_bounds__(256) amax_rows_kernel(AmaxParams p) {
  __shared__ float s_red[33];
  pdl_launch_dependents();  // the next launch may start its own reads meanwhile
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  float m = amax_rows_share<RHT>(p, gw, ((int64_t)gridDim.x * blockDim.x) >> 5);
  m = block_max(m, s_red);
  if (threadIdx.x == 0) p.partials[blockIdx.x] = m;
}

// The thread's maximum over column warp tasks gw, gw + nwarps, ... of p (the
// transform down the columns, its 1/4 applied); with PLAIN, *plain gets the
// maximum of the untransformed values.
template <bool PLAIN>
__device__ __forceinline__ float amax_cols_share(const AmaxParams& p, int64_t gw, int64_t nwarps, float* plain) {
  constexpr int W = kAmaxColCPL / 2;  // words per row and lane
  const int lane = threadIdx.x & 31;
  const uint32_t rht_mask = rht_sign_mask(p.hk0, p.hk1);
  const int64_t ngroups = (p.cols + kAmaxColTask - 1) / kAmaxColTask;
  const int64_t n_tasks = (p.rows >> 4) * ngroups;
  float m = 0.0f, mp = 0.0f;  // mp: PLAIN's maximum
  for (int64_t t = gw; t < n_tasks; t += nwarps) {
    int64_t rb = t / ngroups, c0 = (t - rb * ngroups) * kAmaxColTask + kAmaxColCPL * lane;
    if (c0 >= p.cols) continue;  // cols % 16 == 0: the lane's columns all exist
    uint32_t d[16][W];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint16_t* src = p.x + (rb * 16 + i) * p.ld + c0;
      if constexpr (W == 4) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
        d[i][0] = v.x; d[i][W - 3] = v.y; d[i][W - 2] = v.z; d[i][W - 1] = v.w;
      } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
        d[i][0] = v.x; d[i][W - 1] = v.y;
      }
    }
#pragma unroll
    for (int k = 0; k < kAmaxColCPL; ++k) {
      float y[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t wv = d[i][k >> 1];
        const uint32_t s = ((rht_mask >> i) & 1u) << 31;
        y[i] = __uint_as_float(((k & 1) ? (wv & 0xFFFF0000u) : (wv << 16)) ^ s);
      }
      if (PLAIN) mp = fmaxf(mp, absmax16(y));
      butterflies16(y);  // 1/4 applied to the maximum below
      m = fmaxf(m, absmax16(y));
    }
  }
  if (PLAIN) *plain = mp;
  return unscaled_to_amax(m);
}

// RHT down columns: a lane owns kAmaxColCPL adjacent columns x 16 rows, so a
// warp reads 64 * kAmaxColCPL contiguous bytes of each of the 16 rows.  With
// PLAIN, the same pass also takes max |x| of the untransformed values (the
// column's magnitudes before the butterflies: the sign flips do not change
// them) into p.partials_plain.  Two CTAs per SM at 128 registers (a few bytes
// spilled) measured faster than one at 142, and than 4 columns per lane (also
// with the next task's loads issued before the current task's reduction).
template <bool PLAIN>
__global__ void __launch_bounds__(256, 2) amax_cols_kernel(AmaxParams p) {
  __shared__ float s_red[33];
  pdl_launch_dependents();  // the quantize launch may start its own reads meanwhile
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  float mp = 0.0f;
  float m = amax_cols_share<PLAIN>(p, gw, ((int64_t)gridDim.x * blockDim.x) >> 5, &mp);
  m = block_max(m, s_red);
  if (threadIdx.x == 0) p.partials[blockIdx.x] = m;
  if (PLAIN) {
    mp = block_max(mp, s_red);
    if (threadIdx.x == 0) p.partials_plain[blockIdx.x] = mp;
  }
}

// The amax passes of several jobs in one launch (a batch of transposed or 2D
// jobs): every CTA takes its share of each job in turn and leaves one partial
// maximum per job, at the job's partials[blockIdx.x].  MODE 0: rows, 1: rows
// with the RHT, 2: the RHT down the columns.
template <int MODE>
__global__ void __launch_bounds__(256, MODE == 2 ? 2 : 0) amax_batch_kernel(const __grid_constant__ AmaxBatch b) {
  __shared__ float s_red[33];
  pdl_launch_dependents();  // the first quantize launch may start its own reads meanwhile
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int j = 0; j < b.n_jobs; ++j) {
    const AmaxParams& p = b.job[j];
    float m;
    if constexpr (MODE == 2)
      m = amax_cols_share<false>(p, gw, nwarps, nullptr);
    else
      m = amax_rows_share<MODE == 1>(p, gw, nwarps);
    m = block_max(m, s_red);
    if (threadIdx.x == 0) p.partials[blockIdx.x] = m;
  }
}

// ------------------------------------------------------- quantize prologue

__device__ __forceinline__ TensorConsts quant_prologue(const QuantParams& p, float* s_red) {
  float amax;
  if (p.n_partials == 0) {
    amax = __ldcg(p.amax_src);
  } else {
    float m = 0.0f;
    for (int i = threadIdx.x; i < p.n_partials; i += blockDim.x) m = fmaxf(m, __ldcg(p.amax_src + i));
    amax = block_max(m, s_red);
  }
  TensorConsts tc = tensor_consts(amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.tensor_scale = tc.s_t;
  return tc;
}

// The stochastic-rounding draws n = w >> 8 (as floats, exact) of the 16
// consecutive source elements starting at index i0.
template <bool SR>
__device__ __forceinline__ void sr_draws16(uint64_t i0, const QuantParams& p, float (&n)[16]) {
  if constexpr (SR) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const U4 u = sr_words4(i0 + 4 * g, p.sr_k0, p.sr_k1);
      n[4 * g] = sr_draw(u.x);
      n[4 * g + 1] = sr_draw(u.y);
      n[4 * g + 2] = sr_draw(u.z);
      n[4 * g + 3] = sr_draw(u.w);
    }
  }
}

// ------------------------------------------------------------ quant_rows
// Warp task = one row and up to 128 consecutive blocks (2048 values, 4 KB of
// bf16).  Each warp streams its tasks through a private ring of shared-memory
// slots filled by bulk copies (issued kRowSlots tasks ahead by lane 0), so the
// HBM reads stay in flight without holding registers.  Lane l owns blocks l,
// l+32, l+64, l+96 of a task: its code stores and the warp's reads of the slot
// are contiguous across lanes.  The two candidates' reciprocal and squared
// effective scale come from a per-CTA table indexed by the E4M3 byte.
constexpr int kRowWarps = 8;
constexpr int kRowSlots = 2;
constexpr int kRowSlotBytes = 128 * 32;
constexpr int kRowSmemBytes = kRowWarps * kRowSlots * kRowSlotBytes;
// chained mode: 2 more warps per CTA stream the next job's input for its
// amax through rings of 4 slots each
constexpr int kAmaxWarps = 2;
constexpr int kAmaxSlots = 4;
constexpr int kChainSmemBytes = kRowSmemBytes + kAmaxWarps * kAmaxSlots * kRowSlotBytes;

// The row kernel's prologue, run by its kRowWarps quantize warps alone: the
// tensor amax from the supplied value or from the partial maxima a previous
// launch wrote (read through L2: that launch may have been running when this
// one started), then the tensor constants.
__device__ __forceinline__ TensorConsts quant_prologue_rows(const QuantParams& p, float* s_red) {
  float amax;
  if (p.n_partials == 0) {
    amax = __ldcg(p.amax_src);
  } else {
    float m = 0.0f;
    for (int i = threadIdx.x; i < p.n_partials; i += 32 * kRowWarps) m = max_nan(m, __ldcg(p.amax_src + i));
    amax = group_max<kRowWarps>(m, s_red);  // a NaN partial (a give-up) makes s_t NaN
  }
  TensorConsts tc = tensor_consts(amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.tensor_scale = tc.s_t;
  return tc;
}

template <int RULE, bool SR>
__device__ __forceinline__ void quant_block_tab(const uint64_t (&yp)[8], float ab, const TensorConsts& tc,
                                                const float2* tab, const float (&n_sr)[16], uint32_t& lo,
                                                uint32_t& hi, uint32_t& sf, bool& four) {
  const uint32_t pair = candidate_scales(ab, tc);
  const uint32_t sf6 = pair & 0xFFu, sf4 = pair >> 8;
  F2 ay[8], sg[8];
  if (SR) sr_split16(yp, ay, sg);
  uint32_t lo6 = 0, hi6 = 0, lo4 = 0, hi4 = 0;
  float E6 = 0.0f, E4 = 0.0f;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (c == 0 && RULE == FOS_SCALE_4) continue;
    if (c == 1 && RULE == FOS_SCALE_6) continue;
    const float2 t = tab[c == 0 ? sf6 : sf4];
    uint32_t l, h;
    float S;
    if (SR) {
      S = cand_sr16(ay, sg, t.x, n_sr, l, h);
    } else {
      const uint64_t inv2 = pack_f2(t.x, t.x);
      uint64_t acc = 0ull;
      const uint64_t a[4] = {yp[0], yp[1], yp[2], yp[3]}, b[4] = {yp[4], yp[5], yp[6], yp[7]};
      l = cand_rne8(a, inv2, acc);
      h = cand_rne8(b, inv2, acc);
      const F2 e = unpack_f2(acc);
      S = __fadd_rn(e.x, e.y);
    }
    if (c == 0) {
      lo6 = l; hi6 = h; E6 = __fmul_rn(S, t.y);
    } else {
      lo4 = l; hi4 = h; E4 = __fmul_rn(S, t.y);
    }
  }
  if (sf6 == 0u || sf4 == 0u) {
    // a zero scale flushes the block to zero codes: its error is sum y^2
    float z[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      F2 v = unpack_f2(yp[k]);
      z[2 * k] = v.x;
      z[2 * k + 1] = v.y;
    }
    const float zz = sumsq16(z);
    if (sf6 == 0u) E6 = zz;
    if (sf4 == 0u) E4 = zz;
  }
  four = (RULE == FOS_SCALE_4) || (RULE == FOS_SCALE_4OVER6 && E4 < E6);
  lo = four ? lo4 : lo6;
  hi = four ? hi4 : hi6;
  sf = four ? sf4 : sf6;
}

// Block maxima of the next job of a batch, by the kAmaxWarps extra warps of a
// chained launch: tasks of 2048 values stream through each warp's ring of
// bulk-copy slots; the CTA's maximum (as bits: non-negative floats order like
// their bit patterns) goes to p.next_partials[blockIdx.x] once both warps are
// done.  A copy that outlasts the time limit makes the partial NaN.
template <bool RHT>
__device__ __forceinline__ void next_job_amax(const QuantParams& p, uint8_t* ring, uint64_t* bars, int aw, int lane,
                                              uint32_t rht_mask, unsigned int* s_max, unsigned int* s_done) {
  const int64_t nb = p.next_cols >> 4;
  const int64_t wpr = (nb + 127) >> 7;
  const int64_t nwarps = (int64_t)gridDim.x * kAmaxWarps;
  const int64_t gw = (int64_t)blockIdx.x * kAmaxWarps + aw;
  const int64_t R = nb > 0 ? p.next_rows : 0;
  const int64_t dr = nwarps / (wpr > 0 ? wpr : 1), dch = nwarps - dr * (wpr > 0 ? wpr : 1);
  uint8_t* slots = ring + aw * (kAmaxSlots * kRowSlotBytes);
  const uint32_t bar0 = smem_addr(&bars[aw * kAmaxSlots]);
  const uint64_t keep = l2_policy_evict_last();  // the job's own launch reads it next
  float m = 0.0f;
  if (wpr > 0) {
    int64_t pr = gw / wpr, pch = gw - pr * wpr;
    auto issue_next = [&](int slot) -> bool {
      if (pr >= R) return false;
      const int64_t c0 = pch * 128;
      const int64_t nblk = nb - c0 < 128 ? nb - c0 : 128;
      bulk_g2s_hint(smem_addr(slots + slot * kRowSlotBytes), p.next_x + pr * p.next_ld + c0 * 16,
                    (uint32_t)(nblk * 32), bar0 + 8u * slot, keep);
      pr += dr;
      pch += dch;
      if (pch >= wpr) {
        pch -= wpr;
        ++pr;
      }
      return true;
    };
    int issued = 0, consumed = 0;
    if (lane == 0)
      for (int k = 0; k < kAmaxSlots; ++k) issued += issue_next(k) ? 1 : 0;
    int slot = 0;
    uint32_t ph = 0;
    bool failed = false;
    int64_t r = gw / wpr, ch = gw - r * wpr;
    for (; r < R; r += dr, ch += dch) {
      if (ch >= wpr) {
        ch -= wpr;
        if (++r >= R) break;
      }
      const int64_t c0 = ch * 128;
      const int nblk = nb - c0 < 128 ? (int)(nb - c0) : 128;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_for(bar0 + 8u * slot, ph, p.timeout_ns))) {
        failed = true;
        break;
      }
      uint32_t wv[4][8];
      const uint8_t* src = slots + slot * kRowSlotBytes + lane * 32;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (lane + 32 * j < nblk) {
          const uint4 a = *reinterpret_cast<const uint4*>(src + 1024 * j);
          const uint4 b = *reinterpret_cast<const uint4*>(src + 1024 * j + 16);
          wv[j][0] = a.x; wv[j][1] = a.y; wv[j][2] = a.z; wv[j][3] = a.w;
          wv[j][4] = b.x; wv[j][5] = b.y; wv[j][6] = b.z; wv[j][7] = b.w;
        }
      }
      __syncwarp();
      ++consumed;
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issued += issue_next(slot) ? 1 : 0;
      }
      if (++slot == kAmaxSlots) {
        slot = 0;
        ph ^= 1u;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (lane + 32 * j >= nblk) break;
        if (RHT) {
          float y[16];
          unpack16(wv[j], rht_mask, y);
          butterflies16(y);  // 1/4 applied to the maximum below
          m = fmaxf(m, absmax16(y));
        } else {
          m = fmaxf(m, absmax16_bf16(wv[j]));
        }
      }
    }
    if (RHT) m = unscaled_to_amax(m);
    if (failed) m = __int_as_float(0x7FC00000);
    if (lane == 0) {
      for (; consumed < issued; ++consumed) {
        mbar_wait_for(bar0 + 8u * slot, ph, p.timeout_ns);
        if (++slot == kAmaxSlots) {
          slot = 0;
          ph ^= 1u;
        }
      }
    }
  }
  m = warp_max_nan(m);
  if (lane == 0) {
    atomicMax(s_max, __float_as_uint(m));
    __threadfence_block();
    if (atomicAdd(s_done, 1u) == kAmaxWarps - 1) p.next_partials[blockIdx.x] = __uint_as_float(atomicMax(s_max, 0u));
  }
}

// MODE kRowsPlain: the tensor amax is supplied, or reduced from partials a
// previous launch wrote.
// MODE kRowsFused: the tensor amax is computed in the same launch.  Pass 1
// reads every task once for its block maxima (keeping the lines in L2), one
// partial per CTA goes to the workspace, a grid barrier (all CTAs resident:
// cooperative launch) publishes them, and pass 2 quantizes, re-reading the
// input mostly from L2 when the matrix fits there.
// MODE kRowsChained: as kRowsPlain, and 2 extra warps per CTA take the block
// maxima of the NEXT job of a batch meanwhile (memory-bound work beside the
// issue-bound quantization), leaving one partial per CTA for that job's launch.
constexpr int kRowsPlain = 0, kRowsFused = 1, kRowsChained = 2;

// End of a one-launch (kRowsFused) CTA, by one thread: a CTA that gave up on a
// wait raises the flag word; the last CTA to finish writes the tensor scale,
// or NaN when any CTA gave up.  Raising the flag comes before the finish count
// (fenced), so the last CTA sees every flag however late a wait ran out.
__device__ __forceinline__ void fused_finish(const QuantParams& p, bool ok, float s_t) {
  unsigned int* const give_up = p.ws_barrier + 1;
  unsigned int* const finished = p.ws_barrier + 2;
  if (!ok) atomicOr(give_up, 1u);
  __threadfence();
  if (atomicAdd(finished, 1u) == gridDim.x - 1) {
    __threadfence();
    const bool any_gave_up = atomicOr(give_up, 0u) != 0u;
    *p.tensor_scale = any_gave_up ? __int_as_float(0x7FC00000) : s_t;  // NaN: the result is not valid
  }
}

template <int RULE, bool RHT, bool SR, int MODE>
__global__ void __launch_bounds__(MODE == kRowsChained ? 320 : 256, MODE == kRowsChained ? 2 : (SR ? 2 : 3))
    quant_rows_kernel(QuantParams p) {
  constexpr bool FUSED = MODE == kRowsFused;
  extern __shared__ __align__(128) uint8_t q_smem[];
  __shared__ float s_red[33];
  __shared__ float2 s_tab[128];
  __shared__ uint64_t s_bar[kRowWarps * kRowSlots + kAmaxWarps * kAmaxSlots];
  __shared__ int s_ok;
  __shared__ unsigned int s_next_max, s_next_done;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < kRowWarps * kRowSlots + kAmaxWarps * kAmaxSlots) mbar_init(smem_addr(&s_bar[threadIdx.x]), 1);
  if (threadIdx.x == 0) {
    s_next_max = 0u;
    s_next_done = 0u;
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if constexpr (!FUSED) __syncthreads();  // the barriers are initialised before the roles split
  pdl_launch_dependents();
  const uint32_t rht_mask = RHT ? rht_sign_mask(p.hk0, p.hk1) : 0u;
  const int64_t nb = p.nb;
  const int64_t wpr = (nb + 127) >> 7;  // warp tasks per row
  const int64_t nwarps = (int64_t)gridDim.x * kRowWarps;
  const int64_t gw = (int64_t)blockIdx.x * kRowWarps + warp;
  // tasks t = gw, gw + nwarps, ... as (row, chunk) pairs advanced without division
  const int64_t dr = nwarps / wpr, dch = nwarps - dr * wpr;
  TensorConsts tc;
  if constexpr (FUSED) {
    const uint64_t keep = l2_policy_evict_last();
    float m = 0.0f;
    int64_t r = gw / wpr, ch = gw - r * wpr;
    for (; r < p.R; r += dr, ch += dch) {
      if (ch >= wpr) {
        ch -= wpr;
        if (++r >= p.R) break;
      }
      const int64_t c0 = ch * 128;
      const int nblk = nb - c0 < 128 ? (int)(nb - c0) : 128;
      const uint16_t* src = p.x + r * p.ld + (c0 + lane) * 16;
      uint32_t wv[4][8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (lane + 32 * j < nblk) {
          if (p.aligned32)
            ldg256_hint(src + 512 * j, wv[j], keep);
          else
            ldg128x2_hint(src + 512 * j, wv[j], keep);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (lane + 32 * j >= nblk) break;
        if (RHT) {
          float y[16];
          unpack16(wv[j], rht_mask, y);
          butterflies16(y);  // 1/4 applied to the maximum below
          m = fmaxf(m, absmax16(y));
        } else {
          m = fmaxf(m, absmax16_bf16(wv[j]));
        }
      }
    }
    if (RHT) m = unscaled_to_amax(m);
    m = block_max(m, s_red);
    if (threadIdx.x == 0) {
      p.ws_partials[blockIdx.x] = m;
      s_ok = grid_barrier(p.ws_barrier, gridDim.x + p.barrier_extra, p.timeout_ns) ? 1 : 0;
    }
    __syncthreads();
    if (!s_ok) {
      if (threadIdx.x == 0) fused_finish(p, false, 0.0f);
      return;
    }
    float mm = 0.0f;
    for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x) mm = fmaxf(mm, __ldcg(p.ws_partials + i));
    tc = tensor_consts(block_max(mm, s_red));  // the same in every CTA; the last to finish stores s_t
  }
  if (MODE == kRowsChained && warp >= kRowWarps) {
    // the next job's block maxima need nothing from earlier launches
    next_job_amax<RHT>(p, q_smem + kRowSmemBytes, &s_bar[kRowWarps * kRowSlots], warp - kRowWarps, lane, rht_mask,
                       &s_next_max, &s_next_done);
    return;
  }
  const uint64_t stream_once = l2_policy_evict_first();
  const bool swz = p.sf_layout == FOS_SF_SWIZZLED_128x4;
  const int64_t sf_step = swz ? 4096 : 32;
  const bool want_choice = p.choice != nullptr;
  const int64_t n_ct = (nb + 3) >> 2;
  uint8_t* slots = q_smem + warp * (kRowSlots * kRowSlotBytes);
  const uint32_t bar0 = smem_addr(&s_bar[warp * kRowSlots]);

  // producer cursor (lane 0): the next task to fetch.  The quantize pass runs
  // the rows from last to first: an amax pass over the same matrix (the one
  // of this launch, or the previous launch's amax warps) read them first to
  // last, so the rows it read last -- the ones most likely still in L2 --
  // are quantized first.
  int64_t pr = gw / wpr, pch = gw - pr * wpr;
  auto issue_next = [&](int slot) -> bool {
    if (pr >= p.R) return false;
    const int64_t c0 = pch * 128;
    const int64_t nblk = nb - c0 < 128 ? nb - c0 : 128;
    bulk_g2s_hint(smem_addr(slots + slot * kRowSlotBytes), p.x + (p.R - 1 - pr) * p.ld + c0 * 16,
                  (uint32_t)(nblk * 32), bar0 + 8u * slot, stream_once);
    pr += dr;
    pch += dch;
    if (pch >= wpr) {
      pch -= wpr;
      ++pr;
    }
    return true;
  };
  int issued = 0, consumed = 0;
  if (lane == 0)
    for (int k = 0; k < kRowSlots; ++k) issued += issue_next(k) ? 1 : 0;
  if constexpr (FUSED) {
    build_scale_table(tc.s_t, s_tab);
    __syncthreads();
  } else {
    // The input is read-only, so its first copies are in flight already; the
    // partial maxima come from the launch before this one, which may still be
    // running.  Everything from here on waits for it.
    pdl_wait();
    tc = quant_prologue_rows(p, s_red);
    build_scale_table(tc.s_t, s_tab);
    bar_sync_first(32 * kRowWarps);
  }

  int slot = 0;
  uint32_t ph = 0;
  bool failed = false;
  int64_t ri = gw / wpr, ch = gw - ri * wpr;
  for (; ri < p.R; ri += dr, ch += dch) {
    if (ch >= wpr) {
      ch -= wpr;
      if (++ri >= p.R) break;
    }
    const int64_t r = p.R - 1 - ri;  // rows run last to first (see the note at the ring)
    const int64_t c0 = ch * 128;
    const int nblk = nb - c0 < 128 ? (int)(nb - c0) : 128;
    // every lane observes the copy's completion itself; the verdict is made
    // warp-uniform so the warp stays converged
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_for(bar0 + 8u * slot, ph, p.timeout_ns))) {
      failed = true;
      break;
    }
    const uint8_t* src = slots + slot * kRowSlotBytes + lane * 32;
    const int64_t b_lane = c0 + lane;
    uint8_t* code_dst = p.codes + r * p.ld_codes + b_lane * 8;
    uint8_t* sf_dst = p.sf + (swz ? ((((r >> 7) * n_ct + (b_lane >> 2)) << 9) + ((r & 31) << 4) +
                                     (((r >> 5) & 3) << 2) + (b_lane & 3))
                                  : r * nb + b_lane);
    uint8_t* choice_dst = want_choice ? p.choice + r * nb + b_lane : nullptr;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (lane + 32 * j >= nblk) break;
      uint32_t wv[8];
      {
        const uint4 a = *reinterpret_cast<const uint4*>(src + 1024 * j);
        const uint4 b = *reinterpret_cast<const uint4*>(src + 1024 * j + 16);
        wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
        wv[4] = b.x; wv[5] = b.y; wv[6] = b.z; wv[7] = b.w;
      }
      uint64_t yp[8];
      float ab;
      if (RHT) {
        float y[16];
        unpack16(wv, rht_mask, y);
        hadamard16(y);
        ab = absmax16(y);
#pragma unroll
        for (int k = 0; k < 8; ++k) yp[k] = pack_f2(y[2 * k], y[2 * k + 1]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) yp[k] = bf16x2_to_f32x2(wv[k]);
        ab = absmax16_bf16(wv);
      }
      float n_sr[16];
      sr_draws16<SR>((uint64_t)r * (uint64_t)p.cols + (uint64_t)(b_lane + 32 * j) * 16, p, n_sr);
      uint32_t lo, hi, sf;
      bool four;
      quant_block_tab<RULE, SR>(yp, ab, tc, s_tab, n_sr, lo, hi, sf, four);
      *reinterpret_cast<uint2*>(code_dst + 256 * j) = make_uint2(lo, hi);
      // 32 blocks further along a row: 8 swizzled tiles (4096 bytes) further
      sf_dst[sf_step * j] = (uint8_t)sf;
      if (want_choice) choice_dst[32 * j] = four ? 1 : 0;
    }
    __syncwarp();
    ++consumed;
    if (lane == 0) {
      // the warp's reads of this slot are done: refill it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issued += issue_next(slot) ? 1 : 0;
    }
    if (++slot == kRowSlots) {
      slot = 0;
      ph ^= 1u;
    }
  }
  if (lane == 0) {
    if (failed) {
      if (FUSED)
        s_ok = 0;  // reported by fused_finish below
      else
        *p.tensor_scale = __int_as_float(0x7FC00000);  // NaN: the result is not valid
    }
    // let copies still in flight land before the CTA exits (bounded)
    for (; consumed < issued; ++consumed) {
      mbar_wait_for(bar0 + 8u * slot, ph, p.timeout_ns);
      if (++slot == kRowSlots) {
        slot = 0;
        ph ^= 1u;
      }
    }
  }
  if constexpr (FUSED) {
    __syncthreads();
    if (threadIdx.x == 0) fused_finish(p, s_ok != 0, tc.s_t);
  }
}

// ------------------------------------------------------------ quant_cols
// Transposed output: a lane owns source columns c0..c0+3 (output rows) and
// the 16 source rows of output block rb.
// Transposed input (blocks run down X's columns; output row c of the result
// is source column c).  A lane owns CPL adjacent source columns (4 with RNE,
// 2 with stochastic rounding, whose words take registers); warp task = 64
// source rows (4 block-rows) x 32*CPL source columns.  Each block-row of the
// task (16 rows x 64*CPL bytes) is one slot of the warp's ring of bulk copies,
// one copy per row issued by lanes 0..15 (the slot's barrier counts their 16
// arrivals); a lane reads each row's 2*CPL bytes from shared memory.
// Stochastic rounding: the Philox call for (row, 4-column group j) serves
// lanes 2j and 2j+1; lane 2j computes rows 0-7 of the block-row and lane
// 2j+1 rows 8-15, and each pair swaps the two words the other needs.  A
// task's 4 block-rows give each output row 32 contiguous code bytes: a lane
// parks each block's 8 bytes in its own entries of the warp's output buffer
// (entry (k, lane) holds output row CPL * lane + k; 40-byte entries, so the
// 8-byte writes of a warp and its 32-byte reads fall on distinct banks) and
// keeps the scale bytes in a word, then stores each output row's 32 code
// bytes and 4 scale bytes at once after the task's last block-row: whole
// sectors rather than four 8-byte pieces each.
constexpr int kColWarps = 8;
constexpr int kColWarpSmem = 8192;   // ring bytes per warp: 4 slots x 2 KB (CPL 2) or 2 x 4 KB (CPL 4)
constexpr int kColOutPitch = 40;     // bytes per output-buffer entry (32 used)
constexpr int kColWarpOut = 4 * 32 * kColOutPitch;  // up to CPL = 4 entries per lane
constexpr int kColSmemBytes = kColWarps * (kColWarpSmem + kColWarpOut);

// 32 bytes to global memory; p 32-byte aligned.
__device__ __forceinline__ void st_v8(void* p, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w),
               "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

template <int RULE, bool RHT, bool SR>
__global__ void __launch_bounds__(256, 2) quant_cols_kernel(QuantParams p) {
  constexpr int CPL = SR ? 2 : 4;                 // source columns per lane
  constexpr int kCW = 32 * CPL;                   // source columns per task
  constexpr int kColSlotBytes = 16 * 2 * kCW;     // one block-row of the task
  constexpr int kColSlots = kColWarpSmem / kColSlotBytes;
  extern __shared__ __align__(128) uint8_t c_smem[];
  __shared__ float s_red[33];
  __shared__ float2 s_tab[128];
  __shared__ uint64_t s_bar[kColWarps * 4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < kColWarps * kColSlots) mbar_init(smem_addr(&s_bar[threadIdx.x]), 16);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();  // the ring barriers are initialised before any copy
  pdl_launch_dependents();  // a dependent launch (the next quantize launch, a GEMM) may start its own reads
  const uint32_t rht_mask = RHT ? rht_sign_mask(p.hk0, p.hk1) : 0u;
  const int64_t nbr = p.rows >> 4;            // block-rows of the source = blocks per output row
  const int64_t ngr = (nbr + 3) >> 2;          // task rows (4 block-rows each)
  const int64_t nch = (p.cols + kCW - 1) / kCW;  // task columns (kCW source columns each)
  const int64_t n_tasks = ngr * nch;
  const int64_t nwarps = (int64_t)gridDim.x * kColWarps;
  const int64_t gw = (int64_t)blockIdx.x * kColWarps + warp;
  const uint64_t stream_once = l2_policy_evict_first();
  uint8_t* slots = c_smem + warp * (kColSlots * kColSlotBytes);
  uint8_t* obuf = c_smem + kColWarps * kColWarpSmem + warp * kColWarpOut + lane * kColOutPitch;
  const uint32_t bar0 = smem_addr(&s_bar[warp * kColSlots]);

  // producer cursor (all lanes): the next (task, block-row) to fetch
  int64_t pt = gw;
  int psub = 0;
  auto issue_next = [&](int slot) -> bool {
    if (pt >= n_tasks) return false;
    const int64_t g = pt / nch, ch = pt - g * nch;
    const int64_t rb = 4 * g + psub;
    const int64_t c0 = ch * kCW;
    const uint32_t bytes = (uint32_t)((p.cols - c0 < kCW ? p.cols - c0 : kCW) * 2);
    if (lane < 16)
      bulk_g2s_hint(smem_addr(slots + slot * kColSlotBytes + lane * (2 * kCW)), p.x + (rb * 16 + lane) * p.ld + c0,
                    bytes, bar0 + 8u * slot, stream_once);
    if (++psub == 4 || 4 * g + psub >= nbr) {
      psub = 0;
      pt += nwarps;
    }
    return true;
  };
  int issued = 0, consumed = 0;
  for (int k = 0; k < kColSlots; ++k) issued += issue_next(k) ? 1 : 0;
  // The input is read-only, so its first copies are in flight already; the
  // partial maxima come from the amax launch before this one, which may still
  // be running (programmatic dependent launch).  Everything after waits.
  pdl_wait();
  const TensorConsts tc = quant_prologue(p, s_red);
  build_scale_table(tc.s_t, s_tab);
  __syncthreads();

  int slot = 0;
  uint32_t ph = 0;
  bool failed = false;
  for (int64_t t = gw; t < n_tasks && !failed; t += nwarps) {
    const int64_t g = t / nch, ch = t - g * nch;
    const int64_t c0 = ch * kCW;
    const int nsub = nbr - 4 * g < 4 ? (int)(nbr - 4 * g) : 4;
    uint32_t sfw[CPL];  // the task's scale bytes of each output row, block-row sub in byte sub
#pragma unroll
    for (int k = 0; k < CPL; ++k) sfw[k] = 0u;
    for (int sub = 0; sub < nsub; ++sub) {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_for(bar0 + 8u * slot, ph, p.timeout_ns))) {
        failed = true;
        break;
      }
      uint32_t v[CPL / 2][16];  // word h of row i: columns 2h, 2h+1 of the lane
      const uint8_t* src = slots + slot * kColSlotBytes + 2 * CPL * lane;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if constexpr (CPL == 2) {
          v[0][i] = *reinterpret_cast<const uint32_t*>(src + 2 * kCW * i);
        } else {
          const uint2 d = *reinterpret_cast<const uint2*>(src + 2 * kCW * i);
          v[0][i] = d.x;
          v[CPL / 2 - 1][i] = d.y;
        }
      }
      __syncwarp();
      ++consumed;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issued += issue_next(slot) ? 1 : 0;
      if (++slot == kColSlots) {
        slot = 0;
        ph ^= 1u;
      }
      const int64_t rb = 4 * g + sub;
      // the two columns' stochastic-rounding draws
      float n0[16], n1[16];
      if (SR) {
        const bool odd = lane & 1;
        const uint64_t grp = (uint64_t)(c0 + 4 * (lane >> 1));
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint64_t r = (uint64_t)(rb * 16 + (odd ? q + 8 : q));
          const U4 u = sr_words4(r * (uint64_t)p.cols + grp, p.sr_k0, p.sr_k1);
          const uint32_t r0 = __shfl_xor_sync(0xFFFFFFFFu, odd ? u.x : u.z, 1);
          const uint32_t r1 = __shfl_xor_sync(0xFFFFFFFFu, odd ? u.y : u.w, 1);
          if (odd) {
            n0[q] = sr_draw(r0); n1[q] = sr_draw(r1); n0[q + 8] = sr_draw(u.z); n1[q + 8] = sr_draw(u.w);
          } else {
            n0[q] = sr_draw(u.x); n1[q] = sr_draw(u.y); n0[q + 8] = sr_draw(r0); n1[q + 8] = sr_draw(r1);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t s = RHT ? (((rht_mask >> i) & 1u) << 31) : 0u;
          const uint32_t wv = v[k >> 1][i];
          y[i] = __uint_as_float(((k & 1) ? (wv & 0xFFFF0000u) : (wv << 16)) ^ s);
        }
        if (RHT) hadamard16(y);
        const float ab = absmax16(y);
        uint64_t yp[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) yp[j] = pack_f2(y[2 * j], y[2 * j + 1]);
        uint32_t lo, hi, sf;
        bool four;
        quant_block_tab<RULE, SR>(yp, ab, tc, s_tab, (k & 1) ? n1 : n0, lo, hi, sf, four);
        *reinterpret_cast<uint2*>(obuf + k * 32 * kColOutPitch + 8 * sub) = make_uint2(lo, hi);
        sfw[k] |= sf << (8 * sub);
        const int64_t orow = c0 + CPL * lane + k;  // output row = source column
        if (p.choice && orow < p.cols) p.choice[orow * nbr + rb] = four ? 1 : 0;
      }
    }
    if (failed) break;
    // the task's output: each row's codes for block-rows 4g .. 4g + nsub - 1
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      const int64_t orow = c0 + CPL * lane + k;
      if (orow >= p.cols) continue;
      const uint8_t* e = obuf + k * 32 * kColOutPitch;
      uint8_t* dst = p.codes + orow * p.ld_codes + 4 * g * 8;
      const uint2 d0 = *reinterpret_cast<const uint2*>(e), d1 = *reinterpret_cast<const uint2*>(e + 8);
      const uint2 d2 = *reinterpret_cast<const uint2*>(e + 16), d3 = *reinterpret_cast<const uint2*>(e + 24);
      if (nsub == 4 && (reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
        st_v8(dst, make_uint4(d0.x, d0.y, d1.x, d1.y), make_uint4(d2.x, d2.y, d3.x, d3.y));
      } else {
        const uint2 d[4] = {d0, d1, d2, d3};
#pragma unroll
        for (int sub = 0; sub < 4; ++sub)
          if (sub < nsub) *reinterpret_cast<uint2*>(dst + 8 * sub) = d[sub];
      }
      // the 4 scale bytes of block-rows 4g .. 4g+3 are one aligned word in both
      // layouts (row-major when the output rows' scale counts are a multiple of 4)
      const int64_t so = sf_off(orow, 4 * g, nbr, p.sf_layout);
      if (nsub == 4 && (p.sf_layout == FOS_SF_SWIZZLED_128x4 || (nbr & 3) == 0)) {
        *reinterpret_cast<uint32_t*>(p.sf + so) = sfw[k];
      } else {
#pragma unroll
        for (int sub = 0; sub < 4; ++sub)
          if (sub < nsub) p.sf[sf_off(orow, 4 * g + sub, nbr, p.sf_layout)] = (uint8_t)(sfw[k] >> (8 * sub));
      }
    }
  }
  if (failed && lane == 0) *p.tensor_scale = __int_as_float(0x7FC00000);  // NaN: the result is not valid
  // let copies still in flight land before the CTA exits (bounded)
  for (; consumed < issued; ++consumed) {
    mbar_wait_for(bar0 + 8u * slot, ph, p.timeout_ns);
    if (++slot == kColSlots) {
      slot = 0;
      ph ^= 1u;
    }
  }
}

// ------------------------------------------------------------ dual (SR)
// One read of x [rows, cols] for both of its stochastic-rounding
// quantizations: pc along the source columns (transposed; with the RHT when
// RHT) and pr along the rows (no RHT).  Element i rounds with the Philox word
// of its source index in both, so each word is computed once: the transposed
// pass computes a block-row's words as the transposed kernel does (a lane pair
// shares each call) and leaves their draws in a per-warp stash, from which the
// row pass reads its own.  Warp task: 64 source rows (4 block-rows) x 64 source
// columns.  Per block-row, the transposed pass takes lane l's two columns
// (2l, 2l + 1) and the row pass lane l's two row blocks (row l/2, columns
// 32 (l & 1) .. + 31).  Slot rows are padded to 144 bytes and stash rows to 68
// words, so that the row pass's reads spread over the banks.
constexpr int kDualRowPitch = 2 * 64 + 16;
constexpr int kDualSlotBytes = 16 * kDualRowPitch;
constexpr int kDualSlots = 2;
constexpr int kDualStashPitch = 68;  // words
constexpr int kDualStashBytes = 16 * kDualStashPitch * 4;
constexpr int kDualOutBytes = 2 * 32 * kColOutPitch;
constexpr int kDualWarpBytes = kDualSlots * kDualSlotBytes + kDualStashBytes + kDualOutBytes;
constexpr int kDualSmemBytes = kColWarps * kDualWarpBytes;

template <int RULE, bool RHT>
__global__ void __launch_bounds__(256, 2) quant_dual_sr_kernel(QuantParams pc, QuantParams pr) {
  extern __shared__ __align__(128) uint8_t d_smem[];
  __shared__ float s_red[33];
  __shared__ float2 s_tab_c[128], s_tab_r[128];
  __shared__ uint64_t s_bar[kColWarps * kDualSlots];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < kColWarps * kDualSlots) mbar_init(smem_addr(&s_bar[threadIdx.x]), 16);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();  // the ring barriers are initialised before any copy
  const uint32_t rht_mask = RHT ? rht_sign_mask(pc.hk0, pc.hk1) : 0u;
  const int64_t nbr = pc.rows >> 4;             // block-rows of the source
  const int64_t ngr = (nbr + 3) >> 2;           // task rows (4 block-rows each)
  const int64_t nch = (pc.cols + 63) >> 6;      // task columns (64 source columns each)
  const int64_t n_tasks = ngr * nch;
  const int64_t nwarps = (int64_t)gridDim.x * kColWarps;
  const int64_t gw = (int64_t)blockIdx.x * kColWarps + warp;
  const uint64_t stream_once = l2_policy_evict_first();
  uint8_t* const wbase = d_smem + warp * kDualWarpBytes;
  uint8_t* const slots = wbase;
  float* const stash = reinterpret_cast<float*>(wbase + kDualSlots * kDualSlotBytes);
  uint8_t* const obuf = wbase + kDualSlots * kDualSlotBytes + kDualStashBytes + lane * kColOutPitch;
  const uint32_t bar0 = smem_addr(&s_bar[warp * kDualSlots]);

  // producer cursor (all lanes): the next (task, block-row) to fetch
  int64_t pt = gw;
  int psub = 0;
  auto issue_next = [&](int slot) -> bool {
    if (pt >= n_tasks) return false;
    const int64_t g = pt / nch, ch = pt - g * nch;
    const int64_t rb = 4 * g + psub;
    const int64_t c0 = ch * 64;
    const uint32_t bytes = (uint32_t)((pc.cols - c0 < 64 ? pc.cols - c0 : 64) * 2);
    if (lane < 16)
      bulk_g2s_hint(smem_addr(slots + slot * kDualSlotBytes + lane * kDualRowPitch),
                    pc.x + (rb * 16 + lane) * pc.ld + c0, bytes, bar0 + 8u * slot, stream_once);
    if (++psub == 4 || 4 * g + psub >= nbr) {
      psub = 0;
      pt += nwarps;
    }
    return true;
  };
  int issued = 0, consumed = 0;
  for (int k = 0; k < kDualSlots; ++k) issued += issue_next(k) ? 1 : 0;
  // Both tensor maxima are supplied (the launch is plain): nothing to wait for
  // but the stream order.
  const TensorConsts tcc = quant_prologue(pc, s_red);
  const TensorConsts tcr = quant_prologue(pr, s_red);
  build_scale_table(tcc.s_t, s_tab_c);
  build_scale_table(tcr.s_t, s_tab_r);
  __syncthreads();

  const bool odd = lane & 1;
  int slot = 0;
  uint32_t ph = 0;
  bool failed = false;
  for (int64_t t = gw; t < n_tasks && !failed; t += nwarps) {
    const int64_t g = t / nch, ch = t - g * nch;
    const int64_t c0 = ch * 64;
    const int nsub = nbr - 4 * g < 4 ? (int)(nbr - 4 * g) : 4;
    uint32_t sfw[2] = {0u, 0u};  // the task's scale bytes of each transposed output row
    for (int sub = 0; sub < nsub; ++sub) {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_for(bar0 + 8u * slot, ph, pc.timeout_ns))) {
        failed = true;
        break;
      }
      const uint8_t* sl = slots + slot * kDualSlotBytes;
      const int64_t rb = 4 * g + sub;

      // ---- the block-row's draws: 8 Philox calls per lane (rows q, or q + 8
      // for the odd lane of a pair, of the pair's 4-column group), each word
      // converted once (sr_draw), into the stash, and swapped with the pair
      // for the transposed pass
      float n0[16], n1[16];
      {
        const uint64_t grp = (uint64_t)(c0 + 4 * (lane >> 1));
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int rr = odd ? q + 8 : q;
          const uint64_t r = (uint64_t)(rb * 16 + rr);
          const U4 u = sr_words4(r * (uint64_t)pc.cols + grp, pc.sr_k0, pc.sr_k1);
          const float f0 = sr_draw(u.x), f1 = sr_draw(u.y), f2 = sr_draw(u.z), f3 = sr_draw(u.w);
          *reinterpret_cast<float4*>(stash + kDualStashPitch * rr + 4 * (lane >> 1)) = make_float4(f0, f1, f2, f3);
          const float r0 = __shfl_xor_sync(0xFFFFFFFFu, odd ? f0 : f2, 1);
          const float r1 = __shfl_xor_sync(0xFFFFFFFFu, odd ? f1 : f3, 1);
          if (odd) {
            n0[q] = r0; n1[q] = r1; n0[q + 8] = f2; n1[q + 8] = f3;
          } else {
            n0[q] = f0; n1[q] = f1; n0[q + 8] = r0; n1[q + 8] = r1;
          }
        }
      }

      // ---- transposed pass: the lane's two source columns
      {
        uint32_t v[16];  // row i: columns 2 lane, 2 lane + 1
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = *reinterpret_cast<const uint32_t*>(sl + kDualRowPitch * i + 4 * lane);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          float y[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t s = RHT ? (((rht_mask >> i) & 1u) << 31) : 0u;
            y[i] = __uint_as_float((k ? (v[i] & 0xFFFF0000u) : (v[i] << 16)) ^ s);
          }
          if (RHT) hadamard16(y);
          const float ab = absmax16(y);
          uint64_t yp[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) yp[j] = pack_f2(y[2 * j], y[2 * j + 1]);
          uint32_t lo, hi, sf;
          bool four;
          quant_block_tab<RULE, true>(yp, ab, tcc, s_tab_c, k ? n1 : n0, lo, hi, sf, four);
          *reinterpret_cast<uint2*>(obuf + k * 32 * kColOutPitch + 8 * sub) = make_uint2(lo, hi);
          sfw[k] |= sf << (8 * sub);
          const int64_t orow = c0 + 2 * lane + k;  // output row = source column
          if (pc.choice && orow < pc.cols) pc.choice[orow * nbr + rb] = four ? 1 : 0;
        }
      }
      __syncwarp();  // the stash is complete

      // ---- row pass: the lane's two blocks of row l/2
      {
        const int rr = lane >> 1, hb = lane & 1;
        const int64_t row = rb * 16 + rr;
        const uint8_t* src = sl + kDualRowPitch * rr + 64 * hb;
        const float* nsrc = stash + kDualStashPitch * rr + 32 * hb;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int64_t blk = (c0 >> 4) + 2 * hb + b;  // the block's index along the row
          if (16 * blk >= pr.cols) break;              // past a ragged task's last column
          uint32_t wv[8];
          const uint4 a = *reinterpret_cast<const uint4*>(src + 32 * b);
          const uint4 c = *reinterpret_cast<const uint4*>(src + 32 * b + 16);
          wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
          wv[4] = c.x; wv[5] = c.y; wv[6] = c.z; wv[7] = c.w;
          uint64_t yp[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) yp[k] = bf16x2_to_f32x2(wv[k]);
          const float ab = absmax16_bf16(wv);
          float n[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 w = *reinterpret_cast<const float4*>(nsrc + 16 * b + 4 * q);
            n[4 * q] = w.x; n[4 * q + 1] = w.y; n[4 * q + 2] = w.z; n[4 * q + 3] = w.w;
          }
          uint32_t lo, hi, sf;
          bool four;
          quant_block_tab<RULE, true>(yp, ab, tcr, s_tab_r, n, lo, hi, sf, four);
          *reinterpret_cast<uint2*>(pr.codes + row * pr.ld_codes + 8 * blk) = make_uint2(lo, hi);
          pr.sf[sf_off(row, blk, pr.nb, pr.sf_layout)] = (uint8_t)sf;
          if (pr.choice) pr.choice[row * pr.nb + blk] = four ? 1 : 0;
        }
      }
      __syncwarp();  // the slot and the stash have been read
      ++consumed;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issued += issue_next(slot) ? 1 : 0;
      if (++slot == kDualSlots) {
        slot = 0;
        ph ^= 1u;
      }
    }
    if (failed) break;
    // the task's transposed output: each row's codes for block-rows 4g .. 4g + nsub - 1
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t orow = c0 + 2 * lane + k;
      if (orow >= pc.cols) continue;
      const uint8_t* e = obuf + k * 32 * kColOutPitch;
      uint8_t* dst = pc.codes + orow * pc.ld_codes + 4 * g * 8;
      const uint2 d0 = *reinterpret_cast<const uint2*>(e), d1 = *reinterpret_cast<const uint2*>(e + 8);
      const uint2 d2 = *reinterpret_cast<const uint2*>(e + 16), d3 = *reinterpret_cast<const uint2*>(e + 24);
      if (nsub == 4 && (reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
        st_v8(dst, make_uint4(d0.x, d0.y, d1.x, d1.y), make_uint4(d2.x, d2.y, d3.x, d3.y));
      } else {
        const uint2 d[4] = {d0, d1, d2, d3};
#pragma unroll
        for (int sub = 0; sub < 4; ++sub)
          if (sub < nsub) *reinterpret_cast<uint2*>(dst + 8 * sub) = d[sub];
      }
      const int64_t so = sf_off(orow, 4 * g, nbr, pc.sf_layout);
      if (nsub == 4 && (pc.sf_layout == FOS_SF_SWIZZLED_128x4 || (nbr & 3) == 0)) {
        *reinterpret_cast<uint32_t*>(pc.sf + so) = sfw[k];
      } else {
#pragma unroll
        for (int sub = 0; sub < 4; ++sub)
          if (sub < nsub) pc.sf[sf_off(orow, 4 * g + sub, nbr, pc.sf_layout)] = (uint8_t)(sfw[k] >> (8 * sub));
      }
    }
  }
  if (failed && lane == 0) {
    *pc.tensor_scale = __int_as_float(0x7FC00000);  // NaN: the results are not valid
    *pr.tensor_scale = __int_as_float(0x7FC00000);
  }
  // let copies still in flight land before the CTA exits (bounded)
  for (; consumed < issued; ++consumed) {
    mbar_wait_for(bar0 + 8u * slot, ph, pc.timeout_ns);
    if (++slot == kDualSlots) {
      slot = 0;
      ph ^= 1u;
    }
  }
}

// -------------------------------------------------------------- quant_2d
// Warp task = 16 source rows x 32 source columns (two tiles); lane l owns
// source row (l & 15) of tile (l >> 4).  Tile reductions use xor-shuffles
// within each 16-lane half; the error tree pairs adjacent rows first.
__device__ __forceinline__ float half_max(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ float half_tree_sum(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// The stochastic-rounding forms are held to three CTAs per SM (80 registers):
// unbounded, the compiler gives the 4/6 one 124 and it runs two.  The RNE
// forms get no bound (0): an explicit one, even 1 or 4, changed their code
// and measured slower.
template <int RULE, bool RHT, bool SR, bool TRANS>
__global__ void __launch_bounds__(256, SR ? 3 : 0) quant_2d_kernel(QuantParams p) {
  __shared__ float s_red[33];
  __shared__ float2 s_tab[128];
  pdl_launch_dependents();  // a dependent launch (the next quantize launch, a GEMM) may start its own reads
  pdl_wait();  // the partial maxima come from the amax launch before this one
  const TensorConsts tc = quant_prologue(p, s_red);
  build_scale_table(tc.s_t, s_tab);
  __syncthreads();
  const uint32_t rht_mask = RHT ? rht_sign_mask(p.hk0, p.hk1) : 0u;
  const int lane = threadIdx.x & 31, i = lane & 15, half = lane >> 4;
  const int64_t ntc = p.cols >> 4;  // tiles along source columns
  // warp task: 16 source rows x 2 * kSteps tiles, two tiles per step (one per
  // half).  With stochastic rounding a row-major task takes 4 tiles, so that
  // each source row's 32 code bytes and 4 scale bytes of the task are stored
  // at once after the second step: whole sectors rather than 8-byte pieces.
  // The RNE form stores per tile: the two steps' registers cost it a CTA per
  // SM and measured slower.  Transposed output rows differ between the
  // halves, so there a task is one step.
  constexpr bool kBand = SR && !TRANS;
  constexpr int kSteps = kBand ? 2 : 1;
  const int64_t ngrp = (ntc + 2 * kSteps - 1) / (2 * kSteps);
  const int64_t n_tasks = (p.rows >> 4) * ngrp;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < n_tasks; t += nwarps) {
    const int64_t tr = t / ngrp, tile0 = (t - tr * ngrp) * 2 * kSteps;
    const int nt = ntc - tile0 < 2 * kSteps ? (int)(ntc - tile0) : 2 * kSteps;  // tiles of this task
    uint32_t lo0 = 0, hi0 = 0, sf0 = 0, lo1 = 0, hi1 = 0, sf1 = 0;  // kBand: each step's results
    auto step = [&](const int s2) {  // tiles tile0 + 2 * s2 (first half) and + 1 (second)
      const int64_t tcol = tile0 + 2 * s2 + half;
      const bool valid = 2 * s2 + half < nt;  // uniform within each 16-lane half
      const int64_t r = tr * 16 + i, c0 = tcol * 16;
      uint32_t wv[8];
      float y[16];
      if (valid) {
        load_block16(p.x + r * p.ld + c0, p.aligned32, wv);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) wv[k] = 0u;
      }
      if (RHT && !TRANS) {
        unpack16(wv, rht_mask, y);
        hadamard16(y);
      } else {
        unpack16(wv, 0u, y);
      }
      if (RHT && TRANS) {
        // transform down the 16 source rows of each column: across lanes
        if ((rht_mask >> i) & 1u) {
#pragma unroll
          for (int j = 0; j < 16; ++j) y[j] = -y[j];
        }
#pragma unroll
        for (int h = 1; h < 16; h <<= 1) {
          const bool upper = (i & h) != 0;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float o = __shfl_xor_sync(0xFFFFFFFFu, y[j], h);
            y[j] = upper ? __fsub_rn(o, y[j]) : __fadd_rn(y[j], o);
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) y[j] = __fmul_rn(y[j], 0.25f);
      }
      const float ab = half_max(absmax16(y));
      float n_sr[16];
      sr_draws16<SR>((uint64_t)r * (uint64_t)p.cols + (uint64_t)c0, p, n_sr);
      const uint32_t pair = candidate_scales(ab, tc);
      const uint32_t sf6 = pair & 0xFFu, sf4 = pair >> 8;
      uint64_t yp[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) yp[j] = pack_f2(y[2 * j], y[2 * j + 1]);
      uint32_t lo6 = 0, hi6 = 0, lo4 = 0, hi4 = 0;
      float E6 = 0.0f, E4 = 0.0f;
#pragma unroll
      for (int cnd = 0; cnd < 2; ++cnd) {
        if (cnd == 0 && RULE == FOS_SCALE_4) continue;
        if (cnd == 1 && RULE == FOS_SCALE_6) continue;
        const uint32_t sfc = cnd == 0 ? sf6 : sf4;
        const float2 tb = s_tab[sfc];
        uint32_t l, h;
        float S;
        if (SR) {
          // split per candidate here: kept across both, it cost this kernel a
          // CTA per SM (125 registers)
          F2 ay[8], sg[8];
          sr_split16(yp, ay, sg);
          S = cand_sr16(ay, sg, tb.x, n_sr, l, h);
        } else {
          const uint64_t inv2 = pack_f2(tb.x, tb.x);
          uint64_t acc = 0ull;
          const uint64_t a[4] = {yp[0], yp[1], yp[2], yp[3]}, b[4] = {yp[4], yp[5], yp[6], yp[7]};
          l = cand_rne8(a, inv2, acc);
          h = cand_rne8(b, inv2, acc);
          const F2 e = unpack_f2(acc);
          S = __fadd_rn(e.x, e.y);
        }
        if (sfc == 0) S = sumsq16(y);  // a zero scale flushes the row: its error is sum y^2
        S = half_tree_sum(S);
        const float E = sfc ? __fmul_rn(S, tb.y) : S;
        if (cnd == 0) {
          lo6 = l; hi6 = h; E6 = E;
        } else {
          lo4 = l; hi4 = h; E4 = E;
        }
      }
      const bool four = (RULE == FOS_SCALE_4) || (RULE == FOS_SCALE_4OVER6 && E4 < E6);
      const uint32_t lo = four ? lo4 : lo6, hi = four ? hi4 : hi6, sf = four ? sf4 : sf6;
      if (kBand) {
        if (valid && p.choice) p.choice[r * p.nb + tcol] = four ? 1 : 0;
        if (s2 == 0) {
          lo0 = lo; hi0 = hi; sf0 = sf;
        } else {
          lo1 = lo; hi1 = hi; sf1 = sf;
        }
      } else if (!TRANS) {
        if (valid) {
          *reinterpret_cast<uint2*>(p.codes + r * p.ld_codes + tcol * 8) = make_uint2(lo, hi);
          p.sf[sf_off(r, tcol, p.nb, p.sf_layout)] = (uint8_t)sf;
          if (p.choice) p.choice[r * p.nb + tcol] = four ? 1 : 0;
        }
      } else {
        // lane i collects output row (source column) c0 + i: nibble i of every
        // source row j of its tile, j = 0..15 in order along the output row
        uint32_t olo = 0, ohi = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          uint32_t slo = __shfl_sync(0xFFFFFFFFu, lo, (half << 4) | j);
          uint32_t shi = __shfl_sync(0xFFFFFFFFu, hi, (half << 4) | j);
          uint32_t nib = ((i < 8 ? slo : shi) >> (4 * (i & 7))) & 15u;
          if (j < 8)
            olo |= nib << (4 * j);
          else
            ohi |= nib << (4 * (j - 8));
        }
        if (valid) {
          const int64_t orow = c0 + i;
          *reinterpret_cast<uint2*>(p.codes + orow * p.ld_codes + tr * 8) = make_uint2(olo, ohi);
          p.sf[sf_off(orow, tr, p.nb, p.sf_layout)] = (uint8_t)sf;
          if (p.choice) p.choice[orow * p.nb + tr] = four ? 1 : 0;
        }
      }
    };
    step(0);
    if (kBand && nt > 2) step(1);
    if (kBand) {
      // lane i of the first half stores source row i's tiles tile0 .. tile0+3:
      // its own (steps 0 and 1) and its partner's in the second half
      const uint32_t plo0 = __shfl_down_sync(0xFFFFFFFFu, lo0, 16), phi0 = __shfl_down_sync(0xFFFFFFFFu, hi0, 16);
      const uint32_t psf0 = __shfl_down_sync(0xFFFFFFFFu, sf0, 16), plo1 = __shfl_down_sync(0xFFFFFFFFu, lo1, 16);
      const uint32_t phi1 = __shfl_down_sync(0xFFFFFFFFu, hi1, 16), psf1 = __shfl_down_sync(0xFFFFFFFFu, sf1, 16);
      if (half == 0) {
        const int64_t r = tr * 16 + i;
        uint8_t* cd = p.codes + r * p.ld_codes + tile0 * 8;
        if (nt == 4 && (reinterpret_cast<uintptr_t>(cd) & 31) == 0) {
          st_v8(cd, make_uint4(lo0, hi0, plo0, phi0), make_uint4(lo1, hi1, plo1, phi1));
        } else {
          const uint2 c[4] = {make_uint2(lo0, hi0), make_uint2(plo0, phi0), make_uint2(lo1, hi1),
                              make_uint2(plo1, phi1)};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (k < nt) *reinterpret_cast<uint2*>(cd + 8 * k) = c[k];
        }
        // tile0 % 4 == 0: the 4 scale bytes are one aligned word in both
        // layouts (row-major when the rows' scale counts are a multiple of 4)
        const uint32_t sfw = sf0 | (psf0 << 8) | (sf1 << 16) | (psf1 << 24);
        if (nt == 4 && (p.sf_layout == FOS_SF_SWIZZLED_128x4 || (p.nb & 3) == 0)) {
          *reinterpret_cast<uint32_t*>(p.sf + sf_off(r, tile0, p.nb, p.sf_layout)) = sfw;
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (k < nt) p.sf[sf_off(r, tile0 + k, p.nb, p.sf_layout)] = (uint8_t)(sfw >> (8 * k));
        }
      }
    }
  }
}

// ------------------------------------------------------------ sf padding

__global__ void sf_pad_zero_kernel(uint8_t* sf, int64_t bytes, int64_t R, int64_t nb) {
  const int64_t n_ct = (nb + 3) >> 2;
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < bytes; o += (int64_t)gridDim.x * blockDim.x) {
    int64_t tile = o >> 9, w = o & 511;
    int64_t rt = tile / n_ct, ct = tile - rt * n_ct;
    int64_t r = rt * 128 + ((w >> 2) & 3) * 32 + (w >> 4);
    int64_t c = ct * 4 + (w & 3);
    if (r >= R || c >= nb) sf[o] = 0;
  }
}

// ----------------------------------------------------------- dequantize

template <bool BF16>
__global__ void __launch_bounds__(256) dequant_kernel(DequantParams p) {
  const int64_t nb = p.cols >> 4;
  const int64_t n = p.rows * nb;
  const float s_t = __ldg(p.tensor_scale);
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / nb, b = t - r * nb;
    const uint2 cw = *reinterpret_cast<const uint2*>(p.codes + r * p.ld_codes + b * 8);
    const uint32_t s = p.sf[sf_off(r, b, nb, p.sf_layout)];
    const float eff = __fmul_rn(e4m3x2_decode(s).x, s_t);
    float v[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t byte = ((k < 4 ? cw.x : cw.y) >> (8 * (k & 3))) & 0xFFu;
      F2 g = e2m1x2_decode(byte);
      F2 x = mul2(g, F2{eff, eff});
      v[2 * k] = x.x;
      v[2 * k + 1] = x.y;
    }
    if (BF16) {
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        o[k] = *reinterpret_cast<uint32_t*>(&h);
      }
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + r * p.ld_out + b * 16);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + r * p.ld_out + b * 16);
#pragma unroll
      for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    }
  }
}

// ---------------------------------------------------------------- codecs

__global__ void e2m1_encode_kernel(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (uint8_t)(e2m1x2(x[i], 0.0f) & 15u);
}

__global__ void e4m3_encode_kernel(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (uint8_t)(e4m3x2(x[i], 0.0f) & 0xFFu);
}

__global__ void philox_kernel(const uint32_t* ctr, int64_t n, uint32_t k0, uint32_t k1, uint32_t* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    U4 u = philox10(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3], k0, k1);
    out[4 * i] = u.x;
    out[4 * i + 1] = u.y;
    out[4 * i + 2] = u.z;
    out[4 * i + 3] = u.w;
  }
}

// ------------------------------------------------------------- launchers

static int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

cudaError_t launch_amax(const AmaxParams& p, bool hadamard, bool transpose, int grid, cudaStream_t s) {
  if (hadamard && transpose)
    if (p.partials_plain)
      amax_cols_kernel<true><<<grid, 256, 0, s>>>(p);
    else
      amax_cols_kernel<false><<<grid, 256, 0, s>>>(p);
  else if (hadamard)
    amax_rows_kernel<true><<<grid, 256, 0, s>>>(p);
  else
    amax_rows_kernel<false><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

// Launch fn(p); with pdl, the launch may begin while the stream's previous
// kernel is still running (programmatic stream serialization): fn must then
// wait (griddepcontrol.wait) before it reads anything that kernel writes.
static cudaError_t launch_params(void (*fn)(QuantParams), int grid, int block, int smem, bool pdl,
                                 const QuantParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

// The dynamic shared-memory opt-in is a property of a kernel on one device:
// it is set once per (kernel, device), and its error is returned.
constexpr int kMaxDevices = 64;

static int current_device() {
  int d = -1;
  return cudaGetDevice(&d) == cudaSuccess ? d : -1;
}

// Resident CTAs per SM of an amax kernel at 256 threads, found once per device.
template <typename Fn>
static int amax_per_sm(Fn fn, std::atomic<int>* per_sm_of) {
  const int dev = current_device();
  int n = (dev >= 0 && dev < kMaxDevices) ? per_sm_of[dev].load(std::memory_order_acquire) : 0;
  if (n == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, 256, 0) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();  // the query's own error: fall back to four per SM
      return 4;
    }
    if (dev >= 0 && dev < kMaxDevices) per_sm_of[dev].store(n, std::memory_order_release);
  }
  return n;
}

int amax_grid(int64_t n_warp_tasks, bool hadamard, bool transpose) {
  static std::atomic<int> rows_plain[kMaxDevices], rows_rht[kMaxDevices], cols[kMaxDevices];
  // one resident wave of the kernel launch_amax picks (the tasks are split
  // evenly over the grid up front)
  const int per_sm = hadamard && transpose ? amax_per_sm(amax_cols_kernel<false>, cols)
                     : hadamard            ? amax_per_sm(amax_rows_kernel<true>, rows_rht)
                                           : amax_per_sm(amax_rows_kernel<false>, rows_plain);
  int64_t g = (n_warp_tasks + 7) / 8;
  int64_t cap = (int64_t)sm_count() * per_sm;
  if (cap > kMaxAmaxPartials) cap = kMaxAmaxPartials;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

template <int MODE>
static cudaError_t launch_amax_batch_mode(const AmaxBatch& b, int64_t total_tasks, int* grid, cudaStream_t s) {
  auto fn = amax_batch_kernel<MODE>;
  static std::atomic<int> per_sm_of[kMaxDevices];
  const int per_sm = amax_per_sm(fn, per_sm_of);
  int64_t g = (total_tasks + 7) / 8;
  int64_t cap = (int64_t)sm_count() * per_sm;
  if (cap > kMaxAmaxPartials) cap = kMaxAmaxPartials;
  if (g > cap) g = cap;
  *grid = (int)(g < 1 ? 1 : g);
  fn<<<*grid, 256, 0, s>>>(b);
  return cudaGetLastError();
}

cudaError_t launch_amax_batch(const AmaxBatch& b, bool hadamard, bool transpose, int64_t total_tasks, int* grid,
                              cudaStream_t s) {
  if (b.n_jobs < 1 || b.n_jobs > kAmaxBatchJobs) return cudaErrorInvalidValue;
  if (hadamard && transpose) return launch_amax_batch_mode<2>(b, total_tasks, grid, s);
  if (hadamard) return launch_amax_batch_mode<1>(b, total_tasks, grid, s);
  return launch_amax_batch_mode<0>(b, total_tasks, grid, s);
}

template <typename Fn>
static cudaError_t smem_opt_in(Fn fn, int bytes, std::atomic<int>* done) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (dev < kMaxDevices && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < kMaxDevices) done[dev].store(1, std::memory_order_release);
  return e;
}

// Cut a quantize launch's grid to the CTAs that fit on the GPU at once (found
// once per device for each kernel).  The kernels split their tasks evenly over
// the grid up front, so CTAs beyond one resident wave run as a later, partly
// filled wave.  Measured on B300: the column kernel 4-5% faster and the RNE 2D
// kernel 1-3%; the row kernel unchanged; the stochastic-rounding 2D kernel 3%
// slower, so it keeps its larger grid.
template <typename Fn>
static cudaError_t one_wave(Fn fn, int smem, std::atomic<int>* per_sm_of, int* grid) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  int per_sm = dev < kMaxDevices ? per_sm_of[dev].load(std::memory_order_acquire) : 0;
  if (per_sm == 0) {
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 256, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (dev < kMaxDevices) per_sm_of[dev].store(per_sm, std::memory_order_release);
  }
  const int64_t cap = (int64_t)per_sm * sm_count();
  if (*grid > cap) *grid = (int)cap;
  return cudaSuccess;
}

template <int RULE, bool RHT, bool SR, bool TRANS>
static cudaError_t launch_2d(const QuantParams& p, int grid, cudaStream_t s, bool pdl) {
  auto fn = quant_2d_kernel<RULE, RHT, SR, TRANS>;
  if constexpr (!SR) {
    static std::atomic<int> per_sm[kMaxDevices];
    const cudaError_t e = one_wave(fn, 0, per_sm, &grid);
    if (e != cudaSuccess) return e;
  }
  return launch_params(fn, grid, 256, 0, pdl, p, s);
}

template <int RULE, bool RHT, bool SR>
static cudaError_t launch_q(const QuantParams& p, int kind, int grid, cudaStream_t s, bool pdl) {
  switch (kind) {
    case 0: {
      auto fn = quant_rows_kernel<RULE, RHT, SR, kRowsPlain>;
      static std::atomic<int> done[kMaxDevices];
      const cudaError_t e = smem_opt_in(fn, kRowSmemBytes, done);
      return e != cudaSuccess ? e : launch_params(fn, grid, 256, kRowSmemBytes, pdl, p, s);
    }
    case 1: {
      auto fn = quant_cols_kernel<RULE, RHT, SR>;
      static std::atomic<int> done[kMaxDevices], per_sm[kMaxDevices];
      cudaError_t e = smem_opt_in(fn, kColSmemBytes, done);
      if (e == cudaSuccess) e = one_wave(fn, kColSmemBytes, per_sm, &grid);
      return e != cudaSuccess ? e : launch_params(fn, grid, 256, kColSmemBytes, pdl, p, s);
    }
    case 2: return launch_2d<RULE, RHT, SR, false>(p, grid, s, pdl);
    default: return launch_2d<RULE, RHT, SR, true>(p, grid, s, pdl);
  }
}

template <int RULE>
static cudaError_t launch_q_rule(const QuantParams& p, int kind, bool rht, bool sr, int grid, cudaStream_t s,
                                 bool pdl) {
  if (rht) return sr ? launch_q<RULE, true, true>(p, kind, grid, s, pdl) : launch_q<RULE, true, false>(p, kind, grid, s, pdl);
  return sr ? launch_q<RULE, false, true>(p, kind, grid, s, pdl) : launch_q<RULE, false, false>(p, kind, grid, s, pdl);
}

int quant_grid(int64_t n_warp_tasks, int kind) {
  int64_t g = (n_warp_tasks + 7) / 8;
  // the row and column kernels keep at most three CTAs per SM resident (their
  // shared-memory rings)
  int64_t cap = (int64_t)sm_count() * (kind <= 1 ? 3 : 8);
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

template <int RULE, bool RHT, bool SR>
static cudaError_t launch_rows_fused(const QuantParams& p, int64_t n_tasks, cudaStream_t s) {
  auto fn = quant_rows_kernel<RULE, RHT, SR, kRowsFused>;
  // resident CTAs per SM, found once per device (the grid barrier needs all
  // CTAs resident at once)
  static std::atomic<int> per_sm_of[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  int per_sm = dev < kMaxDevices ? per_sm_of[dev].load(std::memory_order_acquire) : 0;
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 256, kRowSmemBytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (dev < kMaxDevices) per_sm_of[dev].store(per_sm, std::memory_order_release);
  }
  int64_t grid = (int64_t)per_sm * sm_count();
  const int64_t want = (n_tasks + kRowWarps - 1) / kRowWarps;
  if (grid > want) grid = want;
  if (grid > kMaxAmaxPartials) grid = kMaxAmaxPartials;
  if (grid < 1) grid = 1;
  QuantParams q = p;
  void* args[] = {&q};
  // the barrier's arrival counter, the give-up flag and the exit counter
  cudaError_t e = cudaMemsetAsync(p.ws_barrier, 0, kBarrierWords * sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fn), dim3((unsigned)grid), dim3(256), args,
                                     kRowSmemBytes, s);
}

template <int RULE>
static cudaError_t launch_rows_fused_rule(const QuantParams& p, bool rht, bool sr, int64_t n_tasks,
                                          cudaStream_t s) {
  if (rht) return sr ? launch_rows_fused<RULE, true, true>(p, n_tasks, s) : launch_rows_fused<RULE, true, false>(p, n_tasks, s);
  return sr ? launch_rows_fused<RULE, false, true>(p, n_tasks, s) : launch_rows_fused<RULE, false, false>(p, n_tasks, s);
}

template <int RULE, bool RHT, bool SR>
static cudaError_t launch_rows_chained(const QuantParams& p, int grid, cudaStream_t s) {
  auto fn = quant_rows_kernel<RULE, RHT, SR, kRowsChained>;
  static std::atomic<int> done[kMaxDevices];
  const cudaError_t e = smem_opt_in(fn, kChainSmemBytes, done);
  if (e != cudaSuccess) return e;
  // always the successor of a launch of the same batch: overlap its tail
  return launch_params(fn, grid, 32 * (kRowWarps + kAmaxWarps), kChainSmemBytes, true, p, s);
}

int chained_grid() {
  int g = sm_count() * 2;
  return g > kMaxAmaxPartials ? kMaxAmaxPartials : g;
}

cudaError_t launch_quant_rows_chained(const QuantParams& p, int rule, bool rht, bool sr, int grid, cudaStream_t s) {
#define FOS_CHAIN(R)                                                                                        \
  return rht ? (sr ? launch_rows_chained<R, true, true>(p, grid, s) : launch_rows_chained<R, true, false>(p, grid, s)) \
             : (sr ? launch_rows_chained<R, false, true>(p, grid, s) : launch_rows_chained<R, false, false>(p, grid, s))
  switch (rule) {
    case FOS_SCALE_6: FOS_CHAIN(FOS_SCALE_6);
    case FOS_SCALE_4: FOS_CHAIN(FOS_SCALE_4);
    default: FOS_CHAIN(FOS_SCALE_4OVER6);
  }
#undef FOS_CHAIN
}

cudaError_t launch_quant_rows_fused(const QuantParams& p, int rule, bool rht, bool sr, int64_t n_tasks,
                                    cudaStream_t s) {
  switch (rule) {
    case FOS_SCALE_6: return launch_rows_fused_rule<FOS_SCALE_6>(p, rht, sr, n_tasks, s);
    case FOS_SCALE_4: return launch_rows_fused_rule<FOS_SCALE_4>(p, rht, sr, n_tasks, s);
    default: return launch_rows_fused_rule<FOS_SCALE_4OVER6>(p, rht, sr, n_tasks, s);
  }
}

template <int RULE, bool RHT>
static cudaError_t launch_dual_rule(const QuantParams& pc, const QuantParams& pr, int64_t n_tasks, cudaStream_t s) {
  auto fn = quant_dual_sr_kernel<RULE, RHT>;
  static std::atomic<int> done[kMaxDevices], per_sm[kMaxDevices];
  const int64_t want = (n_tasks + kColWarps - 1) / kColWarps;
  int grid = want < 1 ? 1 : (want > (1 << 20) ? (1 << 20) : (int)want);
  cudaError_t e = smem_opt_in(fn, kDualSmemBytes, done);
  if (e == cudaSuccess) e = one_wave(fn, kDualSmemBytes, per_sm, &grid);
  if (e != cudaSuccess) return e;
  fn<<<grid, 32 * kColWarps, kDualSmemBytes, s>>>(pc, pr);
  return cudaGetLastError();
}

cudaError_t launch_quant_dual_sr(const QuantParams& pc, const QuantParams& pr, int rule, bool rht, int64_t n_tasks,
                                 cudaStream_t s) {
#define FOS_DUAL(R) return rht ? launch_dual_rule<R, true>(pc, pr, n_tasks, s) : launch_dual_rule<R, false>(pc, pr, n_tasks, s)
  switch (rule) {
    case FOS_SCALE_6: FOS_DUAL(FOS_SCALE_6);
    case FOS_SCALE_4: FOS_DUAL(FOS_SCALE_4);
    default: FOS_DUAL(FOS_SCALE_4OVER6);
  }
#undef FOS_DUAL
}

cudaError_t launch_quant(const QuantParams& p, int rule, int kind, bool rht, bool sr, int grid, cudaStream_t s,
                         bool pdl) {
  switch (rule) {
    case FOS_SCALE_6: return launch_q_rule<FOS_SCALE_6>(p, kind, rht, sr, grid, s, pdl);
    case FOS_SCALE_4: return launch_q_rule<FOS_SCALE_4>(p, kind, rht, sr, grid, s, pdl);
    default: return launch_q_rule<FOS_SCALE_4OVER6>(p, kind, rht, sr, grid, s, pdl);
  }
}

cudaError_t launch_sf_pad(uint8_t* sf, int64_t bytes, int64_t R, int64_t nb, cudaStream_t s) {
  int64_t g = (bytes + 255) / 256;
  if (g > 1024) g = 1024;
  sf_pad_zero_kernel<<<(int)(g < 1 ? 1 : g), 256, 0, s>>>(sf, bytes, R, nb);
  return cudaGetLastError();
}

__global__ void nan_to_status_kernel(const float* ts, int32_t* out) {
  *out = isnan(*ts) ? (int32_t)FOS_ERR_TIMEOUT : (int32_t)FOS_OK;
}

cudaError_t launch_nan_to_status(const float* tensor_scale, int32_t* out, cudaStream_t s) {
  nan_to_status_kernel<<<1, 1, 0, s>>>(tensor_scale, out);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const DequantParams& p, bool bf16, cudaStream_t s) {
  int64_t n = p.rows * (p.cols >> 4);
  int64_t g = (n + 255) / 256;
  int64_t cap = (int64_t)sm_count() * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  if (bf16)
    dequant_kernel<true><<<(int)g, 256, 0, s>>>(p);
  else
    dequant_kernel<false><<<(int)g, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_e2m1_encode(const float* x, int64_t n, uint8_t* out, cudaStream_t s) {
  e2m1_encode_kernel<<<(int)((n + 255) / 256 < 4096 ? (n + 255) / 256 + 1 : 4096), 256, 0, s>>>(x, n, out);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_encode(const float* x, int64_t n, uint8_t* out, cudaStream_t s) {
  e4m3_encode_kernel<<<(int)((n + 255) / 256 < 4096 ? (n + 255) / 256 + 1 : 4096), 256, 0, s>>>(x, n, out);
  return cudaGetLastError();
}

cudaError_t launch_philox(const uint32_t* ctr, int64_t n, uint64_t key, uint32_t* out, cudaStream_t s) {
  philox_kernel<<<(int)((n + 255) / 256 < 4096 ? (n + 255) / 256 + 1 : 4096), 256, 0, s>>>(
      ctr, n, (uint32_t)key, (uint32_t)(key >> 32), out);
  return cudaGetLastError();
}

}  // namespace fos
