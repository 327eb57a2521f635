// MXFP4 with the Four Over Six choice, for sm_103a.
//
// "FP4" (Ultralytics glossary), "FP4 Nasıl Çalışır": MXFP4 groups 32 values
// under one 8-bit power-of-two scale (E8M0 in the OCP Microscaling
// specification: byte X + 127 means 2^X) and has no tensor scale.  Each
// 32-value block gets two candidate exponents: the specification's own,
// X6 = floor(log2 amax) - 2, which maps the block maximum into [4, 8) and lets
// values above 6 saturate, and X4 = X6 + 1, which maps it below 4 and
// saturates nothing.  Each candidate's codes are the E2M1 round-to-nearest-even
// roundings of q = y * 2^-X; its error S is the sum of (q - g)^2, taken per
// 16-value half in the order of the NVFP4 path (even and odd FMA chains, then
// one add) and the halves added.  Keep 4 iff 4 * S_4 < S_6 (both in the
// 6-candidate's units, exact), ties to 6.  An all-zero block gets byte 0.
//
// No tensor scale means no amax pass: one launch reads each value once.  One
// thread owns one 32-value block (64 contiguous bytes; a warp reads 2 KB).
// Scales go row-major or into the 128x4 tiles the block-scaled MMA reads
// (one tile: 128 rows x 4 scales = 128 values of K).  For the tiles, thread t
// takes the block whose scale byte is byte t of the buffer, so a warp stores
// 32 contiguous scale bytes (and reads 8 rows x 4 neighbouring blocks, 256
// contiguous bytes a row); a thread whose byte is padding writes a zero.
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "fos.h"
#include "fos_device.cuh"
#include "fos_internal.h"

namespace fos {
namespace {

__device__ __forceinline__ float max_nan_f32(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

struct MxParams {
  const uint16_t* x;
  int64_t rows, cols, ld;  // cols % 32 == 0
  uint8_t* codes;
  int64_t ld_codes;
  uint8_t* scales;  // [rows][cols / 32] or 128x4 tiles over cols / 32 scale columns
  uint8_t* choice;  // optional, [rows][cols / 32]
  int codes16;      // codes 16-byte aligned with ld_codes % 16 == 0
  int layout;       // fos_sf_layout
};

// max |x| of 16 bf16 values held as 8 words, NaN-propagating: a NaN input
// gives NaN, an infinity gives infinity (the sign bit of the bf16 maxima is
// junk from xorsign and is dropped).
__device__ __forceinline__ float absmax16_bf16_nan(const uint32_t (&w)[8]) {
  uint32_t m[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[k]) : "r"(w[2 * k]), "r"(w[2 * k + 1]));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(m[1]));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[2]) : "r"(m[2]), "r"(m[3]));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(m[2]));
  return max_nan_f32(fabsf(__uint_as_float(m[0] << 16)), fabsf(__uint_as_float(m[0] & 0xFFFF0000u)));
}

// floor(log2 a) for a finite float a > 0, from its bits (exact).
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t b = __float_as_uint(a);
  const int ef = (int)(b >> 23);
  if (ef != 0) return ef - 127;
  return (31 - __clz((int)b)) - 149;  // subnormal: a = mantissa * 2^-149
}

// 2^-X as a float for X in [-127, 126] (always a normal number).
__device__ __forceinline__ float exp2_neg(int X) { return __uint_as_float((uint32_t)(127 - X) << 23); }

// One candidate on a 32-value block: its 16 code bytes (as 4 words) and S.
__device__ __forceinline__ float mx_candidate(const uint64_t (&yp)[16], float inv, uint32_t (&w)[4]) {
  const uint64_t inv2 = pack_f2(inv, inv);
  float S = 0.0f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint64_t acc = 0ull;
    const uint64_t a[4] = {yp[8 * h], yp[8 * h + 1], yp[8 * h + 2], yp[8 * h + 3]};
    const uint64_t b[4] = {yp[8 * h + 4], yp[8 * h + 5], yp[8 * h + 6], yp[8 * h + 7]};
    w[2 * h] = cand_rne8(a, inv2, acc);
    w[2 * h + 1] = cand_rne8(b, inv2, acc);
    const F2 e = unpack_f2(acc);
    const float Sh = __fadd_rn(e.x, e.y);
    S = h ? __fadd_rn(S, Sh) : Sh;
  }
  return S;
}

template <int RULE>
__global__ void __launch_bounds__(256) quant_mx_kernel(MxParams p) {
  const int64_t nb = p.cols >> 5;
  const bool tiled = p.layout == FOS_SF_SWIZZLED_128x4;
  const int64_t n_ct = (nb + 3) >> 2;  // 4-scale column tiles
  const int64_t n = tiled ? (((p.rows + 127) >> 7) * n_ct) << 9 : p.rows * nb;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    int64_t r, b;
    if (tiled) {
      // byte t of the tiles: tile t/512, and inside it (r%32)*16 + ((r%128)/32)*4 + b%4
      const int64_t tile = t >> 9, w = t & 511, rt = tile / n_ct;
      r = (rt << 7) + (((w >> 2) & 3) << 5) + (w >> 4);
      b = ((tile - rt * n_ct) << 2) + (w & 3);
      if (r >= p.rows || b >= nb) {
        p.scales[t] = 0;
        continue;
      }
    } else {
      r = t / nb;
      b = t - r * nb;
    }
    const uint4* src = reinterpret_cast<const uint4*>(p.x + r * p.ld + b * 32);
    uint32_t wv[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = __ldg(src + k);
      wv[4 * k] = v.x;
      wv[4 * k + 1] = v.y;
      wv[4 * k + 2] = v.z;
      wv[4 * k + 3] = v.w;
    }
    const uint32_t lo8[8] = {wv[0], wv[1], wv[2], wv[3], wv[4], wv[5], wv[6], wv[7]};
    const uint32_t hi8[8] = {wv[8], wv[9], wv[10], wv[11], wv[12], wv[13], wv[14], wv[15]};
    const float a = max_nan_f32(absmax16_bf16_nan(lo8), absmax16_bf16_nan(hi8));
    // a block holding a NaN or an infinity gets the E8M0 NaN scale 0xFF (its
    // every value decodes to NaN) with zero codes
    const bool finite = a <= FLT_MAX;
    int X6 = -127, X4 = -127;
    if (a > 0.0f) {
      const int e = floor_log2(a);
      X6 = max(-127, e - 2);
      X4 = max(-127, e - 1);
    }
    uint64_t yp[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) yp[k] = bf16x2_to_f32x2(wv[k]);
    uint32_t c6[4] = {0u, 0u, 0u, 0u}, c4[4] = {0u, 0u, 0u, 0u};
    float S6 = 0.0f, S4 = 0.0f;
    if (RULE != FOS_SCALE_4) S6 = mx_candidate(yp, exp2_neg(X6), c6);
    if (RULE != FOS_SCALE_6) S4 = mx_candidate(yp, exp2_neg(X4), c4);
    const float S4u = X4 > X6 ? __fmul_rn(S4, 4.0f) : S4;
    const bool four = finite && ((RULE == FOS_SCALE_4) || (RULE == FOS_SCALE_4OVER6 && S4u < S6));
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) c[k] = finite ? (four ? c4[k] : c6[k]) : 0u;
    uint8_t* dst = p.codes + r * p.ld_codes + b * 16;
    if (p.codes16) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(c[0], c[1], c[2], c[3]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) reinterpret_cast<uint32_t*>(dst)[k] = c[k];
    }
    p.scales[t] = finite ? (uint8_t)((four ? X4 : X6) + 127) : (uint8_t)0xFF;
    if (p.choice) p.choice[r * nb + b] = four ? 1 : 0;
  }
}

struct MxDequantParams {
  const uint8_t* codes;
  const uint8_t* scales;
  int64_t rows, cols, ld_codes, ld_out;
  void* out;
  int layout;
};

// x_hat = g * 2^X (exact in FP32; bf16 output is that value rounded to
// nearest even).
template <bool BF16>
__global__ void __launch_bounds__(256) dequant_mx_kernel(MxDequantParams p) {
  const int64_t nb = p.cols >> 5;
  const int64_t n = p.rows * nb;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / nb, b = t - r * nb;
    const int X = (int)p.scales[sf_off(r, b, nb, p.layout)] - 127;
    // 2^X: normal for X >= -126; 2^-127 is the subnormal 0x00400000; byte
    // 0xFF is the NaN scale (every value of the block NaN)
    const float s = X == 128 ? __uint_as_float(0x7FC00000u)
                  : X >= -126 ? __uint_as_float((uint32_t)(X + 127) << 23) : __uint_as_float(0x00400000u);
    const uint8_t* cw = p.codes + r * p.ld_codes + b * 16;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const F2 g = e2m1x2_decode(cw[k]);
      const float v0 = __fmul_rn(g.x, s), v1 = __fmul_rn(g.y, s);
      const int64_t o = r * p.ld_out + b * 32 + 2 * k;
      if (BF16) {
        reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(v0);
        reinterpret_cast<__nv_bfloat16*>(p.out)[o + 1] = __float2bfloat16_rn(v1);
      } else {
        reinterpret_cast<float*>(p.out)[o] = v0;
        reinterpret_cast<float*>(p.out)[o + 1] = v1;
      }
    }
  }
}

int mx_grid(int64_t n_blocks) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t g = (n_blocks + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace
}  // namespace fos

extern "C" {

fos_status fos_mxfp4_sf_bytes(int64_t rows, int64_t cols, int32_t sf_layout, size_t* bytes) {
  if (!bytes || rows < 0 || cols < 0 || cols % 32 != 0) return FOS_ERR_INVALID_ARG;
  if (sf_layout != FOS_SF_SWIZZLED_128x4 && sf_layout != FOS_SF_ROWMAJOR) return FOS_ERR_INVALID_ARG;
  const int64_t nb = cols / 32;
  *bytes = sf_layout == FOS_SF_ROWMAJOR ? (size_t)(rows * nb)
                                        : (size_t)(((rows + 127) / 128) * 128 * ((nb + 3) / 4) * 4);
  return FOS_OK;
}

fos_status fos_quantize_mxfp4(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int32_t scale_rule,
                              int32_t sf_layout, uint8_t* codes, int64_t ld_codes, uint8_t* scales,
                              uint8_t* choice, cudaStream_t stream) {
  using fos::aligned;
  if (rows < 0 || cols < 0 || cols % 32 != 0 || ld_x < cols || ld_x % 8 != 0) return FOS_ERR_INVALID_ARG;
  if (scale_rule < FOS_SCALE_4OVER6 || scale_rule > FOS_SCALE_4) return FOS_ERR_INVALID_ARG;
  if (sf_layout != FOS_SF_SWIZZLED_128x4 && sf_layout != FOS_SF_ROWMAJOR) return FOS_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FOS_OK;
  if (!x || !aligned(x, 16) || !codes || !scales) return FOS_ERR_INVALID_ARG;
  if (ld_codes < cols / 2 || ld_codes % 4 != 0 || !aligned(codes, 4)) return FOS_ERR_INVALID_ARG;
  fos::MxParams p{};
  p.x = static_cast<const uint16_t*>(x);
  p.rows = rows;
  p.cols = cols;
  p.ld = ld_x;
  p.codes = codes;
  p.ld_codes = ld_codes;
  p.scales = scales;
  p.choice = choice;
  p.codes16 = aligned(codes, 16) && ld_codes % 16 == 0;
  p.layout = sf_layout;
  const int g = fos::mx_grid(rows * (cols / 32));
  switch (scale_rule) {
    case FOS_SCALE_6: fos::quant_mx_kernel<FOS_SCALE_6><<<g, 256, 0, stream>>>(p); break;
    case FOS_SCALE_4: fos::quant_mx_kernel<FOS_SCALE_4><<<g, 256, 0, stream>>>(p); break;
    default: fos::quant_mx_kernel<FOS_SCALE_4OVER6><<<g, 256, 0, stream>>>(p); break;
  }
  return cudaGetLastError() == cudaSuccess ? FOS_OK : FOS_ERR_CUDA;
}

fos_status fos_dequantize_mxfp4(const fos_mxfp4_tensor* q, void* out, int32_t out_dtype, int64_t ld_out,
                                cudaStream_t stream) {
  if (!q || q->rows < 0 || q->cols < 0 || q->cols % 32 != 0 || q->ld_codes < q->cols / 2 || ld_out < q->cols)
    return FOS_ERR_INVALID_ARG;
  if (q->sf_layout != FOS_SF_SWIZZLED_128x4 && q->sf_layout != FOS_SF_ROWMAJOR) return FOS_ERR_INVALID_ARG;
  if (out_dtype != FOS_DTYPE_F32 && out_dtype != FOS_DTYPE_BF16) return FOS_ERR_INVALID_ARG;
  if (q->rows == 0 || q->cols == 0) return FOS_OK;
  if (!q->codes || !q->sf || !out) return FOS_ERR_INVALID_ARG;
  if (!fos::aligned(out, out_dtype == FOS_DTYPE_F32 ? 4 : 2)) return FOS_ERR_INVALID_ARG;
  fos::MxDequantParams p{q->codes, q->sf, q->rows, q->cols, q->ld_codes, ld_out, out, q->sf_layout};
  const int g = fos::mx_grid(q->rows * (q->cols / 32));
  if (out_dtype == FOS_DTYPE_BF16)
    fos::dequant_mx_kernel<true><<<g, 256, 0, stream>>>(p);
  else
    fos::dequant_mx_kernel<false><<<g, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? FOS_OK : FOS_ERR_CUDA;
}

}  // extern "C"
