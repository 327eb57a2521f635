// Device building blocks for the NVFP4 Four Over Six quantizer (sm_103a).
//
// Every floating-point step that decides a code is written with an explicit
// rounding (the __f*_rn intrinsics, or PTX .rn instructions) and the library is
// compiled with --fmad=false, so no expression is contracted behind our back.
#pragma once

#include <cfloat>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fos {

// ---------------------------------------------------------------- Philox
// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11): each round multiplies words 0 and 2 by
// two fixed odd multipliers, exchanges the high halves with words 1 and 3 and
// the round key; the key advances by two Weyl constants per round.
struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                       uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
    uint32_t h0 = __umulhi(m0, c0), l0 = m0 * c0;
    uint32_t h1 = __umulhi(m1, c2), l1 = m1 * c2;
    uint32_t n0 = h1 ^ c1 ^ k0;
    uint32_t n2 = h0 ^ c3 ^ k1;
    c0 = n0;
    c1 = l1;
    c2 = n2;
    c3 = l0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return {c0, c1, c2, c3};
}

// RHT sign vector of a tensor: bit j of word 0 of Philox(counter (0,0,0,1),
// key = hadamard seed); bit j set means s_j = -1.
__device__ __forceinline__ uint32_t rht_sign_mask(uint32_t k0, uint32_t k1) {
  return philox10(0u, 0u, 0u, 1u, k0, k1).x & 0xFFFFu;
}

// Stochastic-rounding words for the 4 consecutive source elements starting at
// index i0 (i0 % 4 == 0): word (i mod 4) of Philox(counter = i/4, key = seed).
__device__ __forceinline__ U4 sr_words4(uint64_t i0, uint32_t k0, uint32_t k1) {
  uint64_t blk = i0 >> 2;
  return philox10((uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u, k0, k1);
}

// ------------------------------------------------------- packed FP32 ops
// Two independent IEEE round-to-nearest operations per instruction.
struct F2 {
  float x, y;
};

__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
  F2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ F2 add2(F2 a, F2 b) {
  F2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ F2 sub2(F2 a, F2 b) {
  F2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) {
  F2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// ------------------------------------------------------------- E2M1 / E4M3
// Hardware conversions.  For the two-element forms the first source operand
// goes to the upper half of the result, so (lo, hi) is passed as (hi, lo).

// codes of (lo, hi): low nibble = E2M1_rne_satfinite(lo), high nibble = ...(hi)
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(lo), "f"(hi));
  return r;
}

// One byte of two codes -> (residual lo, residual hi) = (qlo - g(lo code),
// qhi - g(hi code)), each one FP32 rounding; also returns the byte.  The code
// values are decoded exactly to f16 and subtracted with a mixed-precision FMA
// (g * -1 + q).
__device__ __forceinline__ uint32_t e2m1x2_residual(float qlo, float qhi, float& rlo, float& rhi) {
  uint32_t byte;
  asm("{\n\t.reg .b8 c;\n\t.reg .b32 h;\n\t.reg .b16 hl, hh, m1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c, %4, %3;\n\t"
      "cvt.rn.f16x2.e2m1x2 h, c;\n\t"
      "mov.b32 {hl, hh}, h;\n\t"
      "mov.b16 m1, 0xBC00;\n\t"
      "fma.rn.f32.f16 %0, hl, m1, %3;\n\t"
      "fma.rn.f32.f16 %1, hh, m1, %4;\n\t"
      "cvt.u32.u8 %2, c;\n\t}"
      : "=f"(rlo), "=f"(rhi), "=r"(byte)
      : "f"(qlo), "f"(qhi));
  return byte;
}

// Value of each nibble of a code byte as two floats (exact).
__device__ __forceinline__ F2 e2m1x2_decode(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b8 c;\n\tcvt.u8.u32 c, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, c;\n\t}" : "=r"(h) : "r"(byte));
  F2 d;
  d.x = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
  d.y = __half2float(__ushort_as_half((unsigned short)(h >> 16)));
  return d;
}

// (lo, hi) -> 16 bits: low byte E4M3(lo), high byte E4M3(hi); RNE, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(lo), "f"(hi));
  return r;
}

// 16 bits of two E4M3 bytes -> their exact values.
__device__ __forceinline__ F2 e4m3x2_decode(uint32_t pair) {
  uint32_t h;
  unsigned short p = (unsigned short)pair;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(p));
  F2 d;
  d.x = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
  d.y = __half2float(__ushort_as_half((unsigned short)(h >> 16)));
  return d;
}

// --------------------------------------------------------------- bf16 unpack
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 256-bit read-only load (sm_100+).
__device__ __forceinline__ void ldg256(const void* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                 "=r"(w[7])
               : "l"(p));
}

__device__ __forceinline__ void ldg128x2(const void* p, uint32_t (&w)[8]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  uint4 a = __ldg(q), b = __ldg(q + 1);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// ------------------------------------------------------------------- RHT
// In place on 16 values: sign flips (bit j of mask), butterflies of stride
// 1, 2, 4, 8 -- (a, b) -> (a + b, a - b) -- then an exact scaling by 1/4.
__device__ __forceinline__ void rht16(float (&v)[16], uint32_t mask) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if ((mask >> j) & 1u) v[j] = -v[j];
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    float a = v[j], b = v[j + 1];
    v[j] = __fadd_rn(a, b);
    v[j + 1] = __fsub_rn(a, b);
  }
#pragma unroll
  for (int h = 2; h < 16; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      if (j & h) continue;
      F2 a{v[j], v[j + 1]}, b{v[j + h], v[j + h + 1]};
      F2 s = add2(a, b), d = sub2(a, b);
      v[j] = s.x; v[j + 1] = s.y;
      v[j + h] = d.x; v[j + h + 1] = d.y;
    }
  }
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    F2 s = mul2(F2{v[j], v[j + 1]}, F2{0.25f, 0.25f});
    v[j] = s.x;
    v[j + 1] = s.y;
  }
}

// ------------------------------------------------------------ per tensor
struct TensorConsts {
  float s_t, k6, k4;
};

// s_t = amax / 2688; k_M = 1 / (M * s_t) (0 when M * s_t is 0).
__device__ __forceinline__ TensorConsts tensor_consts(float amax) {
  TensorConsts t;
  t.s_t = __fdiv_rn(amax, 2688.0f);
  float t6 = __fmul_rn(6.0f, t.s_t), t4 = __fmul_rn(4.0f, t.s_t);
  t.k6 = t6 > 0.0f ? __frcp_rn(t6) : 0.0f;
  t.k4 = t4 > 0.0f ? __frcp_rn(t4) : 0.0f;
  return t;
}

// ------------------------------------------------------------ per block
// The two candidate scales of a block with magnitude max `ab`.
struct Cands {
  uint32_t sf6, sf4;   // E4M3 bytes
  float eff6, eff4;    // float(sf) * s_t
  float inv6, inv4;    // min(1/eff, FLT_MAX), or 0 when sf == 0
};

__device__ __forceinline__ Cands candidates(float ab, const TensorConsts& tc) {
  Cands c;
  uint32_t pair = e4m3x2(__fmul_rn(ab, tc.k6), __fmul_rn(ab, tc.k4));
  c.sf6 = pair & 0xFFu;
  c.sf4 = pair >> 8;
  F2 v = e4m3x2_decode(pair);
  F2 e = mul2(v, F2{tc.s_t, tc.s_t});
  c.eff6 = e.x;
  c.eff4 = e.y;
  c.inv6 = c.sf6 ? fminf(__frcp_rn(c.eff6), FLT_MAX) : 0.0f;
  c.inv4 = c.sf4 ? fminf(__frcp_rn(c.eff4), FLT_MAX) : 0.0f;
  return c;
}

// Fixed-order sum of 16 squares: FMA chains over even and odd positions, then one add.
__device__ __forceinline__ float sumsq16(const float (&r)[16]) {
  F2 acc{0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < 8; ++k) acc = fma2(F2{r[2 * k], r[2 * k + 1]}, F2{r[2 * k], r[2 * k + 1]}, acc);
  return __fadd_rn(acc.x, acc.y);
}

// RNE codes of one candidate for 16 values: returns the scaled-domain sum of
// squared residuals and the 8 code bytes in (lo, hi) words.
__device__ __forceinline__ float cand_rne16(const float (&y)[16], float inv, uint32_t& lo, uint32_t& hi) {
  F2 acc{0.0f, 0.0f};
  uint32_t b[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    F2 q = mul2(F2{y[2 * k], y[2 * k + 1]}, F2{inv, inv});
    F2 r;
    b[k] = e2m1x2_residual(q.x, q.y, r.x, r.y);
    acc = fma2(r, r, acc);
  }
  lo = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  hi = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
  return __fadd_rn(acc.x, acc.y);
}

// Stochastic rounding of one value to an E2M1 grid magnitude: lo <= a < hi,
// up iff u < (a - lo) / (hi - lo) with u = (w >> 8) * 2^-24 (all exact).
__device__ __forceinline__ float sr_mag(float a, uint32_t w) {
  float step = a < 2.0f ? 0.5f : (a < 4.0f ? 1.0f : 2.0f);
  float inv_step = a < 2.0f ? 2.0f : (a < 4.0f ? 1.0f : 0.5f);
  float lo = a < 4.0f ? __fmul_rn(floorf(__fmul_rn(a, inv_step)), step) : 4.0f;
  float p = __fmul_rn(__fsub_rn(a, lo), inv_step);
  float u = __fmul_rn((float)(w >> 8), 5.9604644775390625e-8f);  // 2^-24
  float g = (u < p) ? __fadd_rn(lo, step) : lo;
  return a >= 6.0f ? 6.0f : g;
}

// Stochastic-rounding codes of one candidate (w: the 16 elements' words).
__device__ __forceinline__ float cand_sr16(const float (&y)[16], float inv, const uint32_t (&w)[16], uint32_t& lo,
                                           uint32_t& hi) {
  F2 acc{0.0f, 0.0f};
  uint32_t b[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    F2 q = mul2(F2{y[2 * k], y[2 * k + 1]}, F2{inv, inv});
    float a0 = fabsf(q.x), a1 = fabsf(q.y);
    float g0 = sr_mag(a0, w[2 * k]), g1 = sr_mag(a1, w[2 * k + 1]);
    // the grid value with q's sign converts exactly
    b[k] = e2m1x2(copysignf(g0, q.x), copysignf(g1, q.y));
    F2 r = sub2(F2{a0, a1}, F2{g0, g1});
    acc = fma2(r, r, acc);
  }
  lo = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  hi = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
  return __fadd_rn(acc.x, acc.y);
}

// Scale-factor byte offset of block (r, c) of a matrix with nb scale columns.
__device__ __forceinline__ int64_t sf_off(int64_t r, int64_t c, int64_t nb, int layout) {
  if (layout == 1) return r * nb + c;
  int64_t n_ct = (nb + 3) >> 2;
  return (((r >> 7) * n_ct + (c >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (c & 3);
}

}  // namespace fos
