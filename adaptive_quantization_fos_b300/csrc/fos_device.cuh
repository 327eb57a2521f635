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

// Four pairs of signed grid values -> one word of E2M1 codes (byte k: pair k,
// the even element in the low nibble); exact for grid values.
__device__ __forceinline__ uint32_t e2m1x8(F2 g0, F2 g1, F2 g2, F2 g3) {
  uint32_t w;
  asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
      : "=r"(w)
      : "f"(g0.x), "f"(g0.y), "f"(g1.x), "f"(g1.y), "f"(g2.x), "f"(g2.y), "f"(g3.x), "f"(g3.y));
  return w;
}

// ------------------------------------------------ float pairs in 64 bits
// A value pair (element 2k in the low half) kept in one 64-bit register, the
// operand form of the packed f32x2 instructions.
__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ F2 unpack_f2(uint64_t v) {
  F2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(v));
  return d;
}

// Two bf16 values of one word -> their exact FP32 pair, as x * 1 + (-0) in
// the mixed-precision FMA (exact for every finite x, signed zeros kept); this
// keeps the conversion on the FMA pipe, off the busier integer/ALU pipe.
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
  uint64_t r;
  asm("{\n\t.reg .b16 l, h, one;\n\t.reg .f32 a, b, z;\n\t"
      "mov.b32 {l, h}, %1;\n\tmov.b16 one, 0x3F80;\n\tmov.f32 z, 0f80000000;\n\t"
      "fma.rn.f32.bf16 a, l, one, z;\n\tfma.rn.f32.bf16 b, h, one, z;\n\tmov.b64 %0, {a, b};\n\t}"
      : "=l"(r)
      : "r"(w));
  return r;
}

// One candidate on 8 consecutive values (4 pairs y[k]): q = y * inv (packed),
// RNE E2M1 codes of q (returned as one word, byte k = codes of pair k), and
// the squared residuals (q - g)^2 added to the two running sums in acc
// (even positions in the low half), one packed FMA per pair in pair order.
__device__ __forceinline__ uint32_t cand_rne8(const uint64_t (&y)[4], uint64_t inv2, uint64_t& acc) {
  uint32_t word;
  asm("{\n\t"
      ".reg .b64 q0, q1, q2, q3, r0, r1, r2, r3;\n\t"
      ".reg .f32 x0, x1, x2, x3, x4, x5, x6, x7, e0, e1, e2, e3, e4, e5, e6, e7;\n\t"
      ".reg .b8 c0, c1, c2, c3;\n\t"
      ".reg .b32 h0, h1, h2, h3;\n\t"
      ".reg .b16 l0, g0, l1, g1, l2, g2, l3, g3, m1;\n\t"
      "mul.rn.f32x2 q0, %2, %6;\n\t"
      "mul.rn.f32x2 q1, %3, %6;\n\t"
      "mul.rn.f32x2 q2, %4, %6;\n\t"
      "mul.rn.f32x2 q3, %5, %6;\n\t"
      "mov.b64 {x0, x1}, q0;\n\tmov.b64 {x2, x3}, q1;\n\tmov.b64 {x4, x5}, q2;\n\tmov.b64 {x6, x7}, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, x1, x0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, x3, x2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, x5, x4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, x7, x6;\n\t"
      "cvt.rn.f16x2.e2m1x2 h0, c0;\n\t"
      "cvt.rn.f16x2.e2m1x2 h1, c1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h2, c2;\n\t"
      "cvt.rn.f16x2.e2m1x2 h3, c3;\n\t"
      "mov.b32 {l0, g0}, h0;\n\tmov.b32 {l1, g1}, h1;\n\tmov.b32 {l2, g2}, h2;\n\tmov.b32 {l3, g3}, h3;\n\t"
      "mov.b16 m1, 0xBC00;\n\t"
      "fma.rn.f32.f16 e0, l0, m1, x0;\n\t"
      "fma.rn.f32.f16 e1, g0, m1, x1;\n\t"
      "fma.rn.f32.f16 e2, l1, m1, x2;\n\t"
      "fma.rn.f32.f16 e3, g1, m1, x3;\n\t"
      "fma.rn.f32.f16 e4, l2, m1, x4;\n\t"
      "fma.rn.f32.f16 e5, g2, m1, x5;\n\t"
      "fma.rn.f32.f16 e6, l3, m1, x6;\n\t"
      "fma.rn.f32.f16 e7, g3, m1, x7;\n\t"
      "mov.b64 r0, {e0, e1};\n\tmov.b64 r1, {e2, e3};\n\tmov.b64 r2, {e4, e5};\n\tmov.b64 r3, {e6, e7};\n\t"
      "fma.rn.f32x2 %1, r0, r0, %1;\n\t"
      "fma.rn.f32x2 %1, r1, r1, %1;\n\t"
      "fma.rn.f32x2 %1, r2, r2, %1;\n\t"
      "fma.rn.f32x2 %1, r3, r3, %1;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
      : "=r"(word), "+l"(acc)
      : "l"(y[0]), "l"(y[1]), "l"(y[2]), "l"(y[3]), "l"(inv2));
  return word;
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

// ------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of the given parity; false once timeout_ns have passed.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 15u) == 0 && globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// Contiguous global -> shared copy on the async (bulk) path, with an L2
// eviction policy (from createpolicy) for the source lines; the calling
// thread arrives on the mbarrier and completion is counted there in bytes.
// Addresses 16-byte aligned, size % 16 == 0.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 32 bytes of read-only global data with an L2 eviction policy.
__device__ __forceinline__ void ldg256_hint(const void* p, uint32_t (&w)[8], uint64_t policy) {
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(p), "l"(policy));
}

__device__ __forceinline__ void ldg128x2_hint(const void* p, uint32_t (&w)[8], uint64_t policy) {
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.b32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "l"(p), "l"(policy));
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.b32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(static_cast<const char*>(p) + 16), "l"(policy));
}

// Grid-wide barrier for a launch whose CTAs are all resident (cooperative
// launch) on an arrival counter that is zero when the launch starts (the host
// clears it in stream order before the launch).  Called by one thread per
// CTA; the wait gives up (returns false) after timeout_ns.
__device__ __forceinline__ bool grid_barrier(unsigned int* word, unsigned int n, uint64_t timeout_ns) {
  __threadfence();
  atomicAdd(word, 1u);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    unsigned int cur;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(cur) : "l"(word) : "memory");
    if (cur >= n) break;
    if ((i & 15u) == 15u && globaltimer_ns() - t0 > timeout_ns) return false;
  }
  __threadfence();
  return true;
}

// ------------------------------------------------------------------- RHT
// In place on 16 values: the butterflies of stride 1, 2, 4, 8 --
// (a, b) -> (a + b, a - b) -- without the final scaling by 1/4.
__device__ __forceinline__ void butterflies16(float (&v)[16]) {
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
}

// In place on 16 values: sign flips (bit j of mask), the butterflies, then an
// exact scaling by 1/4.
__device__ __forceinline__ void rht16(float (&v)[16], uint32_t mask) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if ((mask >> j) & 1u) v[j] = -v[j];
  butterflies16(v);
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    F2 s = mul2(F2{v[j], v[j + 1]}, F2{0.25f, 0.25f});
    v[j] = s.x;
    v[j + 1] = s.y;
  }
}

// ------------------------------------------------------------ per tensor
// A block's candidate scale maps its maximum a_b to M = 6 or 4:
// sf_M = E4M3(a_b / t_M) with t_M = M * s_t, the product and the quotient each
// rounded once in FP32.  The quotient is formed without a division, by one
// correction step after a reciprocal multiply (Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): with k = RN(1/t) and q = RN(a * k) within an ulp of a/t,
// the residual r = a - q*t is exact in one FMA and RN(q + r*k) is RN(a/t),
// provided nothing underflows.  To keep every quantity normal, a_b and t_M are
// first scaled by P = 2^sigma with s_t * P in [1, 2) (sigma clamped to
// [-126, 126]); the scaling is exact and leaves the quotient unchanged.  a_b * P
// is clamped to 4096 * t_4 * P (a quotient of 1024 or more saturates to 448
// either way), so a caller-supplied amax below a block's maximum cannot
// overflow the steps.
struct TensorConsts {
  float s_t;
  float p;          // 2^sigma
  float nt6, nt4;   // -t_M * P
  float k6, k4;     // RN(1 / (t_M * P)), 0 when t_M is 0
  float clamp;      // 4096 * t_4 * P
};

// s_t = amax / 2688 and the constants of the candidate-scale quotients.
__device__ __forceinline__ TensorConsts tensor_consts(float amax) {
  TensorConsts t;
  t.s_t = __fdiv_rn(amax, 2688.0f);
  const int e = (int)((__float_as_uint(t.s_t) >> 23) & 0xFFu) - 127;  // exponent of a normal s_t
  int sigma = t.s_t > 0.0f ? -e : 0;
  sigma = sigma > 126 ? 126 : (sigma < -126 ? -126 : sigma);  // a subnormal s_t gives 126
  t.p = __uint_as_float((uint32_t)(sigma + 127) << 23);
  const float T6 = __fmul_rn(__fmul_rn(6.0f, t.s_t), t.p), T4 = __fmul_rn(__fmul_rn(4.0f, t.s_t), t.p);
  t.nt6 = -T6;
  t.nt4 = -T4;
  t.k6 = T6 > 0.0f ? __frcp_rn(T6) : 0.0f;
  t.k4 = T4 > 0.0f ? __frcp_rn(T4) : 0.0f;
  t.clamp = __fmul_rn(4096.0f, T4);
  return t;
}

// The two candidate scale bytes of a block with maximum ab: low byte
// E4M3(ab / t_6), high byte E4M3(ab / t_4), both quotients correctly rounded.
__device__ __forceinline__ uint32_t candidate_scales(float ab, const TensorConsts& tc) {
  const float a = fminf(__fmul_rn(ab, tc.p), tc.clamp);
  const F2 aa{a, a}, k{tc.k6, tc.k4};
  const F2 q = mul2(aa, k);
  const F2 r = fma2(q, F2{tc.nt6, tc.nt4}, aa);  // a - q * t, exact
  const F2 raw = fma2(r, k, q);
  return e4m3x2(raw.x, raw.y);
}

// Fixed-order sum of 16 squares: FMA chains over even and odd positions, then one add.
__device__ __forceinline__ float sumsq16(const float (&r)[16]) {
  F2 acc{0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < 8; ++k) acc = fma2(F2{r[2 * k], r[2 * k + 1]}, F2{r[2 * k], r[2 * k + 1]}, acc);
  return __fadd_rn(acc.x, acc.y);
}

// Stochastic rounding to E2M1 grid magnitudes, two values at a time.
//
// For a in [0, 6] let step be the grid spacing of a's interval (0.5 below 2,
// 1 in [2, 4), 2 in [4, 6]) and t = a / step (exact: step is a power of 2),
// so the interval's ends are lo = floor(t) * step and hi = lo + step.  The
// rule "up iff u < p" with p = t - floor(t) and u = n * 2^-24 (n = w >> 8)
// picks ceil(t - u) * step: t - u lies in (floor(t), floor(t) + 1) when
// u < p, and in (floor(t) - 1, floor(t)] otherwise.  t - u is one FMA rounded
// toward +inf, and ceil(.) the round-up addition of M = 1.5 * 2^23, then M
// subtracted: t - u lies in (-1, 4), so M + (t - u) stays inside
// [2^23, 2^24), where the spacing of floats is exactly 1.  Both roundings
// are exact for ceil's purpose: rounding up never passes an integer, and the
// integers involved are floats.
// Evaluated scaled by step: rounding toward +inf commutes with multiplying
// by a power of two while the results stay normal, so
// fma.rp(n, -step * 2^-24, a) = step * fma.rp(-n, 2^-24, t), and the
// round-up addition of step * M lands on multiples of step.  (With n = 0
// nothing is rounded; with n >= 1 a nonzero a - n * step * 2^-24 is a
// multiple of ulp(a) >= 2^-49, since a >= 2^-26 whenever it comes that
// close to n * step * 2^-24 >= 2^-25: never subnormal.)  The products
// -step * 2^-24 and step * M come from P = 2^e (e the exponent of
// max(a, 1), step = P / 2) by two exact multiplies, so t, 1/step and the
// final multiply by step are not needed.
// a >= 6 is clamped to 6 first (t = 3 gives 6 for every u), as the rule
// saturates.
__device__ __forceinline__ F2 sr_mag2(F2 aq, F2 n) {
  const float a0 = fminf(aq.x, 6.0f), a1 = fminf(aq.y, 6.0f);
  const F2 P{__uint_as_float(__float_as_uint(fmaxf(a0, 1.0f)) & 0x7F800000u),
             __uint_as_float(__float_as_uint(fmaxf(a1, 1.0f)) & 0x7F800000u)};
  F2 g;
  asm("{\n\t.reg .b64 rn, rp, ra, rk, rs, rm, rx, rc;\n\t"
      "mov.b64 rn, {%2, %3};\n\tmov.b64 rp, {%4, %5};\n\tmov.b64 ra, {%6, %7};\n\t"
      "mov.b64 rk, {%8, %8};\n\tmov.b64 rm, {%9, %9};\n\t"
      "mul.rn.f32x2 rs, rp, rk;\n\t"    // -step * 2^-24
      "mul.rn.f32x2 rm, rp, rm;\n\t"    // step * M
      "fma.rp.f32x2 rx, rn, rs, ra;\n\t"
      "add.rp.f32x2 rc, rx, rm;\n\t"
      "sub.rn.f32x2 rc, rc, rm;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "=f"(g.x), "=f"(g.y)
      : "f"(n.x), "f"(n.y), "f"(P.x), "f"(P.y), "f"(a0), "f"(a1), "f"(-2.98023223876953125e-8f),
        "f"(6291456.0f));
  return g;
}

// The draw of one element: n = w >> 8 of its Philox word, as a float (exact:
// n < 2^24).  Both candidates round with the same u = n * 2^-24.
__device__ __forceinline__ float sr_draw(uint32_t w) { return (float)(w >> 8); }

// A block's magnitudes |y| and signs (+-1.0 with y's sign bit) as pairs,
// once per block: both stochastic-rounding candidates use them.
__device__ __forceinline__ void sr_split16(const uint64_t (&yp)[8], F2 (&ay)[8], F2 (&sg)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const F2 v = unpack_f2(yp[k]);
    ay[k] = F2{fabsf(v.x), fabsf(v.y)};
    sg[k] = F2{copysignf(1.0f, v.x), copysignf(1.0f, v.y)};
  }
}

// Stochastic-rounding codes of one candidate (ay, sg from sr_split16; n the
// elements' draws, sr_draw).  |q| = |y| * inv exactly (inv > 0), and the
// signed grid value g * sign carries q's sign, zeros included, as the codes
// need.
__device__ __forceinline__ float cand_sr16(const F2 (&ay)[8], const F2 (&sg)[8], float inv, const float (&n)[16],
                                           uint32_t& lo, uint32_t& hi) {
  F2 acc{0.0f, 0.0f};
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // each code word as soon as its 4 pairs are done
    F2 gs[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = 4 * h + j;
      const F2 aq = mul2(ay[k], F2{inv, inv});
      const F2 g = sr_mag2(aq, F2{n[2 * k], n[2 * k + 1]});
      gs[j] = mul2(g, sg[k]);
      const F2 r = sub2(aq, g);
      acc = fma2(r, r, acc);
    }
    (h ? hi : lo) = e2m1x8(gs[0], gs[1], gs[2], gs[3]);
  }
  return __fadd_rn(acc.x, acc.y);
}

// Per-tensor table over the 128 non-negative finite E4M3 bytes b (0x7F is NaN
// and never produced): x = min(1/eff, FLT_MAX) (0 for b = 0) and y = eff*eff,
// eff = float(b) * s_t, each one IEEE rounding -- the candidate's reciprocal
// scale and the factor of its error, computed once per CTA instead of per block.
__device__ __forceinline__ void build_scale_table(float s_t, float2* tab) {
  for (int b = threadIdx.x; b < 128; b += blockDim.x) {
    const float v = e4m3x2_decode((uint32_t)b).x;
    const float eff = __fmul_rn(v, s_t);
    const float inv = b ? fminf(__frcp_rn(eff), FLT_MAX) : 0.0f;
    tab[b] = make_float2(inv, __fmul_rn(eff, eff));
  }
}

// max |x| of 16 bf16 values held as 8 words: max.xorsign.abs keeps the larger
// magnitude of each half (its sign bit is junk and is dropped at the end).
__device__ __forceinline__ float absmax16_bf16(const uint32_t (&w)[8]) {
  uint32_t m[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[k]) : "r"(w[2 * k]), "r"(w[2 * k + 1]));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(m[1]));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[2]) : "r"(m[2]), "r"(m[3]));
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(m[2]));
  return fmaxf(fabsf(__uint_as_float(m[0] << 16)), fabsf(__uint_as_float(m[0] & 0xFFFF0000u)));
}

// Scale-factor byte offset of block (r, c) of a matrix with nb scale columns.
__device__ __forceinline__ int64_t sf_off(int64_t r, int64_t c, int64_t nb, int layout) {
  if (layout == 1) return r * nb + c;
  int64_t n_ct = (nb + 3) >> 2;
  return (((r >> 7) * n_ct + (c >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (c & 3);
}

}  // namespace fos
