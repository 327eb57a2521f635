// Block-scaled NVFP4 GEMM on the fifth-generation tensor cores (sm_103a).
//
// C[m][n] = bf16( (s_tA * s_tB) * sum_k (gA[m,k] sfA[m,k/16]) (gB[n,k] sfB[n,k/16]) )
//
// This is the contraction of the quantized linear layer: "FP4" (Ultralytics
// glossary), "FP4 ile Çıkarım ve Eğitim", notes that FP4 matrix products
// accumulate at higher precision; here the products and the FP32 accumulation
// run in tcgen05.mma kind::mxf4nvf4 (E2M1 operands, one E4M3 scale per 16
// values along K, "scale_vec::4X"), with the accumulator in tensor memory.
//
// Structure (one persistent CTA per SM, static round-robin over output tiles):
//   warp 0      TMA producer: codes of A (128 x 256 values) and B (BN x 256)
//               per stage with 128-byte swizzle, plus the stage's scale bytes
//               (contiguous 512-byte chunks of the 128x4 layout) by bulk copy.
//   warp 1      allocates tensor memory; one thread issues 4 MMAs of K = 64 per
//               stage once the stage's codes and scales are in place;
//               tcgen05.commit frees the stage and, after the last stage,
//               signals the accumulator.
//   warps 2..   scales and epilogue: they write each stage's scale words into
//               tensor memory (tcgen05.st), and at the end of a tile each
//               reads 32 accumulator lanes x 128 columns into registers, hands
//               the accumulator back at once (so the next tile's MMAs start
//               while it stores), scales, rounds to bf16 and stores.
// The MXFP4 form (gemm_mxfp4_kernel) is the same kernel with E8M0 scales, one
// per 32 values: its 512-byte scale chunks each span 128 values of K (two MMA
// steps), and the staging warps give each 32-value scale to both 16-value
// halves it covers, so the MMA reads the same tensor-memory scale image.
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel records
// FOS_ERR_TIMEOUT, all roles stop, in-flight copies and MMAs are drained
// (again bounded) and the tensor memory is freed before the CTA exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>
#include <type_traits>

#include "fos.h"

namespace {

// ------------------------------------------------------------ constants
constexpr int kBM = 128;              // rows of A per tile (= tensor-memory lanes)
constexpr int kBKBytes = 128;         // codes bytes per row per stage (256 values)
constexpr int kKPerMma = 64;          // values of K per MMA
constexpr int kSfChunk = 512;         // scale bytes of 128 rows x 4 scales (64 NVFP4 / 128 MXFP4 values)
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait

template <int BN>
struct Cfg {
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr int kABytes = kBM * kBKBytes;
  static constexpr int kBBytes = BN * kBKBytes;
  static constexpr int kSfaBytes = 4 * kSfChunk;
  static constexpr int kSfbBytes = (BN / 128) * 4 * kSfChunk;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kEpiWarps = 4 * (BN / 128);
  static constexpr int kThreads = 32 * (2 + kEpiWarps);
  // tensor-memory columns: accumulator, then per stage 4 MMAs x (4 + BN/32)
  static constexpr int kSfaCols = 16;
  static constexpr int kSfbColsPerMma = BN / 32;
  static constexpr int kSfStageCols = kSfaCols + 4 * kSfbColsPerMma;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
  static_assert((4 * kStages + 5) * 8 <= 256, "barrier area");
  static_assert(kStageBytes % 1024 == 0, "stage buffers stay 1024-byte aligned");
  static_assert(BN + kStages * kSfStageCols <= (int)kTmemCols, "tensor memory budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct GemmArgs {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* sta;
  const float* stb;
  uint16_t* c;
  int64_t ldc;
  int32_t c32;           // C 32-byte aligned with ldc % 16 == 0: 32-byte stores
  int32_t m, n, k;       // k in values
  int32_t tiles_m, tiles_n, num_kb;
  int64_t sf_ktiles;     // 512-byte scale chunks per 128-row tile (K / 64 NVFP4, ceil(K / 128) MXFP4)
  int32_t* status;
  uint64_t timeout_ns;
  int32_t stall_test;    // 1: the producer never fills a stage (bounded-wait self test)
  int32_t pre_a;         // under programmatic launch: A's first stages before the wait (B's after)
};

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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

// Wait for the phase with the given parity to complete.  Gives up (returns
// false) when the wait outlasts timeout_ns or, if abort is not null, when
// another role has raised *abort.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          volatile int* abort) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (abort && *abort) return false;
      if (globaltimer() - t0 > timeout_ns) return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start >> 4 in bits 0-13, leading
// byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45, the fixed
// version 1 in 46-47, swizzle mode in 61-63 (2 = 128-byte, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46) | ((uint64_t)swizzle << 61);
}

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B (format 1), both
// K-major, N >> 3 at bit 17, the scale format at bit 23 (0: E4M3, 1: E8M0),
// M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t mma_idesc(int m, int n, bool e8m0 = false) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((e8m0 ? 1u : 0u) << 23) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// 32 lanes x 32 columns of 32-bit accumulator -> 32 registers per thread.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&v)[32], int off) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr + off));
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Registers -> tensor memory: lane L of the warp's quadrant writes its 8 (16)
// words to columns taddr .. taddr+7 (+15) of lane L.
__device__ __forceinline__ void tc_st8(uint32_t taddr, const uint4& a, const uint4& b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(a.x),
               "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint4& a, const uint4& b, const uint4& c,
                                       const uint4& d) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w), "r"(c.x), "r"(c.y), "r"(c.z),
      "r"(c.w), "r"(d.x), "r"(d.y), "r"(d.z), "r"(d.w)
      : "memory");
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// E8M0 scale words of one MXFP4 chunk row (4 scales of 32 values) for the
// MMA step `step` (0 or 1) of the two it spans: each 32-value scale serves
// both 16-value quarters of the step it covers, [s0 s0 s1 s1] or [s2 s2 s3 s3].
__device__ __forceinline__ uint4 mx_step_words(const uint4& w, int step) {
  const uint32_t sel = step ? 0x3322u : 0x1100u;
  return make_uint4(__byte_perm(w.x, 0u, sel), __byte_perm(w.y, 0u, sel), __byte_perm(w.z, 0u, sel),
                    __byte_perm(w.w, 0u, sel));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// 32 bytes to global memory with the streaming (evict-first) hint; p 32-byte aligned.
__device__ __forceinline__ void st_cs_v8(void* p, const uint4& a, const uint4& b) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
               "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// Programmatic dependent launch: wait until the kernel this launch depends on
// (the stream's previous one, when launched with programmatic serialization)
// has completed and its writes are visible; a no-op otherwise.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void raise_timeout(const GemmArgs& a, volatile int* abort) {
  *abort = 1;
  if (a.status) atomicExch(a.status, (int)FOS_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ kernel
// MX: E8M0 scales per 32 values (MXFP4) instead of E4M3 per 16 (NVFP4).
template <int BN, bool MX>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const GemmArgs& args) {
  using C = Cfg<BN>;
  // 512-byte scale chunks per 128 rows per stage, and those a stage of kkc MMA steps uses
  constexpr int kChunksPerStage = MX ? 2 : 4;
  auto n_chunks = [](int kkc) { return MX ? (kkc + 1) >> 1 : kkc; };
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  // bars[0, S): stage codes landed; [S, 2S): stage empty; 2S: acc full; 2S+1: acc empty;
  // 2S+2: drain; [2S+3, 3S+3): stage scales in tensor memory; [3S+3, 4S+3): stage scale
  // bytes landed
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 4 * C::kStages + 3);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4 * C::kStages + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * C::kStages);
  const uint32_t acc_empty = acc_full + 8u;
  const uint32_t drain_bar = acc_full + 16u;
  auto sf_ready = [&](int s) { return acc_full + 24u + 8u * s; };
  auto sf_full = [&](int s) { return acc_full + 24u + 8u * (C::kStages + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, C::kEpiWarps);
    mbar_init(drain_bar, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(sf_ready(s), C::kEpiWarps);
      mbar_init(sf_full(s), 1);
    }
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_tiles = args.tiles_m * args.tiles_n;
  const int kmma_total = args.k / kKPerMma;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool ok = true;
      // The operand that no earlier kernel of the stream writes (B, or A with
      // pre_a) is requested for the first tile's first stages before this
      // CTA waits for the previous kernel (the other operand's producer,
      // under programmatic dependent launch); the other operand follows the
      // wait.  Stage slots start empty, so these stages need no empty-barrier
      // wait.
      const int pre = (!args.stall_test && (int)blockIdx.x < n_tiles) ? min(C::kStages, args.num_kb) : 0;
      {
        const int mb = (int)blockIdx.x % args.tiles_m, nb = (int)blockIdx.x / args.tiles_m;
        int halves = 0;
        for (int h = 0; h < BN / 128; ++h)
          if ((nb * (BN / 128) + h) * 128 < args.n) ++halves;
        auto load_b = [&](int kb) {
          const int nch = n_chunks(min(4, kmma_total - 4 * kb));
          const uint32_t st = smem_u32(smem + kb * C::kStageBytes);
          const uint32_t sfa_dst = st + C::kABytes + C::kBBytes;
          for (int h = 0; h < halves; ++h)
            bulk_load(sfa_dst + C::kSfaBytes + h * 4 * kSfChunk,
                      args.sfb + ((int64_t)(nb * (BN / 128) + h) * args.sf_ktiles + kChunksPerStage * kb) * kSfChunk,
                      nch * kSfChunk, sf_full(kb));
          tma_load_2d(st + C::kABytes, &tm_b, kb * kBKBytes, nb * BN, full_bar(kb));
        };
        auto load_a = [&](int kb) {
          const int nch = n_chunks(min(4, kmma_total - 4 * kb));
          const uint32_t st = smem_u32(smem + kb * C::kStageBytes);
          bulk_load(st + C::kABytes + C::kBBytes,
                    args.sfa + ((int64_t)mb * args.sf_ktiles + kChunksPerStage * kb) * kSfChunk, nch * kSfChunk,
                    sf_full(kb));
          tma_load_2d(st, &tm_a, kb * kBKBytes, mb * kBM, full_bar(kb));
        };
        for (int kb = 0; kb < pre; ++kb) {
          const int nch = n_chunks(min(4, kmma_total - 4 * kb));
          mbar_expect_tx(sf_full(kb), (1 + halves) * nch * kSfChunk);
          mbar_expect_tx(full_bar(kb), C::kABytes + C::kBBytes);
          if (args.pre_a)
            load_a(kb);
          else
            load_b(kb);
        }
        pdl_wait();
        for (int kb = 0; kb < pre; ++kb) {
          if (args.pre_a)
            load_b(kb);
          else
            load_a(kb);
          ++issued;
        }
        s = pre % C::kStages;
        ph = pre == C::kStages ? 1u : 0u;
      }
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        const int mb = t % args.tiles_m, nb = t / args.tiles_m;
        for (int kb = t == (int)blockIdx.x ? pre : 0; kb < args.num_kb; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, args.timeout_ns, abort)) {
            raise_timeout(args, abort);
            ok = false;
            break;
          }
          if (!args.stall_test) {
            const int nch = n_chunks(min(4, kmma_total - 4 * kb));
            int halves = 0;
            for (int h = 0; h < BN / 128; ++h)
              if ((nb * (BN / 128) + h) * 128 < args.n) ++halves;
            const uint32_t st = smem_u32(smem + s * C::kStageBytes);
            // the small scale copies first, on their own barrier, so the
            // scales reach tensor memory while the code tiles are in flight
            const uint32_t sfa_dst = st + C::kABytes + C::kBBytes;
            mbar_expect_tx(sf_full(s), (1 + halves) * nch * kSfChunk);
            bulk_load(sfa_dst, args.sfa + ((int64_t)mb * args.sf_ktiles + kChunksPerStage * kb) * kSfChunk,
                      nch * kSfChunk, sf_full(s));
            for (int h = 0; h < halves; ++h)
              bulk_load(sfa_dst + C::kSfaBytes + h * 4 * kSfChunk,
                        args.sfb + ((int64_t)(nb * (BN / 128) + h) * args.sf_ktiles + kChunksPerStage * kb) *
                                       kSfChunk,
                        nch * kSfChunk, sf_full(s));
            mbar_expect_tx(full_bar(s), C::kABytes + C::kBBytes);
            tma_load_2d(st, &tm_a, kb * kBKBytes, mb * kBM, full_bar(s));
            tma_load_2d(st + C::kABytes, &tm_b, kb * kBKBytes, nb * BN, full_bar(s));
            ++issued;
          }
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // let the copies in flight land before the CTA can exit (bounded)
      if (!ok) {
        for (int j = 0; j < C::kStages && j < issued; ++j) {
          if (--s < 0) {
            s = C::kStages - 1;
            ph ^= 1u;
          }
          mbar_wait(full_bar(s), ph, args.timeout_ns, nullptr);
          mbar_wait(sf_full(s), ph, args.timeout_ns, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = mma_idesc(kBM, BN, MX);
      const uint32_t acc = tmem;
      int s = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        if (!mbar_wait(acc_empty, acc_ph ^ 1u, args.timeout_ns, abort)) {
          raise_timeout(args, abort);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < args.num_kb; ++kb) {
          // the stage's codes are in shared memory and its scales in tensor memory
          if (!mbar_wait(full_bar(s), ph, args.timeout_ns, abort) ||
              !mbar_wait(sf_ready(s), ph, args.timeout_ns, abort)) {
            raise_timeout(args, abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const int kkc = min(4, kmma_total - 4 * kb);
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const uint32_t sf_col = tmem + BN + s * C::kSfStageCols;
          const uint64_t adesc = smem_desc(st, 16, 1024, 2);
          const uint64_t bdesc = smem_desc(st + C::kABytes, 16, 1024, 2);
          for (int kk = 0; kk < kkc; ++kk) {
            // +32 bytes of K per MMA inside the 128-byte swizzle atom
            tc_mma(acc, adesc + 2 * kk, bdesc + 2 * kk, idesc, sf_col + 4 * kk,
                   sf_col + C::kSfaCols + C::kSfbColsPerMma * kk, (kb | kk) != 0);
          }
          tc_commit(empty_bar(s));
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(acc_full);
        acc_ph ^= 1u;
      }
      // all MMAs and copies issued so far complete before the memory is freed
      tc_commit(drain_bar);
      mbar_wait(drain_bar, 0, args.timeout_ns, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue + scales
    // Between tiles these warps put each stage's scale words into tensor
    // memory with tcgen05.st (the tcgen05.cp route costs the MMA pipe a fixed
    // time per copy): lane j of the warp on lane quadrant q reads row j of a
    // 512-byte scale chunk (16 bytes = the 4-scale words of rows j, 32+j,
    // 64+j, 96+j) and writes them as 4 columns of tensor-memory lane 32q+j --
    // in every quadrant the image a 32x128b.warpx4 copy of that chunk makes.
    // With 256-column tiles the two warps of a quadrant split a stage's chunks
    // by K step; the MMA waits until all epilogue warps have signalled.
    const int q = warp & 3;                    // tensor-memory lane quadrant of this warp
    const int h = (warp - 2) / 4;              // which 128-column half of the tile
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + 128 * h;
    const uint32_t quad = (uint32_t)(32 * q) << 16;
    pdl_wait();  // A's tensor scale comes from the previous kernel under programmatic launch
    const float alpha = MX ? 1.0f : __fmul_rn(__ldcg(args.sta), __ldcg(args.stb));
    uint32_t acc_ph = 0;
    // scale-staging cursor: the next stage (tile, k block) in this CTA's sequence
    int sf_s = 0, sf_t = blockIdx.x, sf_kb = 0;
    uint32_t sf_ph = 0;
    bool ok = true;
    // stage the next stage in sequence; with only_if_ready, return false at
    // once (staging nothing) when its scale bytes have not landed yet
    auto stage_scales = [&](bool only_if_ready) -> bool {
      int go = 1;
      if (lane == 0)
        go = only_if_ready ? (mbar_try(sf_full(sf_s), sf_ph) ? 1 : 0)
                           : (mbar_wait(sf_full(sf_s), sf_ph, args.timeout_ns, abort) ? 1 : 0);
      go = __shfl_sync(0xFFFFFFFFu, go, 0);
      if (!go) {
        if (only_if_ready) return false;
        if (lane == 0) raise_timeout(args, abort);
        ok = false;
        return false;
      }
      const uint32_t st = smem_u32(smem + sf_s * C::kStageBytes);
      const uint32_t sfa_s = st + C::kABytes + C::kBBytes + 16u * lane, sfb_s = sfa_s + C::kSfaBytes;
      const uint32_t sf_col = tmem + quad + BN + sf_s * C::kSfStageCols;
      if (MX) {
        // one chunk spans two K steps: this warp (256-column tiles) stages
        // steps 2h, 2h+1 from chunk h, a 128-column tile all four from chunks 0, 1
        if (BN == 256) {
          const uint4 a = lds128(sfa_s + h * kSfChunk), b0 = lds128(sfb_s + h * kSfChunk),
                      b1 = lds128(sfb_s + 4 * kSfChunk + h * kSfChunk);
          tc_st8(sf_col + 8 * h, mx_step_words(a, 0), mx_step_words(a, 1));
          tc_st16(sf_col + 16 + 16 * h, mx_step_words(b0, 0), mx_step_words(b1, 0), mx_step_words(b0, 1),
                  mx_step_words(b1, 1));
        } else {
          const uint4 a0 = lds128(sfa_s), a1 = lds128(sfa_s + kSfChunk), b0 = lds128(sfb_s),
                      b1 = lds128(sfb_s + kSfChunk);
          tc_st16(sf_col, mx_step_words(a0, 0), mx_step_words(a0, 1), mx_step_words(a1, 0), mx_step_words(a1, 1));
          tc_st16(sf_col + 16, mx_step_words(b0, 0), mx_step_words(b0, 1), mx_step_words(b1, 0),
                  mx_step_words(b1, 1));
        }
      } else if (BN == 256) {
        // this warp: K steps 2h, 2h+1 of A (columns 8h..8h+7) and of both B halves
        // (columns 16+16h .. 16+16h+15: [B0 k][B1 k][B0 k+1][B1 k+1])
        const uint32_t k0 = 2u * h;
        tc_st8(sf_col + 8 * h, lds128(sfa_s + k0 * kSfChunk), lds128(sfa_s + (k0 + 1) * kSfChunk));
        tc_st16(sf_col + 16 + 16 * h, lds128(sfb_s + k0 * kSfChunk), lds128(sfb_s + 4 * kSfChunk + k0 * kSfChunk),
                lds128(sfb_s + (k0 + 1) * kSfChunk), lds128(sfb_s + 4 * kSfChunk + (k0 + 1) * kSfChunk));
      } else {
        tc_st16(sf_col, lds128(sfa_s), lds128(sfa_s + kSfChunk), lds128(sfa_s + 2 * kSfChunk),
                lds128(sfa_s + 3 * kSfChunk));
        tc_st16(sf_col + 16, lds128(sfb_s), lds128(sfb_s + kSfChunk), lds128(sfb_s + 2 * kSfChunk),
                lds128(sfb_s + 3 * kSfChunk));
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sf_ready(sf_s));
      if (++sf_kb == args.num_kb) {
        sf_kb = 0;
        sf_t += gridDim.x;
      }
      if (++sf_s == C::kStages) {
        sf_s = 0;
        sf_ph ^= 1u;
      }
      return true;
    };
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const int mb = t % args.tiles_m, nb = t / args.tiles_m;
      while (ok && sf_t == t) stage_scales(false);  // the rest of this tile's stages
      if (!ok) break;
      // one lane waits and the warp follows its verdict, so the warp stays
      // converged for the .sync.aligned tensor-memory loads
      int go = 1;
      if (lane == 0) go = mbar_wait(acc_full, acc_ph, args.timeout_ns, abort) ? 1 : 0;
      go = __shfl_sync(0xFFFFFFFFu, go, 0);
      if (!go) {
        if (lane == 0) raise_timeout(args, abort);
        break;
      }
      tc_fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int j = 0; j < 4; ++j) tc_ld32(lane_base, v[j], 32 * j);
      tc_wait_ld();
      // the loaded registers are valid only after the wait: tie every use to it
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(v[j][i]));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      acc_ph ^= 1u;
      // the next tile's first stages are (or soon will be) loaded: give the
      // MMA their scales before spending time on the stores.  Only that tile:
      // its stages depend on nothing but this tile's finished MMAs, while a
      // later tile's would wait on an accumulator this warp has yet to free.
      for (int i = 0; i < C::kStages && ok && sf_t < n_tiles && sf_t == t + (int)gridDim.x; ++i)
        stage_scales(false);
      // between store groups, stage any further stage of the next tile whose
      // scale bytes have landed, so the MMA is not kept waiting by the stores
      auto stage_ready_ones = [&]() {
        while (ok && sf_t < n_tiles && sf_t == t + (int)gridDim.x && stage_scales(true)) {
        }
      };

      const int row = mb * kBM + 32 * q + lane;
      const int col0 = nb * BN + 128 * h;
      uint16_t* dst = args.c + (int64_t)row * args.ldc + col0;
#pragma unroll
      for (int jh = 0; jh < 8; ++jh) {
        const int j = jh >> 1;
        if (row < args.m) {
          // columns 16 * (jh & 1) .. +15 of this 32-column group: 32 bytes of C
          uint4 o[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int g = 2 * (jh & 1) + e;
            o[e].x = pack_bf16x2(__fmul_rn(__uint_as_float(v[j][8 * g + 0]), alpha),
                                 __fmul_rn(__uint_as_float(v[j][8 * g + 1]), alpha));
            o[e].y = pack_bf16x2(__fmul_rn(__uint_as_float(v[j][8 * g + 2]), alpha),
                                 __fmul_rn(__uint_as_float(v[j][8 * g + 3]), alpha));
            o[e].z = pack_bf16x2(__fmul_rn(__uint_as_float(v[j][8 * g + 4]), alpha),
                                 __fmul_rn(__uint_as_float(v[j][8 * g + 5]), alpha));
            o[e].w = pack_bf16x2(__fmul_rn(__uint_as_float(v[j][8 * g + 6]), alpha),
                                 __fmul_rn(__uint_as_float(v[j][8 * g + 7]), alpha));
          }
          // streaming stores: C is written once, and keeping it out of L2's
          // way keeps the operand tiles there for the next tiles; a whole
          // 32-byte sector per store where C's alignment allows it
          const int col = col0 + 32 * j + 16 * (jh & 1);
          uint16_t* p = dst + 32 * j + 16 * (jh & 1);
          if (args.c32 && col + 16 <= args.n) {
            st_cs_v8(p, o[0], o[1]);
          } else {
            if (col < args.n) __stcs(reinterpret_cast<uint4*>(p), o[0]);
            if (col + 8 < args.n) __stcs(reinterpret_cast<uint4*>(p + 8), o[1]);
          }
        }
        __syncwarp();
        stage_ready_ones();  // warp-uniform: outside the per-lane row test
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int BN>
__global__ void __launch_bounds__(Cfg<BN>::kThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ GemmArgs args) {
  gemm_body<BN, false>(tm_a, tm_b, args);
}

template <int BN>
__global__ void __launch_bounds__(Cfg<BN>::kThreads, 1)
    gemm_mxfp4_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ GemmArgs args) {
  gemm_body<BN, true>(tm_a, tm_b, args);
}

// ------------------------------------------------- tensor-pipe rate probe
// The MMA instruction of the GEMM (kind::mxf4nvf4, E4M3 scales per 16 values,
// M = 128, N = BN, K = 64) issued `iters` x 4 times back to back by one
// thread per CTA on operands that stay in shared memory (zeros) with scale
// columns of E4M3 1.0: no loads, no scale staging, no stores.  It measures
// the instruction's throughput on this part, the ceiling the GEMM's operand
// pipeline is compared with.  Nothing asynchronous but the MMAs is ever in
// flight; their completion is awaited (bounded) before the tensor memory is
// freed.  The dynamic shared memory (over half an SM's) keeps one CTA per SM.
constexpr int kRateSmemBytes = 120 * 1024;

template <int BN>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int64_t iters, uint64_t timeout_ns, int32_t* status) {
  constexpr int kA = kBM * kBKBytes, kB = BN * kBKBytes;
  constexpr uint32_t kCols = BN == 256 ? 512 : 256;  // accumulator + 48 scale columns, a power of 2
  static_assert(BN + 48 <= (int)kCols, "tensor memory budget");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (kA + kB) / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // the operands were written through the generic proxy; the MMA reads them through the async proxy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // scale columns [BN, BN + 48) of this warp's lane quadrant: E4M3 1.0 in every byte
  {
    const uint4 one = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    const uint32_t col = tmem + ((uint32_t)(32 * warp) << 16) + BN;
    tc_st16(col, one, one, one, one);
    tc_st16(col + 16, one, one, one, one);
    tc_st16(col + 32, one, one, one, one);
    tc_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 32) {
    constexpr uint32_t idesc = mma_idesc(kBM, BN);
    const uint64_t adesc = smem_desc(smem_u32(smem), 16, 1024, 2);
    const uint64_t bdesc = smem_desc(smem_u32(smem + kA), 16, 1024, 2);
    const uint32_t sfa = tmem + BN, sfb = sfa + 16;
    for (int64_t it = 0; it < iters; ++it)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc_mma(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, sfa + 4 * kk, sfb + (BN / 32) * kk, (it | kk) != 0);
    tc_commit(smem_u32(&bar));
    if (!mbar_wait(smem_u32(&bar), 0, timeout_ns, nullptr) && status) atomicExch(status, (int)FOS_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
  }
}

}  // namespace

// ---------------------------------------------------------------- host side
namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// One FP4 operand of either format (tensor_scale null for MXFP4).
struct Operand {
  const uint8_t* codes;
  const uint8_t* sf;
  const float* tensor_scale;
  int64_t rows, cols, ld_codes;
};

bool valid_codes_and_scales(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t cols, int64_t ld_codes,
                            int32_t sf_layout) {
  if (!codes || !sf) return false;
  if (rows < 0 || rows > INT32_MAX || cols <= 0 || cols % kKPerMma != 0 || cols > INT32_MAX) return false;
  if (ld_codes < cols / 2 || ld_codes % 16 != 0 || !aligned(codes, 16) || !aligned(sf, 16)) return false;
  return sf_layout == FOS_SF_SWIZZLED_128x4;
}

bool valid_operand(const fos_nvfp4_tensor* t) {
  return t && t->tensor_scale && valid_codes_and_scales(t->codes, t->sf, t->rows, t->cols, t->ld_codes, t->sf_layout);
}

bool valid_operand(const fos_mxfp4_tensor* t) {
  return t && valid_codes_and_scales(t->codes, t->sf, t->rows, t->cols, t->ld_codes, t->sf_layout);
}

Operand operand(const fos_nvfp4_tensor* t) { return {t->codes, t->sf, t->tensor_scale, t->rows, t->cols, t->ld_codes}; }
Operand operand(const fos_mxfp4_tensor* t) { return {t->codes, t->sf, nullptr, t->rows, t->cols, t->ld_codes}; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major u8 matrix [rows][row_bytes] (stride ld bytes), box 128 bytes x
// box_rows rows, 128-byte swizzle (the K-major layout the MMA descriptors name).
bool make_codes_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes, int64_t ld,
                    uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {(cuuint32_t)kBKBytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
    return 148;
  return n > 0 ? n : 148;
}

template <int BN, bool MX>
fos_status launch_gemm(const Operand& A, const Operand& B, void* Cout, int64_t ldc, int32_t* dev_status,
                       uint64_t timeout_ns, int stall_test, int grid_cap, int pdl, cudaStream_t stream) {
  using C = Cfg<BN>;
  CUtensorMap ta, tb;
  const int64_t kbytes = A.cols / 2;
  if (!make_codes_map(&ta, A.codes, A.rows, kbytes, A.ld_codes, kBM) ||
      !make_codes_map(&tb, B.codes, B.rows, kbytes, B.ld_codes, BN))
    return FOS_ERR_CUDA;
  GemmArgs a{};
  a.sfa = A.sf;
  a.sfb = B.sf;
  a.sta = A.tensor_scale;
  a.stb = B.tensor_scale;
  a.c = static_cast<uint16_t*>(Cout);
  a.ldc = ldc;
  a.c32 = aligned(Cout, 32) && ldc % 16 == 0;
  a.m = (int32_t)A.rows;
  a.n = (int32_t)B.rows;
  a.k = (int32_t)A.cols;
  a.tiles_m = (int32_t)((A.rows + kBM - 1) / kBM);
  a.tiles_n = (int32_t)((B.rows + BN - 1) / BN);
  a.num_kb = (int32_t)((A.cols + 255) / 256);
  // scale chunks of 4 scales per 128-row tile: 64 values each (NVFP4) or 128 (MXFP4, the last one padded)
  a.sf_ktiles = MX ? (A.cols + 127) / 128 : A.cols / kKPerMma;
  a.status = dev_status;
  a.timeout_ns = timeout_ns;
  a.stall_test = stall_test;
  a.pre_a = pdl == 2;
  const int64_t tiles = (int64_t)a.tiles_m * a.tiles_n;
  if (tiles > INT32_MAX) return FOS_ERR_INVALID_ARG;
  int grid = sm_count();
  if (grid_cap > 0 && grid > grid_cap) grid = grid_cap;
  if (grid > tiles) grid = (int)tiles;
  const auto kernel = MX ? gemm_mxfp4_kernel<BN> : gemm_nvfp4_kernel<BN>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return FOS_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)C::kThreads);
  cfg.dynamicSmemBytes = (size_t)C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, ta, tb, a) == cudaSuccess ? FOS_OK : FOS_ERR_CUDA;
}

// pdl: 0 a plain launch; 1 a programmatic dependent of A's producer; 2 of B's.
template <typename T>
fos_status gemm_checked(const T* A, const T* B, void* C, int64_t ldc, int32_t* dev_status, uint64_t timeout_ns,
                        int stall_test, int pdl, cudaStream_t stream) {
  constexpr bool MX = std::is_same<T, fos_mxfp4_tensor>::value;
  if (!valid_operand(A) || !valid_operand(B) || !C) return FOS_ERR_INVALID_ARG;
  if (A->cols != B->cols || B->rows % 8 != 0) return FOS_ERR_INVALID_ARG;
  if (ldc < B->rows || ldc % 8 != 0 || !aligned(C, 16)) return FOS_ERR_INVALID_ARG;
  if (dev_status && !aligned(dev_status, 4)) return FOS_ERR_INVALID_ARG;
  if (A->rows == 0 || B->rows == 0) return FOS_OK;
  const Operand a = operand(A), b = operand(B);
  // 256-column tiles unless the last one would be half empty
  if (B->rows % 256 == 0 || B->rows % 256 > 128)
    return launch_gemm<256, MX>(a, b, C, ldc, dev_status, timeout_ns, stall_test, 0, pdl, stream);
  return launch_gemm<128, MX>(a, b, C, ldc, dev_status, timeout_ns, stall_test, 0, pdl, stream);
}

}  // namespace

namespace fos {
fos_status gemm_stall_selftest(void* scratch, size_t scratch_bytes, uint64_t timeout_ns, int32_t* status,
                               cudaStream_t s) {
  // A [128 x 256] and B [128 x 256] codes (16 KB each), their scales (2 KB
  // each), two tensor scales and C [128 x 128] bf16 (32 KB): 70 KB
  if (scratch_bytes < (72u << 10)) return FOS_ERR_INVALID_ARG;
  uint8_t* b = static_cast<uint8_t*>(scratch);
  fos_nvfp4_tensor A{b, b + 32768, reinterpret_cast<float*>(b + 36864), 128, 256, 128, FOS_SF_SWIZZLED_128x4, 0};
  fos_nvfp4_tensor B{b + 16384, b + 34816, reinterpret_cast<float*>(b + 36864), 128, 256, 128,
                     FOS_SF_SWIZZLED_128x4, 0};
  if (cudaMemsetAsync(b, 0, 40960, s) != cudaSuccess) return FOS_ERR_CUDA;
  return launch_gemm<128, false>(operand(&A), operand(&B), b + 40960, 128, status, timeout_ns, 1, 1, 0, s);
}

fos_status gemm_after_producer_of_a(const fos_nvfp4_tensor* A, const fos_nvfp4_tensor* B, void* C, int64_t ldc,
                                    int32_t* dev_status, cudaStream_t stream) {
  return gemm_checked(A, B, C, ldc, dev_status, kDefaultTimeoutNs, 0, 1, stream);
}

fos_status gemm_after_producer_of_b(const fos_nvfp4_tensor* A, const fos_nvfp4_tensor* B, void* C, int64_t ldc,
                                    int32_t* dev_status, cudaStream_t stream) {
  return gemm_checked(A, B, C, ldc, dev_status, kDefaultTimeoutNs, 0, 2, stream);
}
}  // namespace fos

extern "C" fos_status fos_selftest_mma_rate(int32_t n_cols, int64_t iters, int32_t grid, int32_t* dev_status,
                                            cudaStream_t stream) {
  if ((n_cols != 128 && n_cols != 256) || iters < 1 || iters > (1ll << 24) || grid < 1) return FOS_ERR_INVALID_ARG;
  if (dev_status && !aligned(dev_status, 4)) return FOS_ERR_INVALID_ARG;
  const int g = grid < sm_count() ? grid : sm_count();
  const void* fn = n_cols == 256 ? reinterpret_cast<const void*>(mma_rate_kernel<256>)
                                 : reinterpret_cast<const void*>(mma_rate_kernel<128>);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmemBytes) != cudaSuccess)
    return FOS_ERR_CUDA;
  if (n_cols == 256)
    mma_rate_kernel<256><<<g, 128, kRateSmemBytes, stream>>>(iters, kDefaultTimeoutNs, dev_status);
  else
    mma_rate_kernel<128><<<g, 128, kRateSmemBytes, stream>>>(iters, kDefaultTimeoutNs, dev_status);
  return cudaGetLastError() == cudaSuccess ? FOS_OK : FOS_ERR_CUDA;
}

extern "C" fos_status fos_gemm(const fos_nvfp4_tensor* A, const fos_nvfp4_tensor* B, void* C, int64_t ldc,
                               int32_t* dev_status, cudaStream_t stream) {
  return gemm_checked(A, B, C, ldc, dev_status, kDefaultTimeoutNs, 0, 0, stream);
}

extern "C" fos_status fos_gemm_mxfp4(const fos_mxfp4_tensor* A, const fos_mxfp4_tensor* B, void* C, int64_t ldc,
                                     int32_t* dev_status, cudaStream_t stream) {
  return gemm_checked(A, B, C, ldc, dev_status, kDefaultTimeoutNs, 0, 0, stream);
}
