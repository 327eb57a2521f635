// fos_quantize_noalloc: fos_quantize without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they quantize.
// Examples are plugin hosts and inference runtimes that hand an operator only
// its inputs and outputs and forbid cudaMalloc after start-up: an allocation
// can synchronize the device, fail under memory pressure at an arbitrary
// moment, or fall outside the runtime's memory accounting.  This entry point
// serves them.  The only scratch the quantizer needs, one partial maximum per
// CTA of the amax pass, lives in a fixed array in device memory that the
// library itself owns.
//
// Limits and behaviour a caller must know:
//   - The array holds kNoAllocScratchFloats floats (8448 bytes: the partial
//     maxima and the words of the one-launch quantizer's grid barrier).  Every
//     GPU that loads the library holds it until the process exits.
//   - The first call on each device looks up the array's device address (with
//     that device current) and caches it.  Make that first call before any
//     stream capture.
//   - All calls share the one array.  Calls that overlap on the GPU (for
//     example on two streams without ordering between them) race on it and
//     may produce wrong scales.
//   - Nothing in the array needs clearing between calls: each call's amax pass
//     writes every slot its quantize pass later reads, and each call clears
//     the one-launch quantizer's three barrier words (a 12-byte
//     cudaMemsetAsync on the caller's stream, which allocates nothing) before
//     its launch.
//   - A call whose scratch need exceeds the array is rejected with
//     FOS_ERR_INVALID_ARG.  The amax pass never runs more than
//     kMaxAmaxPartials CTAs, so every call fos_quantize accepts fits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fos.h"
#include "fos_internal.h"

namespace {

constexpr int kNoAllocScratchFloats = (int)(fos::kQuantWorkspaceBytes / sizeof(float));
static_assert(kNoAllocScratchFloats * sizeof(float) >= fos::kQuantWorkspaceBytes,
              "the fixed scratch must cover the quantizer's workspace");

// In host code this name stands in for the array; it is not a device address.
// Host code passes the address from cudaGetSymbolAddress to the kernels.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
fos_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FOS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FOS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FOS_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FOS_OK;
}

}  // namespace

extern "C" fos_status fos_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                           const fos_quant_options* opt, uint8_t* codes, int64_t ld_codes,
                                           uint8_t* sf, float* tensor_scale, uint8_t* choice,
                                           cudaStream_t stream) {
  size_t need = 0;
  if (fos_quantize_workspace_size(rows, cols, opt, &need) != FOS_OK) return FOS_ERR_INVALID_ARG;
  if (need > sizeof(float) * kNoAllocScratchFloats) return FOS_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (need > 0) {
    fos_status s = scratch_address(&scratch);
    if (s != FOS_OK) return s;
  }
  return fos_quantize(x, rows, cols, ld_x, opt, codes, ld_codes, sf, tensor_scale, choice, scratch,
                      need > 0 ? sizeof(float) * kNoAllocScratchFloats : 0, stream);
}
