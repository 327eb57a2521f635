// Block-scaled NVFP4 GEMM (tcgen05) -- argument validation; the kernel follows.
#include <cstdint>

#include "fos.h"

namespace {
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_operand(const fos_nvfp4_tensor* t) {
  if (!t || !t->codes || !t->sf || !t->tensor_scale) return false;
  if (t->rows < 0 || t->cols <= 0 || t->cols % 256 != 0) return false;
  if (t->ld_codes < t->cols / 2 || t->ld_codes % 16 != 0 || !aligned(t->codes, 16) || !aligned(t->sf, 16))
    return false;
  return t->sf_layout == FOS_SF_SWIZZLED_128x4;
}
}  // namespace

extern "C" fos_status fos_gemm(const fos_nvfp4_tensor* A, const fos_nvfp4_tensor* B, void* C, int64_t ldc,
                               int32_t* dev_status, cudaStream_t stream) {
  (void)dev_status;
  (void)stream;
  if (!valid_operand(A) || !valid_operand(B) || !C) return FOS_ERR_INVALID_ARG;
  if (A->cols != B->cols || A->rows % 128 != 0 || B->rows % 256 != 0) return FOS_ERR_INVALID_ARG;
  if (ldc < B->rows || ldc % 8 != 0 || !aligned(C, 16)) return FOS_ERR_INVALID_ARG;
  return FOS_ERR_UNSUPPORTED;
}
