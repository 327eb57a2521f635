// The quantized linear layer's forward and backward passes as compositions of
// the library's own calls: quantizations (fos_quantize) and block-scaled
// products (fos_gemm), all enqueued on the caller's stream.
//
// "Four Over Six" ("Training"): the quantized linear layer carries a backward
// pass.  "FP4" (Ultralytics glossary, "FP4 ile Çıkarım ve Eğitim"): FP4
// training spreads outliers with random Hadamard transforms and rounds
// gradients stochastically.  For Y = X W^T the two products are
//   dgrad  dX = dY W      (contraction over N: dY along its rows, W^T along N)
//   wgrad  dW = dY^T X    (contraction over M: both operands along M)
// and both operands of a product must be blocked along its contraction, so
// dY is quantized twice (along N and along M) and W and X along N and M.
#include <cuda_runtime.h>

#include <cstdint>

#include "fos.h"
#include "fos_internal.h"

namespace {

constexpr size_t kAlign = 256;

size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t codes_ld(int64_t cols) { return ((cols / 2 + 15) / 16) * 16; }

int64_t sf_bytes(int64_t rows, int64_t cols) { return ((rows + 127) / 128) * 128 * ((cols / 16 + 3) / 4) * 4; }

// Where each part of the workspace lies.
struct Layout {
  int64_t rows[4], cols[4];
  size_t codes[4], sf[4], scales, amax, scratch, total;
};

bool valid_shape(int64_t M, int64_t N, int64_t K) {
  return M > 0 && N > 0 && K > 0 && M % 64 == 0 && N % 64 == 0 && K % 16 == 0 && M <= INT32_MAX &&
         N <= INT32_MAX && K <= INT32_MAX;
}

Layout layout(int64_t M, int64_t N, int64_t K) {
  Layout L{};
  const int64_t r[4] = {M, K, N, K}, c[4] = {N, N, M, M};
  size_t o = 0;
  for (int i = 0; i < 4; ++i) {
    L.rows[i] = r[i];
    L.cols[i] = c[i];
    L.codes[i] = o;
    o = up(o + (size_t)(r[i] * codes_ld(c[i])));
    L.sf[i] = o;
    o = up(o + (size_t)sf_bytes(r[i], c[i]));
  }
  L.scales = o;
  o = up(o + 4 * sizeof(float));
  L.amax = o;  // dY's two tensor maxima when both products are computed
  o = up(o + 2 * sizeof(float));
  L.scratch = o;
  L.total = o + fos::kQuantWorkspaceBytes;
  return L;
}

bool valid_bf16(const void* p, int64_t ld, int64_t row_len) {
  return p && aligned(p, 16) && ld >= row_len && ld % 8 == 0;
}

}  // namespace

// ------------------------------------------------------------ forward
// Y = X W^T with W already quantized (offline, along K; with the RHT of the
// same seed when X gets it, so that the transform cancels in the product):
// X is quantized into the workspace, then the GEMM runs as the quantizer's
// programmatic dependent, loading W's first stages during the quantizer's
// tail.  The quantizer is not folded into the GEMM's producer: every 128-row
// tile of X feeds all N/256 output-column tiles, so it would be quantized
// that many times over.

namespace {

struct FwdLayout {
  size_t codes, sf, scale, scratch, total;
};

FwdLayout fwd_layout(int64_t M, int64_t K) {
  FwdLayout L{};
  L.codes = 0;
  L.sf = up((size_t)(M * codes_ld(K)));
  L.scale = up(L.sf + (size_t)sf_bytes(M, K));
  L.scratch = up(L.scale + sizeof(float));
  L.total = L.scratch + fos::kQuantWorkspaceBytes;
  return L;
}

bool valid_fwd_shape(int64_t M, int64_t K) { return M > 0 && K > 0 && K % 64 == 0 && M <= INT32_MAX && K <= INT32_MAX; }

}  // namespace

extern "C" {

fos_status fos_linear_backward_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
  if (!bytes || !valid_shape(M, N, K)) return FOS_ERR_INVALID_ARG;
  *bytes = layout(M, N, K).total;
  return FOS_OK;
}

fos_status fos_linear_backward_operands(int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                                        fos_nvfp4_tensor ops[4]) {
  if (!ops || !workspace || !valid_shape(M, N, K) || !aligned(workspace, kAlign)) return FOS_ERR_INVALID_ARG;
  const Layout L = layout(M, N, K);
  if (workspace_bytes < L.total) return FOS_ERR_INVALID_ARG;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  for (int i = 0; i < 4; ++i) {
    ops[i].codes = base + L.codes[i];
    ops[i].sf = base + L.sf[i];
    ops[i].tensor_scale = reinterpret_cast<const float*>(base + L.scales) + i;
    ops[i].rows = L.rows[i];
    ops[i].cols = L.cols[i];
    ops[i].ld_codes = codes_ld(L.cols[i]);
    ops[i].sf_layout = FOS_SF_SWIZZLED_128x4;
    ops[i].reserved = 0;
  }
  return FOS_OK;
}

fos_status fos_linear_backward(const void* dy, int64_t ld_dy, const void* x, int64_t ld_x, const void* w,
                               int64_t ld_w, int64_t M, int64_t N, int64_t K, const fos_backward_options* opt,
                               void* dx, int64_t ld_dx, void* dw, int64_t ld_dw, void* workspace,
                               size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream) {
  // ---- every check first: nothing is enqueued unless all of them pass
  if (!opt || opt->struct_size < sizeof(fos_backward_options) || opt->reserved != 0) return FOS_ERR_INVALID_ARG;
  if (opt->scale_rule < FOS_SCALE_4OVER6 || opt->scale_rule > FOS_SCALE_4) return FOS_ERR_INVALID_ARG;
  if (opt->grad_rounding != FOS_ROUND_RNE && opt->grad_rounding != FOS_ROUND_STOCHASTIC) return FOS_ERR_INVALID_ARG;
  if ((opt->wgrad_hadamard | opt->weight_2d) & ~1) return FOS_ERR_INVALID_ARG;
  if (!valid_shape(M, N, K)) return FOS_ERR_INVALID_ARG;
  if (!valid_bf16(dy, ld_dy, N)) return FOS_ERR_INVALID_ARG;
  if (dx && (!valid_bf16(w, ld_w, K) || !valid_bf16(dx, ld_dx, K))) return FOS_ERR_INVALID_ARG;
  if (dw && (!valid_bf16(x, ld_x, K) || !valid_bf16(dw, ld_dw, K))) return FOS_ERR_INVALID_ARG;
  if (dev_status && !aligned(dev_status, 4)) return FOS_ERR_INVALID_ARG;
  fos_nvfp4_tensor ops[4];
  fos_status st = fos_linear_backward_operands(M, N, K, workspace, workspace_bytes, ops);
  if (st != FOS_OK) return st;
  const Layout L = layout(M, N, K);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  void* scratch = base + L.scratch;
  const size_t scratch_bytes = fos::kQuantWorkspaceBytes;

  auto opts = [&](int32_t rounding, int32_t transpose, int32_t hadamard, int32_t block_2d) {
    fos_quant_options o{};
    o.struct_size = sizeof(fos_quant_options);
    o.scale_rule = opt->scale_rule;
    o.rounding = rounding;
    o.block_2d = block_2d;
    o.transpose = transpose;
    o.hadamard = hadamard;
    o.sf_layout = FOS_SF_SWIZZLED_128x4;
    o.sr_seed = opt->sr_seed;
    o.hadamard_seed = opt->hadamard_seed;
    return o;
  };
  // quantize src [rows, cols] into operand i
  auto quant = [&](int i, const void* src, int64_t rows, int64_t cols, int64_t ld, const fos_quant_options& o) {
    return fos_quantize(src, rows, cols, ld, &o, const_cast<uint8_t*>(ops[i].codes), ops[i].ld_codes,
                        const_cast<uint8_t*>(ops[i].sf), const_cast<float*>(ops[i].tensor_scale), nullptr, scratch,
                        scratch_bytes, stream);
  };

  // With both products, dY is quantized twice (along N and, transposed, along
  // M).  Its two tensor maxima -- of dY, and of its RHT down the columns when
  // the wgrad operands get the RHT -- then come from one read of dY, and both
  // quantizations take them as supplied maxima (the same values their own
  // amax passes would find).
  const bool both = dx && dw;
  // With both products under stochastic rounding, dY's two quantizations come
  // from one launch: one read of dY, and each element's Philox word computed
  // once for both (they draw from the same word).
  const bool dual = both && opt->grad_rounding == FOS_ROUND_STOCHASTIC;
  float* amax_dy = reinterpret_cast<float*>(base + L.amax);  // [max|dY|, max|RHT_M(dY)|]
  // the fused launch with the RHT reduces the amax pass's partial maxima itself
  int dual_partials = 0;
  if (both) {
    if (opt->wgrad_hadamard) {
      if (fos::amax_plain_and_rht_cols(dy, M, N, ld_dy, opt->hadamard_seed, amax_dy, scratch, stream,
                                       dual ? &dual_partials : nullptr) != cudaSuccess)
        return FOS_ERR_CUDA;
    } else if ((st = fos_tensor_amax(dy, M, N, ld_dy, 0, 0, 0, amax_dy, scratch, scratch_bytes, stream)) != FOS_OK) {
      return st;
    }
  }
  fos_quant_options o_dy = opts(opt->grad_rounding, 0, 0, 0);
  fos_quant_options o_dyt = opts(opt->grad_rounding, 1, opt->wgrad_hadamard, 0);
  if (both) {
    o_dy.tensor_amax = amax_dy;
    o_dyt.tensor_amax = opt->wgrad_hadamard ? amax_dy + 1 : amax_dy;
  }
  if (dual) {
    // the maxima: one value each, or the amax pass's partials (max |RHT(dY)|
    // at the scratch, max |dY| half-way into its partial region)
    const float* part = static_cast<const float*>(scratch);
    const float* src_r = dual_partials ? part + fos::kMaxAmaxPartials / 2 : o_dy.tensor_amax;
    const float* src_c = dual_partials ? part : o_dyt.tensor_amax;
    const auto qr = fos::quant_launch(dy, M, N, ld_dy, &o_dy, const_cast<uint8_t*>(ops[0].codes), ops[0].ld_codes,
                                      const_cast<uint8_t*>(ops[0].sf), const_cast<float*>(ops[0].tensor_scale),
                                      nullptr, src_r, dual_partials);
    const auto qc = fos::quant_launch(dy, M, N, ld_dy, &o_dyt, const_cast<uint8_t*>(ops[2].codes), ops[2].ld_codes,
                                      const_cast<uint8_t*>(ops[2].sf), const_cast<float*>(ops[2].tensor_scale),
                                      nullptr, src_c, dual_partials);
    if (fos::launch_quant_dual_sr(qc.p, qr.p, opt->scale_rule, opt->wgrad_hadamard != 0, qc.tasks, stream) !=
            cudaSuccess ||
        fos::pad_scales(qr.p, stream) != cudaSuccess || fos::pad_scales(qc.p, stream) != cudaSuccess)
      return FOS_ERR_CUDA;
  }
  if (dx) {
    const fos_quant_options o_w = opts(FOS_ROUND_RNE, 1, 0, opt->weight_2d);
    if (!dual && (st = quant(0, dy, M, N, ld_dy, o_dy)) != FOS_OK) return st;
    if ((st = quant(1, w, N, K, ld_w, o_w)) != FOS_OK) return st;
    // W^T's quantize launch comes right before and dY's operand is complete:
    // the GEMM loads dY's first stages while that launch finishes
    if ((st = fos::gemm_after_producer_of_b(&ops[0], &ops[1], dx, ld_dx, dev_status, stream)) != FOS_OK) return st;
  }
  if (dw) {
    const fos_quant_options o_xt = opts(FOS_ROUND_RNE, 1, opt->wgrad_hadamard, 0);
    if (!dual && (st = quant(2, dy, M, N, ld_dy, o_dyt)) != FOS_OK) return st;
    if ((st = quant(3, x, M, K, ld_x, o_xt)) != FOS_OK) return st;
    // likewise after X^T's quantize launch, with dY^T's operand complete
    if ((st = fos::gemm_after_producer_of_b(&ops[2], &ops[3], dw, ld_dw, dev_status, stream)) != FOS_OK) return st;
  }
  return FOS_OK;
}


fos_status fos_linear_forward_workspace_size(int64_t M, int64_t K, size_t* bytes) {
  if (!bytes || !valid_fwd_shape(M, K)) return FOS_ERR_INVALID_ARG;
  *bytes = fwd_layout(M, K).total;
  return FOS_OK;
}

fos_status fos_linear_forward_operand(int64_t M, int64_t K, void* workspace, size_t workspace_bytes,
                                      fos_nvfp4_tensor* xq) {
  if (!xq || !workspace || !valid_fwd_shape(M, K) || !aligned(workspace, kAlign)) return FOS_ERR_INVALID_ARG;
  const FwdLayout L = fwd_layout(M, K);
  if (workspace_bytes < L.total) return FOS_ERR_INVALID_ARG;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  xq->codes = base + L.codes;
  xq->sf = base + L.sf;
  xq->tensor_scale = reinterpret_cast<const float*>(base + L.scale);
  xq->rows = M;
  xq->cols = K;
  xq->ld_codes = codes_ld(K);
  xq->sf_layout = FOS_SF_SWIZZLED_128x4;
  xq->reserved = 0;
  return FOS_OK;
}

fos_status fos_linear_forward(const void* x, int64_t ld_x, int64_t M, int64_t K, const fos_quant_options* x_opt,
                              const fos_nvfp4_tensor* w, void* y, int64_t ld_y, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream) {
  if (!x_opt || !w || x_opt->transpose || x_opt->sf_layout != FOS_SF_SWIZZLED_128x4) return FOS_ERR_INVALID_ARG;
  if (w->cols != K || w->sf_layout != FOS_SF_SWIZZLED_128x4) return FOS_ERR_INVALID_ARG;
  if (!valid_bf16(y, ld_y, w->rows) || (dev_status && !aligned(dev_status, 4))) return FOS_ERR_INVALID_ARG;
  fos_nvfp4_tensor xq;
  fos_status st = fos_linear_forward_operand(M, K, workspace, workspace_bytes, &xq);
  if (st != FOS_OK) return st;
  // the GEMM's own checks, on the operand the quantizer is about to write
  if (!w->codes || !w->sf || !w->tensor_scale || w->rows <= 0 || w->rows % 8 != 0 || w->ld_codes % 16 != 0 ||
      w->ld_codes < K / 2 || !aligned(w->codes, 16) || !aligned(w->sf, 16))
    return FOS_ERR_INVALID_ARG;
  const FwdLayout L = fwd_layout(M, K);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  st = fos_quantize(x, M, K, ld_x, x_opt, base + L.codes, xq.ld_codes, base + L.sf,
                    reinterpret_cast<float*>(base + L.scale), nullptr, base + L.scratch, fos::kQuantWorkspaceBytes,
                    stream);
  if (st != FOS_OK) return st;
  return fos::gemm_after_producer_of_a(&xq, w, y, ld_y, dev_status, stream);
}

}  // extern "C"
