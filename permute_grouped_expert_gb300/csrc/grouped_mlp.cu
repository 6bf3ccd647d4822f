// grouped_mlp.cu -- workspace sizing and per-format dispatch of the grouped
// SwiGLU expert MLP (FC1 -> SwiGLU -> FC2).
#include "moe_internal.h"

namespace moe {

cudaError_t launch_grouped_mlp_bf16(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                    const void* perm_tokens, const void* w13, const void* w2, void* act,
                                    void* ready, void* out_fc2, const float* fc2_probs, cudaStream_t st,
                                    int64_t silent_token_tile);
size_t grouped_mlp_bf16_ready_bytes(const moe_shape& s, const moe_layout& l);

cudaError_t launch_grouped_mlp_bf16_pair(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                         const void* perm_tokens, const void* w13, const void* w2, void* act,
                                         void* out_fc2, const float* fc2_probs, cudaStream_t st);

cudaError_t launch_grouped_mlp_fp8(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                   const void* perm_codes, const void* perm_scales, const void* w13,
                                   const void* w13_scales, const void* w2, const void* w2_scales, void* workspace,
                                   void* out_fc2, int32_t out_format, void* out_fc2_scales, const float* fc2_probs,
                                   cudaStream_t st);

cudaError_t launch_grouped_mlp_nvfp4(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                     const void* perm_packed, const void* perm_scales, const void* w13,
                                     const void* w13_scales, const void* w2, const void* w2_scales,
                                     const moe_nvfp4_globals& g, void* workspace, void* out_fc2,
                                     const float* fc2_probs, cudaStream_t st);

namespace {
constexpr int64_t kPairMinRowsPerExpert = 4096;
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
}  // namespace

size_t grouped_mlp_workspace_bytes(const moe_shape& s, const moe_layout& l, int32_t w_dtype) {
  const size_t cap = (size_t)l.capacity, I = (size_t)s.I;
  switch (w_dtype) {
    case MOE_DTYPE_BF16:  // bf16 intermediate + FC1 completion counters per M tile
      return round_up(cap * I * 2, 1024) + round_up(grouped_mlp_bf16_ready_bytes(s, l), 1024) + 1024;
    case MOE_DTYPE_FP8_E4M3_B128:  // E4M3 intermediate + fp32 scales per 128 elements
      return round_up(cap * I, 1024) + round_up(cap * (I / 128) * 4, 1024) + 1024;
    case MOE_DTYPE_NVFP4:  // packed E2M1 intermediate + E4M3 scales per 16 elements
      return round_up(cap * I / 2, 1024) + round_up(cap * (I / 16), 1024) + 1024;
  }
  return 0;
}

bool grouped_mlp_bf16_uses_pairs(const moe_shape& s, const moe_layout& l) {
  // Experts with thousands of rows (capacity >= 4096 rows per expert) run each
  // MMA across an SM pair (256-row tiles, half the operand bytes per MAC of a
  // single SM); below that the single-SM fused kernel (no kernel boundary,
  // ragged expert ends at 16-row granularity) is faster: at 2048 rows per
  // expert 0.166 ms against 0.189 ms, at ~6000 rows 0.611 ms against 0.559 ms.
  return l.capacity >= kPairMinRowsPerExpert * s.E;
}

int grouped_mlp_kernel_count(const moe_shape& s, const moe_layout& l, int32_t w_dtype) {
  switch (w_dtype) {
    case MOE_DTYPE_BF16:  // one fused FC1 + FC2 kernel on single SMs; two kernels on SM pairs
      return l.capacity == 0 ? 0 : grouped_mlp_bf16_uses_pairs(s, l) ? 2 : 1;
    case MOE_DTYPE_FP8_E4M3_B128:
    case MOE_DTYPE_NVFP4:
      return l.capacity == 0 ? 0 : 2;
  }
  return -1;
}

cudaError_t launch_grouped_mlp(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                               int32_t w_dtype, const void* perm_tokens, const void* perm_scales,
                               const void* w13, const void* w13_scales, const void* w2,
                               const void* w2_scales, const moe_nvfp4_globals* globals,
                               void* workspace, void* out_fc2, int32_t out_format, void* out_fc2_scales,
                               const float* fc2_probs, cudaStream_t st) {
  const int64_t silent = take_debug_mlp_silent_tile();  // testing hook: only the fused bf16 kernel uses it
  // MX combine formats are written by the FP8 path's FC2 epilogue only
  if (out_format != MOE_COMBINE_BF16 && w_dtype != MOE_DTYPE_FP8_E4M3_B128) return cudaErrorNotSupported;
  switch (w_dtype) {
    case MOE_DTYPE_BF16:
      if (grouped_mlp_bf16_uses_pairs(s, l))
        return launch_grouped_mlp_bf16_pair(h, s, l, perm_tokens, w13, w2, workspace, out_fc2, fc2_probs, st);
      return launch_grouped_mlp_bf16(h, s, l, perm_tokens, w13, w2, workspace,
                                     static_cast<uint8_t*>(workspace) + round_up((size_t)l.capacity * s.I * 2, 1024),
                                     out_fc2, fc2_probs, st, silent);
    case MOE_DTYPE_FP8_E4M3_B128:
      return launch_grouped_mlp_fp8(h, s, l, perm_tokens, perm_scales, w13, w13_scales, w2, w2_scales, workspace,
                                    out_fc2, out_format, out_fc2_scales, fc2_probs, st);
    case MOE_DTYPE_NVFP4:
      return launch_grouped_mlp_nvfp4(h, s, l, perm_tokens, perm_scales, w13, w13_scales, w2, w2_scales, *globals,
                                      workspace, out_fc2, fc2_probs, st);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace moe
