// grouped_mlp.cu -- placeholder until the tcgen05 grouped GEMMs land.
#include "moe_internal.h"

namespace moe {

size_t grouped_mlp_workspace_bytes(const moe_shape& s, const moe_layout& l, int32_t w_dtype) {
  (void)w_dtype;
  return (size_t)l.capacity * (size_t)s.I * 2 + 1024;
}

cudaError_t launch_grouped_mlp(const moe_handle_dev&, const moe_shape&, const moe_layout&, int32_t,
                               const void*, const void*, const void*, const void*, const void*,
                               const void*, const moe_nvfp4_globals*, void*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace moe
