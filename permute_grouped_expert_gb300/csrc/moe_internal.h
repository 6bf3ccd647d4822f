// moe_internal.h -- launchers shared between the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "moe.h"

namespace moe {

// Preprocess tiling: about kPreTargetTiles tiles, each holding at most
// kPreMaxEntries routes and at most kPreStageBytes bytes of routing map.
constexpr int kPreMaxEntries = 4096;
constexpr int kPreStageBytes = 32768;
constexpr int kPreTargetTiles = 64;
constexpr int kPreThreads = 256;
constexpr int kPreWarps = kPreThreads / 32;

inline int64_t pre_tokens_per_tile(int64_t T, int64_t E, int64_t K) {
  int64_t t = (T + kPreTargetTiles - 1) / kPreTargetTiles;
  if (t > kPreMaxEntries / K) t = kPreMaxEntries / K;
  if (t > kPreStageBytes / E) t = kPreStageBytes / E;
  return t < 1 ? 1 : t;
}
inline int64_t pre_num_tiles(int64_t T, int64_t E, int64_t K) {
  int64_t tpt = pre_tokens_per_tile(T, E, K);
  int64_t n = (T + tpt - 1) / tpt;
  return n < 1 ? 1 : n;  // a zero-token call still runs one (empty) tile
}

struct PreWorkspace {
  int32_t* tile_counter;       // [1]
  uint64_t* lookback;          // [num_tiles][E]
  int16_t* route_expert;       // [T*K]
  size_t memset_bytes;         // leading bytes to clear per call (counter + lookback)
};

size_t preprocess_workspace_bytes(int64_t T, int64_t E, int64_t K);
PreWorkspace preprocess_workspace_carve(void* ws, int64_t T, int64_t E, int64_t K);

cudaError_t launch_preprocess(const moe_routing& r, const moe_shape& s, const moe_layout& l,
                              const moe_handle_dev& h, const PreWorkspace& ws, cudaStream_t st,
                              int64_t silent_tile = -1);

cudaError_t launch_dispatch(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                            int32_t in_dtype, const void* x, const void* x_scales,
                            const moe_routing& r, void* out_tokens, float* out_probs,
                            void* out_scales, cudaStream_t st);

cudaError_t launch_combine(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                           const void* expert_out, const float* perm_probs, void* y,
                           cudaStream_t st);

cudaError_t launch_combine_backward(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                    const void* grad_y, const void* expert_out, const float* perm_probs,
                                    void* grad_expert_out, float* grad_perm_probs, cudaStream_t st);
cudaError_t launch_dispatch_backward(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                     int32_t routing_format, const void* grad_perm_tokens,
                                     const float* grad_perm_probs, void* grad_x, float* grad_probs,
                                     cudaStream_t st);

cudaError_t launch_quantize_fp8_blocks(const void* w, int64_t G, int64_t N, int64_t Kd, void* codes,
                                       float* scales, cudaStream_t st);
cudaError_t launch_quantize_nvfp4_rows(const void* x, int64_t R, int64_t Kd, const float* global,
                                       void* packed, void* scales, cudaStream_t st);

// Grouped MLP (bf16 / FP8 / NVFP4), defined in the GEMM translation units.
size_t grouped_mlp_workspace_bytes(const moe_shape& s, const moe_layout& l, int32_t w_dtype);
int grouped_mlp_kernel_count(const moe_shape& s, const moe_layout& l, int32_t w_dtype);
cudaError_t launch_grouped_mlp(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                               int32_t w_dtype, const void* perm_tokens, const void* perm_scales,
                               const void* w13, const void* w13_scales, const void* w2,
                               const void* w2_scales, const moe_nvfp4_globals* globals,
                               void* workspace, void* out_fc2, int32_t out_format, void* out_fc2_scales,
                               const float* fc2_row_probs, cudaStream_t st);
cudaError_t launch_combine_mx(const moe_handle_dev& h, const moe_shape& s, int32_t in_format,
                              const void* codes, const void* scales, const float* perm_probs, void* y,
                              cudaStream_t st);
cudaError_t launch_quantize_mx_rows(const void* x, int64_t R, int64_t H, int32_t format, void* codes, void* scales,
                                    cudaStream_t st);

int device_sm_count();

// Runs a per-device setup step (a kernel attribute such as its dynamic
// shared-memory limit, which CUDA keeps per device) once for each device it is
// called on, with that device current.  Thread-safe; a failed step is retried
// on the next call.
class PerDeviceOnce {
 public:
  static constexpr int kMaxDevices = 64;
  template <class F>
  cudaError_t run(F&& step) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mutex_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = step();
    if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
    return e;
  }

 private:
  std::mutex mutex_;
  std::atomic<bool> done_[kMaxDevices] = {};
};

// Host-side argument checks of moe_preprocess (shape, routing, layout, padded
// total, handle), in that order; MOE_OK or MOE_ERR_INVALID_ARG.
moe_status validate_preprocess_args(const moe_routing* routing, const moe_shape* shape, const moe_layout* layout,
                                    const moe_handle_dev* handle);

// Records a CUDA error for moe_last_cuda_error() (the caller returns MOE_ERR_CUDA).
void record_cuda_error(cudaError_t e);

// Events the next grouped-MLP launch on this thread records (see
// moe_profile_next_grouped_mlp); consumed and cleared by that launch.
struct ProfileEvents {
  cudaEvent_t before_fc1 = nullptr, after_fc1 = nullptr, after_fc2 = nullptr;
};
ProfileEvents take_profile_events();
// Records a profiling event on `st`; under stream capture the record becomes an
// event-record node of the graph (recorded again on every replay).
cudaError_t record_profile_event(cudaEvent_t ev, cudaStream_t st);
// Testing hook (moe_debug_next_grouped_mlp_silent_token_tile); consumed and
// cleared by the next fused bf16 grouped-MLP launch of this host thread.
int64_t take_debug_mlp_silent_tile();
void set_debug_mlp_silent_tile(int64_t token_tile);
void set_profile_events(const ProfileEvents& ev);

}  // namespace moe
