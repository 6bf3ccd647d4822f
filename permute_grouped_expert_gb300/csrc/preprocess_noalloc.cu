// preprocess_noalloc.cu -- moe_preprocess for callers that cannot allocate
// device memory: the scratch space the preprocessing kernels need lives in a
// fixed, file-scope device array instead of a caller-provided workspace.
//
// Some callers have no way to obtain a device workspace: a plugin running
// inside a host application that owns every device allocation and hands its
// plugins no allocator, or a latency-critical loop that sized its memory once
// up front and must not call cudaMalloc (which can synchronise the device).
// This entry point serves them.  The array below is part of the library's
// device image, so every GPU that loads the library holds it until the process
// exits.
#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = MOE_PREPROCESS_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  Host code must not pass `g_preprocess_scratch` to a
// kernel: on the host that name denotes a host-side stand-in, not the device
// address.  The device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_preprocess_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  Outside stream
// capture it is looked up afresh (with the device current), so a module that
// was reloaded after cudaDeviceReset gives its new address; during capture the
// address cached by the last lookup on this device is used, because a capture
// must not depend on a call that may load the module.
cudaError_t scratch_for_current_device(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(stream, &cap)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (cap == cudaStreamCaptureStatusNone || !g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_preprocess_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_preprocess_noalloc(const moe_routing* routing, const moe_shape* shape,
                                             const moe_layout* layout, const moe_handle_dev* handle,
                                             void* stream) {
  // Argument checks first (as moe_preprocess makes them), then the size rule.
  moe_status st = moe::validate_preprocess_args(routing, shape, layout, handle);
  if (st != MOE_OK) return st;
  size_t need = 0;
  if ((st = moe_preprocess_workspace_size(shape, &need)) != MOE_OK) return st;
  if (need > moe::kNoAllocScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;  // shape beyond the fixed scratch
  void* scratch = nullptr;
  cudaError_t e = moe::scratch_for_current_device(static_cast<cudaStream_t>(stream), &scratch);
  if (e != cudaSuccess) {
    moe::record_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  // The ordinary entry point clears the scratch bytes that must start at zero
  // (on `stream`) and launches the same kernels.
  return moe_preprocess(routing, shape, layout, handle, scratch, moe::kNoAllocScratchBytes, stream);
}
