// moe_api.cu -- the extern "C" entry points declared in moe.h: host-side
// argument validation (nothing is enqueued when it fails), workspace queries,
// launches, error reporting and the host-side output-buffer ring.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include "moe_internal.h"

#define MOE_TRY_INTERNAL(expr)          \
  do {                                   \
    moe_status _st = (expr);             \
    if (_st != MOE_OK) return _st;       \
  } while (0)

namespace moe {

namespace {
thread_local char g_last_error[256] = "no error";

moe_status cuda_fail(cudaError_t e) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_shape(const moe_shape* s, bool need_h) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->E < 1 || s->E > 1024 || s->K < 1 || s->K > 128 || s->K > s->E) return MOE_ERR_INVALID_ARG;
  if (s->T * s->K >= (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;  // row ids are int32
  if (need_h && (s->H <= 0 || s->H % 128 != 0)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status check_layout(const moe_layout* l) {
  if (!l || l->pad_multiple < 1 || l->pad_multiple >= (int64_t(1) << 31) || l->capacity < 0 ||
      l->capacity >= (int64_t(1) << 31))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// The padded total sum_e ceil(count[e]/m)*m is at most T*K + E*(m-1); offsets,
// total_rows and row ids are int32, so that bound must stay below 2^31.
moe_status check_padded_total(const moe_shape* s, const moe_layout* l) {
  if (s->T * s->K + s->E * (l->pad_multiple - 1) >= (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status check_handle(const moe_handle_dev* h) {
  if (!h || !h->tokens_per_expert || !h->padded_offsets || !h->row_of || !h->token_of || !h->slot_of ||
      !h->total_rows || !h->overflow || !h->status)
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status check_routing(const moe_routing* r, int64_t T) {
  if (!r || (T > 0 && !r->map)) return MOE_ERR_INVALID_ARG;
  if (r->format != MOE_ROUTING_DENSE_I16 && r->format != MOE_ROUTING_SPARSE_BOOL) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}
}  // namespace

namespace {
thread_local ProfileEvents g_profile;
}

void record_cuda_error(cudaError_t e) { cuda_fail(e); }

moe_status validate_preprocess_args(const moe_routing* routing, const moe_shape* shape, const moe_layout* layout,
                                    const moe_handle_dev* handle) {
  MOE_TRY_INTERNAL(check_shape(shape, false));
  MOE_TRY_INTERNAL(check_routing(routing, shape->T));
  MOE_TRY_INTERNAL(check_layout(layout));
  MOE_TRY_INTERNAL(check_padded_total(shape, layout));
  MOE_TRY_INTERNAL(check_handle(handle));
  return MOE_OK;
}

ProfileEvents take_profile_events() {
  ProfileEvents e = g_profile;
  g_profile = ProfileEvents();
  return e;
}

void set_profile_events(const ProfileEvents& ev) { g_profile = ev; }

cudaError_t record_profile_event(cudaEvent_t ev, cudaStream_t st) {
  return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
}

thread_local int64_t g_debug_mlp_silent = -1;

int64_t take_debug_mlp_silent_tile() {
  const int64_t v = g_debug_mlp_silent;
  g_debug_mlp_silent = -1;
  return v;
}

void set_debug_mlp_silent_tile(int64_t token_tile) { g_debug_mlp_silent = token_tile; }

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

}  // namespace moe

using namespace moe;

#define MOE_TRY(expr)                    \
  do {                                   \
    moe_status _st = (expr);             \
    if (_st != MOE_OK) return _st;       \
  } while (0)

extern "C" {

const char* moe_last_cuda_error(void) { return g_last_error; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_RING_EARLY_REUSE: return "MOE_ERR_RING_EARLY_REUSE";
    case MOE_ERR_RING_DOUBLE_RELEASE: return "MOE_ERR_RING_DOUBLE_RELEASE";
  }
  return "unknown moe_status";
}

moe_status moe_capacity(int64_t rows, double factor, int64_t align, int64_t* capacity_out) {
  if (!capacity_out || rows < 0 || !(factor > 0.0) || !std::isfinite(factor) || align < 1)
    return MOE_ERR_INVALID_ARG;
  const double prod = std::ceil((double)rows * factor);
  if (prod > 9.0e15) return MOE_ERR_INVALID_ARG;
  int64_t c = (int64_t)prod;
  c = (c + align - 1) / align * align;
  *capacity_out = c;
  return MOE_OK;
}

moe_status moe_decode_bucket(int64_t tokens, const int64_t* ladder, int32_t n, int64_t* bucket_out) {
  if (!ladder || !bucket_out || n < 1 || tokens < 0) return MOE_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; i++)
    if (ladder[i] < 1 || (i > 0 && ladder[i] <= ladder[i - 1])) return MOE_ERR_INVALID_ARG;
  const int64_t want = tokens > 0 ? tokens : 1;  // zero tokens keep the smallest non-empty bucket
  for (int32_t i = 0; i < n; i++)
    if (ladder[i] >= want) {
      *bucket_out = ladder[i];
      return MOE_OK;
    }
  return MOE_ERR_INVALID_ARG;  // above the largest bucket
}

moe_status moe_routing_map_bytes(int32_t format, int64_t T, int64_t E, int64_t K, size_t* bytes_out) {
  if (!bytes_out || T < 0 || E < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (format == MOE_ROUTING_SPARSE_BOOL)
    *bytes_out = (size_t)T * (size_t)E;
  else if (format == MOE_ROUTING_DENSE_I16)
    *bytes_out = (size_t)T * (size_t)K * 2;
  else
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status moe_preprocess_workspace_size(const moe_shape* shape, size_t* bytes_out) {
  MOE_TRY(check_shape(shape, false));
  if (!bytes_out) return MOE_ERR_INVALID_ARG;
  *bytes_out = preprocess_workspace_bytes(shape->T, shape->E, shape->K);
  return MOE_OK;
}

moe_status moe_preprocess(const moe_routing* routing, const moe_shape* shape, const moe_layout* layout,
                          const moe_handle_dev* handle, void* workspace, size_t workspace_bytes,
                          void* stream) {
  MOE_TRY(check_shape(shape, false));
  MOE_TRY(check_routing(routing, shape->T));
  MOE_TRY(check_layout(layout));
  MOE_TRY(check_padded_total(shape, layout));
  MOE_TRY(check_handle(handle));
  if (!workspace || !aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < preprocess_workspace_bytes(shape->T, shape->E, shape->K))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  const PreWorkspace ws = preprocess_workspace_carve(workspace, shape->T, shape->E, shape->K);
  cudaError_t e = launch_preprocess(*routing, *shape, *layout, *handle, ws, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_debug_preprocess_silent_tile(const moe_routing* routing, const moe_shape* shape,
                                            const moe_layout* layout, const moe_handle_dev* handle, void* workspace,
                                            size_t workspace_bytes, int64_t silent_tile, void* stream) {
  MOE_TRY(check_shape(shape, false));
  MOE_TRY(check_routing(routing, shape->T));
  MOE_TRY(check_layout(layout));
  MOE_TRY(check_padded_total(shape, layout));
  MOE_TRY(check_handle(handle));
  if (!workspace || !aligned16(workspace) || silent_tile < 0) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < preprocess_workspace_bytes(shape->T, shape->E, shape->K))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  const PreWorkspace ws = preprocess_workspace_carve(workspace, shape->T, shape->E, shape->K);
  cudaError_t e = launch_preprocess(*routing, *shape, *layout, *handle, ws, static_cast<cudaStream_t>(stream),
                                    silent_tile);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_dispatch_permute(const moe_handle_dev* handle, const moe_shape* shape,
                                const moe_layout* layout, int32_t in_dtype, const void* x,
                                const void* x_scales, const moe_routing* routing, void* out_tokens,
                                float* out_probs, void* out_scales, void* stream) {
  MOE_TRY(check_handle(handle));
  MOE_TRY(check_shape(shape, true));
  MOE_TRY(check_layout(layout));
  MOE_TRY(check_padded_total(shape, layout));
  MOE_TRY(check_routing(routing, shape->T));
  if ((shape->T > 0 && !x) || !out_tokens || !aligned16(x) || !aligned16(out_tokens))
    return MOE_ERR_INVALID_ARG;
  switch (in_dtype) {
    case MOE_DTYPE_BF16:
      break;
    case MOE_DTYPE_FP8_E4M3_B128:
      if ((shape->T > 0 && !x_scales) || !out_scales) return MOE_ERR_INVALID_ARG;
      break;
    case MOE_DTYPE_BF16_TO_FP8:
      if (!out_scales) return MOE_ERR_INVALID_ARG;
      break;
    case MOE_DTYPE_BF16_TO_NVFP4:
      if (!x_scales || !out_scales) return MOE_ERR_INVALID_ARG;
      break;
    default:
      return MOE_ERR_INVALID_ARG;
  }
  cudaError_t e = launch_dispatch(*handle, *shape, *layout, in_dtype, x, x_scales, *routing, out_tokens,
                                  out_probs, out_scales, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_combine_unpermute(const moe_handle_dev* handle, const moe_shape* shape,
                                 const moe_layout* layout, const void* expert_out,
                                 const float* perm_probs, void* y, void* stream) {
  MOE_TRY(check_handle(handle));
  MOE_TRY(check_shape(shape, true));
  MOE_TRY(check_layout(layout));
  MOE_TRY(check_padded_total(shape, layout));
  if (!expert_out || (shape->T > 0 && !y) || !aligned16(expert_out) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_combine(*handle, *shape, *layout, expert_out, perm_probs, y,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_combine_unpermute_fmt(const moe_handle_dev* handle, const moe_shape* shape,
                                     const moe_layout* layout, int32_t in_format, const void* expert_out,
                                     const void* expert_out_scales, const float* perm_probs, void* y,
                                     void* stream) {
  if (in_format == MOE_COMBINE_BF16)
    return moe_combine_unpermute(handle, shape, layout, expert_out, perm_probs, y, stream);
  if (in_format != MOE_COMBINE_MXFP8 && in_format != MOE_COMBINE_MXFP4) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_handle(handle));
  MOE_TRY(check_shape(shape, true));
  MOE_TRY(check_layout(layout));
  MOE_TRY(check_padded_total(shape, layout));
  if (!expert_out || !expert_out_scales || (shape->T > 0 && !y) || !aligned16(expert_out) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_combine_mx(*handle, *shape, in_format, expert_out, expert_out_scales, perm_probs, y,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_quantize_mx_rows(const void* x, int64_t R, int64_t H, int32_t format, void* codes, void* scales,
                                void* stream) {
  if (R < 0 || H <= 0 || H % 32 || (format != MOE_COMBINE_MXFP8 && format != MOE_COMBINE_MXFP4))
    return MOE_ERR_INVALID_ARG;
  if (R == 0) return MOE_OK;
  if (!x || !codes || !scales || !aligned16(x) || !aligned16(codes)) return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_quantize_mx_rows(x, R, H, format, codes, scales, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_combine_backward(const moe_handle_dev* handle, const moe_shape* shape, const moe_layout* layout,
                                const void* grad_y, const void* expert_out, const float* perm_probs,
                                void* grad_expert_out, float* grad_perm_probs, void* stream) {
  MOE_TRY(check_handle(handle));
  MOE_TRY(check_shape(shape, true));
  MOE_TRY(check_layout(layout));
  MOE_TRY(check_padded_total(shape, layout));
  if ((shape->T > 0 && !grad_y) || !grad_expert_out || !aligned16(grad_y) || !aligned16(grad_expert_out))
    return MOE_ERR_INVALID_ARG;
  if (grad_perm_probs && (!expert_out || !perm_probs || !aligned16(expert_out))) return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_combine_backward(*handle, *shape, *layout, grad_y, grad_perm_probs ? expert_out : nullptr,
                                          perm_probs, grad_expert_out, grad_perm_probs,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_dispatch_backward(const moe_handle_dev* handle, const moe_shape* shape, const moe_layout* layout,
                                 int32_t routing_format, const void* grad_perm_tokens, const float* grad_perm_probs,
                                 void* grad_x, float* grad_probs, void* stream) {
  MOE_TRY(check_handle(handle));
  MOE_TRY(check_shape(shape, true));
  MOE_TRY(check_layout(layout));
  MOE_TRY(check_padded_total(shape, layout));
  if (routing_format != MOE_ROUTING_DENSE_I16 && routing_format != MOE_ROUTING_SPARSE_BOOL)
    return MOE_ERR_INVALID_ARG;
  if (!grad_perm_tokens || (shape->T > 0 && !grad_x) || !aligned16(grad_perm_tokens) || !aligned16(grad_x))
    return MOE_ERR_INVALID_ARG;
  if ((grad_perm_probs == nullptr) != (grad_probs == nullptr)) return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_dispatch_backward(*handle, *shape, *layout, routing_format, grad_perm_tokens,
                                           grad_perm_probs, grad_x, grad_probs, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_grouped_mlp_workspace_size(const moe_shape* shape, const moe_layout* layout,
                                          int32_t w_dtype, size_t* bytes_out) {
  MOE_TRY(check_shape(shape, true));
  MOE_TRY(check_layout(layout));
  MOE_TRY(check_padded_total(shape, layout));
  if (!bytes_out || shape->I <= 0 || shape->I % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (w_dtype != MOE_DTYPE_BF16 && w_dtype != MOE_DTYPE_FP8_E4M3_B128 && w_dtype != MOE_DTYPE_NVFP4)
    return MOE_ERR_INVALID_ARG;
  *bytes_out = grouped_mlp_workspace_bytes(*shape, *layout, w_dtype);
  return MOE_OK;
}

moe_status moe_grouped_mlp_kernel_count(const moe_shape* shape, const moe_layout* layout, int32_t w_dtype,
                                        int32_t* count_out) {
  MOE_TRY(check_shape(shape, true));
  MOE_TRY(check_layout(layout));
  MOE_TRY(check_padded_total(shape, layout));
  if (!count_out || shape->I <= 0 || shape->I % 128 != 0) return MOE_ERR_INVALID_ARG;
  const int n = grouped_mlp_kernel_count(*shape, *layout, w_dtype);
  if (n < 0) return MOE_ERR_INVALID_ARG;
  *count_out = n;
  return MOE_OK;
}

moe_status moe_grouped_mlp(const moe_handle_dev* handle, const moe_shape* shape, const moe_layout* layout,
                           int32_t w_dtype, const void* perm_tokens, const void* perm_scales,
                           const void* w13, const void* w13_scales, const void* w2,
                           const void* w2_scales, const moe_nvfp4_globals* globals, void* workspace,
                           size_t workspace_bytes, void* out_fc2, void* stream) {
  return moe_grouped_mlp_ex(handle, shape, layout, w_dtype, perm_tokens, perm_scales, w13, w13_scales, w2,
                            w2_scales, globals, workspace, workspace_bytes, MOE_COMBINE_BF16, out_fc2, nullptr,
                            nullptr, stream);
}

moe_status moe_grouped_mlp_ex(const moe_handle_dev* handle, const moe_shape* shape, const moe_layout* layout,
                              int32_t w_dtype, const void* perm_tokens, const void* perm_scales,
                              const void* w13, const void* w13_scales, const void* w2,
                              const void* w2_scales, const moe_nvfp4_globals* globals, void* workspace,
                              size_t workspace_bytes, int32_t out_format, void* out_fc2, void* out_fc2_scales,
                              const float* fc2_row_probs, void* stream) {
  if (out_format != MOE_COMBINE_BF16 && out_format != MOE_COMBINE_MXFP8 && out_format != MOE_COMBINE_MXFP4)
    return MOE_ERR_INVALID_ARG;
  if (out_format != MOE_COMBINE_BF16 && (!out_fc2_scales || (reinterpret_cast<uintptr_t>(out_fc2_scales) & 3u)))
    return MOE_ERR_INVALID_ARG;
  if (fc2_row_probs && (reinterpret_cast<uintptr_t>(fc2_row_probs) & 3u)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_handle(handle));
  MOE_TRY(check_shape(shape, true));
  MOE_TRY(check_layout(layout));
  MOE_TRY(check_padded_total(shape, layout));
  if (shape->I <= 0 || shape->I % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (!perm_tokens || !w13 || !w2 || !out_fc2 || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned16(perm_tokens) || !aligned16(w13) || !aligned16(w2) || !aligned16(out_fc2) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_INVALID_ARG;
  switch (w_dtype) {
    case MOE_DTYPE_BF16:
      break;
    case MOE_DTYPE_FP8_E4M3_B128:
      if (!perm_scales || !w13_scales || !w2_scales) return MOE_ERR_INVALID_ARG;
      break;
    case MOE_DTYPE_NVFP4:
      if (!perm_scales || !w13_scales || !w2_scales || !globals || !globals->fc1_input_scale ||
          !globals->fc2_input_scale || !globals->w13_scale_2 || !globals->w2_scale_2)
        return MOE_ERR_INVALID_ARG;
      // the NVFP4 kernels stage 256 K elements at a time (FC1: K = H, FC2: K = I)
      if (shape->H % 256 != 0 || shape->I % 256 != 0) return MOE_ERR_UNSUPPORTED;
      break;
    default:
      return MOE_ERR_INVALID_ARG;
  }
  if (workspace_bytes < grouped_mlp_workspace_bytes(*shape, *layout, w_dtype)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaError_t e = launch_grouped_mlp(*handle, *shape, *layout, w_dtype, perm_tokens, perm_scales, w13,
                                     w13_scales, w2, w2_scales, globals, workspace, out_fc2, out_format,
                                     out_fc2_scales, fc2_row_probs, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_debug_next_grouped_mlp_silent_token_tile(int64_t token_tile) {
  if (token_tile < -1) return MOE_ERR_INVALID_ARG;
  set_debug_mlp_silent_tile(token_tile);
  return MOE_OK;
}

moe_status moe_profile_next_grouped_mlp(void* ev_before_fc1, void* ev_after_fc1, void* ev_after_fc2) {
  ProfileEvents e;
  e.before_fc1 = static_cast<cudaEvent_t>(ev_before_fc1);
  e.after_fc1 = static_cast<cudaEvent_t>(ev_after_fc1);
  e.after_fc2 = static_cast<cudaEvent_t>(ev_after_fc2);
  if ((e.before_fc1 || e.after_fc1 || e.after_fc2) && !(e.before_fc1 && e.after_fc1 && e.after_fc2))
    return MOE_ERR_INVALID_ARG;
  set_profile_events(e);
  return MOE_OK;
}

moe_status moe_quantize_fp8_blocks(const void* w, int64_t G, int64_t N, int64_t Kd, void* codes,
                                   float* scales, void* stream) {
  if (G < 0 || N < 0 || Kd < 0 || N % 128 || Kd % 128) return MOE_ERR_INVALID_ARG;
  if (G * N * Kd > 0 && (!w || !codes || !scales || !aligned16(w) || !aligned16(codes)))
    return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_quantize_fp8_blocks(w, G, N, Kd, codes, scales, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status moe_quantize_nvfp4_rows(const void* x, int64_t R, int64_t Kd, const float* global,
                                   void* packed, void* scales, void* stream) {
  if (R < 0 || Kd <= 0 || Kd % 16) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!x || !global || !packed || !scales || !aligned16(x) ||
                (reinterpret_cast<uintptr_t>(packed) & 7u)))
    return MOE_ERR_INVALID_ARG;
  if (R == 0) return MOE_OK;
  cudaError_t e =
      launch_quantize_nvfp4_rows(x, R, Kd, global, packed, scales, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

/* ------------------------------------------------------------ buffer ring */

struct moe_ring {
  int32_t n;
  int32_t next;
  int32_t use_events;
  bool* held;
  bool* recorded;
  cudaEvent_t* events;
};

moe_status moe_ring_create(int32_t n_slots, int32_t use_events, moe_ring** ring_out) {
  if (!ring_out || n_slots < 1 || n_slots > 4096) return MOE_ERR_INVALID_ARG;
  moe_ring* r = new (std::nothrow) moe_ring;
  if (!r) return MOE_ERR_INVALID_ARG;
  r->n = n_slots;
  r->next = 0;
  r->use_events = use_events ? 1 : 0;
  r->held = new bool[n_slots]();
  r->recorded = new bool[n_slots]();
  r->events = new cudaEvent_t[n_slots]();
  if (r->use_events) {
    for (int32_t i = 0; i < n_slots; i++) {
      cudaError_t e = cudaEventCreateWithFlags(&r->events[i], cudaEventDisableTiming);
      if (e != cudaSuccess) {
        for (int32_t j = 0; j < i; j++) cudaEventDestroy(r->events[j]);
        delete[] r->held;
        delete[] r->recorded;
        delete[] r->events;
        delete r;
        return cuda_fail(e);
      }
    }
  }
  *ring_out = r;
  return MOE_OK;
}

moe_status moe_ring_acquire(moe_ring* r, void* stream, int32_t* slot_out) {
  if (!r || !slot_out) return MOE_ERR_INVALID_ARG;
  const int32_t s = r->next;
  if (r->held[s]) return MOE_ERR_RING_EARLY_REUSE;
  if (r->use_events && r->recorded[s]) {
    cudaError_t e = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), r->events[s], 0);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  r->held[s] = true;
  r->next = (s + 1) % r->n;
  *slot_out = s;
  return MOE_OK;
}

moe_status moe_ring_release(moe_ring* r, int32_t slot, void* stream) {
  if (!r || slot < 0 || slot >= r->n) return MOE_ERR_INVALID_ARG;
  if (!r->held[slot]) return MOE_ERR_RING_DOUBLE_RELEASE;
  if (r->use_events) {
    cudaError_t e = cudaEventRecord(r->events[slot], static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    r->recorded[slot] = true;
  }
  r->held[slot] = false;
  return MOE_OK;
}

moe_status moe_ring_destroy(moe_ring* r) {
  if (!r) return MOE_ERR_INVALID_ARG;
  if (r->use_events)
    for (int32_t i = 0; i < r->n; i++) cudaEventDestroy(r->events[i]);
  delete[] r->held;
  delete[] r->recorded;
  delete[] r->events;
  delete r;
  return MOE_OK;
}

}  // extern "C"
