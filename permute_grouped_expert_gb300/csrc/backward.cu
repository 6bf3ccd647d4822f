// backward.cu -- the backward of combine and of dispatch (HBM-bound gathers and
// scatters of gradient rows, 128-bit vectors).
//
// Follows DeepEP PR #716 "perf: reuse HybridEP routing allgather buffer"
// (Testing, output and gradient regression: hidden-state and probability
// gradients for the backward of the combine and of the dispatch) and NeMo
// Automodel PR #3931 "perf(moe): sync-free HybridEP dispatch" (What does this PR
// do?: the combine's backward is a dispatch sized by the same host capacity).
//
// combine forward:  y[t] = sum_k w(r) * O[r],  r = row_of[t][k] kept
// combine backward: gO[r] = bf16(w(r) * gy[t]);  gw[r] = sum_h gy[t][h] * O[r][h]
//   one warp per route (t, k): the token's gradient row is read once per route
//   (the K routes of a token are neighbouring work items, so the repeats hit
//   L1/L2), the expert row read once and the gradient row written once; the dot
//   product is a per-lane fp32 sum in a fixed order reduced by a fixed shuffle
//   tree, so results do not depend on scheduling.  One warp per expert zeroes
//   its pad rows.
// dispatch forward:  Y[r] = x[t],  Yp[r] = p(t, k)
// dispatch backward: gx[t] = bf16(sum_k gY[r]) -- the combine kernel with
//   weight 1 -- and gp(t, k) = gYp[r] gathered into the routing layout by one
//   warp per token.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_reused(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_vec(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

struct CombineBwdParams {
  int64_t T, H, E, K, cap;
  const int32_t* row_of;
  const int32_t* offsets;
  const int32_t* counts;
  const uint8_t* gy;        // bf16 [T][H]
  const uint8_t* o;         // bf16 [cap][H] (read only when gw is formed)
  const float* perm_probs;  // [cap] or NULL (weight 1)
  uint8_t* g_o;             // bf16 [cap][H]
  float* g_w;               // [cap] or NULL
};

__device__ __forceinline__ uint32_t scale_pair(float w, uint32_t packed) {
  const float a = w * bf16_bits_to_float(packed & 0xffffu);
  const float b = w * bf16_bits_to_float(packed >> 16);
  return float_to_bf16_bits(a) | (float_to_bf16_bits(b) << 16);
}

__device__ __forceinline__ float dot_pair(uint32_t g, uint32_t o, float acc) {
  acc = fmaf(bf16_bits_to_float(g & 0xffffu), bf16_bits_to_float(o & 0xffffu), acc);
  return fmaf(bf16_bits_to_float(g >> 16), bf16_bits_to_float(o >> 16), acc);
}

__global__ void __launch_bounds__(kThreads) combine_backward_kernel(CombineBwdParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nvec = p.H / 8;
  const int64_t routes = p.T * p.K;
  const int64_t items = routes + p.E;
  for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; it < items; it += (int64_t)gridDim.x * kWarps) {
    if (it >= routes) {
      // pad rows of expert e: zero gradient rows and zero probability gradients
      const int64_t e = it - routes;
      const int64_t beg = (int64_t)p.offsets[e] + p.counts[e];
      const int64_t end = min64(p.offsets[e + 1], p.cap);
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int64_t r = beg; r < end; r++) {
        for (int64_t v = lane; v < nvec; v += 32) st_vec(p.g_o + (r * nvec + v) * 16, z);
        if (p.g_w && lane == 0) p.g_w[r] = 0.0f;
      }
      continue;
    }
    const int64_t t = it / p.K;
    const int32_t r = p.row_of[it];
    if (r < 0) continue;  // dropped route or empty slot: no row
    const float w = p.perm_probs ? p.perm_probs[r] : 1.0f;
    const uint8_t* grow = p.gy + t * nvec * 16;
    const uint8_t* orow = p.o + (int64_t)r * nvec * 16;
    uint8_t* drow = p.g_o + (int64_t)r * nvec * 16;
    const bool want_dot = p.g_w != nullptr;
    float dot = 0.0f;
    for (int64_t base = 0; base < nvec; base += 32 * kUnroll) {
      uint4 g[kUnroll], o[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; u++) {
        const int64_t idx = base + u * 32 + lane;
        if (idx < nvec) {
          g[u] = ld_reused(grow + idx * 16);
          if (want_dot) o[u] = ld_stream(orow + idx * 16);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; u++) {
        const int64_t idx = base + u * 32 + lane;
        if (idx < nvec) {
          st_vec(drow + idx * 16, make_uint4(scale_pair(w, g[u].x), scale_pair(w, g[u].y), scale_pair(w, g[u].z),
                                             scale_pair(w, g[u].w)));
          if (want_dot) {
            dot = dot_pair(g[u].x, o[u].x, dot);
            dot = dot_pair(g[u].y, o[u].y, dot);
            dot = dot_pair(g[u].z, o[u].z, dot);
            dot = dot_pair(g[u].w, o[u].w, dot);
          }
        }
      }
    }
    if (want_dot) {
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, d);
      if (lane == 0) p.g_w[r] = dot;
    }
  }
}

// The same results for hidden sizes up to 2048 (a gradient row fits in four
// or eight 16-byte registers a lane): one warp per token, whose gradient row is read
// from HBM once and kept in registers for all K routes, instead of once per
// route through L2.  The expert rows of two routes are loaded before either
// is processed, so two routes' loads are in flight at a time; each route's
// rounding and dot-product order are those of combine_backward_kernel.
template <int kTokVec>  // 16-byte vectors a lane holds: H <= 32 * kTokVec * 8
__device__ __forceinline__ void load_route(const CombineBwdParams& p, int64_t nvec, int lane, int32_t r,
                                           uint4 (&o)[kTokVec]) {
  const uint8_t* orow = p.o + (int64_t)r * nvec * 16;
#pragma unroll
  for (int u = 0; u < kTokVec; u++) {
    const int64_t idx = u * 32 + lane;
    if (idx < nvec) o[u] = ld_stream(orow + idx * 16);
  }
}

template <int kTokVec>
__device__ __forceinline__ void finish_route(const CombineBwdParams& p, int64_t nvec, int lane, int32_t r, float w,
                                             const uint4 (&g)[kTokVec], const uint4 (&o)[kTokVec], bool want_dot) {
  uint8_t* drow = p.g_o + (int64_t)r * nvec * 16;
  float dot = 0.0f;
#pragma unroll
  for (int u = 0; u < kTokVec; u++) {
    const int64_t idx = u * 32 + lane;
    if (idx < nvec) {
      st_vec(drow + idx * 16, make_uint4(scale_pair(w, g[u].x), scale_pair(w, g[u].y), scale_pair(w, g[u].z),
                                         scale_pair(w, g[u].w)));
      if (want_dot) {
        dot = dot_pair(g[u].x, o[u].x, dot);
        dot = dot_pair(g[u].y, o[u].y, dot);
        dot = dot_pair(g[u].z, o[u].z, dot);
        dot = dot_pair(g[u].w, o[u].w, dot);
      }
    }
  }
  if (want_dot) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, d);
    if (lane == 0) p.g_w[r] = dot;
  }
}

template <int kTokVec>
__global__ void __launch_bounds__(kThreads, kTokVec == 4 ? 3 : 2) combine_backward_token_kernel(CombineBwdParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nvec = p.H / 8;
  const int64_t items = p.T + p.E;
  const bool want_dot = p.g_w != nullptr;
  for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; it < items; it += (int64_t)gridDim.x * kWarps) {
    if (it >= p.T) {
      // pad rows of expert e: zero gradient rows and zero probability gradients
      const int64_t e = it - p.T;
      const int64_t beg = (int64_t)p.offsets[e] + p.counts[e];
      const int64_t end = min64(p.offsets[e + 1], p.cap);
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int64_t r = beg; r < end; r++) {
        for (int64_t v = lane; v < nvec; v += 32) st_vec(p.g_o + (r * nvec + v) * 16, z);
        if (p.g_w && lane == 0) p.g_w[r] = 0.0f;
      }
      continue;
    }
    const int64_t t = it;
    uint4 g[kTokVec];
#pragma unroll
    for (int u = 0; u < kTokVec; u++) {
      const int64_t idx = u * 32 + lane;
      if (idx < nvec) g[u] = ld_stream(p.gy + (t * nvec + idx) * 16);
    }
    for (int64_t k0 = 0; k0 < p.K; k0 += 32) {
      // lane j holds route k0 + j: its row and weight
      const int64_t kk = k0 + lane;
      const int32_t rr = kk < p.K ? p.row_of[t * p.K + kk] : -1;
      const float ww = rr >= 0 && p.perm_probs ? p.perm_probs[rr] : 1.0f;
      const int n = (int)min64(32, p.K - k0);
      for (int j = 0; j < n; j += 2) {
        const int32_t r0 = __shfl_sync(0xffffffffu, rr, j);
        const float w0 = __shfl_sync(0xffffffffu, ww, j);
        const int32_t r1 = j + 1 < n ? __shfl_sync(0xffffffffu, rr, j + 1) : -1;
        const float w1 = __shfl_sync(0xffffffffu, ww, (j + 1) & 31);
        uint4 o0[kTokVec], o1[kTokVec];
        if (want_dot && r0 >= 0) load_route(p, nvec, lane, r0, o0);  // warp-uniform conditions
        if (want_dot && r1 >= 0) load_route(p, nvec, lane, r1, o1);
        if (r0 >= 0) finish_route(p, nvec, lane, r0, w0, g, o0, want_dot);
        if (r1 >= 0) finish_route(p, nvec, lane, r1, w1, g, o1, want_dot);
      }
    }
  }
}

struct ProbGradParams {
  int format;
  int64_t T, E, K;
  const int32_t* row_of;
  const int32_t* offsets;
  const float* g_yp;  // [cap]
  float* g_p;         // dense [T][K] or sparse [T][E]
};

// gp(t, k) = gYp[row_of[t][k]] (0 for a dropped route or an empty slot), in the
// routing layout; the sparse layout's entries of unrouted experts are 0.
__global__ void __launch_bounds__(kThreads) prob_grad_gather_kernel(ProbGradParams p) {
  extern __shared__ int32_t soff[];  // [E+1] (sparse layout only)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (p.format == MOE_ROUTING_SPARSE_BOOL) {
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) soff[i] = p.offsets[i];
    __syncthreads();
  }
  for (int64_t t = (int64_t)blockIdx.x * kWarps + warp; t < p.T; t += (int64_t)gridDim.x * kWarps) {
    if (p.format == MOE_ROUTING_DENSE_I16) {
      for (int64_t k = lane; k < p.K; k += 32) {
        const int32_t r = p.row_of[t * p.K + k];
        p.g_p[t * p.K + k] = r >= 0 ? p.g_yp[r] : 0.0f;
      }
    } else {
      float* row = p.g_p + t * p.E;
      for (int64_t e = lane; e < p.E; e += 32) row[e] = 0.0f;
      __syncwarp();
      for (int64_t k = lane; k < p.K; k += 32) {
        const int32_t r = p.row_of[t * p.K + k];
        if (r >= 0) row[expert_of_row(soff, (int)p.E, r)] = p.g_yp[r];
      }
    }
    __syncwarp();
  }
}

unsigned grid_for_warps(int64_t warps) {
  int64_t blocks = (warps + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)device_sm_count() * (2048 / kThreads);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (unsigned)blocks;
}

}  // namespace

cudaError_t launch_combine_backward(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                    const void* grad_y, const void* expert_out, const float* perm_probs,
                                    void* grad_expert_out, float* grad_perm_probs, cudaStream_t st) {
  CombineBwdParams p;
  p.T = s.T;
  p.H = s.H;
  p.E = s.E;
  p.K = s.K;
  p.cap = l.capacity;
  p.row_of = h.row_of;
  p.offsets = h.padded_offsets;
  p.counts = h.tokens_per_expert;
  p.gy = static_cast<const uint8_t*>(grad_y);
  p.o = static_cast<const uint8_t*>(expert_out);
  p.perm_probs = perm_probs;
  p.g_o = static_cast<uint8_t*>(grad_expert_out);
  p.g_w = grad_perm_probs;
  if (s.H <= 32 * 4 * 8)
    combine_backward_token_kernel<4><<<grid_for_warps(s.T + s.E), kThreads, 0, st>>>(p);
  else if (s.H <= 32 * 8 * 8)
    combine_backward_token_kernel<8><<<grid_for_warps(s.T + s.E), kThreads, 0, st>>>(p);
  else
    combine_backward_kernel<<<grid_for_warps(s.T * s.K + s.E), kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_backward(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                     int32_t routing_format, const void* grad_perm_tokens,
                                     const float* grad_perm_probs, void* grad_x, float* grad_probs,
                                     cudaStream_t st) {
  // gx[t] = bf16(sum over kept k, ascending, of gY[row]): the combine with weight 1
  cudaError_t e = launch_combine(h, s, l, grad_perm_tokens, nullptr, grad_x, st);
  if (e != cudaSuccess || !grad_probs || s.T == 0) return e;
  ProbGradParams p;
  p.format = routing_format;
  p.T = s.T;
  p.E = s.E;
  p.K = s.K;
  p.row_of = h.row_of;
  p.offsets = h.padded_offsets;
  p.g_yp = grad_perm_probs;
  p.g_p = grad_probs;
  const size_t smem = routing_format == MOE_ROUTING_SPARSE_BOOL ? (size_t)(s.E + 1) * 4 : 0;
  prob_grad_gather_kernel<<<grid_for_warps(s.T), kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
