// permute.cu -- dispatch_with_permute, combine with unpermute, and the FP8 /
// NVFP4 quantizers.  All HBM-bound: 128-bit vector loads and stores, one warp
// per (token, row chunk) work item so that even a decode batch of 64 tokens
// keeps every SM busy, grids sized to fill every SM.
//
// Follows Megatron-LM PR #6800 "Reuse caller-owned HybridEP dispatch and expert
// output buffers" (Summary: dispatch writes permuted tokens into a caller
// buffer; combine performs the final read), DeepEP PR #716 "perf: reuse HybridEP
// routing allgather buffer" (Testing: dispatch with permutation and combine with
// unpermutation, with and without probabilities, BF16 and FP8; bitwise
// dispatched rows) and TensorRT-LLM PR #16190 "Update CuTeDSL MegaMoE kernels"
// (TopkReduce combine; NVFP4 block scales with a global scale).
#include <algorithm>

#include <cuda_fp16.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxK = 128;
constexpr int kUnroll = 4;  // 16-byte vectors in flight per lane per chunk

struct DispatchParams {
  int format;
  const float* probs;
  int64_t T, H, E, K, cap;
  const int32_t* row_of;
  const int32_t* offsets;
  const int32_t* counts;
  const uint8_t* x;
  const float* x_scales;  // FP8 passthrough scales, or the NVFP4 global scale
  uint8_t* out;
  float* out_probs;
  uint8_t* out_scales;
  int64_t row_bytes;    // bytes of one output row
  int64_t scale_bytes;  // bytes of one output scale row
  int64_t nchunks;      // work items per token (row chunks)
  int64_t chunk_steps;  // loop steps of the row per chunk
  int32_t* status;      // handle status word (bounds-checked builds report there)
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_vec(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Destination rows of token t into this warp's shared slots; with
// write_probs also writes the dispatched probabilities (once per token: by the
// warp that copies the token's first chunk).
__device__ __forceinline__ void load_dests(const DispatchParams& p, const int32_t* soff, int64_t t,
                                           int32_t* sdest, bool write_probs) {
  const int lane = threadIdx.x & 31;
  for (int k = lane; k < p.K; k += 32) {
    int32_t d = p.row_of[t * p.K + k];
    if (d >= 0 && !MOE_IN_BOUNDS(1, d, p.cap, p.status)) d = -1;
    sdest[k] = d;
    if (write_probs && d >= 0 && p.out_probs && p.probs) {
      float pr;
      if (p.format == MOE_ROUTING_DENSE_I16)
        pr = p.probs[t * p.K + k];
      else
        pr = p.probs[t * p.E + expert_of_row(soff, (int)p.E, d)];
      p.out_probs[d] = pr;
    }
  }
  __syncwarp();
}

// Zero the pad rows of expert e (tokens, scales, probabilities).
__device__ __forceinline__ void zero_pads(const DispatchParams& p, const int32_t* soff, int e) {
  const int lane = threadIdx.x & 31;
  const int64_t beg = (int64_t)soff[e] + p.counts[e];
  const int64_t end = min64(soff[e + 1], p.cap);
  const uint4 z = make_uint4(0, 0, 0, 0);
  if (beg < end && !MOE_IN_BOUNDS(2, beg, p.cap, p.status)) return;
  for (int64_t r = beg; r < end; r++) {
    uint8_t* row = p.out + r * p.row_bytes;
    for (int64_t v = lane; v < p.row_bytes / 16; v += 32) st_vec(row + v * 16, z);
    if (p.out_scales) {
      uint8_t* srow = p.out_scales + r * p.scale_bytes;
      for (int64_t b = lane; b < p.scale_bytes; b += 32) srow[b] = 0;
    }
    if (p.out_probs && lane == 0) p.out_probs[r] = 0.0f;
  }
}

// BF16 or FP8 rows copied bit for bit (plus FP8 scale rows).
__global__ void __launch_bounds__(kThreads) dispatch_copy_kernel(DispatchParams p) {
  __shared__ int32_t s_dest[kWarps][kMaxK];
  extern __shared__ int32_t soff[];
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) soff[i] = p.offsets[i];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nvec = p.row_bytes / 16;
  const int64_t nsc = p.scale_bytes / 4;
  const int64_t nchunks = p.nchunks;
  const int64_t items = p.T * nchunks + p.E;
  for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; it < items; it += (int64_t)gridDim.x * kWarps) {
    if (it >= p.T * nchunks) {
      zero_pads(p, soff, (int)(it - p.T * nchunks));
      continue;
    }
    const int64_t t = it / nchunks, chunk = it - t * nchunks;
    load_dests(p, soff, t, s_dest[warp], chunk == 0);
    const uint8_t* src = p.x + t * p.row_bytes;
    const int64_t vend = min64(nvec, (chunk + 1) * p.chunk_steps * 32 * kUnroll);
    for (int64_t base = chunk * p.chunk_steps * 32 * kUnroll; base < vend; base += 32 * kUnroll) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; u++) {
        const int64_t idx = base + u * 32 + lane;
        if (idx < vend) v[u] = ld_stream(src + idx * 16);
      }
      for (int k = 0; k < p.K; k++) {
        const int32_t d = s_dest[warp][k];
        if (d < 0) continue;
        uint8_t* dst = p.out + (int64_t)d * p.row_bytes;
#pragma unroll
        for (int u = 0; u < kUnroll; u++) {
          const int64_t idx = base + u * 32 + lane;
          if (idx < vend) st_vec(dst + idx * 16, v[u]);
        }
      }
    }
    if (nsc && chunk == 0) {
      const float* ssrc = p.x_scales + t * nsc;
      for (int64_t b = lane; b < nsc; b += 32) {
        const float sv = ssrc[b];
        for (int k = 0; k < p.K; k++) {
          const int32_t d = s_dest[warp][k];
          if (d >= 0) reinterpret_cast<float*>(p.out_scales + (int64_t)d * p.scale_bytes)[b] = sv;
        }
      }
    }
    __syncwarp();
  }
}

// bf16 rows quantized to E4M3 with one fp32 scale per 128 elements, then
// scattered.  A lane holds 8 elements; 16 lanes hold one 128-element block.
__global__ void __launch_bounds__(kThreads) dispatch_fp8_kernel(DispatchParams p) {
  __shared__ int32_t s_dest[kWarps][kMaxK];
  extern __shared__ int32_t soff[];
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) soff[i] = p.offsets[i];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t H = p.H;
  const int64_t kChunk = p.chunk_steps * 512;  // elements of a row one work item quantizes
  const int64_t nchunks = p.nchunks;
  const int64_t items = p.T * nchunks + p.E;
  for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; it < items; it += (int64_t)gridDim.x * kWarps) {
    if (it >= p.T * nchunks) {
      zero_pads(p, soff, (int)(it - p.T * nchunks));
      continue;
    }
    const int64_t t = it / nchunks, chunk = it - t * nchunks;
    load_dests(p, soff, t, s_dest[warp], chunk == 0);
    const uint8_t* src = p.x + t * H * 2;
    const int64_t chunk_end = min64(H, (chunk + 1) * kChunk);
    // each lane encodes 16 consecutive elements (one 16-byte code store a
    // destination); eight lanes share a 128-element scale block
    for (int64_t base = chunk * kChunk; base < chunk_end; base += 512 * 2) {
      uint4 q[2];
      float sc[2];
      bool live[2];
#pragma unroll
      for (int u = 0; u < 2; u++) {
        const int64_t e0 = base + u * 512 + lane * 16;
        live[u] = e0 < chunk_end;  // H and the chunk are multiples of 128: an 8-lane block is live or dead as a whole
        const uint4 v0 = live[u] ? ld_stream(src + e0 * 2) : make_uint4(0, 0, 0, 0);
        const uint4 v1 = live[u] ? ld_stream(src + e0 * 2 + 16) : make_uint4(0, 0, 0, 0);
        float f[16];
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int j = 0; j < 8; j++) {
          f[2 * j] = bf16_bits_to_float(w[j] & 0xffffu);
          f[2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
        }
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; j++) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
        for (int d = 4; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
        const float rs = __frcp_rn(s);
        sc[u] = s;
        uint32_t c[8];
#pragma unroll
        for (int j = 0; j < 8; j++) c[j] = e4m3x2(div_by_scale(f[2 * j], s, rs), div_by_scale(f[2 * j + 1], s, rs));
        q[u] = make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16), c[6] | (c[7] << 16));
      }
      for (int k = 0; k < p.K; k++) {
        const int32_t d = s_dest[warp][k];
        if (d < 0) continue;
        uint8_t* dst = p.out + (int64_t)d * H;
        float* sdst = reinterpret_cast<float*>(p.out_scales + (int64_t)d * p.scale_bytes);
#pragma unroll
        for (int u = 0; u < 2; u++) {
          if (!live[u]) continue;
          const int64_t e0 = base + u * 512 + lane * 16;
          st_vec(dst + e0, q[u]);
          if ((lane & 7) == 0) sdst[e0 / 128] = sc[u];
        }
      }
    }
    __syncwarp();
  }
}

// bf16 rows quantized to NVFP4 (E2M1 + one E4M3 scale per 16 elements + the
// fp32 global scale), then scattered.  A lane holds 8 elements; 2 lanes hold
// one 16-element block.
__global__ void __launch_bounds__(kThreads) dispatch_nvfp4_kernel(DispatchParams p) {
  __shared__ int32_t s_dest[kWarps][kMaxK];
  extern __shared__ int32_t soff[];
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) soff[i] = p.offsets[i];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t H = p.H;
  const float g = *p.x_scales;
  const int64_t kChunk = p.chunk_steps * 256;  // elements of a row one work item quantizes
  const int64_t nchunks = p.nchunks;
  const int64_t items = p.T * nchunks + p.E;
  for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; it < items; it += (int64_t)gridDim.x * kWarps) {
    if (it >= p.T * nchunks) {
      zero_pads(p, soff, (int)(it - p.T * nchunks));
      continue;
    }
    const int64_t t = it / nchunks, chunk = it - t * nchunks;
    load_dests(p, soff, t, s_dest[warp], chunk == 0);
    const uint8_t* src = p.x + t * H * 2;
    const int64_t chunk_end = min64(H, (chunk + 1) * kChunk);
    for (int64_t base = chunk * kChunk; base < chunk_end; base += 256) {
      const int64_t e0 = base + lane * 8;
      const bool live = e0 < chunk_end;
      uint4 v = live ? ld_stream(src + e0 * 2) : make_uint4(0, 0, 0, 0);
      float f[8];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        f[2 * j] = bf16_bits_to_float(w[j] & 0xffffu);
        f[2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
      }
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; j++) amax = fmaxf(amax, fabsf(f[j]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      const uint32_t scode = e4m3x2(__fdiv_rn(amax, 6.0f * g), 0.0f) & 0xffu;
      const float denom = e4m3_to_float(scode) * g;
      uint32_t packed = 0;
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const uint32_t b = (denom == 0.0f)
                               ? 0u
                               : e2m1x2(__fdiv_rn(f[2 * j], denom), __fdiv_rn(f[2 * j + 1], denom));
        packed |= b << (8 * j);
      }
      for (int k = 0; k < p.K; k++) {
        const int32_t d = s_dest[warp][k];
        if (d < 0 || !live) continue;
        if (!MOE_IN_BOUNDS(3, e0 + 8, H + 1, p.status)) continue;
        *reinterpret_cast<uint32_t*>(p.out + (int64_t)d * (H / 2) + e0 / 2) = packed;
        if ((lane & 1) == 0) p.out_scales[(int64_t)d * (H / 16) + e0 / 16] = (uint8_t)scode;
      }
    }
    __syncwarp();
  }
}

struct CombineParams {
  int64_t T, H, K;
  int64_t nchunks, chunk_steps;  // work items per token; 64-vector steps per item
  const int32_t* row_of;
  const uint8_t* o;
  const float* perm_probs;
  uint8_t* y;
};

// y[t] = bf16(sum_k w_k * O[row_k]) with fp32 accumulation in ascending k.
__global__ void __launch_bounds__(kThreads) combine_kernel(CombineParams p) {
  __shared__ int32_t s_row[kWarps][kMaxK];
  __shared__ float s_w[kWarps][kMaxK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nvec = p.H / 8;
  const int64_t nchunks = p.nchunks;
  const int64_t items = p.T * nchunks;
  for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; it < items; it += (int64_t)gridDim.x * kWarps) {
    const int64_t t = it / nchunks, chunk = it - t * nchunks;
    int nk = 0;
    for (int k0 = 0; k0 < p.K; k0 += 32) {
      const int k = k0 + lane;
      int32_t r = (k < p.K) ? p.row_of[t * p.K + k] : -1;
      const unsigned keep = __ballot_sync(0xffffffffu, r >= 0);
      if (r >= 0) {
        const int slot = nk + __popc(keep & lanemask_lt());  // kept routes, ascending k
        s_row[warp][slot] = r;
        s_w[warp][slot] = p.perm_probs ? p.perm_probs[r] : 1.0f;
      }
      nk += __popc(keep);
    }
    __syncwarp();
    const int64_t vend = min64(nvec, (chunk + 1) * p.chunk_steps * 64);
    for (int64_t base = chunk * p.chunk_steps * 64; base < vend; base += 64) {
      float acc[2][8];
#pragma unroll
      for (int u = 0; u < 2; u++)
#pragma unroll
        for (int j = 0; j < 8; j++) acc[u][j] = 0.0f;
      for (int k0 = 0; k0 < nk; k0 += 8) {
        uint4 v[8][2];
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          if (k0 + kk < nk) {
            const uint8_t* row = p.o + (int64_t)s_row[warp][k0 + kk] * p.H * 2;
#pragma unroll
            for (int u = 0; u < 2; u++) {
              const int64_t idx = base + u * 32 + lane;
              if (idx < nvec) v[kk][u] = ld_stream(row + idx * 16);
            }
          }
        }
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          if (k0 + kk < nk) {
            const float wk = s_w[warp][k0 + kk];
#pragma unroll
            for (int u = 0; u < 2; u++) {
              const uint32_t w4[4] = {v[kk][u].x, v[kk][u].y, v[kk][u].z, v[kk][u].w};
#pragma unroll
              for (int j = 0; j < 4; j++) {
                acc[u][2 * j] = fmaf(wk, bf16_bits_to_float(w4[j] & 0xffffu), acc[u][2 * j]);
                acc[u][2 * j + 1] = fmaf(wk, bf16_bits_to_float(w4[j] >> 16), acc[u][2 * j + 1]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 2; u++) {
        const int64_t idx = base + u * 32 + lane;
        if (idx < nvec) {
          uint4 out;
          out.x = float_to_bf16_bits(acc[u][0]) | (float_to_bf16_bits(acc[u][1]) << 16);
          out.y = float_to_bf16_bits(acc[u][2]) | (float_to_bf16_bits(acc[u][3]) << 16);
          out.z = float_to_bf16_bits(acc[u][4]) | (float_to_bf16_bits(acc[u][5]) << 16);
          out.w = float_to_bf16_bits(acc[u][6]) | (float_to_bf16_bits(acc[u][7]) << 16);
          st_vec(p.y + t * p.H * 2 + idx * 16, out);
        }
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------- MX combine formats
// E4M3 (MXFP8) or E2M1 (MXFP4) elements with one E8M0 scale 2^X per 32: X =
// floor(log2(amax)) - emax (8 for E4M3, 2 for E2M1) clamped to [-127, 127], 0
// for an all-zero block; element = x / 2^X rounded to nearest even, saturating.

// 2^(code - 127) for an E8M0 code in [0, 254] (code 0 is the fp32 subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_float(uint32_t code) {
  return code ? __uint_as_float(code << 23) : __uint_as_float(0x00400000u);
}

// Shared exponent X of a block with magnitude maximum amax (exact, from the fp32 bits).
__device__ __forceinline__ int mx_exponent(float amax, int emax) {
  if (amax == 0.0f) return 0;
  const int field = (int)((__float_as_uint(amax) >> 23) & 0xff);  // 0 for a subnormal: floor(log2) <= -127
  const int X = (field == 0 ? -127 : field - 127) - emax;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// Two E4M3 codes (low byte first) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t pair) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(pair));
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Two E2M1 codes in one byte (low nibble first) -> two floats.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(byte));
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

struct CombineMxParams {
  int64_t T, H, K;
  int64_t nchunks, chunk_steps;  // work items per token; loop steps per item
  const int32_t* row_of;
  const uint8_t* codes;   // E4M3 [cap][H] or packed E2M1 [cap][H/2]
  const uint8_t* scales;  // E8M0 [cap][H/32]
  const float* perm_probs;
  uint8_t* y;
};

// y[t] = bf16(sum_k w_k * decoded O[row_k]), fp32 accumulation in ascending k.
// A lane handles one MX block (32 consecutive elements, one scale byte) per
// step and loads it for up to 8 routes at once: 8 x 32 bytes in flight per lane
// for MXFP8, 8 x 16 for MXFP4.
template <int kElem>
__global__ void __launch_bounds__(kThreads, 2) combine_mx_kernel(CombineMxParams p) {
  __shared__ int32_t s_row[kWarps][kMaxK];
  __shared__ float s_w[kWarps][kMaxK];
  constexpr int kKC = 8;                       // routes loaded together
  constexpr int kVec = kElem == 0 ? 2 : 1;     // 16-byte vectors per block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nblk = p.H / 32;
  const int64_t row_bytes = kElem == 0 ? p.H : p.H / 2;
  const int64_t items = p.T * p.nchunks;
  for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; it < items; it += (int64_t)gridDim.x * kWarps) {
    const int64_t t = it / p.nchunks, chunk = it - t * p.nchunks;
    int nk = 0;
    for (int k0 = 0; k0 < p.K; k0 += 32) {
      const int k = k0 + lane;
      int32_t r = (k < p.K) ? p.row_of[t * p.K + k] : -1;
      const unsigned keep = __ballot_sync(0xffffffffu, r >= 0);
      if (r >= 0) {
        const int slot = nk + __popc(keep & lanemask_lt());
        s_row[warp][slot] = r;
        s_w[warp][slot] = p.perm_probs ? p.perm_probs[r] : 1.0f;
      }
      nk += __popc(keep);
    }
    __syncwarp();
    const int64_t bend = min64(nblk, (chunk + 1) * p.chunk_steps * 32);
    for (int64_t b = chunk * p.chunk_steps * 32 + lane; b < bend; b += 32) {
      float acc[32];
#pragma unroll
      for (int j = 0; j < 32; j++) acc[j] = 0.0f;
      for (int k0 = 0; k0 < nk; k0 += kKC) {
        uint4 v[kKC][kVec];
        uint32_t sc[kKC];
#pragma unroll
        for (int kk = 0; kk < kKC; kk++) {
          if (k0 + kk < nk) {
            const int64_t r = s_row[warp][k0 + kk];
#pragma unroll
            for (int q = 0; q < kVec; q++) v[kk][q] = ld_stream(p.codes + r * row_bytes + b * 16 * kVec + 16 * q);
            sc[kk] = __ldg(p.scales + r * nblk + b);
          }
        }
#pragma unroll
        for (int kk = 0; kk < kKC; kk++) {
          if (k0 + kk < nk) {
            const float ws = e8m0_to_float(sc[kk]) * s_w[warp][k0 + kk];
            if (kElem == 0) {
#pragma unroll
              for (int q = 0; q < 2; q++) {
                const uint32_t w4[4] = {v[kk][q].x, v[kk][q].y, v[kk][q].z, v[kk][q].w};
#pragma unroll
                for (int i = 0; i < 4; i++) {
                  const float2 a = e4m3x2_to_float2(w4[i] & 0xffffu), c = e4m3x2_to_float2(w4[i] >> 16);
                  float* d = acc + 16 * q + 4 * i;
                  d[0] = fmaf(ws, a.x, d[0]);
                  d[1] = fmaf(ws, a.y, d[1]);
                  d[2] = fmaf(ws, c.x, d[2]);
                  d[3] = fmaf(ws, c.y, d[3]);
                }
              }
            } else {
              const uint32_t w4[4] = {v[kk][0].x, v[kk][0].y, v[kk][0].z, v[kk][0].w};
#pragma unroll
              for (int q = 0; q < 16; q++) {
                const float2 a = e2m1x2_to_float2((w4[q >> 2] >> (8 * (q & 3))) & 0xffu);
                acc[2 * q] = fmaf(ws, a.x, acc[2 * q]);
                acc[2 * q + 1] = fmaf(ws, a.y, acc[2 * q + 1]);
              }
            }
          }
        }
      }
      uint8_t* dst = p.y + (t * p.H + b * 32) * 2;
#pragma unroll
      for (int q = 0; q < 4; q++) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; j++)
          o[j] = float_to_bf16_bits(acc[8 * q + 2 * j]) | (float_to_bf16_bits(acc[8 * q + 2 * j + 1]) << 16);
        st_vec(dst + 16 * q, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
    __syncwarp();
  }
}

// One thread per 32-element block of bf16 rows [R][H] -> MX codes + E8M0 scale.
template <int kElem>
__global__ void __launch_bounds__(256) quantize_mx_rows_kernel(const uint8_t* x, int64_t R, int64_t H, uint8_t* codes,
                                                               uint8_t* scales) {
  const int64_t nblk = R * (H / 32);
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += (int64_t)gridDim.x * blockDim.x) {
    float f[32];
#pragma unroll
    for (int v = 0; v < 4; v++) {
      const uint4 q = ld_stream(x + b * 64 + v * 16);
      const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        f[v * 8 + 2 * j] = bf16_bits_to_float(w4[j] & 0xffffu);
        f[v * 8 + 2 * j + 1] = bf16_bits_to_float(w4[j] >> 16);
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; j++) amax = fmaxf(amax, fabsf(f[j]));
    const int X = mx_exponent(amax, kElem == 0 ? 8 : 2);
    const float inv = X < 127 ? __uint_as_float((uint32_t)(127 - X) << 23) : __uint_as_float(0x00400000u);
    if (kElem == 0) {
      uint32_t c[16];
#pragma unroll
      for (int j = 0; j < 16; j++) c[j] = e4m3x2(f[2 * j] * inv, f[2 * j + 1] * inv);
      uint8_t* dst = codes + b * 32;
      st_vec(dst, make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16), c[6] | (c[7] << 16)));
      st_vec(dst + 16,
             make_uint4(c[8] | (c[9] << 16), c[10] | (c[11] << 16), c[12] | (c[13] << 16), c[14] | (c[15] << 16)));
    } else {
      uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
      for (int j = 0; j < 16; j++) w[j >> 2] |= e2m1x2(f[2 * j] * inv, f[2 * j + 1] * inv) << (8 * (j & 3));
      st_vec(codes + b * 16, make_uint4(w[0], w[1], w[2], w[3]));
    }
    scales[b] = (uint8_t)(X + 127);
  }
}

// One CTA per 128x128 block of a bf16 weight [G][N][Kd]: fp32 scale amax/448
// (1 for an all-zero block) and E4M3 codes of w / scale.
__global__ void __launch_bounds__(256) quantize_fp8_blocks_kernel(const uint8_t* w, int64_t N,
                                                                  int64_t Kd, uint8_t* codes,
                                                                  float* scales) {
  __shared__ float s_max[8];
  const int64_t kb = blockIdx.x, nb = blockIdx.y, g = blockIdx.z;
  const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int64_t r = g * N + nb * 128 + row;
  const uint8_t* src = w + (r * Kd + kb * 128 + half * 64) * 2;
  float f[64];
  float amax = 0.0f;
#pragma unroll
  for (int v = 0; v < 8; v++) {
    const uint4 q = ld_stream(src + v * 16);
    const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
      f[v * 8 + 2 * j] = bf16_bits_to_float(w4[j] & 0xffffu);
      f[v * 8 + 2 * j + 1] = bf16_bits_to_float(w4[j] >> 16);
    }
  }
#pragma unroll
  for (int j = 0; j < 64; j++) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = s_max[0];
#pragma unroll
  for (int i = 1; i < 8; i++) amax = fmaxf(amax, s_max[i]);
  const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
  uint8_t* dst = codes + r * Kd + kb * 128 + half * 64;
#pragma unroll
  for (int v = 0; v < 4; v++) {
    uint4 o;
    uint32_t c[8];
#pragma unroll
    for (int j = 0; j < 8; j++) c[j] = e4m3x2(__fdiv_rn(f[v * 16 + 2 * j], s), __fdiv_rn(f[v * 16 + 2 * j + 1], s));
    o.x = c[0] | (c[1] << 16);
    o.y = c[2] | (c[3] << 16);
    o.z = c[4] | (c[5] << 16);
    o.w = c[6] | (c[7] << 16);
    st_vec(dst + v * 16, o);
  }
  if (threadIdx.x == 0) scales[(g * (N / 128) + nb) * (Kd / 128) + kb] = s;
}

// One thread per 16-element block of bf16 rows [R][Kd] -> NVFP4.
__global__ void __launch_bounds__(256) quantize_nvfp4_rows_kernel(const uint8_t* x, int64_t R, int64_t Kd,
                                                                  const float* global, uint8_t* packed,
                                                                  uint8_t* scales) {
  const float g = *global;
  const int64_t nblk = R * (Kd / 16);
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const uint8_t* src = x + b * 32;
    float f[16];
#pragma unroll
    for (int v = 0; v < 2; v++) {
      const uint4 q = ld_stream(src + v * 16);
      const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        f[v * 8 + 2 * j] = bf16_bits_to_float(w4[j] & 0xffffu);
        f[v * 8 + 2 * j + 1] = bf16_bits_to_float(w4[j] >> 16);
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; j++) amax = fmaxf(amax, fabsf(f[j]));
    const uint32_t scode = e4m3x2(__fdiv_rn(amax, 6.0f * g), 0.0f) & 0xffu;
    const float denom = e4m3_to_float(scode) * g;
    uint32_t w0 = 0, w1 = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const uint32_t c =
          (denom == 0.0f) ? 0u : e2m1x2(__fdiv_rn(f[2 * j], denom), __fdiv_rn(f[2 * j + 1], denom));
      if (j < 4)
        w0 |= c << (8 * j);
      else
        w1 |= c << (8 * (j - 4));
    }
    *reinterpret_cast<uint2*>(packed + b * 8) = make_uint2(w0, w1);
    scales[b] = (uint8_t)scode;
  }
}

// Work items per token: a row of `steps` loop steps is split into chunks only
// when the tokens alone would leave SMs idle (fewer than ~16 warps of work per
// SM, as in decode batches); long runs of work per warp keep more loads in
// flight, so large batches keep one item per token.
void row_split(int64_t T, int64_t steps, int64_t* nchunks, int64_t* chunk_steps) {
  const int64_t want = (int64_t)device_sm_count() * 16;
  int64_t n = T > 0 ? (want + T - 1) / T : 1;
  if (n > steps) n = steps;
  if (n < 1) n = 1;
  const int64_t cs = steps > 0 ? (steps + n - 1) / n : 1;
  *chunk_steps = cs;
  *nchunks = steps > 0 ? (steps + cs - 1) / cs : 1;
}

unsigned grid_for(int64_t items_warps) {
  const int64_t per_sm = 2048 / kThreads;
  int64_t blocks = (items_warps + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (unsigned)blocks;
}

}  // namespace

cudaError_t launch_dispatch(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                            int32_t in_dtype, const void* x, const void* x_scales,
                            const moe_routing& r, void* out_tokens, float* out_probs,
                            void* out_scales, cudaStream_t st) {
  DispatchParams p;
  p.format = r.format;
  p.probs = r.probs;
  p.T = s.T;
  p.H = s.H;
  p.E = s.E;
  p.K = s.K;
  p.cap = l.capacity;
  p.row_of = h.row_of;
  p.offsets = h.padded_offsets;
  p.counts = h.tokens_per_expert;
  p.x = static_cast<const uint8_t*>(x);
  p.x_scales = static_cast<const float*>(x_scales);
  p.out = static_cast<uint8_t*>(out_tokens);
  p.out_probs = out_probs;
  p.out_scales = static_cast<uint8_t*>(out_scales);
  p.status = h.status;
  const size_t smem = (size_t)(s.E + 1) * 4;
  // one warp per (token, row chunk) work item, plus one per expert for its pad rows
  switch (in_dtype) {
    case MOE_DTYPE_BF16:
      p.row_bytes = s.H * 2;
      p.scale_bytes = 0;
      p.out_scales = nullptr;
      row_split(s.T, (p.row_bytes / 16 + 32 * kUnroll - 1) / (32 * kUnroll), &p.nchunks, &p.chunk_steps);
      dispatch_copy_kernel<<<grid_for(s.T * p.nchunks + s.E), kThreads, smem, st>>>(p);
      break;
    case MOE_DTYPE_FP8_E4M3_B128:
      p.row_bytes = s.H;
      p.scale_bytes = (s.H / 128) * 4;
      row_split(s.T, (p.row_bytes / 16 + 32 * kUnroll - 1) / (32 * kUnroll), &p.nchunks, &p.chunk_steps);
      dispatch_copy_kernel<<<grid_for(s.T * p.nchunks + s.E), kThreads, smem, st>>>(p);
      break;
    case MOE_DTYPE_BF16_TO_FP8:
      p.row_bytes = s.H;
      p.scale_bytes = (s.H / 128) * 4;
      row_split(s.T, (s.H + 511) / 512, &p.nchunks, &p.chunk_steps);
      dispatch_fp8_kernel<<<grid_for(s.T * p.nchunks + s.E), kThreads, smem, st>>>(p);
      break;
    case MOE_DTYPE_BF16_TO_NVFP4:
      p.row_bytes = s.H / 2;
      p.scale_bytes = s.H / 16;
      row_split(s.T, (s.H + 255) / 256, &p.nchunks, &p.chunk_steps);
      dispatch_nvfp4_kernel<<<grid_for(s.T * p.nchunks + s.E), kThreads, smem, st>>>(p);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                           const void* expert_out, const float* perm_probs, void* y,
                           cudaStream_t st) {
  (void)l;
  CombineParams p;
  p.T = s.T;
  p.H = s.H;
  p.K = s.K;
  p.row_of = h.row_of;
  p.o = static_cast<const uint8_t*>(expert_out);
  p.perm_probs = perm_probs;
  p.y = static_cast<uint8_t*>(y);
  row_split(s.T, (s.H / 8 + 63) / 64, &p.nchunks, &p.chunk_steps);
  combine_kernel<<<grid_for(s.T * p.nchunks), kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_combine_mx(const moe_handle_dev& h, const moe_shape& s, int32_t in_format,
                              const void* codes, const void* scales, const float* perm_probs, void* y,
                              cudaStream_t st) {
  CombineMxParams p;
  p.T = s.T;
  p.H = s.H;
  p.K = s.K;
  p.row_of = h.row_of;
  p.codes = static_cast<const uint8_t*>(codes);
  p.scales = static_cast<const uint8_t*>(scales);
  p.perm_probs = perm_probs;
  p.y = static_cast<uint8_t*>(y);
  row_split(s.T, (s.H / 32 + 31) / 32, &p.nchunks, &p.chunk_steps);
  if (in_format == MOE_COMBINE_MXFP8)
    combine_mx_kernel<0><<<grid_for(s.T * p.nchunks), kThreads, 0, st>>>(p);
  else
    combine_mx_kernel<1><<<grid_for(s.T * p.nchunks), kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quantize_mx_rows(const void* x, int64_t R, int64_t H, int32_t format, void* codes, void* scales,
                                    cudaStream_t st) {
  const int64_t nblk = R * (H / 32);
  int64_t blocks = (nblk + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (format == MOE_COMBINE_MXFP8)
    quantize_mx_rows_kernel<0><<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint8_t*>(x), R, H,
                                                                 static_cast<uint8_t*>(codes),
                                                                 static_cast<uint8_t*>(scales));
  else
    quantize_mx_rows_kernel<1><<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint8_t*>(x), R, H,
                                                                 static_cast<uint8_t*>(codes),
                                                                 static_cast<uint8_t*>(scales));
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp8_blocks(const void* w, int64_t G, int64_t N, int64_t Kd, void* codes,
                                       float* scales, cudaStream_t st) {
  if (G == 0 || N == 0 || Kd == 0) return cudaSuccess;
  dim3 grid((unsigned)(Kd / 128), (unsigned)(N / 128), (unsigned)G);
  quantize_fp8_blocks_kernel<<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(w), N, Kd,
                                                   static_cast<uint8_t*>(codes), scales);
  return cudaGetLastError();
}

cudaError_t launch_quantize_nvfp4_rows(const void* x, int64_t R, int64_t Kd, const float* global,
                                       void* packed, void* scales, cudaStream_t st) {
  const int64_t nblk = R * (Kd / 16);
  int64_t blocks = (nblk + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  quantize_nvfp4_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(
      static_cast<const uint8_t*>(x), R, Kd, global, static_cast<uint8_t*>(packed),
      static_cast<uint8_t*>(scales));
  return cudaGetLastError();
}

}  // namespace moe
