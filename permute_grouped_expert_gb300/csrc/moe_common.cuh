// moe_common.cuh -- device helpers shared by the sm_103a kernels of the MoE
// library: bounded waits, acquire/release accesses, bf16 / FP8 / FP4 packing.
#pragma once

#include <cstdio>

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

#define MOE_DEVICE __device__ __forceinline__

namespace moe {

// Bounded waits give up after this many nanoseconds of %globaltimer; the wait
// then records MOE_DEV_ERR_TIMEOUT and returns, so no kernel can hang the GPU.
constexpr uint64_t kWaitLimitNs = 2000ull * 1000ull * 1000ull;

MOE_DEVICE int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
MOE_DEVICE int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

MOE_DEVICE uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

MOE_DEVICE void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

MOE_DEVICE int32_t ld_acquire_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

MOE_DEVICE void set_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Bounds-checked build (-DMOE_CHECKED): MOE_IN_BOUNDS(site, index, limit,
// status) guards a computed index before the access it feeds; a failed check
// sets MOE_DEV_ERR_BOUNDS, prints the site, index and limit (the first few
// failures of a translation unit) and returns false so the caller skips the
// access.  In the ordinary build the check is the constant true.
#ifdef MOE_CHECKED
static __device__ int g_moe_bounds_prints;
MOE_DEVICE bool moe_in_bounds(int site, int64_t index, int64_t limit, int32_t* status) {
  if (index >= 0 && index < limit) return true;
  set_status(status, MOE_DEV_ERR_BOUNDS);
  if (atomicAdd(&g_moe_bounds_prints, 1) < 16)
    printf("moe bounds check %d failed: index %lld, limit %lld (block %d, thread %d)\n", site, (long long)index,
           (long long)limit, (int)blockIdx.x, (int)threadIdx.x);
  return false;
}
#define MOE_IN_BOUNDS(site, index, limit, status) \
  ::moe::moe_in_bounds((site), (int64_t)(index), (int64_t)(limit), (status))
#else
#define MOE_IN_BOUNDS(site, index, limit, status) true
#endif

MOE_DEVICE unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Expert owning permuted row r: largest e with offsets[e] <= r (offsets in shared memory).
MOE_DEVICE int expert_of_row(const int32_t* offsets, int E, int64_t r) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((int64_t)offsets[mid] <= r)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

MOE_DEVICE float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Round-to-nearest-even fp32 -> bf16 bit pattern (the cuda_bf16 intrinsic).
MOE_DEVICE uint32_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return (uint32_t)(*reinterpret_cast<unsigned short*>(&h));
}

// x / s from the reciprocal rs = RN(1/s): one product and one FMA correction
// step (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  For a 1x128 FP8
// block scale s = RN(amax / 448) and |x| <= amax it equals the correctly
// rounded quotient, i.e. an IEEE division; the FP8 encoders divide a block's
// values by one scale, so one reciprocal and three instructions replace a
// division per value.
MOE_DEVICE float div_by_scale(float x, float s, float rs) {
  const float q = x * rs;
  return fmaf(fmaf(-q, s, x), rs, q);
}

// Two fp32 -> E4M3 codes, nearest even, saturating (low byte = a).
MOE_DEVICE uint16_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// Two fp32 -> E2M1 codes packed in one byte, nearest even, saturating (low nibble = a).
MOE_DEVICE uint32_t e2m1x2(float a, float b) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(b), "f"(a));
  return r;
}

MOE_DEVICE float e4m3_to_float(uint32_t code) {
  __nv_fp8_e4m3 v;
  *reinterpret_cast<uint8_t*>(&v) = (uint8_t)code;
  return float(v);
}

}  // namespace moe
