// gemm_nvfp4.cu -- persistent grouped GEMMs of the expert MLP with NVFP4
// operands (E2M1 values, one E4M3 scale per 16 consecutive K elements, one fp32
// global scale per tensor), shaped for decode batches: a few tokens per expert,
// so the work is bound by streaming the expert weights from HBM.
//
// Follows TensorRT-LLM PR #16190 "Update CuTeDSL MegaMoE kernels" (commit
// list: NVFP4 w3_w1_weight / w2_weight with block scales, weight_scale_2 and
// input_scale with the epilogue alpha derived from both; decode launches sized
// by the real token count instead of the prefill maximum).
//
// Orientation ("swap AB"): the weight tile is the MMA's M = 128 side and the
// expert's tokens the N = 32 side, D^T = W . X^T, so no MMA lane is wasted on
// the handful of rows a decode batch routes to each expert.  E2M1 x E4M3 is
// exactly representable in f16 (at most 6 significant bits, magnitudes in
// [2^-10, 2688]), so converter warps expand both operands to f16 in shared
// memory exactly and tcgen05.mma kind::f16 accumulates in fp32; the two fp32
// global scales (alpha = activation global x expert weight global) are applied
// in the epilogue.
//
// One CTA per SM, 14 warps:
//   warp 0      TMA producer: raw stages of 256 K elements (packed weights
//               128 rows x 128 B, their scales 128 x 16 B, packed tokens 32 x 128 B,
//               their scales 32 x 16 B), 4 stages
//   warp 1      TMEM allocation (2 x 32 fp32 columns) and MMA issue
//   warps 2..9  converters: E2M1 + E4M3 -> f16, written in the 128-byte swizzled
//               K-major layout the MMA reads, 64 K elements per converted stage
//               (5 stages);
//               each thread expands half a weight row (plus, for 64 threads, half
//               a token row; token rows past the expert's end are skipped)
//   warps 10..13 epilogue: FC1 exchanges gate rows through shared memory, applies
//               SwiGLU and re-encodes the intermediate to NVFP4; FC2 writes bf16.
// Every wait is bounded (MOE_DEV_ERR_TIMEOUT, then a clean exit).
#include "moe_internal.h"
#include "sm100_ptx.cuh"
#include "tensor_map.h"

namespace moe {

namespace {

using namespace sm100;

constexpr int BMW = 128;        // weight rows per tile (MMA M)
constexpr int BNT = 32;         // tokens per tile (MMA N)
static_assert(BNT == 32, "the FC2 epilogue hands one token per lane");
constexpr int BKR = 256;        // K elements per raw stage
constexpr int BKC = 64;         // K elements per converted slice (one 128-byte swizzle atom of f16)
constexpr int kRawStages = 4;
constexpr int kCvtWarps = 8;
constexpr int kThreads = 64 + 32 * kCvtWarps + 128;
constexpr uint32_t kRawW = BMW * (BKR / 2);        // 16 KB packed weights
constexpr uint32_t kRawWS = BMW * (BKR / 16);      // 2 KB weight scales
constexpr uint32_t kRawX = BNT * (BKR / 2);        // 4 KB packed tokens
constexpr uint32_t kRawXS = BNT * (BKR / 16);      // 512 B token scales
constexpr uint32_t kRawBytes = kRawW + kRawWS + kRawX + kRawXS;
constexpr uint32_t kRawStride = 23552;             // kRawBytes rounded up to 1024
constexpr uint32_t kCvtW = BMW * BKC * 2;          // 16 KB
constexpr uint32_t kCvtX = BNT * BKC * 2;          // 4 KB
constexpr uint32_t kCvtSlice = kCvtW + kCvtX;      // 20 KB: one slice, weights then tokens
// Converted stages.  FC2 hands two slices (128 K) to the tensor cores per stage,
// one proxy fence and one barrier arrival per 128 K per converter warp (3
// stages); FC1, which keeps 25 KB of static shared memory for its gate
// exchange, runs five one-slice stages, which measured faster there than two
// two-slice stages.
template <int kMode>
constexpr int slices_per_cvt() { return kMode == 0 ? 1 : 2; }
template <int kMode>
constexpr int cvt_stages() { return kMode == 0 ? 5 : 3; }
template <int kMode>
constexpr uint32_t cvt_stride() { return slices_per_cvt<kMode>() * kCvtSlice; }
constexpr uint32_t kTmemCols = 64;
constexpr int kMaxE = 1024;
template <int kMode>
constexpr size_t dyn_smem() {
  return 1024 + (size_t)kRawStages * kRawStride + (size_t)cvt_stages<kMode>() * cvt_stride<kMode>();
}
static_assert(kRawBytes <= kRawStride, "raw stage layout");

enum Mode { kFc1SwiGLU = 0, kFc2 = 1 };

// Instruction descriptor: f16 x f16 -> fp32, K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

MOE_DEVICE uint32_t e4m3_pair_to_f16x2(uint32_t code) {
  uint32_t r;
  const uint16_t pair = (uint16_t)(code | (code << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(pair));
  return r;
}

MOE_DEVICE uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Eight packed E2M1 elements -> four f16x2 words (element pairs in order); the
// word is split into its bytes by one vector move so each convert reads a byte
// register directly.
MOE_DEVICE uint4 e2m1x8_to_f16x8(uint32_t w) {
  uint4 o;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w)
      : "r"(w));
  return o;
}

struct Fp4Params {
  const int32_t* offsets;  // [E+1]
  int32_t* status;
  uint8_t* out;            // FC1: packed E2M1 [cap][I/2]; FC2: bf16 [cap][H]
  uint8_t* out_scales;     // FC1: E4M3 [cap][I/16]
  const float* x_global;   // [1] global scale of the token operand
  const float* w_global;   // [E] global scale of the weights
  const float* out_global; // FC1: [1] global scale the intermediate is encoded with
  const float* row_probs;  // FC2: [cap] probability multiplied into each token row, or NULL
  int64_t ld_out;          // elements per output row
  int64_t w_rows_per_expert;
  int64_t gate_offset;     // FC1: I
  int E, cap, nmt, nkr;    // weight-row tiles per expert, raw stages per tile
};

struct TileInfo {
  int e, mt, nt;
  int64_t row0, row_end;
};

__device__ __forceinline__ TileInfo decode_tile(int t, const int* prefix, const int* ntt, const Fp4Params& p) {
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  TileInfo ti;
  ti.e = lo;
  const int local = t - prefix[lo];
  ti.mt = local / ntt[lo];
  ti.nt = local % ntt[lo];
  const int64_t seg_b = min64(p.offsets[lo], p.cap);
  ti.row_end = min64(p.offsets[lo + 1], p.cap);
  ti.row0 = seg_b + (int64_t)ti.nt * BNT;
  return ti;
}

// Expand half of one 64-element K slice of a packed row: 32 elements = one
// 16-byte chunk of the 128-byte-swizzled raw row (K slice s, half h) plus its
// two scale codes -> four swizzled 16-byte chunks of f16 in the converted tile.
__device__ __forceinline__ void convert_half_row(const uint8_t* raw_row_base, int r, int s, int h,
                                                 const uint8_t* scales_row, uint8_t* cvt_row_base) {
  const int sw = r & 7;
  const uint4 c = *reinterpret_cast<const uint4*>(raw_row_base + (((2 * s + h) ^ sw) << 4));
  const uint32_t sc2 = *reinterpret_cast<const uint16_t*>(scales_row + 4 * s + 2 * h);
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int g = 0; g < 2; g++) {  // 16 elements share one scale
    const uint32_t sh = e4m3_pair_to_f16x2((sc2 >> (8 * g)) & 0xffu);
#pragma unroll
    for (int i = 0; i < 2; i++) {  // one 16-byte output chunk = 8 elements = 4 packed bytes
      const uint32_t w = words[2 * g + i];
      uint4 o = e2m1x8_to_f16x8(w);
      o.x = hmul2(o.x, sh);
      o.y = hmul2(o.y, sh);
      o.z = hmul2(o.z, sh);
      o.w = hmul2(o.w, sh);
      const int chunk = 4 * h + 2 * g + i;
      *reinterpret_cast<uint4*>(cvt_row_base + ((chunk ^ sw) << 4)) = o;
    }
  }
}

MOE_DEVICE uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

MOE_DEVICE uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

MOE_DEVICE void sts128(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Where one thread's half row of a 64-element K slice lives, as shared-memory
// byte offsets fixed for the whole kernel: the row's 128-byte swizzle permutes
// 16-byte chunks by row & 7, so the input chunk of slice s and the four output
// chunks of the half are precomputed once.
struct HalfRow {
  uint32_t in_off[BKR / BKC];  // raw 16-byte chunk of slice s (half h) within the row
  uint32_t out_off[4];         // converted chunks 4h .. 4h+3 within the row
  uint32_t scale_off;          // this half's two scale bytes within a slice's four
};

__device__ __forceinline__ HalfRow half_row(int r, int h) {
  HalfRow hr;
  const int sw = r & 7;
#pragma unroll
  for (int s = 0; s < BKR / BKC; s++) hr.in_off[s] = (uint32_t)(((2 * s + h) ^ sw) << 4);
#pragma unroll
  for (int j = 0; j < 4; j++) hr.out_off[j] = (uint32_t)(((4 * h + j) ^ sw) << 4);
  hr.scale_off = (uint32_t)(2 * h);
  return hr;
}

// convert_half_row with 32-bit shared-memory addresses and precomputed swizzle
// offsets (the form FC2 measured faster with; FC1 measured slower with it).
__device__ __forceinline__ void convert_half_row_sh(uint32_t raw_row, uint32_t scales_row, uint32_t cvt_row, int s,
                                                    const HalfRow& hr) {
  const uint4 c = lds128(raw_row + hr.in_off[s]);
  const uint32_t sc2 = lds16(scales_row + 4 * s + hr.scale_off);
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int g = 0; g < 2; g++) {
    const uint32_t sh = e4m3_pair_to_f16x2((sc2 >> (8 * g)) & 0xffu);
#pragma unroll
    for (int i = 0; i < 2; i++) {
      uint4 o = e2m1x8_to_f16x8(words[2 * g + i]);
      o.x = hmul2(o.x, sh);
      o.y = hmul2(o.y, sh);
      o.z = hmul2(o.z, sh);
      o.w = hmul2(o.w, sh);
      sts128(cvt_row + hr.out_off[2 * g + i], o);
    }
  }
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_ws,
                              const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xs,
                              Fp4Params p) {
  extern __shared__ uint8_t dyn_smem[];
  constexpr int kCvtStages = cvt_stages<kMode>();
  constexpr int kSlicesPerCvt = slices_per_cvt<kMode>();
  constexpr uint32_t kCvtStride = cvt_stride<kMode>();
  __shared__ __align__(8) uint64_t s_rfull[kRawStages], s_rempty[kRawStages], s_cfull[kCvtStages],
      s_cempty[kCvtStages], s_tfull[2], s_tempty[2], s_xbar[2], s_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_prefix[kMaxE + 1];
  __shared__ int s_nt[kMaxE];
  __shared__ float s_gate[2][64][BNT + 1];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = smem;
  uint8_t* cvt = smem + (size_t)kRawStages * kRawStride;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s_abort;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kRawStages; s++) {
      mbar_init(&s_rfull[s], 1);
      mbar_init(&s_rempty[s], kCvtWarps);
    }
    for (int s = 0; s < kCvtStages; s++) {
      mbar_init(&s_cfull[s], kCvtWarps);
      mbar_init(&s_cempty[s], 1);
    }
    for (int a = 0; a < 2; a++) {
      mbar_init(&s_tfull[a], 1);
      mbar_init(&s_tempty[a], 4);
      mbar_init(&s_xbar[a], 4);
    }
    mbar_init(&s_drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_ws);
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_xs);
  }
  if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
  if (warp == 0) {
    const int per = (p.E + 31) / 32;
    int local = 0;
    for (int j = 0; j < per; j++) {
      const int e = lane * per + j;
      if (e < p.E) {
        const int64_t b = min64(p.offsets[e], p.cap), en = min64(p.offsets[e + 1], p.cap);
        const int n = en > b ? (int)((en - b + BNT - 1) / BNT) : 0;
        s_nt[e] = n;
        local += n;
      }
    }
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int run = incl - local;
    for (int j = 0; j < per; j++) {
      const int e = lane * per + j;
      if (e < p.E) {
        s_prefix[e] = run * p.nmt;
        run += s_nt[e];
      }
    }
    if (lane == 31) s_prefix[p.E] = incl * p.nmt;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;
  const int total = s_prefix[p.E];

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_parity[kRawStages];
      bool issued[kRawStages];
      for (int s = 0; s < kRawStages; s++) issued[s] = false;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile(t, s_prefix, s_nt, p);
        const int64_t wbase = (int64_t)ti.e * p.w_rows_per_expert;
        for (int kr = 0; kr < p.nkr; kr++) {
          if (!mbar_wait(&s_rempty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* st = raw + (size_t)stage * kRawStride;
          mbar_arrive_expect_tx(&s_rfull[stage], kRawBytes);
          const int32_t cx = kr * (BKR / 2), cs = kr * (BKR / 16);
          if (kMode == kFc1SwiGLU) {
            const int64_t up = wbase + (int64_t)ti.mt * 64, gate = up + p.gate_offset;
            tma_load_2d(st, &tm_w, cx, (int32_t)up, &s_rfull[stage]);
            tma_load_2d(st + kRawW / 2, &tm_w, cx, (int32_t)gate, &s_rfull[stage]);
            tma_load_2d(st + kRawW, &tm_ws, cs, (int32_t)up, &s_rfull[stage]);
            tma_load_2d(st + kRawW + kRawWS / 2, &tm_ws, cs, (int32_t)gate, &s_rfull[stage]);
          } else {
            const int64_t r0 = wbase + (int64_t)ti.mt * BMW;
            tma_load_2d(st, &tm_w, cx, (int32_t)r0, &s_rfull[stage]);
            tma_load_2d(st + kRawW, &tm_ws, cs, (int32_t)r0, &s_rfull[stage]);
          }
          tma_load_2d(st + kRawW + kRawWS, &tm_x, cx, (int32_t)ti.row0, &s_rfull[stage]);
          tma_load_2d(st + kRawW + kRawWS + kRawX, &tm_xs, cs, (int32_t)ti.row0, &s_rfull[stage]);
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == kRawStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < kRawStages; s++) {
          if (!issued[s]) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&s_rfull[s], issued_parity[s]) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BMW, BNT);
      int cst = 0, acc = 0;
      uint32_t cphase = 0, acc_phase = 0;
      bool ok = true;
      const int nsub = p.nkr * (BKR / BKC) / kSlicesPerCvt;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        if (!mbar_wait(&s_tempty[acc], acc_phase ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BNT);
        for (int ks = 0; ks < nsub; ks++) {
          if (!mbar_wait(&s_cfull[cst], cphase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int sl = 0; sl < kSlicesPerCvt; sl++) {
            const uint32_t cw = smem_u32(cvt + (size_t)cst * kCvtStride + (size_t)sl * kCvtSlice);
            const uint64_t wdesc = smem_desc_sw128(cw);
            const uint64_t xdesc = smem_desc_sw128(cw + kCvtW);
#pragma unroll
            for (int k = 0; k < BKC / 16; k++)
              mma_bf16(d_tmem, wdesc + 2 * k, xdesc + 2 * k, idesc, (ks | sl | k) != 0 ? 1u : 0u);
          }
          mma_commit(&s_cempty[cst]);
          if (++cst == kCvtStages) {
            cst = 0;
            cphase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&s_tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok) {
        mma_commit(&s_drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&s_drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp < 2 + kCvtWarps) {
    // ---------------------------------------------------------- converters
    const int c = threadIdx.x - 64;  // 0..255: weight row c & 127, half c >> 7
    const int wrow = c & 127, whalf = c >> 7;
    const int xrow = c >> 1, xhalf = c & 1;  // token half-rows for c < 64: rows 0..15 in warp 2
    const HalfRow whr = half_row(wrow, whalf), xhr = half_row(xrow, xhalf);
    const uint32_t raw_base = smem_u32(raw), cvt_base = smem_u32(cvt);
    int rst = 0, cst = 0;
    uint32_t rphase = 0, cphase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      // Token rows past the expert's end are not converted: the accumulator
      // column of a token row depends on that row alone, and the epilogue stores
      // valid rows only, so whatever those columns of the converted stage hold
      // never reaches the output.  Whole warps skip when their rows are all past it.
      const TileInfo ti = decode_tile(t, s_prefix, s_nt, p);
      const bool x_conv = c < 2 * BNT && (int64_t)xrow < ti.row_end - ti.row0;
      for (int kr = 0; kr < p.nkr && ok; kr++) {
        int w_ok = 0;
        if (lane == 0) w_ok = mbar_wait(&s_rfull[rst], rphase, abort_flag, p.status) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        const uint8_t* st = raw + (size_t)rst * kRawStride;
        for (int s0 = 0; s0 < BKR / BKC; s0 += kSlicesPerCvt) {
          int c_ok = 0;
          if (lane == 0) c_ok = mbar_wait(&s_cempty[cst], cphase ^ 1, abort_flag, p.status) ? 1 : 0;
          c_ok = __shfl_sync(0xffffffffu, c_ok, 0);
          if (!c_ok) {
            ok = false;
            break;
          }
#pragma unroll
          for (int sl = 0; sl < kSlicesPerCvt; sl++) {
            const int s = s0 + sl;
            if (kMode == kFc2) {
              const uint32_t sts = raw_base + (uint32_t)rst * kRawStride;
              const uint32_t cs = cvt_base + (uint32_t)cst * kCvtStride + (uint32_t)sl * kCvtSlice;
              convert_half_row_sh(sts + wrow * (BKR / 2), sts + kRawW + wrow * (BKR / 16), cs + wrow * (BKC * 2), s,
                                  whr);
              if (x_conv)
                convert_half_row_sh(sts + kRawW + kRawWS + xrow * (BKR / 2),
                                    sts + kRawW + kRawWS + kRawX + xrow * (BKR / 16), cs + kCvtW + xrow * (BKC * 2),
                                    s, xhr);
            } else {
              uint8_t* cs = cvt + (size_t)cst * kCvtStride + (size_t)sl * kCvtSlice;
              convert_half_row(st + wrow * (BKR / 2), wrow, s, whalf, st + kRawW + wrow * (BKR / 16),
                               cs + wrow * (BKC * 2));
              if (x_conv)
                convert_half_row(st + kRawW + kRawWS + xrow * (BKR / 2), xrow, s, xhalf,
                                 st + kRawW + kRawWS + kRawX + xrow * (BKR / 16), cs + kCvtW + xrow * (BKC * 2));
            }
          }
          // make the generic-proxy stores visible to the tensor cores, then publish
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_cfull[cst]);
          if (++cst == kCvtStages) {
            cst = 0;
            cphase ^= 1;
          }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_rempty[rst]);
        if (++rst == kRawStages) {
          rst = 0;
          rphase ^= 1;
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;             // TMEM lane quarter: weight rows 32q .. 32q+31
    const int wr = 32 * q + lane;       // weight row of this thread within the tile
    int acc = 0;
    uint32_t acc_phase = 0;
    int tile_iter = 0;
    const float xg = *p.x_global;
    for (int t = blockIdx.x; t < total; t += gridDim.x, tile_iter++) {
      const TileInfo ti = decode_tile(t, s_prefix, s_nt, p);
      int ok = 0;
      // FC2: a tile's whole K loop passes before its accumulator is full; poll
      // rarely so that the converter warps sharing the schedulers get the issue
      // slots (FC1 measured slower with it)
      if (lane == 0)
        ok = (kMode == kFc2 ? mbar_wait_sleep(&s_tfull[acc], acc_phase, abort_flag, p.status, 256)
                            : mbar_wait(&s_tfull[acc], acc_phase, abort_flag, p.status))
                 ? 1
                 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      float v[32];
      tmem_ld32(tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BNT), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
      const float alpha = xg * p.w_global[ti.e];
      if (kMode == kFc2) {
        const int64_t col = (int64_t)ti.mt * BMW + wr;
        uint16_t* out = reinterpret_cast<uint16_t*>(p.out);
        if (p.row_probs) {
          // lane j fetches token j's probability; every lane scales its feature of the 32 tokens
          const float pr = ti.row0 + lane < ti.row_end ? __ldg(p.row_probs + ti.row0 + lane) : 0.0f;
#pragma unroll
          for (int j = 0; j < BNT; j++) v[j] *= __shfl_sync(0xffffffffu, pr, j);
        }
#pragma unroll
        for (int j = 0; j < BNT; j++) {
          const int64_t row = ti.row0 + j;
          if (row < ti.row_end) out[row * p.ld_out + col] = (uint16_t)float_to_bf16_bits(alpha * v[j]);
        }
      } else {
        // rows 0..63 of the tile are up (w3), rows 64..127 gate (w1) of columns mt*64 + (wr & 63)
        float (*gbuf)[BNT + 1] = s_gate[tile_iter & 1];
        if (q >= 2) {
#pragma unroll
          for (int j = 0; j < BNT; j++) gbuf[wr - 64][j] = alpha * v[j];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_xbar[tile_iter & 1]);
        int x_ok = 0;
        if (lane == 0) x_ok = mbar_wait(&s_xbar[tile_iter & 1], (tile_iter >> 1) & 1, abort_flag, p.status) ? 1 : 0;
        x_ok = __shfl_sync(0xffffffffu, x_ok, 0);
        if (!x_ok) break;
        if (q < 2) {
          const float g2 = *p.out_global;
          const int64_t col = (int64_t)ti.mt * 64 + wr;  // intermediate column of this thread
          const int64_t nvalid = ti.row_end - ti.row0;    // token columns of this tile that exist
#pragma unroll
          for (int j = 0; j < BNT; j++) {
            if (j >= nvalid) break;  // warp-uniform
            const float gt = gbuf[wr][j];
            const float a = gt / (1.0f + __expf(-gt)) * (alpha * v[j]);
            // NVFP4 block = 16 consecutive columns = 16 consecutive lanes
            float amax = fabsf(a);
#pragma unroll
            for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
            const uint32_t scode = e4m3x2(__fdiv_rn(amax, 6.0f * g2), 0.0f) & 0xffu;
            const float denom = e4m3_to_float(scode) * g2;
            const float partner = __shfl_xor_sync(0xffffffffu, a, 1);
            const int64_t row = ti.row0 + j;
            if ((lane & 1) == 0) {
              const uint32_t b = (denom == 0.0f) ? 0u : e2m1x2(__fdiv_rn(a, denom), __fdiv_rn(partner, denom));
              p.out[row * (p.ld_out / 2) + col / 2] = (uint8_t)b;
            }
            if ((lane & 15) == 0) p.out_scales[row * (p.ld_out / 16) + col / 16] = (uint8_t)scode;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int kMode>
cudaError_t launch_one(const CUtensorMap& tw, const CUtensorMap& tws, const CUtensorMap& tx, const CUtensorMap& txs,
                       const Fp4Params& p, int64_t max_tiles, cudaStream_t st) {
  static PerDeviceOnce attr_once;
  cudaError_t e = attr_once.run([] {
    return cudaFuncSetAttribute(grouped_gemm_nvfp4_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)dyn_smem<kMode>());
  });
  if (e != cudaSuccess) return e;
  int64_t grid = device_sm_count();
  if (grid > max_tiles) grid = max_tiles;
  if (grid < 1) grid = 1;
  grouped_gemm_nvfp4_kernel<kMode><<<(unsigned)grid, kThreads, dyn_smem<kMode>(), st>>>(tw, tws, tx, txs, p);
  return cudaGetLastError();
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

cudaError_t launch_grouped_mlp_nvfp4(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                     const void* perm_packed, const void* perm_scales, const void* w13,
                                     const void* w13_scales, const void* w2, const void* w2_scales,
                                     const moe_nvfp4_globals& g, void* workspace, void* out_fc2,
                                     const float* fc2_probs, cudaStream_t st) {
  if (l.capacity == 0) return cudaSuccess;
  if (s.E > kMaxE || s.H % BKR != 0 || s.I % BKR != 0) return cudaErrorNotSupported;
  const uint64_t cap = (uint64_t)l.capacity;
  uint8_t* act = static_cast<uint8_t*>(workspace);
  uint8_t* act_scales = act + round_up(cap * s.I / 2, 1024);
  CUtensorMap w1, w1s, x1, x1s, w2m, w2s, x2, x2s;
  cudaError_t e;
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  const auto NO = CU_TENSOR_MAP_SWIZZLE_NONE;
  const uint64_t rows13 = (uint64_t)s.E * 2 * s.I, rows2 = (uint64_t)s.E * s.H;
  if ((e = make_tensor_map_2d(&w1, w13, U8, 1, rows13, s.H / 2, 64, BKR / 2, SW)) != cudaSuccess) return e;
  if ((e = make_tensor_map_2d(&w1s, w13_scales, U8, 1, rows13, s.H / 16, 64, BKR / 16, NO)) != cudaSuccess) return e;
  if ((e = make_tensor_map_2d(&x1, perm_packed, U8, 1, cap, s.H / 2, BNT, BKR / 2, SW)) != cudaSuccess) return e;
  if ((e = make_tensor_map_2d(&x1s, perm_scales, U8, 1, cap, s.H / 16, BNT, BKR / 16, NO)) != cudaSuccess) return e;
  if ((e = make_tensor_map_2d(&w2m, w2, U8, 1, rows2, s.I / 2, BMW, BKR / 2, SW)) != cudaSuccess) return e;
  if ((e = make_tensor_map_2d(&w2s, w2_scales, U8, 1, rows2, s.I / 16, BMW, BKR / 16, NO)) != cudaSuccess) return e;
  if ((e = make_tensor_map_2d(&x2, act, U8, 1, cap, s.I / 2, BNT, BKR / 2, SW)) != cudaSuccess) return e;
  if ((e = make_tensor_map_2d(&x2s, act_scales, U8, 1, cap, s.I / 16, BNT, BKR / 16, NO)) != cudaSuccess) return e;
  const int64_t n_tiles_bound = (l.capacity + BNT - 1) / BNT + s.E;
  const ProfileEvents prof = take_profile_events();
  if (prof.before_fc1 && (e = record_profile_event(prof.before_fc1, st)) != cudaSuccess) return e;

  Fp4Params p1;
  p1.offsets = h.padded_offsets;
  p1.status = h.status;
  p1.out = act;
  p1.out_scales = act_scales;
  p1.x_global = g.fc1_input_scale;
  p1.w_global = g.w13_scale_2;
  p1.out_global = g.fc2_input_scale;
  p1.row_probs = nullptr;
  p1.ld_out = s.I;
  p1.w_rows_per_expert = 2 * s.I;
  p1.gate_offset = s.I;
  p1.E = (int)s.E;
  p1.cap = (int)l.capacity;
  p1.nmt = (int)(s.I / 64);
  p1.nkr = (int)(s.H / BKR);
  if ((e = launch_one<kFc1SwiGLU>(w1, w1s, x1, x1s, p1, n_tiles_bound * p1.nmt, st)) != cudaSuccess) return e;
  if (prof.after_fc1 && (e = record_profile_event(prof.after_fc1, st)) != cudaSuccess) return e;

  Fp4Params p2 = p1;
  p2.out = static_cast<uint8_t*>(out_fc2);
  p2.out_scales = nullptr;
  p2.x_global = g.fc2_input_scale;
  p2.w_global = g.w2_scale_2;
  p2.out_global = nullptr;
  p2.row_probs = fc2_probs;
  p2.ld_out = s.H;
  p2.w_rows_per_expert = s.H;
  p2.gate_offset = 0;
  p2.nmt = (int)(s.H / BMW);
  p2.nkr = (int)(s.I / BKR);
  if ((e = launch_one<kFc2>(w2m, w2s, x2, x2s, p2, n_tiles_bound * p2.nmt, st)) != cudaSuccess) return e;
  if (prof.after_fc2 && (e = record_profile_event(prof.after_fc2, st)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace moe
