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
// [2^-10, 2688]), so converter warps expand both operands to f16 exactly and
// tcgen05.mma kind::f16 accumulates in fp32; the two fp32 global scales
// (alpha = activation global x expert weight global) are applied in the
// epilogue.  The expanded weights are stored straight into tensor memory
// (tcgen05.st), where the MMA reads its A operand; the expanded tokens go to
// shared memory (the B operand).
//
// One CTA per SM, 16 warps:
//   warp 0      TMA producer: stages of 256 K elements (packed weights 128 rows
//               x 128 B, their scales 128 x 16 B, packed tokens 32 x 128 B, their
//               scales 32 x 16 B); 6 stages (FC1) / 7 (FC2)
//   warp 1      TMEM allocation (512 columns: two 32-column fp32 accumulators,
//               three 128-column f16 weight stages) and MMA issue
//   warps 2..9  weight converters, two per TMEM lane quarter, two 64-K slices
//               each per stage, software pipelined
//   warps 10..13 epilogue: FC1 exchanges gate rows through shared memory, applies
//               SwiGLU and encodes the intermediate to NVFP4 one (token, 16-column
//               block) per thread; FC2 writes bf16
//   warps 14..15 token converters: each thread expands half a token row (rows
//               past the expert's end are skipped) into a two-slot f16 ring
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
constexpr int BKR = 256;        // K elements per stage
constexpr int BKC = 64;         // K elements per slice: one 128-byte swizzle atom of f16 tokens,
                                // 32 tensor-memory columns of f16 weights
constexpr int kSlices = BKR / BKC;
// Shared-memory stages of packed weights and tokens (the bytes in flight from
// HBM): FC1 keeps 41 KB of static shared memory (gate exchange, activation
// transpose, tile prefix) and runs six, FC2 seven.
template <int kMode>
constexpr int stages() { return kMode == 0 ? 6 : 7; }
constexpr int kAStages = 3;     // converted weight stages in tensor memory
constexpr int kCvtWarps = 8;    // weight converters, two per TMEM lane quarter
constexpr int kTokWarps = 2;    // token converters
constexpr int kThreads = 64 + 32 * kCvtWarps + 128 + 32 * kTokWarps;
constexpr int kFirstTokWarp = 2 + kCvtWarps + 4;
constexpr uint32_t kRawW = BMW * (BKR / 2);        // 16 KB packed weights
constexpr uint32_t kRawWS = BMW * (BKR / 16);      // 2 KB weight scales
constexpr uint32_t kRawX = BNT * (BKR / 2);        // 4 KB packed tokens
constexpr uint32_t kRawXS = BNT * (BKR / 16);      // 512 B token scales
constexpr uint32_t kTmaBytes = kRawW + kRawWS + kRawX + kRawXS;
constexpr uint32_t kStageStride = 23552;           // one TMA stage, rounded up to 1024 bytes
constexpr uint32_t kXf16Slice = BNT * BKC * 2;     // 4 KB: 32 rows x 128 B, 128-byte swizzle
constexpr uint32_t kXf16Slot = kSlices * kXf16Slice;  // f16 tokens of one stage
constexpr int kXSlots = 2;                         // f16 token slots, a ring of their own
static_assert(kTmaBytes <= kStageStride && kStageStride % 1024 == 0, "stage layout");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAColBase = 2 * BNT;            // two fp32 accumulators of N = 32 columns come first
constexpr uint32_t kAStageCols = kSlices * (BKC / 2);  // 128 columns: 256 f16 weights per lane
static_assert(kAColBase + kAStages * kAStageCols <= kTmemCols, "tensor memory layout");
constexpr int kMaxE = 1024;
template <int kMode>
constexpr size_t dyn_smem() { return 1024 + (size_t)stages<kMode>() * kStageStride + (size_t)kXSlots * kXf16Slot; }

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
  const int n_tok = MOE_IN_BOUNDS(31, ntt[lo] - 1, 1 << 30, p.status) ? ntt[lo] : 1;  // >= 1 token tile
  ti.mt = local / n_tok;
  ti.nt = local % n_tok;
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

// One 64-element K slice of a packed weight row, already in registers (two
// 16-byte chunks: elements 0..31 and 32..63; four scale codes, one per 16
// elements) -> 32 f16x2 words for the tensor-memory A operand, word j =
// elements 2j, 2j+1.
__device__ __forceinline__ void convert_row_slice_regs(const uint4 (&c)[2], uint32_t sc4, uint32_t (&o)[32]) {
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const uint32_t words[4] = {c[h].x, c[h].y, c[h].z, c[h].w};
#pragma unroll
    for (int g = 0; g < 2; g++) {
      const uint32_t sh = e4m3_pair_to_f16x2((sc4 >> (8 * (2 * h + g))) & 0xffu);
#pragma unroll
      for (int i = 0; i < 2; i++) {
        const uint4 v = e2m1x8_to_f16x8(words[2 * g + i]);
        const int j = 16 * h + 8 * g + 4 * i;
        o[j] = hmul2(v.x, sh);
        o[j + 1] = hmul2(v.y, sh);
        o[j + 2] = hmul2(v.z, sh);
        o[j + 3] = hmul2(v.w, sh);
      }
    }
  }
}

MOE_DEVICE uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

MOE_DEVICE uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_ws,
                              const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xs,
                              Fp4Params p) {
  extern __shared__ uint8_t dyn_smem_buf[];
  constexpr int kStages = stages<kMode>();
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages], s_afull[kAStages], s_aempty[kAStages],
      s_xfree[kXSlots],
      s_tfull[2], s_tempty[2], s_xbar[2], s_ybar[2], s_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_prefix[kMaxE + 1];
  __shared__ int s_nt[kMaxE];
  __shared__ float s_gate[2][64][BNT + 1];  // FC1: gate rows of the tile, [row][token]
  __shared__ float s_act[2][BNT][64 + 1];    // FC1: silu(gate) * up, [token][column]

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem_buf) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s_abort;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; s++) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kCvtWarps + kTokWarps);  // both converter kinds have read the packed data
    }
    for (int a = 0; a < kAStages; a++) {
      mbar_init(&s_afull[a], kCvtWarps + kTokWarps);
      mbar_init(&s_aempty[a], 1);
    }
    for (int x = 0; x < kXSlots; x++) mbar_init(&s_xfree[x], 1);
    for (int a = 0; a < 2; a++) {
      mbar_init(&s_tfull[a], 1);
      mbar_init(&s_tempty[a], 4);
      mbar_init(&s_xbar[a], 4);
      mbar_init(&s_ybar[a], 2);
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
      uint32_t issued_parity[kStages];
      bool issued[kStages];
      for (int s = 0; s < kStages; s++) issued[s] = false;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile(t, s_prefix, s_nt, p);
        (void)MOE_IN_BOUNDS(32, ti.row0, p.cap, p.status);  // a tile starts inside the capacity
        const int64_t wbase = (int64_t)ti.e * p.w_rows_per_expert;
        for (int kr = 0; kr < p.nkr; kr++) {
          // off the critical path (six stages ahead): poll with sleeps, leaving the
          // issue slots to the weight converters (FC1 on decode64 1.128 -> 1.100 ms
          // with this and the token converters' sleeping polls)
          if (!mbar_wait_sleep(&s_empty[stage], phase ^ 1, abort_flag, p.status, 256)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + (size_t)stage * kStageStride;
          mbar_arrive_expect_tx(&s_full[stage], kTmaBytes);
          const int32_t cx = kr * (BKR / 2), cs = kr * (BKR / 16);
          if (kMode == kFc1SwiGLU) {
            const int64_t up = wbase + (int64_t)ti.mt * 64, gate = up + p.gate_offset;
            tma_load_2d(st, &tm_w, cx, (int32_t)up, &s_full[stage]);
            tma_load_2d(st + kRawW / 2, &tm_w, cx, (int32_t)gate, &s_full[stage]);
            tma_load_2d(st + kRawW, &tm_ws, cs, (int32_t)up, &s_full[stage]);
            tma_load_2d(st + kRawW + kRawWS / 2, &tm_ws, cs, (int32_t)gate, &s_full[stage]);
          } else {
            const int64_t r0 = wbase + (int64_t)ti.mt * BMW;
            tma_load_2d(st, &tm_w, cx, (int32_t)r0, &s_full[stage]);
            tma_load_2d(st + kRawW, &tm_ws, cs, (int32_t)r0, &s_full[stage]);
          }
          tma_load_2d(st + kRawW + kRawWS, &tm_x, cx, (int32_t)ti.row0, &s_full[stage]);
          tma_load_2d(st + kRawW + kRawWS + kRawX, &tm_xs, cs, (int32_t)ti.row0, &s_full[stage]);
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < kStages; s++) {
          if (!issued[s]) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&s_full[s], issued_parity[s]) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // A = the converted weight stage in tensor memory, B = the stage's f16
    // token slot in shared memory.  The whole warp runs the loop; one elected
    // lane issues.
    {
      const bool lead = elect_one_lane();
      constexpr uint32_t idesc = idesc_f16_f32(BMW, BNT);
      const uint32_t smem_base = smem_u32(smem);
      int xs = 0, ast = 0, acc = 0;
      uint32_t aphase = 0, acc_phase = 0;
      const uint32_t xbase = smem_base + (uint32_t)kStages * kStageStride;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int w_ok = 0;
        if (lane == 0) w_ok = mbar_wait(&s_tempty[acc], acc_phase ^ 1, abort_flag, p.status) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BNT);
        for (int kr = 0; kr < p.nkr; kr++) {
          int a_ok = 0;
          if (lane == 0) a_ok = mbar_wait(&s_afull[ast], aphase, abort_flag, p.status) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, a_ok, 0)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = tmem_base + kAColBase + (uint32_t)ast * kAStageCols;
          const uint32_t x0 = xbase + (uint32_t)xs * kXf16Slot;
          if (lead) {
#pragma unroll
            for (int sl = 0; sl < kSlices; sl++) {
              const uint64_t xdesc = smem_desc_sw128(x0 + (uint32_t)sl * kXf16Slice);
#pragma unroll
              for (int k = 0; k < BKC / 16; k++)
                mma_f16_tmem_a(d_tmem, a0 + (uint32_t)(sl * (BKC / 2) + 8 * k), xdesc + 2 * k, idesc,
                               (kr | sl | k) != 0 ? 1u : 0u);
            }
            mma_commit(&s_aempty[ast]);
            mma_commit(&s_xfree[xs]);
          }
          __syncwarp();
          if (++ast == kAStages) {
            ast = 0;
            aphase ^= 1;
          }
          if (++xs == kXSlots) xs = 0;
        }
        if (!ok) break;
        if (lead) mma_commit(&s_tfull[acc]);
        __syncwarp();
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok && lead) {
        mma_commit(&s_drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&s_drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp < 2 + kCvtWarps) {
    // ---------------------------------------------------------- weight converters
    // Thread = weight row of the tile = TMEM lane (warp w reaches lane quarter
    // w & 3); the two warps of a quarter take two slices each of a stage.  The
    // converted row is stored straight into tensor memory, where the MMA reads
    // its A operand: no shared-memory round trip and no proxy fence.  Software
    // pipelined: a stage's packed data is released as soon as it is in
    // registers, and its TMEM stores complete while the next stage is loaded
    // and converted; the stage is published after that.
    const int q = warp & 3, grp = (warp - 2) >> 2;
    const int row = 32 * q + lane, sw = row & 7;
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t lane_field = (uint32_t)(32 * q) << 16;
    int stage = 0, ast = 0, prev_ast = -1;
    uint32_t phase = 0, aphase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      for (int kr = 0; kr < p.nkr; kr++) {
        int w_ok = 0;
        if (lane == 0)
          w_ok = (mbar_wait(&s_full[stage], phase, abort_flag, p.status) &&
                  mbar_wait(&s_aempty[ast], aphase ^ 1, abort_flag, p.status))
                     ? 1
                     : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sbase = smem_base + (uint32_t)stage * kStageStride;
        const uint32_t raw_row = sbase + (uint32_t)row * (BKR / 2);
        const uint32_t sc_row = sbase + kRawW + (uint32_t)row * (BKR / 16);
        // this thread's packed data of the stage: two slices x (two 16-byte chunks, four scale codes)
        uint4 c[2][2];
        uint32_t sc[2];
#pragma unroll
        for (int i = 0; i < 2; i++) {
          const int sl = 2 * grp + i;
          sc[i] = lds32(sc_row + 4 * sl);
          c[i][0] = lds128(raw_row + (uint32_t)(((2 * sl) ^ sw) << 4));
          c[i][1] = lds128(raw_row + (uint32_t)(((2 * sl + 1) ^ sw) << 4));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[stage]);
        uint32_t o[2][32];
#pragma unroll
        for (int i = 0; i < 2; i++) convert_row_slice_regs(c[i], sc[i], o[i]);
        if (prev_ast >= 0) {
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_afull[prev_ast]);
        }
        const uint32_t a_cols = tmem_base + lane_field + kAColBase + (uint32_t)ast * kAStageCols;
#pragma unroll
        for (int i = 0; i < 2; i++)
          if (MOE_IN_BOUNDS(41, kAColBase + ast * kAStageCols + (2 * grp + i + 1) * (BKC / 2) - 1, kTmemCols,
                            p.status))
            tmem_st32(a_cols + (uint32_t)((2 * grp + i) * (BKC / 2)), o[i]);
        prev_ast = ast;
        if (++ast == kAStages) {
          ast = 0;
          aphase ^= 1;
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    tmem_wait_st();
    if (ok && prev_ast >= 0) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_afull[prev_ast]);
    }
  } else if (warp >= kFirstTokWarp) {
    // ---------------------------------------------------------- token converters
    // Thread c (0..63) expands half c & 1 of token row c >> 1 for the stage's
    // four slices into the next f16 token slot.  Token rows past the
    // expert's end are not converted: the accumulator column of a token row
    // depends on that row alone, and the epilogue stores valid rows only, so
    // whatever those rows of the area hold never reaches the output.
    const int c = (int)threadIdx.x - 32 * kFirstTokWarp;
    const int row = c >> 1, half = c & 1;
    uint8_t* xslots = smem + (size_t)kStages * kStageStride;
    int stage = 0, ast = 0, xs = 0;
    uint32_t phase = 0, aphase = 0, xphase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = decode_tile(t, s_prefix, s_nt, p);
      const bool conv = (int64_t)row < ti.row_end - ti.row0;
      for (int kr = 0; kr < p.nkr; kr++) {
        // the tensor-memory stage is waited for too, so that this warp's arrival
        // on its full barrier cannot run a phase ahead of the weight converters;
        // a decode tile has a handful of token rows, so these warps mostly wait:
        // they sleep between polls
        int w_ok = 0;
        if (lane == 0)
          w_ok = (mbar_wait_sleep(&s_full[stage], phase, abort_flag, p.status, 256) &&
                  mbar_wait_sleep(&s_aempty[ast], aphase ^ 1, abort_flag, p.status, 256) &&
                  mbar_wait_sleep(&s_xfree[xs], xphase ^ 1, abort_flag, p.status, 256))
                     ? 1
                     : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        const uint8_t* st = smem + (size_t)stage * kStageStride;
        uint8_t* xslot = xslots + (size_t)xs * kXf16Slot;
        if (conv) {
#pragma unroll
          for (int sl = 0; sl < kSlices; sl++)
            convert_half_row(st + kRawW + kRawWS + row * (BKR / 2), row, sl, half,
                             st + kRawW + kRawWS + kRawX + row * (BKR / 16),
                             xslot + sl * kXf16Slice + row * (BKC * 2));
        }
        // make the generic-proxy stores visible to the tensor cores, then publish
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s_afull[ast]);
          mbar_arrive(&s_empty[stage]);
        }
        if (++ast == kAStages) {
          ast = 0;
          aphase ^= 1;
        }
        if (++xs == kXSlots) {
          xs = 0;
          xphase ^= 1;
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
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
      const float alpha = MOE_IN_BOUNDS(13, ti.e, p.E, p.status) ? xg * p.w_global[ti.e] : 0.0f;
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
          if (row < ti.row_end && MOE_IN_BOUNDS(21, row, p.cap, p.status) &&
              MOE_IN_BOUNDS(22, col, p.ld_out, p.status))
            out[row * p.ld_out + col] = (uint16_t)float_to_bf16_bits(alpha * v[j]);
        }
      } else {
        // rows 0..63 of the tile are up (w3), rows 64..127 gate (w1) of columns mt*64 + (wr & 63)
        // rows 0..63 of the tile are up (w3), rows 64..127 gate (w1) of
        // intermediate columns mt*64 + (wr & 63).  (1) the gate rows go to shared
        // memory; (2) the up rows form silu(gate) * up and write it token-major;
        // (3) each thread encodes one (token, 16-column block) of it to NVFP4,
        // all tokens of the tile in parallel.  Buffers alternate by tile and
        // every tile passes both barriers, so a buffer is rewritten only after
        // all four warps have finished the tile that used it before.
        const int buf = tile_iter & 1;
        const uint32_t bphase = (uint32_t)(tile_iter >> 1) & 1u;
        float (*gbuf)[BNT + 1] = s_gate[buf];
        float (*abuf)[64 + 1] = s_act[buf];
        if (q >= 2) {
#pragma unroll
          for (int j = 0; j < BNT; j++) gbuf[wr - 64][j] = alpha * v[j];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_xbar[buf]);
        const int64_t nvalid = ti.row_end - ti.row0;  // token columns of this tile that exist
        if (q < 2) {
          int x_ok = 0;
          if (lane == 0) x_ok = mbar_wait(&s_xbar[buf], bphase, abort_flag, p.status) ? 1 : 0;
          x_ok = __shfl_sync(0xffffffffu, x_ok, 0);
          if (!x_ok) break;
#pragma unroll
          for (int j = 0; j < BNT; j++) {
            if (j >= nvalid) break;  // warp-uniform
            const float gt = gbuf[wr][j];
            abuf[j][wr] = gt / (1.0f + __expf(-gt)) * (alpha * v[j]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_ybar[buf]);
        }
        int y_ok = 0;
        if (lane == 0) y_ok = mbar_wait(&s_ybar[buf], bphase, abort_flag, p.status) ? 1 : 0;
        y_ok = __shfl_sync(0xffffffffu, y_ok, 0);
        if (!y_ok) break;
        // token j = lane, columns 16q .. 16q+15 of the tile
        if (lane < nvalid) {
          const float g2 = *p.out_global;
          float a[16];
          float amax = 0.0f;
#pragma unroll
          for (int c = 0; c < 16; c++) {
            a[c] = abuf[lane][16 * q + c];
            amax = fmaxf(amax, fabsf(a[c]));
          }
          const uint32_t scode = e4m3x2(__fdiv_rn(amax, 6.0f * g2), 0.0f) & 0xffu;
          const float denom = e4m3_to_float(scode) * g2;
          uint32_t packed[2] = {0u, 0u};
          if (denom != 0.0f) {
#pragma unroll
            for (int k = 0; k < 8; k++)
              packed[k >> 2] |= e2m1x2(__fdiv_rn(a[2 * k], denom), __fdiv_rn(a[2 * k + 1], denom)) << (8 * (k & 3));
          }
          const int64_t row = ti.row0 + lane;
          const int64_t col0 = (int64_t)ti.mt * 64 + 16 * q;  // first intermediate column of the block
          if (MOE_IN_BOUNDS(11, row, p.cap, p.status) && MOE_IN_BOUNDS(12, col0 + 15, p.ld_out, p.status)) {
            *reinterpret_cast<uint2*>(p.out + row * (p.ld_out / 2) + col0 / 2) = make_uint2(packed[0], packed[1]);
            p.out_scales[row * (p.ld_out / 16) + col0 / 16] = (uint8_t)scode;
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
