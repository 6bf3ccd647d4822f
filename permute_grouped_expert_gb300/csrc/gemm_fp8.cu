// gemm_fp8.cu -- persistent grouped GEMMs of the expert MLP with FP8 E4M3
// operands and fp32 block scales (one per 128 consecutive elements of an
// activation row, one per 128x128 block of a weight), on the 5th-generation
// tensor cores: FC1 with the SwiGLU epilogue and FP8 re-encoding of the
// intermediate, then FC2 to bf16.
//
// Follows DeepEP PR #716 "perf: reuse HybridEP routing allgather buffer"
// (Testing: BF16 and FP8 dispatch) and Megatron-LM PR #6800 "Reuse caller-owned
// HybridEP dispatch and expert output buffers" (Summary: FP8 expert GEMMs
// consume the dispatch output; grouped FC2 writes into a caller buffer).
//
// The scales are arbitrary fp32 values, which the tensor cores' block-scaled
// MMA kinds (power-of-two or E4M3 scale factors) cannot apply.  So each 128-K
// block is its own MMA chain (tcgen05.mma kind::f8f6f4, M=128, N=256, K=32)
// into one of two TMEM partial buffers, and the epilogue warps fold every
// partial into fp32 register accumulators with the product of the row's and
// the weight block's scales while the tensor cores fill the other buffer.
//
// CTA pairs (clusters of two, one CTA per SM).  A pair takes two tiles that
// share an operand: two token tiles of one expert with the same weight tile,
// or, for an expert's last odd token tile, two output tiles of that token
// tile.  Each CTA loads its own operand and half of the shared one, which TMA
// multicasts into both CTAs' shared memory, so the pair reads the shared tile
// from L2 once; each CTA's MMA commit releases a stage in both CTAs.
//
// 10 warps per CTA:
//   warp 0      TMA producer (A 128 x 128 B, B 256 x 128 B per stage, 4 stages)
//   warp 1      TMEM allocation (512 columns = 2 partials of 128 x 256 fp32) and
//               MMA issue from one thread
//   warps 2..9  two groups of four: group h holds TMEM columns [128h, 128h+128)
//               of every row, one row per thread; 128 fp32 accumulators each,
//               folded in with packed fp32x2 FMAs from 16-column TMEM loads
//               (the 10-warp CTA is budgeted 168 registers a thread; wider loads
//               spill accumulators to local memory inside the K loop).
// FC1's weight tile interleaves up and gate rows in 64-row boxes so that each
// thread ends a tile holding the up and gate values of the same 64 output
// columns.  Every wait is bounded (MOE_DEV_ERR_TIMEOUT, then a clean exit of
// both CTAs).
#include "moe_internal.h"
#include "sm100_ptx.cuh"
#include "tensor_map.h"

namespace moe {

namespace {

using namespace sm100;

constexpr int BM = 128, BN = 256, BK = 128;  // BK in elements = bytes
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTileABytes = BM * BK;
constexpr uint32_t kTileBBytes = BN * BK;
constexpr uint32_t kStageBytes = kTileABytes + kTileBBytes;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxE = 1024;
constexpr size_t kDynSmem = 1024 + (size_t)kStages * kStageBytes;

enum Mode { kFc1SwiGLU = 0, kFc2 = 1 };

// Instruction descriptor of a dense kind::f8f6f4 MMA, E4M3 x E4M3 -> fp32,
// K-major operands: [4,6) D format 1 = f32, [7,10) A format 0 = E4M3,
// [10,13) B format 0 = E4M3, [17,23) N>>3, [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

MOE_DEVICE void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}


// 16 consecutive fp32 columns of this warp's 32 TMEM lanes, load and wait in one statement.
MOE_DEVICE void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}


struct Fp8Params {
  const int32_t* offsets;    // [E+1]
  int32_t* status;
  const float* a_scales;     // [cap][K/128]
  const float* b_scales;     // [E][N/128][K/128]
  uint8_t* out;              // FC1: E4M3 codes [cap][I]; FC2: bf16 [cap][H]
  float* out_scales;         // FC1: fp32 [cap][I/128]
  int64_t ld_out;            // elements per output row
  int64_t out_cols;
  int64_t b_rows_per_expert; // 2I (FC1) or H (FC2)
  int64_t gate_offset;       // FC1: I (rows of w1 after w3)
  int E, cap, nt, nkb, n_blocks_b;  // n_blocks_b = weight rows / 128 per expert
  int out_format;            // FC2: MOE_COMBINE_BF16 / _MXFP8 / _MXFP4
  uint8_t* out_mx_scales;    // FC2 in an MX format: E8M0 [cap][H/32]
  const float* row_probs;    // FC2: [cap] probability multiplied into each output row, or NULL
};

// Shared exponent X of an MX block with magnitude maximum amax: floor(log2(amax))
// - emax (8 for E4M3, 2 for E2M1) from the fp32 bits, clamped to [-127, 127];
// 0 for an all-zero block.
MOE_DEVICE int mx_exponent(float amax, int emax) {
  if (amax == 0.0f) return 0;
  const int field = (int)((__float_as_uint(amax) >> 23) & 0xff);  // 0 for a subnormal: floor(log2) <= -127
  const int X = (field == 0 ? -127 : field - 127) - emax;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

struct TileInfo {
  int e, m, n;
  int64_t row0, row_end;
  bool shares_b;  // the pair shares the weight tile (two M tiles), else the token tile (two N tiles)
  bool masked;    // the second tile of a pair past the last N tile: computed, never stored
};

// Work units of a CTA pair.  Expert e with mt token tiles and nt output tiles
// has (mt / 2) * nt units of two token tiles (m, m+1) that share one weight
// tile, and, for an odd mt, ceil(nt / 2) units of two output tiles (n, n+1)
// of its last token tile that share the token tile.  CTA `rank` of the pair
// takes the unit's tile number `rank`.  Within an expert the units sharing a
// weight tile come first, token-tile pairs innermost, so neighbouring CTA
// pairs read the same weight tile while it is in L2.
__device__ __forceinline__ int units_of(int mt, int nt) { return (mt / 2) * nt + (mt & 1) * ((nt + 1) / 2); }

__device__ __forceinline__ TileInfo decode_unit(int u, uint32_t rank, const int* prefix, const int* mt,
                                                const Fp8Params& p) {
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  TileInfo ti;
  ti.e = lo;
  const int local = u - prefix[lo];
  const int mpairs = mt[lo] / 2;
  ti.masked = false;
  if (local < mpairs * p.nt) {
    ti.shares_b = true;
    ti.n = local / mpairs;
    ti.m = 2 * (local % mpairs) + (int)rank;
  } else {
    ti.shares_b = false;
    ti.m = mt[lo] - 1;
    ti.n = 2 * (local - mpairs * p.nt) + (int)rank;
    if (ti.n >= p.nt) {
      ti.n = p.nt - 1;
      ti.masked = true;
    }
  }
  const int64_t seg_b = min64(p.offsets[lo], p.cap);
  ti.row_end = min64(p.offsets[lo + 1], p.cap);
  ti.row0 = seg_b + (int64_t)ti.m * BM;
  return ti;
}

// Spin (bounded) until `ns` nanoseconds have passed: lets this CTA's own
// multicast copies land after an abort, when part of their completion is
// counted on the peer's barriers and cannot be observed here.
__device__ __forceinline__ void settle(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) __nanosleep(1000);
}

template <int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a64,
                            const __grid_constant__ CUtensorMap tm_b, Fp8Params p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages], s_pfull[2], s_pempty[2], s_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_prefix[kMaxE + 1];
  __shared__ int s_mt[kMaxE];
  __shared__ float s_amax[2][2][BM];  // [tile parity][column group][row]
  __shared__ __align__(8) uint64_t s_xbar[2];  // amax exchange between the two column groups

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  volatile int* abort_flag = &s_abort;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; s++) {
      mbar_init(&s_full[s], 1);   // own producer's arrive; bytes from both CTAs' copies
      mbar_init(&s_empty[s], 2);  // both CTAs' MMA commits: the peer's copies also write this stage
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&s_pfull[b], 1);
      mbar_init(&s_pempty[b], kEpiWarps);
    }
    mbar_init(&s_drain, 1);
    mbar_init(&s_xbar[0], kEpiWarps);
    mbar_init(&s_xbar[1], kEpiWarps);
    fence_barrier_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_a64);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
  if (warp == 0) {
    const int per = (p.E + 31) / 32;
    int local = 0;
    for (int j = 0; j < per; j++) {
      const int e = lane * per + j;
      if (e < p.E) {
        const int64_t b = min64(p.offsets[e], p.cap), en = min64(p.offsets[e + 1], p.cap);
        const int m = en > b ? (int)((en - b + BM - 1) / BM) : 0;
        s_mt[e] = m;
        local += units_of(m, p.nt);
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
        s_prefix[e] = run;
        run += units_of(s_mt[e], p.nt);
      }
    }
    if (lane == 31) s_prefix[p.E] = incl;
  }
  // both CTAs' barriers exist before either CTA's copies or commits reach the peer
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
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
      for (int u = cluster; u < total && ok; u += nclusters) {
        const TileInfo ti = decode_unit(u, rank, s_prefix, s_mt, p);
        const int64_t ebase = (int64_t)ti.e * p.b_rows_per_expert;
        for (int kb = 0; kb < p.nkb; kb++) {
          if (!mbar_wait(&s_empty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * kStageBytes;
          uint8_t* sb = sa + kTileABytes;
          // every stage receives a whole A and B tile in each CTA: this CTA's own
          // operand, half of the shared one from each CTA of the pair
          mbar_arrive_expect_tx(&s_full[stage], kStageBytes);
          if (ti.shares_b) {
            tma_load_2d(sa, &tm_a, kb * BK, (int32_t)ti.row0, &s_full[stage]);
            if (kMode == kFc1SwiGLU) {
              // 64-row boxes up[0:64), gate[0:64), up[64:128), gate[64:128): this CTA loads pair `rank`
              const int64_t up = ebase + (int64_t)ti.n * 128 + 64 * rank, gate = up + p.gate_offset;
              tma_load_2d_mc(sb + (2 * rank) * 8192, &tm_b, kb * BK, (int32_t)up, &s_full[stage], 0x3);
              tma_load_2d_mc(sb + (2 * rank + 1) * 8192, &tm_b, kb * BK, (int32_t)gate, &s_full[stage], 0x3);
            } else {
              const int64_t r0 = ebase + (int64_t)ti.n * BN + 128 * rank;
              tma_load_2d_mc(sb + rank * (kTileBBytes / 2), &tm_b, kb * BK, (int32_t)r0, &s_full[stage], 0x3);
            }
          } else {
            // rows [64 rank, 64 rank + 64) of the shared token tile
            tma_load_2d_mc(sa + rank * (kTileABytes / 2), &tm_a64, kb * BK, (int32_t)(ti.row0 + 64 * rank),
                           &s_full[stage], 0x3);
            if (kMode == kFc1SwiGLU) {
              const int64_t up = ebase + (int64_t)ti.n * 128, gate = up + p.gate_offset;
              tma_load_2d(sb + 0 * 8192, &tm_b, kb * BK, (int32_t)up, &s_full[stage]);
              tma_load_2d(sb + 1 * 8192, &tm_b, kb * BK, (int32_t)gate, &s_full[stage]);
              tma_load_2d(sb + 2 * 8192, &tm_b, kb * BK, (int32_t)(up + 64), &s_full[stage]);
              tma_load_2d(sb + 3 * 8192, &tm_b, kb * BK, (int32_t)(gate + 64), &s_full[stage]);
            } else {
              const int64_t r0 = ebase + (int64_t)ti.n * BN;
              tma_load_2d(sb, &tm_b, kb * BK, (int32_t)r0, &s_full[stage]);
              tma_load_2d(sb + kTileBBytes / 2, &tm_b, kb * BK, (int32_t)(r0 + 128), &s_full[stage]);
            }
          }
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (ok) {
        // every stage this CTA filled (here and, by multicast, in the peer) has
        // been released by both CTAs' MMAs: no copy or commit of this pair is
        // still on its way to either CTA when they leave
        for (int s = 0; s < kStages && ok; s++) {
          if (!mbar_wait(&s_empty[stage], phase ^ 1, abort_flag, p.status)) ok = false;
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
        settle(2000000);  // 2 ms: far longer than any single copy takes
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
      int stage = 0, buf = 0;
      uint32_t phase = 0, buf_phase = 0;
      bool ok = true;
      for (int u = cluster; u < total && ok; u += nclusters) {
        for (int kb = 0; kb < p.nkb; kb++) {
          if (!mbar_wait(&s_pempty[buf], buf_phase ^ 1, abort_flag, p.status) ||
              !mbar_wait(&s_full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes);
          const uint64_t adesc = smem_desc_sw128(sa);
          const uint64_t bdesc = smem_desc_sw128(sa + kTileABytes);
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
          for (int k = 0; k < BK / 32; k++) mma_e4m3(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k != 0 ? 1u : 0u);
          mma_commit_mc(&s_empty[stage], 0x3);  // releases the stage in both CTAs
          mma_commit(&s_pfull[buf]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
          if (++buf == 2) {
            buf = 0;
            buf_phase ^= 1;
          }
        }
      }
      if (!ok) {
        // no MMA may still write TMEM once it is freed
        mma_commit(&s_drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&s_drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int grp = ew >> 2;             // column group: TMEM columns [128 grp, 128 grp + 128)
    const int lane_base = 32 * (warp & 3);
    const int r_local = lane_base + lane;
    const int nsb = p.nkb;               // scale blocks along K
    int buf = 0;
    uint32_t buf_phase = 0;
    int tile_iter = 0;
    bool ok = true;
    for (int u = cluster; u < total && ok; u += nclusters, tile_iter++) {
      const TileInfo ti = decode_unit(u, rank, s_prefix, s_mt, p);
      const int64_t row = ti.row0 + r_local;
      const bool row_in = row < p.cap;
      const float* arow = p.a_scales + (row_in ? row : 0) * (int64_t)nsb;
      // weight scale rows for this thread's two 64-column halves (FC1: up / gate) or its 128 columns (FC2)
      const float* bs0;
      const float* bs1;
      if (kMode == kFc1SwiGLU) {
        bs0 = p.b_scales + ((int64_t)ti.e * p.n_blocks_b + ti.n) * nsb;
        bs1 = p.b_scales + ((int64_t)ti.e * p.n_blocks_b + p.gate_offset / 128 + ti.n) * nsb;
      } else {
        const int64_t blk = (int64_t)ti.n * 2 + grp;
        const int64_t blk_c = blk < p.n_blocks_b ? blk : p.n_blocks_b - 1;
        bs0 = p.b_scales + ((int64_t)ti.e * p.n_blocks_b + blk_c) * nsb;
        bs1 = bs0;
      }
      float2 acc2[64];
#pragma unroll
      for (int j = 0; j < 64; j++) acc2[j] = make_float2(0.0f, 0.0f);
      // scales of the next K block are loaded while this one is folded in
      float sa_next = row_in ? __ldg(arow) : 0.0f;
      float sb0_next = __ldg(bs0), sb1_next = __ldg(bs1);
      for (int kb = 0; kb < p.nkb; kb++) {
        const float sa = sa_next, sb0 = sb0_next, sb1 = sb1_next;
        if (kb + 1 < p.nkb) {
          sa_next = row_in ? __ldg(arow + kb + 1) : 0.0f;
          sb0_next = __ldg(bs0 + kb + 1);
          sb1_next = __ldg(bs1 + kb + 1);
        }
        int w_ok = 0;
        if (lane == 0) w_ok = mbar_wait(&s_pfull[buf], buf_phase, abort_flag, p.status) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)(buf * BN + grp * 128);
        const float s0 = sa * sb0, s1 = sa * sb1;
#pragma unroll
        for (int c = 0; c < 8; c++) {
          float v[16];
          tmem_ld16(taddr + c * 16, v);
          const float s = (kMode == kFc1SwiGLU) ? (c < 4 ? s0 : s1) : s0;
          const float2 s2 = make_float2(s, s);
#pragma unroll
          for (int j = 0; j < 8; j++)
            acc2[c * 8 + j] = __ffma2_rn(s2, make_float2(v[2 * j], v[2 * j + 1]), acc2[c * 8 + j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_pempty[buf]);
        if (++buf == 2) {
          buf = 0;
          buf_phase ^= 1;
        }
      }
      if (!ok) break;
      const bool valid = row < ti.row_end && !ti.masked;
      float* acc = reinterpret_cast<float*>(acc2);
      if (kMode == kFc2 && p.row_probs) {
        // the route's probability scales the row before it is rounded to the output format
        const float pr = valid ? __ldg(p.row_probs + row) : 0.0f;
        const float2 pr2 = make_float2(pr, pr);
#pragma unroll
        for (int j = 0; j < 64; j++) acc2[j] = __fmul2_rn(acc2[j], pr2);
      }
      if (kMode == kFc1SwiGLU) {
        // acc[0..63] = up, acc[64..127] = gate of output columns n*128 + 64*grp + j
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 64; j++) {
          const float g = acc[64 + j];
          const float a = __fdividef(g, 1.0f + __expf(-g)) * acc[j];
          acc[j] = a;
          amax = fmaxf(amax, fabsf(a));
        }
        // the 128-column scale block spans both column groups: exchange row maxima
        s_amax[tile_iter & 1][grp][r_local] = amax;
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_xbar[tile_iter & 1]);
        int x_ok = 0;
        if (lane == 0) x_ok = mbar_wait(&s_xbar[tile_iter & 1], (tile_iter >> 1) & 1, abort_flag, p.status) ? 1 : 0;
        x_ok = __shfl_sync(0xffffffffu, x_ok, 0);
        if (!x_ok) break;
        amax = fmaxf(s_amax[tile_iter & 1][0][r_local], s_amax[tile_iter & 1][1][r_local]);
        const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
        const float rs = __frcp_rn(s);
        if (valid && MOE_IN_BOUNDS(61, row, p.cap, p.status) &&
            MOE_IN_BOUNDS(62, (int64_t)ti.n * 128 + 64 * grp + 63, p.ld_out, p.status)) {
          uint8_t* dst = p.out + row * p.ld_out + (int64_t)ti.n * 128 + 64 * grp;
#pragma unroll
          for (int q = 0; q < 4; q++) {
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const int j = q * 16 + i * 4;
              w4[i] = (uint32_t)e4m3x2(div_by_scale(acc[j], s, rs), div_by_scale(acc[j + 1], s, rs)) |
                      ((uint32_t)e4m3x2(div_by_scale(acc[j + 2], s, rs), div_by_scale(acc[j + 3], s, rs)) << 16);
            }
            *reinterpret_cast<uint4*>(dst + q * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
          if (grp == 0) p.out_scales[row * (p.ld_out / 128) + ti.n] = s;
        }
      } else if (p.out_format != MOE_COMBINE_BF16) {
        // MX combine format: the thread's 128 columns are four blocks of 32,
        // each with its E8M0 scale; x / 2^X is exact in fp32, then rounded
        // to the element format (nearest even, saturating)
        const int64_t col0 = (int64_t)ti.n * BN + grp * 128;
        if (valid && col0 < p.out_cols && MOE_IN_BOUNDS(63, row, p.cap, p.status)) {
          const bool fp8 = p.out_format == MOE_COMBINE_MXFP8;
          uint32_t sc4 = 0;
#pragma unroll
          for (int b = 0; b < 4; b++) {
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; j++) amax = fmaxf(amax, fabsf(acc[32 * b + j]));
            const int X = mx_exponent(amax, fp8 ? 8 : 2);
            sc4 |= (uint32_t)(X + 127) << (8 * b);
            const float inv = X < 127 ? __uint_as_float((uint32_t)(127 - X) << 23) : __uint_as_float(0x00400000u);
            if (fp8) {
              uint8_t* dst = p.out + row * p.ld_out + col0 + 32 * b;
#pragma unroll
              for (int q = 0; q < 2; q++) {
                uint32_t w4[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                  const int j = 32 * b + 16 * q + 4 * i;
                  w4[i] = (uint32_t)e4m3x2(acc[j] * inv, acc[j + 1] * inv) |
                          ((uint32_t)e4m3x2(acc[j + 2] * inv, acc[j + 3] * inv) << 16);
                }
                *reinterpret_cast<uint4*>(dst + 16 * q) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
              }
            } else {
              uint32_t w4[4] = {0, 0, 0, 0};
#pragma unroll
              for (int j = 0; j < 16; j++)
                w4[j >> 2] |= e2m1x2(acc[32 * b + 2 * j] * inv, acc[32 * b + 2 * j + 1] * inv) << (8 * (j & 3));
              *reinterpret_cast<uint4*>(p.out + row * (p.ld_out / 2) + (col0 + 32 * b) / 2) =
                  make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
          *reinterpret_cast<uint32_t*>(p.out_mx_scales + row * (p.ld_out / 32) + col0 / 32) = sc4;
        }
      } else {
        const int64_t col0 = (int64_t)ti.n * BN + grp * 128;
        if (valid && col0 < p.out_cols && MOE_IN_BOUNDS(64, row, p.cap, p.status) &&
            MOE_IN_BOUNDS(65, col0 + 127, p.ld_out, p.status)) {
          uint8_t* dst = p.out + (row * p.ld_out + col0) * 2;
#pragma unroll
          for (int q = 0; q < 16; q++) {
            uint4 w;
            w.x = float_to_bf16_bits(acc[8 * q + 0]) | (float_to_bf16_bits(acc[8 * q + 1]) << 16);
            w.y = float_to_bf16_bits(acc[8 * q + 2]) | (float_to_bf16_bits(acc[8 * q + 3]) << 16);
            w.z = float_to_bf16_bits(acc[8 * q + 4]) | (float_to_bf16_bits(acc[8 * q + 5]) << 16);
            w.w = float_to_bf16_bits(acc[8 * q + 6]) | (float_to_bf16_bits(acc[8 * q + 7]) << 16);
            *reinterpret_cast<uint4*>(dst + q * 16) = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the peer may still write its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int kMode>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& ta64, const CUtensorMap& tb, const Fp8Params& p,
                       int64_t max_units, cudaStream_t st) {
  static PerDeviceOnce attr_once;
  cudaError_t e = attr_once.run([] {
    return cudaFuncSetAttribute(grouped_gemm_fp8_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem);
  });
  if (e != cudaSuccess) return e;
  // CTA pairs (clusters of two), at most one pair per two SMs
  int64_t clusters = device_sm_count() / 2;
  if (clusters > max_units) clusters = max_units;
  if (clusters < 1) clusters = 1;
  grouped_gemm_fp8_kernel<kMode><<<(unsigned)(2 * clusters), kThreads, kDynSmem, st>>>(ta, ta64, tb, p);
  return cudaGetLastError();
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

cudaError_t launch_grouped_mlp_fp8(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                   const void* perm_codes, const void* perm_scales, const void* w13,
                                   const void* w13_scales, const void* w2, const void* w2_scales, void* workspace,
                                   void* out_fc2, int32_t out_format, void* out_fc2_scales,
                                   const float* fc2_probs, cudaStream_t st) {
  if (l.capacity == 0) return cudaSuccess;
  if (s.E > kMaxE) return cudaErrorNotSupported;
  const uint64_t cap = (uint64_t)l.capacity;
  uint8_t* act = static_cast<uint8_t*>(workspace);
  float* act_scales = reinterpret_cast<float*>(act + round_up(cap * s.I, 1024));
  CUtensorMap ta1, ta1h, tb1, ta2, ta2h, tb2;
  cudaError_t e;
  if ((e = make_tensor_map_2d(&ta1, perm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, cap, s.H, BM, BK)) != cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&ta1h, perm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, cap, s.H, BM / 2, BK)) !=
      cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&tb1, w13, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)s.E * 2 * s.I, s.H, 64, BK)) !=
      cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&ta2, act, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, cap, s.I, BM, BK)) != cudaSuccess) return e;
  if ((e = make_tensor_map_2d(&ta2h, act, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, cap, s.I, BM / 2, BK)) != cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&tb2, w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)s.E * s.H, s.I, 128, BK)) !=
      cudaSuccess)
    return e;
  const int64_t m_tiles_bound = (l.capacity + BM - 1) / BM + s.E;
  const ProfileEvents prof = take_profile_events();
  if (prof.before_fc1 && (e = record_profile_event(prof.before_fc1, st)) != cudaSuccess) return e;

  Fp8Params p1;
  p1.offsets = h.padded_offsets;
  p1.status = h.status;
  p1.a_scales = static_cast<const float*>(perm_scales);
  p1.b_scales = static_cast<const float*>(w13_scales);
  p1.out = act;
  p1.out_scales = act_scales;
  p1.ld_out = s.I;
  p1.out_cols = s.I;
  p1.b_rows_per_expert = 2 * s.I;
  p1.gate_offset = s.I;
  p1.E = (int)s.E;
  p1.cap = (int)l.capacity;
  p1.nt = (int)(s.I / 128);
  p1.nkb = (int)(s.H / BK);
  p1.n_blocks_b = (int)(2 * s.I / 128);
  p1.out_format = MOE_COMBINE_BF16;
  p1.out_mx_scales = nullptr;
  p1.row_probs = nullptr;
  if ((e = launch_one<kFc1SwiGLU>(ta1, ta1h, tb1, p1, m_tiles_bound * p1.nt, st)) != cudaSuccess) return e;
  if (prof.after_fc1 && (e = record_profile_event(prof.after_fc1, st)) != cudaSuccess) return e;

  Fp8Params p2 = p1;
  p2.a_scales = act_scales;
  p2.b_scales = static_cast<const float*>(w2_scales);
  p2.out = static_cast<uint8_t*>(out_fc2);
  p2.out_scales = nullptr;
  p2.ld_out = s.H;
  p2.out_cols = s.H;
  p2.b_rows_per_expert = s.H;
  p2.gate_offset = 0;
  p2.nt = (int)((s.H + BN - 1) / BN);
  p2.nkb = (int)(s.I / BK);
  p2.n_blocks_b = (int)(s.H / 128);
  p2.out_format = out_format;
  p2.out_mx_scales = static_cast<uint8_t*>(out_fc2_scales);
  p2.row_probs = fc2_probs;
  if ((e = launch_one<kFc2>(ta2, ta2h, tb2, p2, m_tiles_bound * p2.nt, st)) != cudaSuccess) return e;
  if (prof.after_fc2 && (e = record_profile_event(prof.after_fc2, st)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace moe
