// gemm_bf16_pair.cu -- the bf16 grouped GEMMs of the expert MLP (FC1 + SwiGLU,
// FC2) with each MMA spread over a pair of SMs (a 2-CTA cluster, tcgen05
// cta_group::2): a 256-row tile of the expert's rows, 128 rows per SM, times a
// 256-column weight tile of which each SM holds half.  Per SM and per K step
// that is 16 KB of activations + 16 KB of weights for 128 x 256 x 64 of MMA
// work, one third less shared-memory traffic than a single-SM 128 x 256 tile,
// which buys a 6-stage TMA ring (192 KB) instead of 4.
//
// Follows Megatron-LM PR #6800 "Reuse caller-owned HybridEP dispatch and expert
// output buffers" (Summary: the fused grouped MLP writes FC2 straight into a
// caller buffer) and TensorRT-LLM PR #16190 "Update CuTeDSL MegaMoE kernels"
// (w3_w1 FC1 weight; a persistent tile scheduler over experts).
//
// Per CTA, warp-specialised (both CTAs run the same code; rank 0 leads):
//   warp 0      TMA producer: its 128 rows of the activation tile and its half
//               of the weight tile (FC1: rank 0 the w3 rows, rank 1 the w1 rows
//               of the same 128 intermediate columns; FC2: rows n*256 + 128*rank).
//               Both CTAs' loads complete on the leader's "full" mbarrier.
//   warp 1      TMEM allocation (both CTAs, 512 columns); on the leader one
//               thread issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16) and
//               multicasts each commit to both CTAs' barriers.
//   warps 2..5  epilogue of this CTA's 128 rows (the same code as the single-SM
//               kernel); they release the accumulator on the leader's barrier.
// Every wait is bounded (MOE_DEV_ERR_TIMEOUT, then a clean exit through the
// final cluster barrier, with in-flight copies and MMAs drained first).
#include "moe_internal.h"
#include "sm100_ptx.cuh"
#include "tensor_map.h"

namespace moe {

namespace {

using namespace sm100;

constexpr int BMC = 128;          // rows per CTA
constexpr int BN = 256, BK = 64;  // N per MMA (both halves), K per stage
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr uint32_t kTileABytes = BMC * BK * 2;        // 16 KB
constexpr uint32_t kTileBBytes = (BN / 2) * BK * 2;   // 16 KB: this CTA's half of the weight tile
constexpr uint32_t kStageBytes = kTileABytes + kTileBBytes;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxE = 1024;
constexpr size_t kDynSmem = 1024 + (size_t)kStages * kStageBytes;

enum Mode { kFc1SwiGLU = 0, kFc2 = 1 };

struct PairParams {
  const int32_t* offsets;     // [E+1] padded segment offsets
  int32_t* status;
  uint8_t* out;               // bf16 output [cap][ld_out]
  const float* row_probs;     // [cap] probability multiplied into each output row (FC2), or NULL
  int64_t ld_out;
  int64_t out_cols;
  int64_t b_rows_per_expert;  // 2I (FC1) or H (FC2)
  int64_t half_offset;        // weight-row offset of rank 1's half (FC1: I, FC2: 128)
  int64_t n_step;             // weight rows per N tile step (FC1: 128, FC2: 256)
  int E, cap, nt, nkb;
};

struct TileInfo {
  int e, m, n;
  int64_t row0, row_end;
};

__device__ __forceinline__ TileInfo decode_tile(int t, const int* prefix, const int* mt, const PairParams& p) {
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
  ti.m = local / p.nt;
  ti.n = local % p.nt;
  const int64_t seg_b = min64(p.offsets[lo], p.cap);
  ti.row_end = min64(p.offsets[lo + 1], p.cap);
  ti.row0 = seg_b + (int64_t)ti.m * (2 * BMC);
  return ti;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  return float_to_bf16_bits(a) | (float_to_bf16_bits(b) << 16);
}

__device__ __forceinline__ void store_row32(uint8_t* dst, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; q++) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4*>(dst + q * 16) = w;
  }
}

// Spin (bounded) until `ns` nanoseconds have passed: lets this CTA's own TMA
// copies land after an abort, when their completion is counted on the peer's
// barrier and cannot be observed here.
__device__ __forceinline__ void settle(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) __nanosleep(1000);
}

template <int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                                  PairParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages], s_tfull[2], s_tempty[2], s_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_prefix[kMaxE + 1];
  __shared__ int s_mt[kMaxE];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  volatile int* abort_flag = &s_abort;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; s++) {
      mbar_init(&s_full[s], 1);   // used on the leader: its producer's arrive + both CTAs' bytes
      mbar_init(&s_empty[s], 1);  // each CTA's own, released by the leader's multicast commit
    }
    for (int a = 0; a < 2; a++) {
      mbar_init(&s_tfull[a], 1);   // each CTA's own, multicast commit
      mbar_init(&s_tempty[a], 8);  // used on the leader: 4 epilogue warps of each CTA
    }
    mbar_init(&s_drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) tmem_alloc_pair(&s_tmem, kTmemCols);
  if (warp == 0) {
    const int per = (p.E + 31) / 32;
    int local = 0;
    for (int j = 0; j < per; j++) {
      const int e = lane * per + j;
      if (e < p.E) {
        const int64_t b = min64(p.offsets[e], p.cap), en = min64(p.offsets[e + 1], p.cap);
        const int m = en > b ? (int)((en - b + 2 * BMC - 1) / (2 * BMC)) : 0;
        s_mt[e] = m;
        local += m;
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
        s_prefix[e] = run * p.nt;
        run += s_mt[e];
      }
    }
    if (lane == 31) s_prefix[p.E] = incl * p.nt;
  }
  // both CTAs' barriers exist before either CTA touches the peer's
  tc_fence_before();
  __syncwarp();
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
      for (int t = cluster; t < total && ok; t += nclusters) {
        const TileInfo ti = decode_tile(t, s_prefix, s_mt, p);
        const int64_t arow = ti.row0 + (int64_t)rank * BMC;
        const int64_t brow = (int64_t)ti.e * p.b_rows_per_expert + (int64_t)ti.n * p.n_step + rank * p.half_offset;
        for (int kb = 0; kb < p.nkb; kb++) {
          if (!mbar_wait(&s_empty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * kStageBytes;
          const uint32_t full_leader = mapa_shared(smem_u32(&s_full[stage]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&s_full[stage], 2 * kStageBytes);
          tma_load_2d_pair(sa, &tm_a, kb * BK, (int32_t)arow, full_leader);
          tma_load_2d_pair(sa + kTileABytes, &tm_b, kb * BK, (int32_t)brow, full_leader);
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        if (rank == 0) {
          for (int s = 0; s < kStages; s++) {
            if (!issued[s]) continue;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&s_full[s], issued_parity[s]) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
          }
        }
        settle(2000000);  // 2 ms: far longer than any single copy takes
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BMC, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = cluster; t < total && ok; t += nclusters) {
        if (!mbar_wait(&s_tempty[acc], acc_phase ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < p.nkb; kb++) {
          if (!mbar_wait(&s_full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes);
          const uint64_t adesc = smem_desc_sw128(sa);
          const uint64_t bdesc = smem_desc_sw128(sa + kTileABytes);
#pragma unroll
          for (int k = 0; k < BK / 16; k++)
            mma_bf16_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
          mma_commit_pair(&s_empty[stage], 0x3);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair(&s_tfull[acc], 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok) {
        // no MMA may still write either CTA's TMEM once it is freed
        mma_commit_pair(&s_drain, 0x1);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&s_drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int lane_base = 32 * (warp & 3);
    const uint32_t tempty_leader[2] = {mapa_shared(smem_u32(&s_tempty[0]), 0),
                                       mapa_shared(smem_u32(&s_tempty[1]), 0)};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = cluster; t < total; t += nclusters) {
      const TileInfo ti = decode_tile(t, s_prefix, s_mt, p);
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&s_tfull[acc], acc_phase, abort_flag, p.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int64_t row = ti.row0 + (int64_t)rank * BMC + lane_base + lane;
      const bool valid = row < ti.row_end;
      const uint32_t taddr = tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)(acc * BN);
      if (kMode == kFc1SwiGLU) {
        uint8_t* dst = p.out + (row * p.ld_out + (int64_t)ti.n * 128) * 2;
#pragma unroll 1
        for (int c = 0; c < 4; c++) {
          float up[32], gate[32];
          tmem_ld32(taddr + c * 32, up);
          tmem_ld32(taddr + 128 + c * 32, gate);
#pragma unroll
          for (int j = 0; j < 32; j++) up[j] = gate[j] / (1.0f + __expf(-gate[j])) * up[j];
          if (valid) store_row32(dst + c * 64, up);
        }
      } else {
        uint8_t* dst = p.out + (row * p.ld_out + (int64_t)ti.n * BN) * 2;
        const float pr = p.row_probs && valid ? p.row_probs[row] : 1.0f;
#pragma unroll 1
        for (int c = 0; c < 8; c++) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          if (p.row_probs) {
#pragma unroll
            for (int j = 0; j < 32; j++) v[j] *= pr;
          }
          if (valid && (int64_t)ti.n * BN + c * 32 < p.out_cols) store_row32(dst + c * 64, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&s_tempty[acc]);
        else
          mbar_arrive_cluster(tempty_leader[acc]);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <int kMode>
cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const PairParams& p, int64_t max_tiles,
                        cudaStream_t st) {
  static PerDeviceOnce attr_once;
  cudaError_t e = attr_once.run([] {
    return cudaFuncSetAttribute(grouped_gemm_bf16_pair_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem);
  });
  if (e != cudaSuccess) return e;
  int64_t clusters = device_sm_count() / 2;
  if (clusters > max_tiles) clusters = max_tiles;
  if (clusters < 1) clusters = 1;
  grouped_gemm_bf16_pair_kernel<kMode><<<(unsigned)(2 * clusters), kThreads, kDynSmem, st>>>(ta, tb, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_mlp_bf16_pair(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                         const void* perm_tokens, const void* w13, const void* w2, void* act,
                                         void* out_fc2, const float* fc2_probs, cudaStream_t st) {
  if (l.capacity == 0) return cudaSuccess;
  if (s.E > kMaxE) return cudaErrorNotSupported;
  const uint64_t cap = (uint64_t)l.capacity;
  CUtensorMap ta1, tb1, ta2, tb2;
  cudaError_t e;
  if ((e = make_tensor_map_2d(&ta1, perm_tokens, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cap, s.H, BMC, BK)) !=
      cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&tb1, w13, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)s.E * 2 * s.I, s.H, 128,
                              BK)) != cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&ta2, act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cap, s.I, BMC, BK)) != cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&tb2, w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)s.E * s.H, s.I, 128, BK)) !=
      cudaSuccess)
    return e;
  const int64_t m_tiles_bound = (l.capacity + 2 * BMC - 1) / (2 * BMC) + s.E;
  const ProfileEvents prof = take_profile_events();
  if (prof.before_fc1 && (e = record_profile_event(prof.before_fc1, st)) != cudaSuccess) return e;

  PairParams p1;
  p1.offsets = h.padded_offsets;
  p1.status = h.status;
  p1.out = static_cast<uint8_t*>(act);
  p1.row_probs = nullptr;
  p1.ld_out = s.I;
  p1.out_cols = s.I;
  p1.b_rows_per_expert = 2 * s.I;
  p1.half_offset = s.I;
  p1.n_step = 128;
  p1.E = (int)s.E;
  p1.cap = (int)l.capacity;
  p1.nt = (int)(s.I / 128);
  p1.nkb = (int)(s.H / BK);
  if ((e = launch_pair<kFc1SwiGLU>(ta1, tb1, p1, m_tiles_bound * p1.nt, st)) != cudaSuccess) return e;
  if (prof.after_fc1 && (e = record_profile_event(prof.after_fc1, st)) != cudaSuccess) return e;

  PairParams p2 = p1;
  p2.out = static_cast<uint8_t*>(out_fc2);
  p2.row_probs = fc2_probs;
  p2.ld_out = s.H;
  p2.out_cols = s.H;
  p2.b_rows_per_expert = s.H;
  p2.half_offset = 128;
  p2.n_step = BN;
  p2.nt = (int)((s.H + BN - 1) / BN);
  p2.nkb = (int)(s.I / BK);
  if ((e = launch_pair<kFc2>(ta2, tb2, p2, m_tiles_bound * p2.nt, st)) != cudaSuccess) return e;
  if (prof.after_fc2 && (e = record_profile_event(prof.after_fc2, st)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace moe
