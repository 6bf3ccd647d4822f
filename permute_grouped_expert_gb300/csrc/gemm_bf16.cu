// gemm_bf16.cu -- persistent grouped GEMMs of the expert MLP in bf16 on the
// 5th-generation tensor cores: FC1 with the SwiGLU epilogue, and FC2.
//
// Follows Megatron-LM PR #6800 "Reuse caller-owned HybridEP dispatch and expert
// output buffers" (Summary: the fused grouped MLP writes FC2 straight into a
// caller buffer) and TensorRT-LLM PR #16190 "Update CuTeDSL MegaMoE kernels"
// (w3_w1 FC1 weight; a persistent tile scheduler over experts).
//
// One persistent launch runs both GEMMs.  The tile list holds every FC1 tile,
// then every FC2 tile; CTAs claim tiles in that order from a global counter
// (one tile ahead), so fast CTAs take more tiles and all finish together.  An
// FC2 tile reads the SwiGLU intermediate rows of one M tile, so its producer
// first waits (bounded) on that M tile's completion counter, which each FC1
// epilogue warp raises with a release add after its rows are stored; no kernel
// boundary separates the two GEMMs, and the tail of FC1 overlaps the start of
// FC2.
//
// One CTA per SM, warp-specialised:
//   warp 0      claims tiles and passes their ids to the other roles through a
//               4-slot shared-memory queue; TMA producer: A tile 128 rows x
//               64 K of the expert's rows, B tile 256 rows x 64 K of its
//               weights (two 128-row boxes), 128-byte swizzle, 4-stage
//               shared-memory ring (48 KB per stage).
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and
//               issues tcgen05.mma (M=128, N=256, K=16) from one thread;
//               tcgen05.commit frees ring stages and publishes accumulators.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one row per thread),
//               SwiGLU (FC1) or plain bf16 conversion (FC2), 16-byte stores.
// Tiles are (GEMM, expert, M tile, N tile), N innermost so that CTAs running
// side by side share the activation tile in L2 (and the N tiles of one M tile
// finish together).  Group sizes live only on the device: each
// CTA derives the tile list from the padded offsets, so the launch shape does
// not depend on the routing and the kernel can be captured in a CUDA graph.
// Every wait is bounded (MOE_DEV_ERR_TIMEOUT, then a clean exit).
#include "moe_internal.h"
#include "sm100_ptx.cuh"
#include "tensor_map.h"

namespace moe {

namespace {

using namespace sm100;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kQueue = 4;  // claimed tile ids in flight from the producer to the MMA and epilogue warps
constexpr uint32_t kTileABytes = BM * BK * 2;
constexpr uint32_t kTileBBytes = BN * BK * 2;
constexpr uint32_t kStageBytes = kTileABytes + kTileBBytes;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxE = 1024;
constexpr size_t kDynSmem = 1024 + (size_t)kStages * kStageBytes;

// One GEMM of the pair: FC1 (phase 0, SwiGLU epilogue) or FC2 (phase 1).
struct PhaseParams {
  uint8_t* out;               // bf16 output [cap][ld_out]
  int64_t ld_out;             // elements per output row
  int64_t out_cols;           // output columns that exist
  int64_t b_rows_per_expert;  // weight rows per expert (2I for FC1, H for FC2)
  int64_t half_offset;        // row offset of the second 128-row weight box
  int64_t n_step;             // weight rows advanced per N tile (128 for FC1, 256 for FC2)
  int nt, nkb;                // N tiles per M tile, 64-wide K blocks
};

struct FusedParams {
  const int32_t* offsets;  // [E+1] padded segment offsets
  int32_t* status;         // device status word (timeouts)
  int32_t* sched;          // tile claim counter, zeroed before the launch
  int32_t* ready;          // [M tiles] FC1 completions per M tile, zeroed before the launch
  PhaseParams ph[2];
  int E, cap;
  int ready_target;  // kEpiWarps * FC1 N tiles: an M tile's intermediate rows are complete
};

struct TileInfo {
  int phase, e, g, n;  // g: M tile index over all experts
  int64_t row0, row_end;
};

// Tiles run FC1 first, then FC2; within a GEMM the order is (expert, M tile,
// N tile), N innermost.  prefix[e] = M tiles of the experts before e.
__device__ __forceinline__ TileInfo decode_tile(int t, int total1, const int* prefix, const FusedParams& p) {
  TileInfo ti;
  ti.phase = t >= total1 ? 1 : 0;
  const int nt = ti.phase ? p.ph[1].nt : p.ph[0].nt;
  const int local = t - (ti.phase ? total1 : 0);
  ti.g = local / nt;
  ti.n = local - ti.g * nt;
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= ti.g)
      lo = mid;
    else
      hi = mid - 1;
  }
  ti.e = lo;
  const int64_t seg_b = min64(p.offsets[lo], p.cap);
  ti.row_end = min64(p.offsets[lo + 1], p.cap);
  ti.row0 = seg_b + (int64_t)(ti.g - prefix[lo]) * BM;
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

// Bounded wait until the FC1 tiles of M tile g have all been published.  The
// acquire load orders the intermediate rows before this thread's later
// accesses; the proxy fence extends that to the TMA loads that read them.
__device__ __forceinline__ bool wait_ready(const int32_t* ready, int target, volatile int* abort_flag,
                                           int32_t* status) {
  if (ld_acquire_s32(ready) < target) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      __nanosleep(128);
      if (ld_acquire_s32(ready) >= target) break;
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        set_status(status, MOE_DEV_ERR_TIMEOUT);
        return false;
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    grouped_mlp_bf16_kernel(const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_b1,
                            const __grid_constant__ CUtensorMap tm_a2, const __grid_constant__ CUtensorMap tm_b2,
                            FusedParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages], s_tfull[2], s_tempty[2], s_drain;
  __shared__ __align__(8) uint64_t s_qfull[kQueue], s_qempty[kQueue];
  __shared__ int s_tile[kQueue];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_prefix[kMaxE + 1];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s_abort;

  // ---- set-up: barriers, TMEM, tile list
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kStages; s++) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 1);
    }
    for (int a = 0; a < 2; a++) {
      mbar_init(&s_tfull[a], 1);
      mbar_init(&s_tempty[a], kEpiWarps);
    }
    for (int q = 0; q < kQueue; q++) {
      mbar_init(&s_qfull[q], 1);
      mbar_init(&s_qempty[q], 1 + kEpiWarps);
    }
    mbar_init(&s_drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_a1);
    tma_prefetch_desc(&tm_b1);
    tma_prefetch_desc(&tm_a2);
    tma_prefetch_desc(&tm_b2);
  }
  if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
  if (warp == 0) {
    // exclusive prefix of M tiles over experts (one warp, `per` experts a lane)
    const int per = (p.E + 31) / 32;
    int local = 0;
    for (int j = 0; j < per; j++) {
      const int e = lane * per + j;
      if (e < p.E) {
        const int64_t b = min64(p.offsets[e], p.cap), en = min64(p.offsets[e + 1], p.cap);
        const int m = en > b ? (int)((en - b + BM - 1) / BM) : 0;
        s_prefix[e] = m;
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
        const int m = s_prefix[e];
        s_prefix[e] = run;
        run += m;
      }
    }
    if (lane == 31) s_prefix[p.E] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;
  const int mtiles = s_prefix[p.E];
  const int total1 = mtiles * p.ph[0].nt;
  const int total = total1 + mtiles * p.ph[1].nt;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_parity[kStages];
      bool issued[kStages];
      for (int s = 0; s < kStages; s++) issued[s] = false;
      bool ok = true;
      int ready_g = -1;
      int q = 0;
      uint32_t qphase = 0;
      int t = atomicAdd(p.sched, 1);
      for (;;) {
        // hand the claimed tile (or the end mark) to the MMA and epilogue warps
        if (!mbar_wait(&s_qempty[q], qphase ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        s_tile[q] = t < total ? t : -1;
        mbar_arrive(&s_qfull[q]);
        if (++q == kQueue) {
          q = 0;
          qphase ^= 1;
        }
        if (t >= total) break;
        // claim the next tile now, so the claim's round trip overlaps this tile's loads
        const int next = atomicAdd(p.sched, 1);
        const TileInfo ti = decode_tile(t, total1, s_prefix, p);
        const bool fc2 = ti.phase != 0;
        if (fc2 && ti.g != ready_g) {
          if (!wait_ready(p.ready + ti.g, p.ready_target, abort_flag, p.status)) {
            ok = false;
            break;
          }
          ready_g = ti.g;
        }
        const CUtensorMap* ma = fc2 ? &tm_a2 : &tm_a1;
        const CUtensorMap* mb = fc2 ? &tm_b2 : &tm_b1;
        const int64_t b_rows = fc2 ? p.ph[1].b_rows_per_expert : p.ph[0].b_rows_per_expert;
        const int64_t n_step = fc2 ? p.ph[1].n_step : p.ph[0].n_step;
        const int64_t half = fc2 ? p.ph[1].half_offset : p.ph[0].half_offset;
        const int nkb = fc2 ? p.ph[1].nkb : p.ph[0].nkb;
        const int64_t brow = (int64_t)ti.e * b_rows + (int64_t)ti.n * n_step;
        for (int kb = 0; kb < nkb; kb++) {
          if (!mbar_wait(&s_empty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * kStageBytes;
          uint8_t* sb = sa + kTileABytes;
          mbar_arrive_expect_tx(&s_full[stage], kStageBytes);
          tma_load_2d(sa, ma, kb * BK, (int32_t)ti.row0, &s_full[stage]);
          tma_load_2d(sb, mb, kb * BK, (int32_t)brow, &s_full[stage]);
          tma_load_2d(sb + kTileBBytes / 2, mb, kb * BK, (int32_t)(brow + half), &s_full[stage]);
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        t = next;
      }
      if (!ok) {
        // drain: every copy issued into this CTA's shared memory must land before exit
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
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      int q = 0;
      uint32_t qphase = 0;
      for (;;) {
        if (!mbar_wait(&s_qfull[q], qphase, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const int t = s_tile[q];
        mbar_arrive(&s_qempty[q]);
        if (++q == kQueue) {
          q = 0;
          qphase ^= 1;
        }
        if (t < 0) break;
        const int nkb = t >= total1 ? p.ph[1].nkb : p.ph[0].nkb;
        if (!mbar_wait(&s_tempty[acc], acc_phase ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nkb; kb++) {
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
            mma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
          mma_commit(&s_empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
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
        // no MMA may still write TMEM once it is freed
        mma_commit(&s_drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&s_drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int lane_base = 32 * (warp & 3);
    int acc = 0;
    uint32_t acc_phase = 0;
    int q = 0;
    uint32_t qphase = 0;
    for (;;) {
      // one lane waits and the warp follows its verdict, so the warp-wide
      // tcgen05.ld below is always executed by all 32 lanes or by none
      int ok = 0, t = -1;
      if (lane == 0 && mbar_wait(&s_qfull[q], qphase, abort_flag, p.status)) {
        ok = 1;
        t = s_tile[q];
        mbar_arrive(&s_qempty[q]);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (++q == kQueue) {
        q = 0;
        qphase ^= 1;
      }
      if (!ok || t < 0) break;
      const TileInfo ti = decode_tile(t, total1, s_prefix, p);
      if (lane == 0) ok = mbar_wait(&s_tfull[acc], acc_phase, abort_flag, p.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int64_t row = ti.row0 + lane_base + lane;
      const bool valid = row < ti.row_end;
      const uint32_t taddr = tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)(acc * BN);
      if (ti.phase == 0) {
        uint8_t* dst = p.ph[0].out + (row * p.ph[0].ld_out + (int64_t)ti.n * 128) * 2;
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
        uint8_t* dst = p.ph[1].out + (row * p.ph[1].ld_out + (int64_t)ti.n * BN) * 2;
#pragma unroll 1
        for (int c = 0; c < 8; c++) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          if (valid && (int64_t)ti.n * BN + c * 32 < p.ph[1].out_cols) store_row32(dst + c * 64, v);
        }
      }
      tc_fence_before();
      if (ti.phase == 0) {
        // publish this warp's 32 intermediate rows of the tile: each lane's
        // stores are fenced (generic and async proxy), then one release add
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        __syncwarp();
        if (lane == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.ready + ti.g) : "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
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

}  // namespace

// Synchronisation words in the workspace: the tile claim counter, padded to
// 128 bytes, then one FC1 completion counter per M tile.
constexpr size_t kSchedBytes = 128;
size_t grouped_mlp_bf16_ready_bytes(const moe_shape& s, const moe_layout& l) {
  return kSchedBytes + (size_t)((l.capacity + BM - 1) / BM + s.E + 1) * sizeof(int32_t);
}

// FC1 and FC2 in one persistent launch.  An FC2 tile waits (bounded) for the
// FC1 tiles of its M tile.  Tiles are claimed in list order and every FC1 tile
// precedes every FC2 tile, so those FC1 tiles were claimed earlier by CTAs
// that hold no FC2 tile in front of them (a CTA's tile claimed after an FC2
// tile is an FC2 tile); with one CTA per SM and the grid no larger than the SM
// count all CTAs are resident together, so every wait is on work that is
// running or done.
cudaError_t launch_grouped_mlp_bf16(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                    const void* perm_tokens, const void* w13, const void* w2, void* act,
                                    void* ready, void* out_fc2, cudaStream_t st) {
  if (l.capacity == 0) return cudaSuccess;
  if (s.E > kMaxE) return cudaErrorNotSupported;
  const uint64_t cap = (uint64_t)l.capacity;
  CUtensorMap ta1, tb1, ta2, tb2;
  cudaError_t e;
  if ((e = make_tensor_map_2d(&ta1, perm_tokens, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cap, s.H, BM, BK)) != cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&tb1, w13, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)s.E * 2 * s.I, s.H, 128, BK)) !=
      cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&ta2, act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cap, s.I, BM, BK)) != cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&tb2, w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)s.E * s.H, s.I, 128, BK)) !=
      cudaSuccess)
    return e;
  static bool attr = false;
  if (!attr) {
    if ((e = cudaFuncSetAttribute(grouped_mlp_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kDynSmem)) != cudaSuccess)
      return e;
    attr = true;
  }
  const size_t ready_bytes = grouped_mlp_bf16_ready_bytes(s, l);
  if ((e = cudaMemsetAsync(ready, 0, ready_bytes, st)) != cudaSuccess) return e;

  FusedParams p;
  p.offsets = h.padded_offsets;
  p.status = h.status;
  p.sched = static_cast<int32_t*>(ready);
  p.ready = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ready) + kSchedBytes);
  p.E = (int)s.E;
  p.cap = (int)l.capacity;
  PhaseParams& p1 = p.ph[0];
  p1.out = static_cast<uint8_t*>(act);
  p1.ld_out = s.I;
  p1.out_cols = s.I;
  p1.b_rows_per_expert = 2 * s.I;
  p1.half_offset = s.I;
  p1.n_step = 128;
  p1.nt = (int)(s.I / 128);
  p1.nkb = (int)(s.H / BK);
  PhaseParams& p2 = p.ph[1];
  p2.out = static_cast<uint8_t*>(out_fc2);
  p2.ld_out = s.H;
  p2.out_cols = s.H;
  p2.b_rows_per_expert = s.H;
  p2.half_offset = 128;
  p2.n_step = BN;
  p2.nt = (int)((s.H + BN - 1) / BN);
  p2.nkb = (int)(s.I / BK);
  p.ready_target = kEpiWarps * p1.nt;

  const int64_t m_tiles_bound = (l.capacity + BM - 1) / BM + s.E;
  int64_t grid = device_sm_count();
  if (grid > m_tiles_bound * (p1.nt + p2.nt)) grid = m_tiles_bound * (p1.nt + p2.nt);
  if (grid < 1) grid = 1;

  const ProfileEvents prof = take_profile_events();
  if (prof.before_fc1 && (e = cudaEventRecord(prof.before_fc1, st)) != cudaSuccess) return e;
  grouped_mlp_bf16_kernel<<<(unsigned)grid, kThreads, kDynSmem, st>>>(ta1, tb1, ta2, tb2, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // one kernel runs both GEMMs: the FC1/FC2 boundary event is recorded with the end
  if (prof.after_fc1 && (e = cudaEventRecord(prof.after_fc1, st)) != cudaSuccess) return e;
  if (prof.after_fc2 && (e = cudaEventRecord(prof.after_fc2, st)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace moe
