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
// FC2 tile reads the SwiGLU intermediate rows of one token tile, so its
// producer first waits (bounded) on that token tile's completion counter,
// which each FC1 epilogue warp raises with a release add after its rows are
// stored; no kernel boundary separates the two GEMMs, and the tail of FC1
// overlaps the start of FC2.
//
// Weights are the MMA's M operand and tokens its N operand (D = W . Y^T, one
// TMEM lane per output feature, one column per token).  A tile is 256 output
// features (two M=128 accumulators: up and gate of the same 128 features for
// FC1, two 128-feature halves for FC2) by up to 128 tokens of one expert; the
// last token tile of an expert runs with N = its rows rounded up to 16, so the
// ragged end of every expert segment costs at most 15 rows of MMA work
// instead of up to 127.
//
// One CTA per SM, warp-specialised:
//   warp 0      claims tiles and passes their ids to the other roles through a
//               4-slot shared-memory queue; TMA producer: two weight boxes of
//               128 rows x 64 K and one token box of 128 rows x 64 K, 128-byte
//               swizzle, 4-stage shared-memory ring (48 KB per stage).
//   warp 1      allocates 512 TMEM columns (two buffers of two 128 x 128 fp32
//               accumulators) and issues tcgen05.mma (M=128, N=tokens, K=16)
//               from one thread, two per K step; tcgen05.commit frees ring
//               stages and publishes accumulators.
//   warps 2..5  epilogue: tcgen05.ld of 32 tokens of the warp's 32 features,
//               SwiGLU (FC1) or plain bf16 conversion (FC2), a transpose
//               through a per-warp shared-memory patch, then each lane stores
//               64 contiguous bytes of one token row.
// Tiles are (GEMM, expert, token tile, feature tile), feature tile innermost
// so that CTAs running side by side share the token tile in L2 (and the
// feature tiles of one token tile finish together).  Group sizes live only on
// the device: each CTA derives the tile list from the padded offsets, so the
// launch shape does not depend on the routing and the kernel can be captured
// in a CUDA graph.  Every wait is bounded (MOE_DEV_ERR_TIMEOUT, then a clean
// exit).
#include "moe_internal.h"
#include "sm100_ptx.cuh"
#include "tensor_map.h"

namespace moe {

namespace {

using namespace sm100;

constexpr int BW = 128;   // weight rows (output features) per accumulator
constexpr int BT = 128;   // tokens per tile (MMA N at most)
constexpr int BK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kQueue = 4;  // claimed tile ids in flight from the producer to the MMA and epilogue warps
constexpr uint32_t kTileWBytes = BW * BK * 2;
constexpr uint32_t kTileTBytes = BT * BK * 2;
constexpr uint32_t kStageBytes = 2 * kTileWBytes + kTileTBytes;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxE = 1024;
constexpr int kPatchStride = 80;  // bytes per token row of a transpose patch (64 B + 16 B against bank conflicts)
constexpr uint32_t kPatchBytes = 32 * kPatchStride;
constexpr size_t kDynSmem = 1024 + (size_t)kStages * kStageBytes + (size_t)kEpiWarps * kPatchBytes;

// One GEMM of the pair: FC1 (phase 0, SwiGLU epilogue) or FC2 (phase 1).
struct PhaseParams {
  uint8_t* out;               // bf16 output [cap][ld_out]
  int64_t ld_out;             // elements per output row
  int64_t out_cols;           // output features that exist
  int64_t w_rows_per_expert;  // weight rows per expert (2I for FC1, H for FC2)
  int64_t second_offset;      // weight row offset of the second accumulator (I: gate; 128: next features)
  int64_t n_step;             // weight rows advanced per feature tile (128 for FC1, 256 for FC2)
  int nt, nkb;                // feature tiles per token tile, 64-wide K blocks
};

struct FusedParams {
  const int32_t* offsets;  // [E+1] padded segment offsets
  int32_t* status;         // device status word (timeouts)
  int32_t* sched;          // tile claim counter, zeroed before the launch
  int32_t* ready;          // [token tiles] FC1 completions per token tile, zeroed before the launch
  const float* fc2_probs;  // [cap] probability multiplied into each FC2 row, or NULL
  PhaseParams ph[2];
  int E, cap;
  int ready_target;  // kEpiWarps * FC1 feature tiles: a token tile's intermediate rows are complete
  int silent_g;      // testing hook: FC1 tiles of this token tile withhold their publication (-1: none)
};

struct TileInfo {
  int phase, e, g, n;  // g: token tile index over all experts, n: feature tile
  int ntok;            // MMA N: the tile's rows rounded up to 16, at most BT
  int64_t row0, row_end;
};

// Tiles run FC1 first, then FC2; within a GEMM the order is (expert, token
// tile, feature tile), feature tile innermost.  prefix[e] = token tiles of
// the experts before e.
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
  ti.row0 = seg_b + (int64_t)(ti.g - prefix[lo]) * BT;
  const int64_t rows = min64(ti.row_end - ti.row0, BT);
  ti.ntok = (int)((rows + 15) & ~int64_t(15));
  return ti;
}

// 32 values of this lane's feature for 32 consecutive tokens -> bf16, turned
// through the warp's patch so that lane j stores the 32 features (64 bytes)
// of token j: dst points at token 0's first feature, rows_valid tokens exist.
__device__ __forceinline__ void transpose_store32(uint8_t* patch, const float (&v)[32], uint8_t* dst,
                                                  int64_t row_bytes, int rows_valid, int lane) {
#pragma unroll
  for (int j = 0; j < 32; j++)
    *reinterpret_cast<uint16_t*>(patch + j * kPatchStride + lane * 2) = (uint16_t)float_to_bf16_bits(v[j]);
  __syncwarp();
  if (lane < rows_valid) {
    const uint4* src = reinterpret_cast<const uint4*>(patch + lane * kPatchStride);
    uint4* d = reinterpret_cast<uint4*>(dst + (int64_t)lane * row_bytes);
#pragma unroll
    for (int q = 0; q < 4; q++) d[q] = src[q];
  }
  __syncwarp();
}

// Bounded wait until the FC1 tiles of token tile g have all been published.
// The acquire load orders the intermediate rows before this thread's later
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
    grouped_mlp_bf16_kernel(const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_w13,
                            const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w2,
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
    tma_prefetch_desc(&tm_y);
    tma_prefetch_desc(&tm_w13);
    tma_prefetch_desc(&tm_act);
    tma_prefetch_desc(&tm_w2);
  }
  if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
  if (warp == 0) {
    // exclusive prefix of token tiles over experts (one warp, `per` experts a lane)
    const int per = (p.E + 31) / 32;
    int local = 0;
    for (int j = 0; j < per; j++) {
      const int e = lane * per + j;
      if (e < p.E) {
        const int64_t b = min64(p.offsets[e], p.cap), en = min64(p.offsets[e + 1], p.cap);
        const int m = en > b ? (int)((en - b + BT - 1) / BT) : 0;
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
  const int ttiles = s_prefix[p.E];
  const int total1 = ttiles * p.ph[0].nt;
  const int total = total1 + ttiles * p.ph[1].nt;

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
        const CUtensorMap* mt = fc2 ? &tm_act : &tm_y;
        const CUtensorMap* mw = fc2 ? &tm_w2 : &tm_w13;
        const PhaseParams& pp = p.ph[fc2 ? 1 : 0];
        const int64_t w0 = (int64_t)ti.e * pp.w_rows_per_expert + (int64_t)ti.n * pp.n_step;
        const int64_t w1 = w0 + pp.second_offset;
        for (int kb = 0; kb < pp.nkb; kb++) {
          if (!mbar_wait(&s_empty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sw = smem + (size_t)stage * kStageBytes;
          mbar_arrive_expect_tx(&s_full[stage], kStageBytes);
          tma_load_2d(sw, mw, kb * BK, (int32_t)w0, &s_full[stage]);
          tma_load_2d(sw + kTileWBytes, mw, kb * BK, (int32_t)w1, &s_full[stage]);
          tma_load_2d(sw + 2 * kTileWBytes, mt, kb * BK, (int32_t)ti.row0, &s_full[stage]);
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
        const TileInfo ti = decode_tile(t, total1, s_prefix, p);
        const int nkb = ti.phase ? p.ph[1].nkb : p.ph[0].nkb;
        const uint32_t idesc = idesc_bf16_f32(BW, (uint32_t)ti.ntok);
        if (!mbar_wait(&s_tempty[acc], acc_phase ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)(acc * 2 * BT);
        const uint32_t d1 = d0 + BT;
        for (int kb = 0; kb < nkb; kb++) {
          if (!mbar_wait(&s_full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sw = smem_u32(smem + (size_t)stage * kStageBytes);
          const uint64_t wdesc0 = smem_desc_sw128(sw);
          const uint64_t wdesc1 = smem_desc_sw128(sw + kTileWBytes);
          const uint64_t tdesc = smem_desc_sw128(sw + 2 * kTileWBytes);
#pragma unroll
          for (int k = 0; k < BK / 16; k++) {
            const uint32_t accumulate = (kb | k) != 0 ? 1u : 0u;
            mma_bf16(d0, wdesc0 + 2 * k, tdesc + 2 * k, idesc, accumulate);
            mma_bf16(d1, wdesc1 + 2 * k, tdesc + 2 * k, idesc, accumulate);
          }
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
    const int quad = warp & 3;  // TMEM lanes [32 quad, 32 quad + 32): this warp's 32 features
    uint8_t* patch = smem + (size_t)kStages * kStageBytes + (size_t)(warp - 2) * kPatchBytes;
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
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * quad) << 16) + (uint32_t)(acc * 2 * BT);
      const int nchunks = (ti.ntok + 31) >> 5;
      if (ti.phase == 0) {
        const PhaseParams& pp = p.ph[0];
        const int64_t row_bytes = pp.ld_out * 2;
        uint8_t* dst0 = pp.out + ti.row0 * row_bytes + ((int64_t)ti.n * BW + 32 * quad) * 2;
#pragma unroll 1
        for (int c = 0; c < nchunks; c++) {
          float up[32], gate[32];
          tmem_ld32(taddr + c * 32, up);
          tmem_ld32(taddr + BT + c * 32, gate);
#pragma unroll
          for (int j = 0; j < 32; j++) up[j] = __fdividef(gate[j], 1.0f + __expf(-gate[j])) * up[j];
          const int rows_valid = (int)min64(ti.row_end - (ti.row0 + c * 32), 32);
          transpose_store32(patch, up, dst0 + (int64_t)c * 32 * row_bytes, row_bytes, rows_valid, lane);
        }
      } else {
        const PhaseParams& pp = p.ph[1];
        const int64_t row_bytes = pp.ld_out * 2;
#pragma unroll 1
        for (int h = 0; h < 2; h++) {
          const int64_t f0 = (int64_t)ti.n * 2 * BW + h * BW + 32 * quad;
          if (f0 >= pp.out_cols) continue;
          uint8_t* dst0 = pp.out + ti.row0 * row_bytes + f0 * 2;
#pragma unroll 1
          for (int c = 0; c < nchunks; c++) {
            float v[32];
            tmem_ld32(taddr + h * BT + c * 32, v);
            const int rows_valid = (int)min64(ti.row_end - (ti.row0 + c * 32), 32);
            if (p.fc2_probs) {
              // lane j fetches token j's probability; every lane scales its feature of the 32 tokens
              const float pr = lane < rows_valid ? p.fc2_probs[ti.row0 + c * 32 + lane] : 0.0f;
#pragma unroll
              for (int j = 0; j < 32; j++) v[j] *= __shfl_sync(0xffffffffu, pr, j);
            }
            transpose_store32(patch, v, dst0 + (int64_t)c * 32 * row_bytes, row_bytes, rows_valid, lane);
          }
        }
      }
      tc_fence_before();
      if (ti.phase == 0) {
        // publish this warp's 32 intermediate features of the tile's rows: each
        // lane's stores are fenced (generic and async proxy), then one release add
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        __syncwarp();
        if (lane == 0 && ti.g != p.silent_g)
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.ready + ti.g) : "memory");
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
// 128 bytes, then one FC1 completion counter per token tile.
constexpr size_t kSchedBytes = 128;
size_t grouped_mlp_bf16_ready_bytes(const moe_shape& s, const moe_layout& l) {
  return kSchedBytes + (size_t)((l.capacity + BT - 1) / BT + s.E + 1) * sizeof(int32_t);
}

// FC1 and FC2 in one persistent launch.  An FC2 tile waits (bounded) for the
// FC1 tiles of its token tile.  Tiles are claimed in list order and every FC1
// tile precedes every FC2 tile, so those FC1 tiles were claimed earlier by
// CTAs that hold no FC2 tile in front of them (a CTA's tile claimed after an
// FC2 tile is an FC2 tile); with one CTA per SM and the grid no larger than
// the SM count all CTAs are resident together, so every wait is on work that
// is running or done.
cudaError_t launch_grouped_mlp_bf16(const moe_handle_dev& h, const moe_shape& s, const moe_layout& l,
                                    const void* perm_tokens, const void* w13, const void* w2, void* act,
                                    void* ready, void* out_fc2, const float* fc2_probs, cudaStream_t st,
                                    int64_t silent_token_tile) {
  if (l.capacity == 0) return cudaSuccess;
  if (s.E > kMaxE) return cudaErrorNotSupported;
  const uint64_t cap = (uint64_t)l.capacity;
  CUtensorMap ty, tw13, tact, tw2;
  cudaError_t e;
  if ((e = make_tensor_map_2d(&ty, perm_tokens, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cap, s.H, BT, BK)) != cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&tw13, w13, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)s.E * 2 * s.I, s.H, BW,
                              BK)) != cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&tact, act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cap, s.I, BT, BK)) != cudaSuccess)
    return e;
  if ((e = make_tensor_map_2d(&tw2, w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)s.E * s.H, s.I, BW, BK)) !=
      cudaSuccess)
    return e;
  static PerDeviceOnce attr_once;
  if ((e = attr_once.run([] {
         return cudaFuncSetAttribute(grouped_mlp_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kDynSmem);
       })) != cudaSuccess)
    return e;
  const size_t ready_bytes = grouped_mlp_bf16_ready_bytes(s, l);
  if ((e = cudaMemsetAsync(ready, 0, ready_bytes, st)) != cudaSuccess) return e;

  FusedParams p;
  p.offsets = h.padded_offsets;
  p.status = h.status;
  p.sched = static_cast<int32_t*>(ready);
  p.ready = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ready) + kSchedBytes);
  p.fc2_probs = fc2_probs;
  p.E = (int)s.E;
  p.cap = (int)l.capacity;
  PhaseParams& p1 = p.ph[0];
  p1.out = static_cast<uint8_t*>(act);
  p1.ld_out = s.I;
  p1.out_cols = s.I;
  p1.w_rows_per_expert = 2 * s.I;
  p1.second_offset = s.I;
  p1.n_step = BW;
  p1.nt = (int)(s.I / BW);
  p1.nkb = (int)(s.H / BK);
  PhaseParams& p2 = p.ph[1];
  p2.out = static_cast<uint8_t*>(out_fc2);
  p2.ld_out = s.H;
  p2.out_cols = s.H;
  p2.w_rows_per_expert = s.H;
  p2.second_offset = BW;
  p2.n_step = 2 * BW;
  p2.nt = (int)((s.H + 2 * BW - 1) / (2 * BW));
  p2.nkb = (int)(s.I / BK);
  p.ready_target = kEpiWarps * p1.nt;
  p.silent_g = silent_token_tile >= 0 && silent_token_tile < (int64_t)INT32_MAX ? (int)silent_token_tile : -1;

  const int64_t t_tiles_bound = (l.capacity + BT - 1) / BT + s.E;
  int64_t grid = device_sm_count();
  if (grid > t_tiles_bound * (p1.nt + p2.nt)) grid = t_tiles_bound * (p1.nt + p2.nt);
  if (grid < 1) grid = 1;

  const ProfileEvents prof = take_profile_events();
  if (prof.before_fc1 && (e = record_profile_event(prof.before_fc1, st)) != cudaSuccess) return e;
  grouped_mlp_bf16_kernel<<<(unsigned)grid, kThreads, kDynSmem, st>>>(ty, tw13, tact, tw2, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // one kernel runs both GEMMs: the FC1/FC2 boundary event is recorded with the end
  if (prof.after_fc1 && (e = record_profile_event(prof.after_fc1, st)) != cudaSuccess) return e;
  if (prof.after_fc2 && (e = record_profile_event(prof.after_fc2, st)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace moe
