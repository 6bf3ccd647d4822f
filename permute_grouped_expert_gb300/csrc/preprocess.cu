// preprocess.cu -- metadata preprocessing on the device: per-expert histogram,
// padded exclusive scan with capacity and overflow flag, and the stable row map.
//
// Follows DeepEP PR #716 "perf: reuse HybridEP routing allgather buffer"
// (Summary: the routing map is consumed by metadata preprocessing on the same
// stream before dispatch; Testing: padding multiple) and NeMo Automodel PR #3931
// "perf(moe): sync-free HybridEP dispatch" (What does this PR do?: real counts
// stay on the device; overflow flag instead of a host sync).
//
// Two kernels, one pass over the routing map each:
//   pre_rank_kernel     tiles of tokens; a warp-aggregated histogram per warp
//                       (__match_any_sync groups lanes routed to one expert, one
//                       shared-memory update per group) yields each route's rank
//                       among earlier routes of its tile; a decoupled lookback over
//                       tiles (per expert, acquire/release flag words, bounded
//                       spin) turns tile aggregates into tile prefixes; the tile
//                       that completes the chain writes counts, padded offsets,
//                       total rows and the overflow flag.
//   pre_finalize_kernel adds each expert's padded offset, applies the capacity,
//                       scatters token_of / slot_of and marks pad rows.
#include <algorithm>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr uint64_t kFlagAggregate = 1ull << 32;
constexpr uint64_t kFlagInclusive = 2ull << 32;

struct PreParams {
  int format;
  const void* map;
  int64_t T, E, K, m, cap;
  int64_t tokens_per_tile, num_tiles;
  int32_t* tile_counter;
  uint64_t* lookback;
  int16_t* route_expert;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_of;
  int32_t* token_of;
  int32_t* slot_of;
  int32_t* total_rows;
  int32_t* overflow;
  int32_t* status;      // the handle's status word: written once, by the finalize kernel
  int32_t* ws_status;   // this call's status bits, gathered in the workspace (cleared with the counters)
  int64_t silent_tile;  // testing hook: this tile never publishes its lookback words (-1: none)
};

// Exclusive scan of one int64 per thread across the block (kPreThreads threads).
__device__ int64_t block_exclusive_scan(int64_t v, int64_t* warp_tot, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int64_t o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t run = 0;
    for (int w = 0; w < kPreWarps; w++) {
      int64_t c = warp_tot[w];
      warp_tot[w] = run;
      run += c;
    }
    *total = run;
  }
  __syncthreads();
  return warp_tot[warp] + incl - v;
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* ptr) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ptr) : "memory");
  return v;
}

// Copy n bytes of global memory into shared memory with the whole block:
// 16-byte vectors over the aligned middle, single bytes at the ends.
__device__ void stage_bytes(uint8_t* dst, const uint8_t* src, int n) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(src);
  int head = (int)((16 - (a & 15)) & 15);
  if (head > n) head = n;
  const int nvec = (n - head) / 16;
  for (int i = threadIdx.x; i < head; i += blockDim.x) dst[i] = src[i];
  for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + head) + i);
    uint32_t* d = reinterpret_cast<uint32_t*>(dst + head + 16 * i);  // dst + head may be unaligned for uint4
    if (((reinterpret_cast<uintptr_t>(d)) & 15) == 0) {
      *reinterpret_cast<uint4*>(d) = v;
    } else {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 16; q++) dst[head + 16 * i + q] = (uint8_t)(w[q >> 2] >> (8 * (q & 3)));
    }
  }
  for (int i = head + 16 * nvec + threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

constexpr int kLookbackWindow = 16;

__global__ void __launch_bounds__(kPreThreads) pre_rank_kernel(PreParams p) {
  extern __shared__ __align__(16) int32_t smem[];
  const int E = (int)p.E, K = (int)p.K;
  int32_t* running = smem;                     // [warps][E]: per-warp counts, then warp bases
  int32_t* agg = running + kPreWarps * E;      // [E] tile aggregate (counts on the last tile)
  int32_t* prefix = agg + E;                   // [E] exclusive prefix of this tile
  int32_t* partial = prefix + E;               // [kPreMaxEntries] rank inside the warp's share
  int16_t* eid = reinterpret_cast<int16_t*>(partial + kPreMaxEntries);  // [kPreMaxEntries]
  uint8_t* stage = reinterpret_cast<uint8_t*>(eid + kPreMaxEntries);    // [kPreStageBytes] routing map of the tile
  __shared__ int s_tile, s_err;
  __shared__ int64_t s_warp_tot[kPreWarps], s_total;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    // Tiles are numbered in the order blocks start, so every predecessor a tile
    // looks back on is already resident: the lookback cannot wait on a block
    // that has not been scheduled.
    s_tile = atomicAdd(p.tile_counter, 1);
    s_err = 0;
  }
  for (int i = tid; i < kPreWarps * E; i += blockDim.x) running[i] = 0;
  __syncthreads();

  const int64_t tile = s_tile;
  const int64_t t0 = tile * p.tokens_per_tile;
  const int64_t t1 = min64(t0 + p.tokens_per_tile, p.T);
  const int ntok = (int)max64(0, t1 - t0);
  // stage this tile's part of the routing map in shared memory (coalesced, vectorised)
  if (p.format == MOE_ROUTING_DENSE_I16)
    stage_bytes(stage, static_cast<const uint8_t*>(p.map) + t0 * K * 2, ntok * K * 2);
  else
    stage_bytes(stage, static_cast<const uint8_t*>(p.map) + t0 * E, ntok * E);
  __syncthreads();

  const int tpw = (ntok + kPreWarps - 1) / kPreWarps;  // tokens per warp
  const int wt0 = min(warp * tpw, ntok), wt1 = min(wt0 + tpw, ntok);
  int32_t* my_run = running + warp * E;
  int err = 0;

  if (p.format == MOE_ROUTING_DENSE_I16) {
    const int16_t* idx = reinterpret_cast<const int16_t*>(stage);
    const int ebeg = wt0 * K, eend = wt1 * K;
    for (int base = ebeg; base < eend; base += 32) {
      const int i = base + lane;
      int e = -1;
      if (i < eend) {
        int v = idx[i];
        if (v != -1 && (v < 0 || v >= E)) {
          err |= MOE_DEV_ERR_BAD_EXPERT;
          v = -1;
        }
        e = v;
      }
      // warp-aggregated histogram: one update per group of lanes with one expert
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & lanemask_lt());
      const int run = (e >= 0) ? my_run[e] : 0;
      __syncwarp();
      if (e >= 0 && rank == 0) my_run[e] = run + __popc(peers);
      __syncwarp();
      if (i < eend) {
        partial[i] = run + rank;
        eid[i] = (int16_t)e;
      }
    }
  } else {
    for (int tl = wt0; tl < wt1; tl++) {
      const uint8_t* row = stage + (size_t)tl * E;
      int k_base = 0;
      for (int c = 0; c < E; c += 32) {
        const int e = c + lane;
        const bool set = (e < E) && row[e] != 0;
        const unsigned mask = __ballot_sync(0xffffffffu, set);
        const int k = k_base + __popc(mask & lanemask_lt());
        if (set) {
          if (k < K) {
            const int run = my_run[e];  // experts are distinct across lanes
            my_run[e] = run + 1;
            partial[tl * K + k] = run;
            eid[tl * K + k] = (int16_t)e;
          } else {
            err |= MOE_DEV_ERR_TOO_MANY_ROUTES;
          }
        }
        k_base += __popc(mask);
      }
      for (int k = k_base + lane; k < K; k += 32) {
        eid[tl * K + k] = -1;
        partial[tl * K + k] = -1;
      }
      __syncwarp();
    }
  }
  if (err) atomicOr(&s_err, err);
  __syncthreads();
  if (tid == 0 && s_err) set_status(p.ws_status, s_err);

  // warp bases and tile aggregate per expert; publish the aggregate at once
  for (int e = tid; e < E; e += blockDim.x) {
    int s = 0;
    for (int w = 0; w < kPreWarps; w++) {
      const int c = running[w * E + e];
      running[w * E + e] = s;
      s += c;
    }
    agg[e] = s;
    uint64_t* word = p.lookback + tile * p.E + e;
    if (tile == 0) prefix[e] = 0;  // set even when the tile stays silent: the rank loop reads it
    if (tile == p.silent_tile) {
      // testing hook: successors find nothing published and their bounded wait runs out
    } else if (tile == 0) {
      st_release_u64(word, kFlagInclusive | (uint32_t)s);
    } else {
      st_release_u64(word, kFlagAggregate | (uint32_t)s);
    }
  }

  // decoupled lookback, one expert column per thread, kLookbackWindow
  // predecessors loaded at once: stop at the nearest inclusive prefix, sum the
  // aggregates in between, and wait (bounded) only on a tile that has not
  // published anything yet
  if (tile > 0) {
    for (int e = tid; e < E; e += blockDim.x) {
      int64_t acc = 0;
      int64_t j = tile - 1;
      uint64_t t_start = 0;
      while (j >= 0) {
        const int n = (int)min64(kLookbackWindow, j + 1);
        uint64_t v[kLookbackWindow];
#pragma unroll
        for (int q = 0; q < kLookbackWindow; q++)
          if (q < n) v[q] = ld_relaxed_u64(p.lookback + (j - q) * p.E + e);
        int64_t sum = 0;
        int stop = n;
        bool inclusive = false, not_ready = false;
#pragma unroll
        for (int q = 0; q < kLookbackWindow; q++) {
          if (q >= n || inclusive || not_ready) continue;
          const uint64_t flag = v[q] & ~0xffffffffull;
          if (flag == 0) {
            not_ready = true;
            stop = q;
          } else {
            sum += (uint32_t)v[q];
            if (flag == kFlagInclusive) inclusive = true;
          }
        }
        acc += sum;
        if (inclusive) break;
        if (not_ready) {
          j -= stop;
          const uint64_t now = globaltimer_ns();
          if (stop > 0 || t_start == 0) {
            t_start = now;
          } else if (now - t_start > kWaitLimitNs) {
            set_status(p.ws_status, MOE_DEV_ERR_TIMEOUT);
            break;
          }
          __nanosleep(32);
          continue;
        }
        j -= n;
        t_start = 0;
      }
      prefix[e] = (int32_t)acc;
      if (tile != p.silent_tile)
        st_release_u64(p.lookback + tile * p.E + e, kFlagInclusive | (uint32_t)(acc + agg[e]));
    }
  }
  __syncthreads();

  // rank of each route among its expert's routes so far (offset added later)
  for (int i = tid; i < ntok * K; i += blockDim.x) {
    const int e = eid[i];
    int32_t out = -1;
    if (e >= 0) out = partial[i] + running[((i / K) / tpw) * E + e] + prefix[e];
    p.row_of[t0 * K + i] = out;
    p.route_expert[t0 * K + i] = (int16_t)e;
  }

  // the tile that completes the chain owns the totals
  if (tile == p.num_tiles - 1) {
    for (int e = tid; e < E; e += blockDim.x) {
      const int c = prefix[e] + agg[e];
      p.counts[e] = c;
      agg[e] = c;
    }
    __syncthreads();
    const int per = (E + blockDim.x - 1) / blockDim.x;
    int64_t local = 0;
    for (int j = 0; j < per; j++) {
      const int e = tid * per + j;
      if (e < E) local += ((agg[e] + p.m - 1) / p.m) * p.m;
    }
    int64_t run = block_exclusive_scan(local, s_warp_tot, &s_total);
    for (int j = 0; j < per; j++) {
      const int e = tid * per + j;
      if (e < E) {
        p.offsets[e] = (int32_t)run;
        run += ((agg[e] + p.m - 1) / p.m) * p.m;
      }
    }
    if (tid == 0) {
      p.offsets[E] = (int32_t)s_total;
      *p.total_rows = (int32_t)s_total;
      *p.overflow = (s_total > p.cap) ? 1 : 0;
    }
  }
}

__global__ void __launch_bounds__(256) pre_finalize_kernel(PreParams p) {
  extern __shared__ __align__(16) int32_t soff[];  // [E+1]
  const int E = (int)p.E;
  // the rank kernel has finished: its status bits replace the handle's status word
  const int32_t ws_status = *p.ws_status;
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.status = ws_status;
  // after a timed-out lookback the ranks and offsets are incomplete: every route is
  // marked dropped and nothing is scattered (the call's outputs are documented invalid)
  const bool valid = (ws_status & MOE_DEV_ERR_TIMEOUT) == 0;
  for (int i = threadIdx.x; i <= E; i += blockDim.x) soff[i] = p.offsets[i];
  __syncthreads();
  const int64_t n = p.T * p.K;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int e = p.route_expert[i];
    int32_t out = -1;
    if (valid && e >= 0) {
      const int64_t dest = (int64_t)soff[e] + p.row_of[i];
      if (dest >= 0 && dest < p.cap) {
        out = (int32_t)dest;
        p.token_of[dest] = (int32_t)(i / p.K);
        p.slot_of[dest] = (int32_t)(i % p.K);
      }
    }
    p.row_of[i] = out;
  }
  // pad rows of each expert segment (fewer than m per expert)
  if (!valid) return;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += stride) {
    const int64_t beg = max64(0, (int64_t)soff[e] + p.counts[e]);
    const int64_t end = min64(soff[e + 1], p.cap);
    for (int64_t r = beg; r < end; r++) {
      p.token_of[r] = -1;
      p.slot_of[r] = -1;
    }
  }
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

size_t preprocess_workspace_bytes(int64_t T, int64_t E, int64_t K) {
  const int64_t tiles = pre_num_tiles(T, E, K);
  return 256 + align_up((size_t)tiles * E * 8, 256) + align_up((size_t)(T * K) * 2, 256);
}

PreWorkspace preprocess_workspace_carve(void* ws, int64_t T, int64_t E, int64_t K) {
  const int64_t tiles = pre_num_tiles(T, E, K);
  char* b = static_cast<char*>(ws);
  PreWorkspace w;
  w.tile_counter = reinterpret_cast<int32_t*>(b);
  w.lookback = reinterpret_cast<uint64_t*>(b + 256);
  w.memset_bytes = 256 + (size_t)tiles * E * 8;
  w.route_expert = reinterpret_cast<int16_t*>(b + 256 + align_up((size_t)tiles * E * 8, 256));
  return w;
}

cudaError_t launch_preprocess(const moe_routing& r, const moe_shape& s, const moe_layout& l,
                              const moe_handle_dev& h, const PreWorkspace& ws, cudaStream_t st, int64_t silent_tile) {
  PreParams p;
  p.silent_tile = silent_tile;
  p.format = r.format;
  p.map = r.map;
  p.T = s.T;
  p.E = s.E;
  p.K = s.K;
  p.m = l.pad_multiple;
  p.cap = l.capacity;
  p.tokens_per_tile = pre_tokens_per_tile(s.T, s.E, s.K);
  p.num_tiles = pre_num_tiles(s.T, s.E, s.K);
  p.tile_counter = ws.tile_counter;
  p.lookback = ws.lookback;
  p.route_expert = ws.route_expert;
  p.counts = h.tokens_per_expert;
  p.offsets = h.padded_offsets;
  p.row_of = h.row_of;
  p.token_of = h.token_of;
  p.slot_of = h.slot_of;
  p.total_rows = h.total_rows;
  p.overflow = h.overflow;
  p.status = h.status;
  p.ws_status = ws.tile_counter + 32;  // inside the cleared header, 128 bytes after the tile counter

  cudaError_t e;
  if ((e = cudaMemsetAsync(ws.tile_counter, 0, ws.memset_bytes, st)) != cudaSuccess) return e;

  const size_t smem_a = (size_t)(kPreWarps + 2) * s.E * 4 + (size_t)kPreMaxEntries * 6 + kPreStageBytes;
  static PerDeviceOnce attr_once;
  e = attr_once.run([] {
    return cudaFuncSetAttribute(pre_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)((kPreWarps + 2) * 1024 * 4 + kPreMaxEntries * 6 + kPreStageBytes));
  });
  if (e != cudaSuccess) return e;
  pre_rank_kernel<<<(unsigned)p.num_tiles, kPreThreads, smem_a, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const int64_t n = s.T * s.K;
  int64_t blocks = (std::max<int64_t>(n, s.E) + 255) / 256;
  const int64_t max_blocks = (int64_t)device_sm_count() * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  pre_finalize_kernel<<<(unsigned)blocks, 256, (size_t)(s.E + 1) * 4, st>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
