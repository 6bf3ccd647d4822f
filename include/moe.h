/*
 * moe.h -- C ABI of the GB300 (sm_103a) single-GPU MoE dispatch -> grouped
 * expert MLP -> combine library.
 *
 * The four calls of one MoE layer forward, in stream order:
 *
 *   moe_preprocess         routing map -> per-expert counts, padded offsets,
 *                          stable row map, overflow flag (all on the device)
 *   moe_dispatch_permute   token rows (+ probabilities, + FP8 / NVFP4 scales)
 *                          -> expert-grouped rows in a caller-owned buffer
 *   moe_grouped_mlp        FC1 -> SwiGLU -> FC2 per expert, FC2 rows written
 *                          into a caller-owned buffer
 *   moe_combine_unpermute  expert rows -> token order, top-k probability-
 *                          weighted sum
 *
 * Sources, by page title and section:
 *   [REUSE-BUF] Megatron-LM PR #6800 "Reuse caller-owned HybridEP dispatch and
 *               expert output buffers" (Summary; Configuration; Known
 *               limitations): dispatch and grouped FC2 write into persistent
 *               caller-owned rings; the final consumer releases a slot; early
 *               reuse and double release fail explicitly; a static output bound
 *               is required.
 *   [ALLGATHER] DeepEP PR #716 "perf: reuse HybridEP routing allgather buffer"
 *               (Memory impact; Testing): sparse Boolean tokens x experts and
 *               dense int16 tokens x topk routing maps; padding multiple;
 *               dispatch with permutation and combine with unpermutation, with
 *               and without probabilities; bitwise-identical dispatched rows.
 *   [SYNC-FREE] NeMo Automodel PR #3931 "perf(moe): sync-free HybridEP dispatch
 *               (capacity mode, equal token counts)" (What does this PR do?;
 *               Validation): non-blocking dispatch sized by a host integer
 *               capacity = ceil(rows x factor), 4-aligned; real counts stay on
 *               the device; an overflow flag in the handle replaces the host
 *               sync; truncation past the capacity is silent.
 *   [ELASTIC]   Megatron-LM PR #4632 "moe: add DeepEP V2 ElasticBuffer support
 *               to MoE flex dispatcher" (Motivation): the per-expert counts live
 *               on the dispatch handle; the layout is inferred from the top-k ids.
 *   [MEGAMOE]   TensorRT-LLM PR #16190 "Update CuTeDSL MegaMoE kernels" (commit
 *               list): NVFP4 expert weights w3_w1 / w2 with block scales,
 *               weight_scale_2 and input_scale; zero-token launches keep a
 *               non-empty grid; int64 offsets into large pools; zero only the
 *               leading workspace bytes that need it.
 *
 * Conventions (all calls):
 *   - Every device buffer is owned by the caller.  The library never allocates
 *     or frees device memory and never synchronises the host with the device.
 *     All work is enqueued on the given CUDA stream (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream), so the four calls can be
 *     captured into one CUDA graph and replayed.
 *   - Arguments are validated on the host before anything is enqueued; a bad
 *     argument returns MOE_ERR_INVALID_ARG and enqueues nothing.
 *   - Capacity overflow is not an error status: it is the device int32 flag
 *     handle->overflow, which the caller reads when it chooses to.
 *   - Device-side anomalies (malformed routing, a bounded wait that ran out)
 *     set bits of the device int32 handle->status; no kernel ever traps.
 *   - Row and byte offsets are computed in 64-bit integers.
 *   - Device pointers to rows must be 16-byte aligned; H must be a multiple of
 *     128 (so every row is a whole number of 16-byte vectors and 128-element
 *     FP8 scale blocks).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* bad pointer, shape, alignment or enum */
  MOE_ERR_UNSUPPORTED = 2,          /* dtype / shape combination not built, or no sm_103 device */
  MOE_ERR_CUDA = 3,                 /* a CUDA call failed; see moe_last_cuda_error() */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,  /* workspace smaller than the *_workspace_size query */
  MOE_ERR_RING_EARLY_REUSE = 5,     /* ring slot acquired again before its release */
  MOE_ERR_RING_DOUBLE_RELEASE = 6   /* ring slot released while not held */
} moe_status;

/* Routing map layouts ([ALLGATHER], Memory impact). */
enum {
  MOE_ROUTING_DENSE_I16 = 0,   /* int16 topk_idx [T][K]; -1 = no route in that slot;
                                  probs (optional) float [T][K] */
  MOE_ROUTING_SPARSE_BOOL = 1  /* uint8 map [T][E], nonzero = routed; slot k of a token
                                  is its k-th routed expert in ascending expert order;
                                  probs (optional) float [T][E] */
};

/* Element formats of dispatched rows and expert weights. */
enum {
  MOE_DTYPE_BF16 = 0,            /* bf16 rows */
  MOE_DTYPE_FP8_E4M3_B128 = 1,   /* E4M3 codes + one fp32 scale per 128 consecutive
                                    elements of a row (activations) or per 128x128
                                    block (weights) */
  MOE_DTYPE_BF16_TO_FP8 = 2,     /* dispatch only: bf16 input quantized to
                                    MOE_DTYPE_FP8_E4M3_B128 on the way */
  MOE_DTYPE_NVFP4 = 3,           /* packed E2M1 (2 per byte, even element in the low
                                    nibble) + one E4M3 scale per 16 consecutive
                                    elements + one fp32 global scale */
  MOE_DTYPE_BF16_TO_NVFP4 = 4    /* dispatch only: bf16 input quantized to NVFP4 */
};

/* Formats of expert-output rows read by the combine ([MEGAMOE], commit list:
 * bf16 / fp8 / fp4 combine formats with E8M0 scale factors and E2M1 fp4
 * vectors).  MX formats (the OCP Microscaling family, whose scales are E8M0):
 * blocks of 32 consecutive elements of a row share a scale 2^X stored as the
 * byte X + 127, X = floor(log2(amax)) - emax (emax 8 for E4M3, 2 for E2M1)
 * clamped to [-127, 127], 0 for an all-zero block; each element is x / 2^X
 * rounded to nearest even and saturated.  Row layouts: MXFP8 codes [cap][H]
 * bytes, MXFP4 packed [cap][H/2] (even element in the low nibble); scales
 * [cap][H/32] bytes. */
enum {
  MOE_COMBINE_BF16 = 0,   /* bf16 [cap][H] */
  MOE_COMBINE_MXFP8 = 1,  /* E4M3 + E8M0 per 32 */
  MOE_COMBINE_MXFP4 = 2   /* E2M1 + E8M0 per 32 */
};

/* Bits of the device status word handle->status. */
#define MOE_DEV_ERR_BAD_EXPERT 1      /* a dense id outside [-1, E): treated as no route */
#define MOE_DEV_ERR_TOO_MANY_ROUTES 2 /* a sparse row with more than K routed experts:
                                         the extra ones are ignored */
#define MOE_DEV_ERR_TIMEOUT 4         /* a bounded inter-CTA wait gave up; outputs of
                                         that call are not valid */
#define MOE_DEV_ERR_BOUNDS 8          /* bounds-checked build only (compiled with
                                         -DMOE_CHECKED): a computed index failed its
                                         check and the access was skipped */

typedef struct moe_shape {
  int64_t T; /* tokens (>= 0) */
  int64_t H; /* hidden size (multiple of 128) */
  int64_t E; /* experts (1..1024) */
  int64_t K; /* routes per token (1..128, K <= E) */
  int64_t I; /* SwiGLU intermediate size (multiple of 128; 0 when no MLP is run) */
} moe_shape;

typedef struct moe_layout {
  int64_t pad_multiple; /* m: each expert's segment is padded to a multiple of m (>= 1);
                           T*K + E*(m-1), the largest padded total, must be < 2^31 */
  int64_t capacity;     /* cap: rows of the dispatch / expert-output buffers (>= 0).
                           Routes whose destination row reaches cap are dropped. */
} moe_layout;

typedef struct moe_routing {
  int32_t format;     /* MOE_ROUTING_* */
  const void* map;    /* device pointer, layout per format */
  const float* probs; /* device pointer or NULL */
} moe_routing;

/* Device arrays written by moe_preprocess and read by the other calls (the
 * "handle" of [SYNC-FREE] / [ELASTIC]).  All caller-owned device memory. */
typedef struct moe_handle_dev {
  int32_t* tokens_per_expert; /* [E]   real routed count per expert (never clamped) */
  int32_t* padded_offsets;    /* [E+1] offsets[e] = sum_{e'<e} ceil(count[e']/m)*m */
  int32_t* row_of;            /* [T*K] destination row of route (t,k), or -1 */
  int32_t* token_of;          /* [cap] source token of each row < min(offsets[E],cap);
                                       -1 for pad rows; rows beyond are not written */
  int32_t* slot_of;           /* [cap] route slot k of each such row; -1 for pad rows */
  int32_t* total_rows;        /* [1]   offsets[E] (unclamped) */
  int32_t* overflow;          /* [1]   1 when offsets[E] > cap, else 0 */
  int32_t* status;            /* [1]   MOE_DEV_ERR_* bits of the last preprocess */
} moe_handle_dev;

/* ---------------------------------------------------------------- helpers */

/* Capacity rule of [SYNC-FREE], What does this PR do?: ceil(rows x factor)
 * rounded up to a multiple of align (the pages use 4).  rows >= 0, factor > 0,
 * align >= 1.  Host only. */
MOE_API moe_status moe_capacity(int64_t rows, double factor, int64_t align, int64_t* capacity_out);

/* Bytes of a routing map ([ALLGATHER], Memory impact): T*E for the sparse
 * Boolean layout, T*K*2 for dense int16 ids.  Host only. */
MOE_API moe_status moe_routing_map_bytes(int32_t format, int64_t T, int64_t E, int64_t K, size_t* bytes_out);

/* Decode-bucket selection ([MEGAMOE], commit list: adaptive max-tokens
 * bucketing, so that a decode batch launches kernels sized for a small bucket
 * instead of the prefill maximum; the full bucket is kept for zero tokens so
 * no launch has an empty grid; a batch above the largest bucket is an error).
 * ladder: n >= 1 strictly increasing positive token counts (host array), the
 * shapes a caller has sized buffers for and captured graphs at.  Returns in
 * *bucket_out the smallest ladder entry >= max(tokens, 1).  The caller runs
 * the layer at T = bucket with the extra tokens' routing set to "no route"
 * (dense id -1, or an all-zero sparse row): they get no rows, and every real
 * token's results are those of the unpadded batch.  Host only.  Errors:
 * MOE_ERR_INVALID_ARG for tokens < 0, tokens above ladder[n-1], or a ladder
 * that is empty, unsorted or not positive. */
MOE_API moe_status moe_decode_bucket(int64_t tokens, const int64_t* ladder, int32_t n, int64_t* bucket_out);

/* Message of the last CUDA error seen by this thread's library calls. */
MOE_API const char* moe_last_cuda_error(void);
MOE_API const char* moe_status_string(moe_status s);

/* ------------------------------------------------------------- preprocess */

/* Device workspace bytes moe_preprocess needs for this shape (host only). */
MOE_API moe_status moe_preprocess_workspace_size(const moe_shape* shape, size_t* bytes_out);

/* Metadata preprocessing ([ALLGATHER], Summary: the routing map is consumed by
 * metadata preprocessing on the same stream before dispatch; [SYNC-FREE]).
 * Computes, on the device, every array of *handle:
 *   tokens_per_expert, padded_offsets, total_rows, overflow: as documented in
 *   moe_handle_dev;
 *   row_of[t*K+k] = padded_offsets[e] + (number of routes (t',k') to the same
 *   expert e that come before (t,k) in (token, slot) order), i.e. a stable sort
 *   of the routes by expert, or -1 when that destination is >= capacity (the
 *   route is dropped) or the slot has no route.
 * routing: map (and probs, unused here) on the device.  workspace: device
 * memory of at least moe_preprocess_workspace_size bytes, 16-byte aligned; its
 * contents need no initialisation and are scratch between calls.
 * Runs 2 memsets and 2 kernels on `stream`; no host sync. */
MOE_API moe_status moe_preprocess(const moe_routing* routing, const moe_shape* shape, const moe_layout* layout,
                          const moe_handle_dev* handle, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Allocation-free variant of moe_preprocess.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory, such
 * as a plugin running inside a host application that owns every device
 * allocation and gives its plugins no allocator, or a latency-critical loop
 * that sized its memory once and must not call cudaMalloc (which can
 * synchronise the device).  It computes exactly what moe_preprocess computes,
 * with the same kernels, but its scratch space is a fixed device array inside
 * the library (MOE_PREPROCESS_NOALLOC_SCRATCH_BYTES, held by every GPU that
 * loads the library until the process exits) instead of a caller workspace.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - Checks, in order: the arguments as moe_preprocess checks them
 *     (MOE_ERR_INVALID_ARG), then the size rule: shapes whose scratch need
 *     (moe_preprocess_workspace_size) exceeds
 *     MOE_PREPROCESS_NOALLOC_SCRATCH_BYTES are rejected with
 *     MOE_ERR_WORKSPACE_TOO_SMALL.  Nothing is enqueued when a check fails.
 *   - Each call outside stream capture looks up the array's device address
 *     on the current device with cudaGetSymbolAddress (so a module reloaded
 *     after cudaDeviceReset is found at its new address) and caches it per
 *     device; a call made during stream capture uses that cached address.
 *     Make at least one call on a device before capturing on it, and none
 *     between a cudaDeviceReset and the next uncaptured call.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents; each call clears the bytes that must start at zero on
 *     its own stream.  Calls whose GPU work overlaps (other streams, other host
 *     threads) race on the array and must be serialised by the caller. */
#define MOE_PREPROCESS_NOALLOC_SCRATCH_BYTES (8u << 20)
MOE_API moe_status moe_preprocess_noalloc(const moe_routing* routing, const moe_shape* shape,
                                          const moe_layout* layout, const moe_handle_dev* handle, void* stream);

/* --------------------------------------------------------------- dispatch */

/* dispatch_with_permute ([REUSE-BUF], Summary; [ALLGATHER], Testing): for every
 * route (t,k) with r = row_of[t*K+k] >= 0:
 *   out_tokens[r] = x[t] (bitwise for BF16 / FP8 input; quantized on the way for
 *                  BF16_TO_FP8 / BF16_TO_NVFP4),
 *   out_scales[r] = that row's scales (FP8: fp32 [H/128]; NVFP4: E4M3 codes [H/16]),
 *   out_probs[r]  = the route's probability (when out_probs and routing->probs
 *                   are both non-NULL).
 * Pad rows [offsets[e]+count[e], offsets[e+1]) below the capacity are written
 * with zeros (tokens, scales and probability).  Rows at or beyond
 * min(offsets[E], cap) are not touched.
 * in_dtype: MOE_DTYPE_BF16 (x bf16 [T][H]), MOE_DTYPE_FP8_E4M3_B128 (x codes
 * [T][H] + x_scales fp32 [T][H/128]), MOE_DTYPE_BF16_TO_FP8 (x bf16; output
 * codes + fp32 scales; scale = amax/448 per 128 elements, 1 for an all-zero
 * block, code = E4M3(x / scale) rounded to nearest even, saturating),
 * MOE_DTYPE_BF16_TO_NVFP4 (x bf16; output packed E2M1 [H/2] + E4M3 scale codes
 * [H/16] with the fp32 global scale *nvfp4_global (device pointer, passed in
 * x_scales): block scale = E4M3(amax / (6 * global)), code = E2M1(x / (block *
 * global))).
 * out_tokens: device [cap][row bytes]; out_scales: device or NULL (required for
 * FP8 / NVFP4 outputs); out_probs: device float [cap] or NULL. */
MOE_API moe_status moe_dispatch_permute(const moe_handle_dev* handle, const moe_shape* shape,
                                const moe_layout* layout, int32_t in_dtype, const void* x,
                                const void* x_scales, const moe_routing* routing, void* out_tokens,
                                float* out_probs, void* out_scales, void* stream);

/* ---------------------------------------------------------------- combine */

/* combine with unpermutation ([ALLGATHER], Testing; [MEGAMOE], TopkReduce):
 *   y[t] = bf16( sum over k ascending with r = row_of[t*K+k] >= 0 of
 *                w(r) * expert_out[r] )
 * with fp32 accumulation, w(r) = perm_probs[r] or 1 when perm_probs is NULL.
 * A token whose routes were all dropped gets zeros.
 * expert_out: device bf16 [cap][H]; perm_probs: device float [cap] or NULL;
 * y: device bf16 [T][H]. */
MOE_API moe_status moe_combine_unpermute(const moe_handle_dev* handle, const moe_shape* shape,
                                 const moe_layout* layout, const void* expert_out,
                                 const float* perm_probs, void* y, void* stream);

/* combine with unpermutation from expert rows in a combine format: as
 * moe_combine_unpermute, with the expert rows decoded from in_format
 * (MOE_COMBINE_BF16 reads expert_out as bf16 and ignores expert_out_scales;
 * the MX formats read codes from expert_out and E8M0 scales from
 * expert_out_scales, layouts as documented with MOE_COMBINE_*):
 *   y[t] = bf16( sum over k ascending of w(r) * decoded O[r] ), fp32 accumulation.
 * Errors: MOE_ERR_INVALID_ARG for an unknown format or a NULL / misaligned
 * buffer (expert_out and y 16-byte aligned). */
MOE_API moe_status moe_combine_unpermute_fmt(const moe_handle_dev* handle, const moe_shape* shape,
                                             const moe_layout* layout, int32_t in_format, const void* expert_out,
                                             const void* expert_out_scales, const float* perm_probs, void* y,
                                             void* stream);

/* bf16 rows [R][H] (H a multiple of 32) -> a combine format's codes and E8M0
 * scales (format MOE_COMBINE_MXFP8 or MOE_COMBINE_MXFP4; layouts as documented
 * with MOE_COMBINE_*).  For expert outputs that were written in bf16. */
MOE_API moe_status moe_quantize_mx_rows(const void* x, int64_t R, int64_t H, int32_t format, void* codes,
                                        void* scales, void* stream);

/* --------------------------------------------------------------- backward */

/* Backward of moe_combine_unpermute ([ALLGATHER], Testing / Output and gradient
 * regression: hidden-state and probability gradients of the combine;
 * [SYNC-FREE], What does this PR do?: the combine's backward is a dispatch sized
 * by the same host capacity).  For the output gradient grad_y and every kept
 * route (t,k) -> r = row_of[t*K+k] >= 0:
 *   grad_expert_out[r] = bf16( w(r) * grad_y[t] )   (fp32 product, rounded once)
 *   grad_perm_probs[r] = sum_h grad_y[t][h] * expert_out[r][h]   (fp32)
 * with w(r) = perm_probs[r], or 1 when perm_probs is NULL.  Pad rows
 * [offsets[e]+count[e], offsets[e+1]) below the capacity get zero gradient rows
 * and zero probability gradients; rows at or beyond min(offsets[E], cap) are
 * not touched.
 * grad_y: device bf16 [T][H]; expert_out: device bf16 [cap][H] (the combine's
 * input; required when grad_perm_probs is non-NULL, else ignored);
 * perm_probs: device float [cap] or NULL; grad_expert_out: device bf16
 * [cap][H]; grad_perm_probs: device float [cap] or NULL (not formed).
 * Errors: MOE_ERR_INVALID_ARG for a NULL or misaligned row buffer, or
 * grad_perm_probs without expert_out and perm_probs. */
MOE_API moe_status moe_combine_backward(const moe_handle_dev* handle, const moe_shape* shape,
                                        const moe_layout* layout, const void* grad_y, const void* expert_out,
                                        const float* perm_probs, void* grad_expert_out, float* grad_perm_probs,
                                        void* stream);

/* Backward of moe_dispatch_permute for bf16 rows ([ALLGATHER], Testing / Output
 * and gradient regression: hidden-state and probability gradients of the
 * dispatch).  For row gradients grad_perm_tokens and probability gradients
 * grad_perm_probs of the dispatched rows:
 *   grad_x[t] = bf16( sum over k ascending with r = row_of[t*K+k] >= 0 of
 *               grad_perm_tokens[r] )   (fp32 accumulation; a token whose
 *               routes were all dropped gets zeros)
 *   grad_probs(t,k) = grad_perm_probs[r] for a kept route, else 0, written in
 *               the routing layout of routing_format: MOE_ROUTING_DENSE_I16
 *               float [T][K]; MOE_ROUTING_SPARSE_BOOL float [T][E] with the
 *               entry of the route's expert set and every other entry 0.
 * grad_perm_tokens: device bf16 [cap][H]; grad_perm_probs: device float [cap]
 * or NULL; grad_x: device bf16 [T][H]; grad_probs: device float or NULL (not
 * formed; required when grad_perm_probs is given).
 * Errors: MOE_ERR_INVALID_ARG for a NULL or misaligned row buffer, an unknown
 * routing format, or exactly one of grad_perm_probs / grad_probs NULL. */
MOE_API moe_status moe_dispatch_backward(const moe_handle_dev* handle, const moe_shape* shape,
                                         const moe_layout* layout, int32_t routing_format,
                                         const void* grad_perm_tokens, const float* grad_perm_probs,
                                         void* grad_x, float* grad_probs, void* stream);

/* ------------------------------------------------------------ grouped MLP */

/* Device workspace bytes of moe_grouped_mlp: the intermediate activation
 * [cap][I] in the FC2 input format, plus its scales, plus (bf16 path) a tile
 * claim counter and one completion counter per token tile, which each call
 * zeroes itself.  Calls that share a workspace must not overlap on the GPU. */
MOE_API moe_status moe_grouped_mlp_workspace_size(const moe_shape* shape, const moe_layout* layout,
                                          int32_t w_dtype, size_t* bytes_out);

/* NVFP4 global scales ([MEGAMOE]: weight_scale_2, input_scale; alpha derives
 * from both).  All device pointers. */
typedef struct moe_nvfp4_globals {
  const float* fc1_input_scale; /* [1] global scale of the dispatched rows */
  const float* fc2_input_scale; /* [1] global scale the intermediate is encoded with */
  const float* w13_scale_2;     /* [E] per-expert global scale of w3_w1 */
  const float* w2_scale_2;      /* [E] per-expert global scale of w2 */
} moe_nvfp4_globals;

/* Grouped SwiGLU expert MLP ([REUSE-BUF], Summary: fused grouped MLP writes FC2
 * into a caller buffer).  For every expert e and every row r of its padded
 * segment [offsets[e], offsets[e+1]) below the capacity:
 *   up   = Y[r] . w13[e][0:I]^T,   gate = Y[r] . w13[e][I:2I]^T   (fp32 accumulate)
 *   act  = silu(gate) * up, stored in the FC2 input format (bf16, FP8 with
 *          1x128 fp32 scales, or NVFP4 with the fc2 input global scale)
 *   out_fc2[r] = bf16( act . w2[e]^T )
 * (w3_w1 order: rows 0..I-1 are w3 = up, rows I..2I-1 are w1 = gate.)  Pad rows
 * hold zero input and so produce zero output.  Rows at or beyond
 * min(offsets[E], cap) are not touched.
 * w_dtype: MOE_DTYPE_BF16 (perm_tokens bf16 [cap][H]; w13 bf16 [E][2I][H]; w2
 *   bf16 [E][H][I]);
 *   MOE_DTYPE_FP8_E4M3_B128 (perm_tokens codes [cap][H] + perm_scales fp32
 *   [cap][H/128]; w13 codes [E][2I][H] + w13_scales fp32 [E][2I/128][H/128]; w2
 *   codes [E][H][I] + w2_scales fp32 [E][H/128][I/128]);
 *   MOE_DTYPE_NVFP4 (perm_tokens packed [cap][H/2] + perm_scales E4M3 [cap][H/16];
 *   w13 packed [E][2I][H/2] + E4M3 [E][2I][H/16]; w2 packed [E][H][I/2] + E4M3
 *   [E][H][I/16]; globals required).
 * Shapes: H and I multiples of 128 (MOE_ERR_INVALID_ARG otherwise); NVFP4 also
 * needs H and I multiples of 256 (MOE_ERR_UNSUPPORTED otherwise).
 * workspace: device, >= moe_grouped_mlp_workspace_size bytes, 256-byte aligned.
 * out_fc2: device bf16 [cap][H]. */
MOE_API moe_status moe_grouped_mlp(const moe_handle_dev* handle, const moe_shape* shape, const moe_layout* layout,
                           int32_t w_dtype, const void* perm_tokens, const void* perm_scales,
                           const void* w13, const void* w13_scales, const void* w2,
                           const void* w2_scales, const moe_nvfp4_globals* globals, void* workspace,
                           size_t workspace_bytes, void* out_fc2, void* stream);

/* moe_grouped_mlp with two extensions.
 * (1) FC2 rows written in a combine format ([MEGAMOE], commit list: "fp8
 * combine may use the bulk fc2 store"): out_format MOE_COMBINE_BF16 writes bf16
 * as moe_grouped_mlp does (out_fc2_scales ignored); MOE_COMBINE_MXFP8 /
 * MOE_COMBINE_MXFP4 make FC2's epilogue encode each row's fp32 sums into codes
 * at out_fc2 and E8M0 scales at out_fc2_scales (device [cap][H/32] bytes,
 * 4-byte aligned), layouts as documented with MOE_COMBINE_*.  The MX formats
 * are written by the FP8 path (w_dtype MOE_DTYPE_FP8_E4M3_B128); other w_dtype
 * values return MOE_ERR_UNSUPPORTED with them (write bf16 and convert with
 * moe_quantize_mx_rows).
 * (2) Probabilities applied inside the MLP ([ALLGATHER], Testing: the
 * dispatched probabilities reach the experts and their gradients flow back
 * through the dispatch): fc2_row_probs, when not NULL, is device fp32 [cap]
 * (4-byte aligned) indexed by permuted row -- the perm_probs that
 * moe_dispatch_permute wrote -- and FC2's epilogue multiplies every row r by
 * fc2_row_probs[r] in fp32 before the row is rounded to its output format:
 *   out_fc2[r] = fmt( fc2_row_probs[r] * (act . w2[e]^T) ).
 * The layer is then completed by a combine without weights
 * (moe_combine_unpermute with perm_probs NULL).  Every w_dtype and out_format
 * supports it.  NULL gives moe_grouped_mlp's rows. */
MOE_API moe_status moe_grouped_mlp_ex(const moe_handle_dev* handle, const moe_shape* shape,
                                      const moe_layout* layout, int32_t w_dtype, const void* perm_tokens,
                                      const void* perm_scales, const void* w13, const void* w13_scales,
                                      const void* w2, const void* w2_scales, const moe_nvfp4_globals* globals,
                                      void* workspace, size_t workspace_bytes, int32_t out_format, void* out_fc2,
                                      void* out_fc2_scales, const float* fc2_row_probs, void* stream);

/* Number of kernels one moe_grouped_mlp call with these arguments launches
 * (host only, no device access): 1 where FC1 and FC2 run in one persistent
 * kernel (bf16 on single SMs), 2 where they are separate launches, 0 for a
 * zero capacity.  The bf16 path also issues one small memset of its
 * workspace counters.  Errors: MOE_ERR_INVALID_ARG for a bad shape, layout or
 * dtype. */
MOE_API moe_status moe_grouped_mlp_kernel_count(const moe_shape* shape, const moe_layout* layout, int32_t w_dtype,
                                                int32_t* count_out);

/* Profiling hook: the next moe_grouped_mlp call made by this host thread
 * records the three given CUDA events (cudaEvent_t passed as void*) on its
 * stream -- before FC1, between FC1 and FC2, and after FC2 -- and then forgets
 * them.  Where one kernel runs both GEMMs (moe_grouped_mlp_kernel_count 1),
 * the between and after events are both recorded after it.  Pass NULLs to
 * cancel.  Under stream capture the records become event-record nodes of the
 * graph (cudaEventRecordExternal), so every replay records them again.  Used to time the two GEMM kernels separately
 * inside a step (TensorRT-LLM PR #16190 "Update CuTeDSL MegaMoE kernels",
 * commit list: the microbench reports kernel-level times). */
MOE_API moe_status moe_profile_next_grouped_mlp(void* ev_before_fc1, void* ev_after_fc1, void* ev_after_fc2);

/* Testing hook for the failure path of the fused grouped MLP's bounded waits:
 * the next moe_grouped_mlp call made by this host thread that runs FC1 and FC2
 * in one kernel (moe_grouped_mlp_kernel_count 1) lets the FC1 tiles of token
 * tile `token_tile` (tiles of up to 128 rows, numbered over all experts in
 * order) withhold their completion publication, so the FC2 tiles that read
 * those rows give up after about 2 s: MOE_DEV_ERR_TIMEOUT is set in
 * handle->status and the kernel returns; no kernel traps and the context stays
 * usable.  That call's outputs are not valid.  -1 cancels.  Other paths clear
 * the setting without using it.  Errors: MOE_ERR_INVALID_ARG for token_tile <
 * -1.  Not for production use. */
MOE_API moe_status moe_debug_next_grouped_mlp_silent_token_tile(int64_t token_tile);

/* Testing hook for the failure path of the bounded inter-CTA waits: runs
 * moe_preprocess with tile `silent_tile` (>= 0) withholding its lookback
 * publication, so every later tile's bounded wait runs out (after about 2 s),
 * MOE_DEV_ERR_TIMEOUT is set in handle->status and the kernel returns; no
 * kernel traps and the context stays usable.  The handle's other outputs of
 * that call are not valid.  Not for production use. */
MOE_API moe_status moe_debug_preprocess_silent_tile(const moe_routing* routing, const moe_shape* shape,
                                                    const moe_layout* layout, const moe_handle_dev* handle,
                                                    void* workspace, size_t workspace_bytes, int64_t silent_tile,
                                                    void* stream);

/* ------------------------------------------------- weight / row quantizers */

/* bf16 [G][N][Kd] -> E4M3 codes [G][N][Kd] + fp32 scales [G][N/128][Kd/128],
 * one scale per 128x128 block: scale = amax/448 (1 for an all-zero block),
 * code = E4M3(w / scale), nearest even, saturating.  N, Kd multiples of 128.
 * A one-time weight preparation step, not part of the per-layer path. */
MOE_API moe_status moe_quantize_fp8_blocks(const void* w, int64_t G, int64_t N, int64_t Kd, void* codes,
                                   float* scales, void* stream);

/* bf16 [R][Kd] -> NVFP4 packed [R][Kd/2] + E4M3 scale codes [R][Kd/16] with
 * the fp32 global scale *global (device pointer):
 * block scale = E4M3(amax/(6*global)), code = E2M1(x/(block*global)). */
MOE_API moe_status moe_quantize_nvfp4_rows(const void* x, int64_t R, int64_t Kd, const float* global,
                                   void* packed, void* scales, void* stream);

/* ------------------------------------------------------------ buffer ring */

/* Host-side ring of N caller-owned output slots ([REUSE-BUF], Summary and
 * Known limitations): the producer acquires the next slot in round-robin
 * order; the final consumer releases it on its stream.  With events enabled,
 * acquire makes `stream` wait (device-side, no host sync) on the event recorded
 * by the slot's last release.  Acquiring a slot that is still held returns
 * MOE_ERR_RING_EARLY_REUSE; releasing a slot that is not held returns
 * MOE_ERR_RING_DOUBLE_RELEASE; neither changes the ring.  The ring only tracks
 * slot indices: the caller maps a slot index to its own buffers. */
typedef struct moe_ring moe_ring;
MOE_API moe_status moe_ring_create(int32_t n_slots, int32_t use_events, moe_ring** ring_out);
MOE_API moe_status moe_ring_acquire(moe_ring* ring, void* stream, int32_t* slot_out);
MOE_API moe_status moe_ring_release(moe_ring* ring, int32_t slot, void* stream);
MOE_API moe_status moe_ring_destroy(moe_ring* ring);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
