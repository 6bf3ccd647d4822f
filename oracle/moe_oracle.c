/*
 * moe_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, literal CPU restatement of the single-GPU core of an MoE layer:
 * routing map -> per-expert counts -> padded exclusive scan with a capacity
 * bound and an overflow flag -> stable permute of token rows and probabilities
 * -> grouped SwiGLU expert MLP (FC1, activation, FC2) -> combine (unpermute and
 * top-k probability-weighted sum).  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library.  It shares no
 * code, header, table or helper with the CUDA library, and includes nothing
 * from it.
 *
 * Floating point is evaluated in double (fp64) unless a step's output format
 * is itself part of the method (bf16 outputs, FP8 / NVFP4 codes); those
 * roundings are written out below from the number formats' definitions.
 *
 * Sources, by page title and section:
 *  [REUSE-BUF]  Megatron-LM PR #6800 "Reuse caller-owned HybridEP dispatch and
 *               expert output buffers" -- Summary (dispatch writes permuted tokens
 *               into a caller buffer; grouped MLP writes FC2 into a caller buffer;
 *               combine performs the final read).
 *  [ALLGATHER]  DeepEP PR #716 "perf: reuse HybridEP routing allgather buffer" --
 *               Memory impact (sparse Boolean tokens x experts bytes, dense int16
 *               tokens x topk ids); Testing / Full HybridEP reference validation
 *               (padding multiple 32, dispatch with permutation, combine with
 *               unpermutation, with and without probabilities).
 *  [SYNC-FREE]  NeMo Automodel PR #3931 "perf(moe): sync-free HybridEP dispatch
 *               (capacity mode, equal token counts)" -- What does this PR do?
 *               (counts stay on the device, capacity ceil(rows x factor) 4-aligned,
 *               overflow flag in the handle); Validation (capacity >= actual: flag
 *               0 and identical rows; capacity = actual/2: flag set, silent
 *               truncation; combine round trip).
 *  [MEGAMOE]    TensorRT-LLM PR #16190 "Update CuTeDSL MegaMoE kernels" -- commit
 *               list: NVFP4 expert tensors w3_w1_weight / w2_weight with block
 *               scales, weight_scale_2 and input_scale (alphas derive from both);
 *               TopkReduce combine.
 *
 * Where the pages leave a step open the reading taken is stated beside the code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* Device-status bits the oracle reports for malformed routing (the CUDA library
 * uses the same numeric values; the values are part of the public contract). */
#define ORACLE_ERR_BAD_EXPERT 1      /* dense id outside [-1, E) */
#define ORACLE_ERR_TOO_MANY_ROUTES 2 /* sparse row with more than K set entries */

/* ------------------------------------------------------------------------- */
/* Number formats                                                              */
/* ------------------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32: 1 sign, 8 exponent, 7 fraction bits. */
ORACLE_API double moe_oracle_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static uint16_t f32_bits_hi(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* Round a double to the nearest bf16, ties to even, straight from the format:
 * a finite bf16 is N * 2^(E-7) with N an 8-bit significand (N in [128,256) for
 * normals, exponents down to -126, and a fixed quantum 2^-133 below that). */
ORACLE_API uint16_t moe_oracle_f64_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  int neg = signbit(v) ? 1 : 0;
  double a = fabs(v);
  if (a == 0.0) return neg ? 0x8000 : 0x0000;
  if (isinf(a)) return neg ? 0xFF80 : 0x7F80;
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): the leading bit has weight 2^(e-1) */
  int lead = e - 1;
  if (lead < -126) lead = -126; /* subnormal range keeps the quantum of 2^-126 normals */
  double quantum = ldexp(1.0, lead - 7);
  double n = nearbyint(a / quantum); /* default rounding mode: to nearest, ties to even */
  double r = n * quantum;
  if (r >= ldexp(1.0, 128)) return neg ? 0xFF80 : 0x7F80;
  uint16_t h = f32_bits_hi((float)r); /* r is exactly representable in bf16, hence in fp32 */
  return neg ? (uint16_t)(h | 0x8000) : h;
}

/* Round a double to the nearest binary32, ties to even (the C conversion does
 * exactly this under the default rounding mode). */
static float f64_to_f32(double v) { return (float)v; }

/* OCP FP8 E4M3 (the "fn" variant): 1 sign, 4 exponent (bias 7), 3 fraction
 * bits; exponent field 0 is subnormal (m/8 * 2^-6); code 0x7F/0xFF is NaN; no
 * infinities; largest finite magnitude 448 (code 0x7E). */
ORACLE_API double moe_oracle_e4m3_to_f64(uint8_t c) {
  int neg = (c & 0x80) != 0;
  int ex = (c >> 3) & 0xF;
  int man = c & 0x7;
  double v;
  if (ex == 0xF && man == 0x7) return NAN;
  if (ex == 0)
    v = ldexp((double)man / 8.0, -6);
  else
    v = ldexp(1.0 + (double)man / 8.0, ex - 7);
  return neg ? -v : v;
}

/* Decoded values of every E4M3 code and every E2M1 code, filled once when the
 * library loads from the decoders above and below (a cache of their results:
 * the searches and operand reads use the same values they would compute). */
ORACLE_API double moe_oracle_e2m1_to_f64(uint8_t c);
static double g_e4m3_value[256];
static double g_e2m1_value[16];
__attribute__((constructor)) static void oracle_fill_code_tables(void) {
  for (int c = 0; c < 256; c++) g_e4m3_value[c] = moe_oracle_e4m3_to_f64((uint8_t)c);
  for (int c = 0; c < 16; c++) g_e2m1_value[c] = moe_oracle_e2m1_to_f64((uint8_t)c);
}

/* Encode a binary32 into E4M3 by rounding to the nearest finite code (ties to the
 * code with an even fraction field, i.e. the even code), saturating magnitudes
 * beyond 448 to 448.  The search runs over the code table, so no library
 * conversion is involved. */
ORACLE_API uint8_t moe_oracle_f32_to_e4m3(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  /* largest code c in [0, 0x7E] whose value is <= a (values increase with the code) */
  int lo = 0, hi = 0x7E;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (g_e4m3_value[mid] <= a)
      lo = mid;
    else
      hi = mid - 1;
  }
  int c = lo;
  double below = g_e4m3_value[c];
  double above = g_e4m3_value[c + 1];
  double d_lo = a - below, d_hi = above - a;
  int pick;
  if (d_lo < d_hi)
    pick = c;
  else if (d_hi < d_lo)
    pick = c + 1;
  else
    pick = (c % 2 == 0) ? c : c + 1;
  return (uint8_t)(sign | pick);
}

/* FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 fraction bit.  Magnitudes of codes
 * 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6.  No NaN or infinity. */
ORACLE_API double moe_oracle_e2m1_to_f64(uint8_t c) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double v = mag[c & 7];
  return (c & 8) ? -v : v;
}

/* Nearest E2M1 code, ties to the even code, saturating at 6. */
ORACLE_API uint8_t moe_oracle_f32_to_e2m1(float v) {
  uint8_t sign = signbit(v) ? 8 : 0;
  double a = fabs((double)v);
  if (a >= 6.0) return (uint8_t)(sign | 7);
  int c = 0;
  while (c < 7 && moe_oracle_e2m1_to_f64((uint8_t)(c + 1)) <= a) c++;
  double below = moe_oracle_e2m1_to_f64((uint8_t)c);
  double above = moe_oracle_e2m1_to_f64((uint8_t)(c + 1));
  double d_lo = a - below, d_hi = above - a;
  int pick;
  if (d_lo < d_hi)
    pick = c;
  else if (d_hi < d_lo)
    pick = c + 1;
  else
    pick = (c % 2 == 0) ? c : c + 1;
  return (uint8_t)(sign | pick);
}

/* ------------------------------------------------------------------------- */
/* Capacity                                                                    */
/* ------------------------------------------------------------------------- */

/* [SYNC-FREE], What does this PR do?: later dispatches are sized to
 * ceil(rows x factor), aligned to 4 tokens.  Reading: ceil is taken of the
 * product computed in double, then rounded up to the next multiple of `align`. */
ORACLE_API int64_t moe_oracle_capacity(int64_t rows, double factor, int64_t align) {
  double prod = (double)rows * factor;
  int64_t c = (int64_t)ceil(prod);
  if (align > 1) c = ((c + align - 1) / align) * align;
  return c;
}

/* ------------------------------------------------------------------------- */
/* Metadata preprocessing: counts, padded offsets, stable row map              */
/* ------------------------------------------------------------------------- */

/* The route table: route[t*K + k] = expert of slot k of token t, or -1 when
 * that slot carries no route.
 * Dense int16 ids ([ALLGATHER], Memory impact: tokens x topk ids): slot k is
 * topk_idx[t][k]; -1 means "no route"; any other id outside [0, E) is reported
 * and treated as no route.
 * Sparse Boolean map ([ALLGATHER], Memory impact: tokens x experts bytes):
 * slot k is the k-th set entry of row t in ascending expert order (reading: the
 * pages fix no slot order for a Boolean map); entries past the K-th set one are
 * reported and ignored.  Returns the status bits. */
static int build_routes(int format, const void* map, int64_t T, int64_t E, int64_t K,
                        int32_t* route) {
  int status = 0;
  for (int64_t t = 0; t < T; t++) {
    if (format == 0) {
      const int16_t* idx = (const int16_t*)map;
      for (int64_t k = 0; k < K; k++) {
        int v = idx[t * K + k];
        if (v != -1 && (v < 0 || v >= E)) {
          status |= ORACLE_ERR_BAD_EXPERT;
          v = -1;
        }
        route[t * K + k] = v;
      }
    } else {
      const uint8_t* m = (const uint8_t*)map;
      int64_t k = 0;
      for (int64_t e = 0; e < E; e++) {
        if (m[t * E + e] == 0) continue;
        if (k < K)
          route[t * K + k++] = (int32_t)e;
        else
          status |= ORACLE_ERR_TOO_MANY_ROUTES;
      }
      for (; k < K; k++) route[t * K + k] = -1;
    }
  }
  return status;
}

/* Outputs, all caller-allocated:
 *   counts[E]       tokens routed to each expert (the real count, never clamped)
 *   offsets[E+1]    offsets[e] = sum over e' < e of ceil(counts[e'] / m) * m
 *   row_of[T*K]     destination row of route (t,k), or -1 (no route / dropped)
 *   token_of[cap]   source token of each row < min(offsets[E], cap); -1 for pad rows
 *   slot_of[cap]    route slot k of each such row; -1 for pad rows
 *   total_rows[1]   offsets[E], unclamped
 *   overflow[1]     1 when offsets[E] > cap, else 0
 * Rows at or beyond min(offsets[E], cap) of token_of / slot_of are not written.
 * Returns the status bits (0 when the routing is well formed).
 *
 * [ALLGATHER], Testing: "padding multiple 32" and "dispatch with permutation";
 * [SYNC-FREE], What does this PR do? / Validation: real counts stay on the
 * device, capacity bounds the output rows, an overflow flag replaces the sync,
 * truncation is silent.  Reading: the permuted order is a stable sort of the
 * routes by expert, then token, then slot; routes whose destination reaches the
 * capacity are the ones dropped (the tail of that order). */
ORACLE_API int moe_oracle_preprocess(int format, const void* map, int64_t T, int64_t E, int64_t K,
                                     int64_t m, int64_t cap, int32_t* counts, int32_t* offsets,
                                     int32_t* row_of, int32_t* token_of, int32_t* slot_of,
                                     int32_t* total_rows, int32_t* overflow) {
  int32_t* route = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T * K + 1));
  int status = build_routes(format, map, T, E, K, route);

  /* 1. histogram: a direct count over every (t, k) */
  for (int64_t e = 0; e < E; e++) counts[e] = 0;
  for (int64_t i = 0; i < T * K; i++)
    if (route[i] >= 0) counts[route[i]] += 1;

  /* 2. exclusive scan of the counts, each padded up to a multiple of m */
  int64_t run = 0;
  for (int64_t e = 0; e < E; e++) {
    offsets[e] = (int32_t)run;
    int64_t padded = ((counts[e] + m - 1) / m) * m;
    run += padded;
  }
  offsets[E] = (int32_t)run;
  total_rows[0] = (int32_t)run;
  overflow[0] = (run > cap) ? 1 : 0;

  /* 3. row map: for each expert in order, visit routes in (token, slot) order */
  for (int64_t i = 0; i < T * K; i++) row_of[i] = -1;
  int64_t valid_end = run < cap ? run : cap;
  for (int64_t r = 0; r < valid_end; r++) {
    token_of[r] = -1; /* pad until a route claims the row */
    slot_of[r] = -1;
  }
  for (int64_t e = 0; e < E; e++) {
    int64_t n_e = 0;
    for (int64_t t = 0; t < T; t++)
      for (int64_t k = 0; k < K; k++) {
        if (route[t * K + k] != e) continue;
        int64_t dest = offsets[e] + n_e;
        n_e++;
        if (dest < cap) {
          row_of[t * K + k] = (int32_t)dest;
          token_of[dest] = (int32_t)t;
          slot_of[dest] = (int32_t)k;
        }
      }
  }
  free(route);
  return status;
}

/* Routing probability of route (t, k) whose expert is e: dense probs are
 * [T][K]; sparse probs are [T][E] and the route's probability sits at its
 * expert's column. */
static double prob_of_route(int format, const float* probs, int64_t t, int64_t k, int64_t e,
                            int64_t E, int64_t K) {
  if (format == 0) return (double)probs[t * K + k];
  return (double)probs[t * E + e];
}

/* ------------------------------------------------------------------------- */
/* dispatch_with_permute                                                       */
/* ------------------------------------------------------------------------- */

/* [REUSE-BUF], Summary: dispatch writes the permuted tokens into a buffer the
 * caller owns.  Each routed row is copied byte for byte:
 *   Y[row_of[t][k]] = X[t]            (row_bytes per row; any element type)
 *   Yp[row_of[t][k]] = p(t, k)        (when probs and out_probs are given)
 * Pad rows [offsets[e] + counts[e], offsets[e+1]) below the capacity are zero
 * (zero bytes, probability 0).  Rows at or beyond min(offsets[E], cap) are not
 * written.  Reading: pads are zero because the pages only state the padding
 * multiple. */
ORACLE_API void moe_oracle_dispatch(int format, const void* map, const float* probs, int64_t T,
                                    int64_t E, int64_t K, int64_t cap, const int32_t* counts,
                                    const int32_t* offsets, const int32_t* row_of,
                                    const uint8_t* x, int64_t row_bytes, uint8_t* y,
                                    float* out_probs) {
  int32_t* route = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T * K + 1));
  build_routes(format, map, T, E, K, route);
  for (int64_t t = 0; t < T; t++)
    for (int64_t k = 0; k < K; k++) {
      int32_t dest = row_of[t * K + k];
      if (dest < 0) continue;
      memcpy(y + (int64_t)dest * row_bytes, x + t * row_bytes, (size_t)row_bytes);
      if (probs && out_probs)
        out_probs[dest] = (float)prob_of_route(format, probs, t, k, route[t * K + k], E, K);
    }
  free(route);
  for (int64_t e = 0; e < E; e++)
    for (int64_t r = (int64_t)offsets[e] + counts[e]; r < offsets[e + 1]; r++) {
      if (r >= cap) break;
      memset(y + r * row_bytes, 0, (size_t)row_bytes);
      if (out_probs) out_probs[r] = 0.0f;
    }
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 with 1x128 (activations) / 128x128 (weights) fp32 block scales      */
/* ------------------------------------------------------------------------- */

/* Quantize one block of n fp32 values with a shared fp32 scale.
 * Reading (the pages fix no rule): scale = amax / 448 in fp32; an all-zero block
 * takes scale 1; each code is E4M3(v / scale) with the quotient in fp32. */
static void quant_block_e4m3(const float* v, int64_t n, int64_t stride, uint8_t* q,
                             int64_t qstride, float* scale) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; i++) {
    float a = fabsf(v[i * stride]);
    if (a > amax) amax = a;
  }
  float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
  for (int64_t i = 0; i < n; i++) q[i * qstride] = moe_oracle_f32_to_e4m3(v[i * stride] / s);
  *scale = s;
}

/* Activations: x bf16 [T][H] -> codes [T][H], scales [T][H/128]. */
ORACLE_API void moe_oracle_quantize_fp8_rows(const uint16_t* x, int64_t T, int64_t H, uint8_t* q,
                                             float* scales) {
  float* row = (float*)malloc(sizeof(float) * (size_t)H);
  for (int64_t t = 0; t < T; t++) {
    for (int64_t h = 0; h < H; h++) row[h] = (float)moe_oracle_bf16_to_f64(x[t * H + h]);
    for (int64_t b = 0; b < H / 128; b++)
      quant_block_e4m3(row + b * 128, 128, 1, q + t * H + b * 128, 1, &scales[t * (H / 128) + b]);
  }
  free(row);
}

/* Weights: w bf16 [G][N][Kd] -> codes [G][N][Kd], scales [G][N/128][Kd/128]
 * (one fp32 scale per 128x128 block). */
ORACLE_API void moe_oracle_quantize_fp8_weight(const uint16_t* w, int64_t G, int64_t N, int64_t Kd,
                                               uint8_t* q, float* scales) {
  /* every 128x128 block is quantized on its own, so blocks run in parallel */
  const int64_t nblk = G * (N / 128) * (Kd / 128);
#pragma omp parallel
  {
    float* blk = (float*)malloc(sizeof(float) * 128 * 128);
    uint8_t* qb = (uint8_t*)malloc(128 * 128);
#pragma omp for schedule(static)
    for (int64_t id = 0; id < nblk; id++) {
      const int64_t g = id / ((N / 128) * (Kd / 128));
      const int64_t nb = (id / (Kd / 128)) % (N / 128);
      const int64_t kb = id % (Kd / 128);
      for (int64_t i = 0; i < 128; i++)
        for (int64_t j = 0; j < 128; j++)
          blk[i * 128 + j] = (float)moe_oracle_bf16_to_f64(w[(g * N + nb * 128 + i) * Kd + kb * 128 + j]);
      float s;
      quant_block_e4m3(blk, 128 * 128, 1, qb, 1, &s);
      for (int64_t i = 0; i < 128; i++)
        for (int64_t j = 0; j < 128; j++)
          q[(g * N + nb * 128 + i) * Kd + kb * 128 + j] = qb[i * 128 + j];
      scales[(g * (N / 128) + nb) * (Kd / 128) + kb] = s;
    }
    free(blk);
    free(qb);
  }
}

/* ------------------------------------------------------------------------- */
/* NVFP4: E2M1 values, one E4M3 scale per 16 consecutive K elements, and one   */
/* fp32 global scale per tensor                                               */
/* ------------------------------------------------------------------------- */

/* [MEGAMOE], commit list: w3_w1_weight / w2_weight carry block scales plus a
 * second-level weight_scale_2, activations an input_scale, and the epilogue
 * alpha derives from both.  Reading: value = e2m1 * e4m3(block) * global; the
 * block scale is E4M3(amax / (6 * global)) with the quotient in fp32, and each
 * code is E2M1(v / (block * global)) with the product and quotient in fp32 (a
 * zero block scale gives code 0).  Two codes per byte, the even element in the
 * low nibble. */
static void quant_block_nvfp4(const float* v, int64_t n, float global, uint8_t* codes,
                              uint8_t* scale_code) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; i++) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  uint8_t sc = moe_oracle_f32_to_e4m3(amax / (6.0f * global));
  float sdec = (float)moe_oracle_e4m3_to_f64(sc);
  float denom = sdec * global;
  for (int64_t i = 0; i < n; i++) codes[i] = (denom == 0.0f) ? 0 : moe_oracle_f32_to_e2m1(v[i] / denom);
  *scale_code = sc;
}

/* Rows of fp32 values [R][Kd] -> packed codes [R][Kd/2], scale codes [R][Kd/16]. */
static void quant_rows_nvfp4_f32(const float* v, int64_t R, int64_t Kd, float global,
                                 uint8_t* packed, uint8_t* scales) {
  uint8_t codes[16];
  for (int64_t r = 0; r < R; r++)
    for (int64_t b = 0; b < Kd / 16; b++) {
      quant_block_nvfp4(v + r * Kd + b * 16, 16, global, codes, &scales[r * (Kd / 16) + b]);
      for (int64_t i = 0; i < 8; i++)
        packed[r * (Kd / 2) + b * 8 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
    }
}

/* bf16 rows [R][Kd] -> NVFP4 with the given global scale. */
ORACLE_API void moe_oracle_quantize_nvfp4_rows(const uint16_t* x, int64_t R, int64_t Kd,
                                               float global, uint8_t* packed, uint8_t* scales) {
  /* rows are independent, so they run in parallel */
#pragma omp parallel
  {
    float* row = (float*)malloc(sizeof(float) * (size_t)Kd);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < R; r++) {
      for (int64_t i = 0; i < Kd; i++) row[i] = (float)moe_oracle_bf16_to_f64(x[r * Kd + i]);
      quant_rows_nvfp4_f32(row, 1, Kd, global, packed + r * (Kd / 2), scales + r * (Kd / 16));
    }
    free(row);
  }
}

static double nvfp4_value(const uint8_t* packed, const uint8_t* scales, int64_t Kd, int64_t r,
                          int64_t i, double global) {
  uint8_t byte = packed[r * (Kd / 2) + i / 2];
  uint8_t code = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);
  return g_e2m1_value[code] * g_e4m3_value[scales[r * (Kd / 16) + i / 16]] * global;
}

/* ------------------------------------------------------------------------- */
/* Grouped SwiGLU expert MLP                                                   */
/* ------------------------------------------------------------------------- */

/* Expert owning permuted row r: the e with offsets[e] <= r < offsets[e+1]. */
static int64_t expert_of_row(const int32_t* offsets, int64_t E, int64_t r) {
  for (int64_t e = 0; e < E; e++)
    if (offsets[e] <= r && r < offsets[e + 1]) return e;
  return -1;
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* Operand access by format.  fmt 0: bf16; fmt 1: FP8 E4M3 with 1x128 scales for
 * activations and 128x128 scales for weights; fmt 2: NVFP4. */
typedef struct {
  int fmt;
  const void* data;   /* bf16 / e4m3 codes / packed e2m1 */
  const void* scales; /* fp32 (FP8) or e4m3 codes (NVFP4) */
  double global;      /* NVFP4 second-level scale */
} operand;

/* Element (r, i) of an activation matrix with row length Kd. */
static double act_value(const operand* a, int64_t Kd, int64_t r, int64_t i) {
  if (a->fmt == 0) return moe_oracle_bf16_to_f64(((const uint16_t*)a->data)[r * Kd + i]);
  if (a->fmt == 1)
    return g_e4m3_value[((const uint8_t*)a->data)[r * Kd + i]] *
           (double)((const float*)a->scales)[r * (Kd / 128) + i / 128];
  return nvfp4_value((const uint8_t*)a->data, (const uint8_t*)a->scales, Kd, r, i, a->global);
}

/* Element (n, i) of expert e's weight [E][N][Kd]; globals[e] is that expert's
 * NVFP4 weight_scale_2. */
static double weight_value(const operand* w, const float* globals, int64_t N, int64_t Kd, int64_t e,
                           int64_t n, int64_t i) {
  int64_t row = e * N + n;
  if (w->fmt == 0) return moe_oracle_bf16_to_f64(((const uint16_t*)w->data)[row * Kd + i]);
  if (w->fmt == 1)
    return g_e4m3_value[((const uint8_t*)w->data)[row * Kd + i]] *
           (double)((const float*)w->scales)[(e * (N / 128) + n / 128) * (Kd / 128) + i / 128];
  return nvfp4_value((const uint8_t*)w->data, (const uint8_t*)w->scales, Kd, row, i,
                     (double)globals[e]);
}

/* FFN of one permuted row r of expert e.
 * [REUSE-BUF], Summary: grouped MLP (FC1, activation, FC2) writes FC2 into the
 * caller's buffer.  [MEGAMOE]: FC1's weight is w3_w1.  Reading: rows 0..I-1 of
 * w3_w1 are w3 (up), rows I..2I-1 are w1 (gate); act = silu(gate) * up.
 * The intermediate is stored in the format FC2 consumes (bf16, or FP8 / NVFP4
 * codes), so that rounding is part of the method: the product is rounded to
 * fp32 (the kernel's accumulator precision) and then encoded.  FC2 accumulates
 * in double and rounds to bf16. */
static void ffn_row(const operand* yin, int64_t r, int64_t e, int64_t H, int64_t I,
                    const operand* w13, const float* w13_global, const operand* w2,
                    const float* w2_global, double fc2_in_global, double* out_acc,
                    double* act_dbg) {
  double* act = (double*)malloc(sizeof(double) * (size_t)I);
  float* actf = (float*)malloc(sizeof(float) * (size_t)I);
  for (int64_t j = 0; j < I; j++) {
    double up = 0.0, gate = 0.0;
    for (int64_t h = 0; h < H; h++) {
      double xv = act_value(yin, H, r, h);
      up += xv * weight_value(w13, w13_global, 2 * I, H, e, j, h);
      gate += xv * weight_value(w13, w13_global, 2 * I, H, e, I + j, h);
    }
    act[j] = silu(gate) * up;
  }
  /* the stored intermediate, decoded back to double */
  if (w2->fmt == 0) {
    for (int64_t j = 0; j < I; j++) act[j] = moe_oracle_bf16_to_f64(moe_oracle_f64_to_bf16(act[j]));
  } else if (w2->fmt == 1) {
    for (int64_t j = 0; j < I; j++) actf[j] = f64_to_f32(act[j]);
    uint8_t q[128];
    for (int64_t b = 0; b < I / 128; b++) {
      float s;
      quant_block_e4m3(actf + b * 128, 128, 1, q, 1, &s);
      for (int64_t i = 0; i < 128; i++) act[b * 128 + i] = moe_oracle_e4m3_to_f64(q[i]) * (double)s;
    }
  } else {
    for (int64_t j = 0; j < I; j++) actf[j] = f64_to_f32(act[j]);
    uint8_t codes[16], sc;
    for (int64_t b = 0; b < I / 16; b++) {
      quant_block_nvfp4(actf + b * 16, 16, (float)fc2_in_global, codes, &sc);
      for (int64_t i = 0; i < 16; i++)
        act[b * 16 + i] =
            moe_oracle_e2m1_to_f64(codes[i]) * moe_oracle_e4m3_to_f64(sc) * fc2_in_global;
    }
  }
  if (act_dbg)
    for (int64_t j = 0; j < I; j++) act_dbg[j] = act[j];
  for (int64_t n = 0; n < H; n++) {
    double acc = 0.0;
    for (int64_t j = 0; j < I; j++) acc += act[j] * weight_value(w2, w2_global, H, I, e, n, j);
    out_acc[n] = acc;
  }
  free(act);
  free(actf);
}

/* Grouped MLP over a list of permuted rows.  Each listed row must lie in some
 * expert's padded segment below the capacity.  out: [nrows][H] bf16;
 * act_out (optional): [nrows][I] decoded intermediate in double.
 * fmt: 0 bf16, 1 FP8 (y_scales fp32 [cap][H/128]; w scales fp32 per 128x128),
 * 2 NVFP4 (y packed [cap][H/2] + e4m3 scales [cap][H/16] with global
 * fc1_in_global; weights packed with e4m3 scales and per-expert globals;
 * the intermediate uses fc2_in_global). */
/* row_probs (optional, [nrows]): probabilities applied inside the MLP -- each
 * FC2 row's sums are multiplied by its probability before they are rounded
 * ([ALLGATHER], Testing: probability gradients flow back through the dispatch,
 * i.e. the experts consume the dispatched probabilities; the combine then sums
 * the rows without weights). */
ORACLE_API int moe_oracle_grouped_mlp_rows(int fmt, const void* y, const void* y_scales,
                                           int64_t H, int64_t I, int64_t E, const int32_t* offsets,
                                           const void* w13, const void* w13_scales,
                                           const float* w13_global, const void* w2,
                                           const void* w2_scales, const float* w2_global,
                                           double fc1_in_global, double fc2_in_global,
                                           const int64_t* rows, int64_t nrows, uint16_t* out,
                                           double* act_out, const float* row_probs) {
  operand yin = {fmt, y, y_scales, fc1_in_global};
  operand ow13 = {fmt, w13, w13_scales, 0.0};
  operand ow2 = {fmt, w2, w2_scales, 0.0};
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t i = 0; i < nrows; i++) {
    int64_t e = expert_of_row(offsets, E, rows[i]);
    if (e < 0) {
      bad = 1;
      continue;
    }
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    ffn_row(&yin, rows[i], e, H, I, &ow13, w13_global, &ow2, w2_global, fc2_in_global, acc,
            act_out ? act_out + i * I : NULL);
    const double pr = row_probs ? (double)row_probs[i] : 1.0;
    for (int64_t n = 0; n < H; n++) out[i * H + n] = moe_oracle_f64_to_bf16(pr * acc[n]);
    free(acc);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* MX combine formats: E4M3 or E2M1 elements with one E8M0 scale per 32        */
/* ------------------------------------------------------------------------- */

/* [MEGAMOE], commit list: the combine reads bf16, fp8 or fp4 expert outputs
 * ("fp8 combine may use the bulk fc2 store"); their scale factors are E8M0
 * bytes and the fp4 vectors E2M1.  Reading (OCP Microscaling Formats (MX)
 * v1.0, the format family with E8M0 scales): blocks of 32 consecutive elements
 * of a row share a scale 2^X stored as the E8M0 code X + 127, with
 * X = floor(log2(amax)) - emax, emax the exponent of the element format's
 * largest normal (8 for E4M3, 2 for E2M1), X clamped to [-127, 127]; an
 * all-zero block takes X = 0.  Each element is x / 2^X rounded to the nearest
 * code, ties to even, saturating at the largest finite magnitude.  The FC2 sums
 * are rounded to fp32 (the kernel's accumulator precision) before encoding.
 * elem: 0 = E4M3 (one code byte per element), 1 = E2M1 (two per byte, the even
 * element in the low nibble). */
ORACLE_API double moe_oracle_e8m0_to_f64(uint8_t c) { return c == 255 ? NAN : ldexp(1.0, (int)c - 127); }

static void quant_block_mx(const float* v, int elem, uint8_t* codes, uint8_t* scale_code) {
  float amax = 0.0f;
  for (int i = 0; i < 32; i++) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  int X = 0;
  if (amax > 0.0f) {
    int e;
    frexp((double)amax, &e); /* amax = f * 2^e, f in [0.5, 1): floor(log2(amax)) = e - 1 */
    X = (e - 1) - (elem == 0 ? 8 : 2);
    if (X < -127) X = -127;
    if (X > 127) X = 127;
  }
  for (int i = 0; i < 32; i++) {
    float q = (float)ldexp((double)v[i], -X); /* exact unless it falls below the fp32 range */
    codes[i] = elem == 0 ? moe_oracle_f32_to_e4m3(q) : moe_oracle_f32_to_e2m1(q);
  }
  *scale_code = (uint8_t)(X + 127);
}

/* fp32 rows [R][H] -> element codes (E4M3 [R][H] or packed E2M1 [R][H/2]) and
 * E8M0 scale codes [R][H/32]. */
ORACLE_API void moe_oracle_quantize_mx_rows(const float* x, int64_t R, int64_t H, int elem, uint8_t* codes,
                                            uint8_t* scales) {
  uint8_t q[32];
  for (int64_t r = 0; r < R; r++)
    for (int64_t b = 0; b < H / 32; b++) {
      quant_block_mx(x + r * H + b * 32, elem, q, &scales[r * (H / 32) + b]);
      for (int i = 0; i < 32; i++) {
        if (elem == 0)
          codes[r * H + b * 32 + i] = q[i];
        else if (i % 2 == 0)
          codes[r * (H / 2) + b * 16 + i / 2] = (uint8_t)(q[i] | (q[i + 1] << 4));
      }
    }
}

static double mx_value(const uint8_t* codes, const uint8_t* scales, int64_t H, int elem, int64_t r, int64_t i) {
  double v;
  if (elem == 0) {
    v = g_e4m3_value[codes[r * H + i]];
  } else {
    uint8_t byte = codes[r * (H / 2) + i / 2];
    v = g_e2m1_value[(i % 2 == 0) ? (byte & 0xF) : (byte >> 4)];
  }
  return v * moe_oracle_e8m0_to_f64(scales[r * (H / 32) + i / 32]);
}

/* The grouped MLP of moe_oracle_grouped_mlp_rows with FC2 rows written in an MX
 * combine format instead of bf16: out_codes [nrows][H] (E4M3) or [nrows][H/2]
 * (E2M1), out_scales [nrows][H/32]. */
ORACLE_API int moe_oracle_grouped_mlp_rows_mx(int fmt, const void* y, const void* y_scales, int64_t H, int64_t I,
                                              int64_t E, const int32_t* offsets, const void* w13,
                                              const void* w13_scales, const float* w13_global, const void* w2,
                                              const void* w2_scales, const float* w2_global, double fc1_in_global,
                                              double fc2_in_global, const int64_t* rows, int64_t nrows, int elem,
                                              uint8_t* out_codes, uint8_t* out_scales, const float* row_probs) {
  operand yin = {fmt, y, y_scales, fc1_in_global};
  operand ow13 = {fmt, w13, w13_scales, 0.0};
  operand ow2 = {fmt, w2, w2_scales, 0.0};
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t i = 0; i < nrows; i++) {
    int64_t e = expert_of_row(offsets, E, rows[i]);
    if (e < 0) {
      bad = 1;
      continue;
    }
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    float* accf = (float*)malloc(sizeof(float) * (size_t)H);
    ffn_row(&yin, rows[i], e, H, I, &ow13, w13_global, &ow2, w2_global, fc2_in_global, acc, NULL);
    const double pr = row_probs ? (double)row_probs[i] : 1.0;
    for (int64_t n = 0; n < H; n++) accf[n] = f64_to_f32(pr * acc[n]);
    moe_oracle_quantize_mx_rows(accf, 1, H, elem, out_codes + i * (elem == 0 ? H : H / 2), out_scales + i * (H / 32));
    free(acc);
    free(accf);
  }
  return bad ? -1 : 0;
}

/* Combine from an MX expert-output buffer: y[t] = bf16( sum over k ascending of
 * w(r) * decoded O[r] ) over the kept routes, as moe_oracle_combine does for
 * bf16 rows. */
ORACLE_API void moe_oracle_combine_mx(const uint8_t* codes, const uint8_t* scales, int64_t H, int elem,
                                      const int32_t* row_of, int64_t T, int64_t K, const float* perm_probs,
                                      uint16_t* y) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; t++)
    for (int64_t h = 0; h < H; h++) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; k++) {
        int32_t r = row_of[t * K + k];
        if (r < 0) continue;
        double w = perm_probs ? (double)perm_probs[r] : 1.0;
        acc += w * mx_value(codes, scales, H, elem, r, h);
      }
      y[t * H + h] = moe_oracle_f64_to_bf16(acc);
    }
}

/* ------------------------------------------------------------------------- */
/* combine with unpermute                                                      */
/* ------------------------------------------------------------------------- */

/* [ALLGATHER], Testing: combine with unpermutation, with and without
 * probabilities; [MEGAMOE]: TopkReduce.  y[t] = bf16( sum over k ascending of
 * w(t,k) * O[row_of[t][k]] ) over the routes that kept a row, where w is the
 * dispatched probability of that row, or 1 when no probabilities are given.
 * Reading: the weighting happens here and only here. */
ORACLE_API void moe_oracle_combine(const uint16_t* o, int64_t H, const int32_t* row_of, int64_t T,
                                   int64_t K, const float* perm_probs, uint16_t* y) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; t++)
    for (int64_t h = 0; h < H; h++) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; k++) {
        int32_t r = row_of[t * K + k];
        if (r < 0) continue;
        double w = perm_probs ? (double)perm_probs[r] : 1.0;
        acc += w * moe_oracle_bf16_to_f64(o[(int64_t)r * H + h]);
      }
      y[t * H + h] = moe_oracle_f64_to_bf16(acc);
    }
}

/* ------------------------------------------------------------------------- */
/* Backward of combine and of dispatch                                         */
/* ------------------------------------------------------------------------- */

/* [ALLGATHER], Testing / Output and gradient regression: hidden-state and
 * probability gradients for the backward of the combine; [SYNC-FREE], What does
 * this PR do?: the combine's backward is a dispatch sized by the same host
 * capacity.  The combine computed y[t] = sum_k w(r) * O[r] over the kept rows
 * r = row_of[t][k], so for an output gradient gy:
 *   gO[r] = bf16( w(r) * gy[t] )            (a dispatch of gy, scaled per row)
 *   gw[r] = sum_h gy[t][h] * O[r][h]        (stored as fp32)
 * with w(r) = perm_probs[r], or 1 when perm_probs is NULL (gw then not formed).
 * Pad rows [offsets[e] + counts[e], offsets[e+1]) below cap get gO = 0 and
 * gw = 0; rows at or beyond min(offsets[E], cap) are not written.
 * o may be NULL when gw is not wanted (gw NULL). */
ORACLE_API void moe_oracle_combine_backward(const uint16_t* gy, int64_t T, int64_t H, int64_t E, int64_t K,
                                            const int32_t* row_of, const int32_t* counts,
                                            const int32_t* offsets, int64_t cap, const uint16_t* o,
                                            const float* perm_probs, uint16_t* g_o, float* g_w) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; t++)
    for (int64_t k = 0; k < K; k++) {
      int32_t r = row_of[t * K + k];
      if (r < 0) continue;
      double w = perm_probs ? (double)perm_probs[r] : 1.0;
      double dot = 0.0;
      for (int64_t h = 0; h < H; h++) {
        double g = moe_oracle_bf16_to_f64(gy[t * H + h]);
        g_o[(int64_t)r * H + h] = moe_oracle_f64_to_bf16(w * g);
        if (o) dot += g * moe_oracle_bf16_to_f64(o[(int64_t)r * H + h]);
      }
      if (g_w) g_w[r] = f64_to_f32(dot);
    }
  for (int64_t e = 0; e < E; e++)
    for (int64_t r = (int64_t)offsets[e] + counts[e]; r < offsets[e + 1] && r < cap; r++) {
      for (int64_t h = 0; h < H; h++) g_o[r * H + h] = 0;
      if (g_w) g_w[r] = 0.0f;
    }
}

/* The dispatch computed Y[r] = x[t] and Yp[r] = p(t,k) for every kept route
 * (t,k) -> r, so for row gradients gY and probability gradients gYp:
 *   gx[t] = bf16( sum over k ascending of gY[row_of[t][k]] )   (a combine with
 *           weight 1; tokens whose routes were all dropped get zeros)
 *   gp(t,k) = gYp[row_of[t][k]], 0 for a dropped route or an empty slot,
 * written in the routing layout: dense [T][K]; sparse [T][E] (the entry of the
 * slot's expert; every other entry 0).  gYp and gp may be NULL together. */
ORACLE_API int moe_oracle_dispatch_backward(int format, const void* map, int64_t T, int64_t E, int64_t K,
                                            int64_t H, const int32_t* row_of, const uint16_t* g_y,
                                            const float* g_yp, uint16_t* g_x, float* g_p) {
  int32_t* route = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T * K + 1));
  int status = build_routes(format, map, T, E, K, route);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; t++) {
    for (int64_t h = 0; h < H; h++) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; k++) {
        int32_t r = row_of[t * K + k];
        if (r >= 0) acc += moe_oracle_bf16_to_f64(g_y[(int64_t)r * H + h]);
      }
      g_x[t * H + h] = moe_oracle_f64_to_bf16(acc);
    }
    if (!g_p) continue;
    if (format == 0) {
      for (int64_t k = 0; k < K; k++) {
        int32_t r = row_of[t * K + k];
        g_p[t * K + k] = (r >= 0) ? g_yp[r] : 0.0f;
      }
    } else {
      for (int64_t e = 0; e < E; e++) g_p[t * E + e] = 0.0f;
      for (int64_t k = 0; k < K; k++) {
        int32_t r = row_of[t * K + k];
        if (r >= 0 && route[t * K + k] >= 0) g_p[t * E + route[t * K + k]] = g_yp[r];
      }
    }
  }
  free(route);
  return status;
}

/* ------------------------------------------------------------------------- */
/* Second, unpermuted formulation of the whole layer                          */
/* ------------------------------------------------------------------------- */

/* The layer written per token, with no permutation, counts or offsets:
 *   y[t] = bf16( sum over k ascending of p(t,k) * bf16(FFN_{e(t,k)}(x_t)) )
 * over the slots that carry a route (all of them are kept: no capacity).  The
 * inner FFN is the same per-row arithmetic as the grouped path, fed the token's
 * own row (x in the activation format).  tokens: the token ids to evaluate;
 * y: [ntok][H]. */
ORACLE_API int moe_oracle_layer_per_token(int fmt, int format, const void* map, const float* probs,
                                          int64_t T, int64_t E, int64_t K, const void* x,
                                          const void* x_scales, int64_t H, int64_t I,
                                          const void* w13, const void* w13_scales,
                                          const float* w13_global, const void* w2,
                                          const void* w2_scales, const float* w2_global,
                                          double fc1_in_global, double fc2_in_global,
                                          const int64_t* tokens, int64_t ntok, uint16_t* y) {
  operand xin = {fmt, x, x_scales, fc1_in_global};
  operand ow13 = {fmt, w13, w13_scales, 0.0};
  operand ow2 = {fmt, w2, w2_scales, 0.0};
  int32_t* route = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T * K + 1));
  int status = build_routes(format, map, T, E, K, route);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < ntok; i++) {
    int64_t t = tokens[i];
    double* row_acc = (double*)malloc(sizeof(double) * (size_t)H);
    double* acc = (double*)calloc((size_t)H, sizeof(double));
    for (int64_t k = 0; k < K; k++) {
      int e = route[t * K + k];
      if (e < 0) continue;
      double p = probs ? prob_of_route(format, probs, t, k, e, E, K) : 1.0;
      ffn_row(&xin, t, e, H, I, &ow13, w13_global, &ow2, w2_global, fc2_in_global, row_acc, NULL);
      for (int64_t h = 0; h < H; h++) acc[h] += p * moe_oracle_bf16_to_f64(moe_oracle_f64_to_bf16(row_acc[h]));
    }
    for (int64_t h = 0; h < H; h++) y[i * H + h] = moe_oracle_f64_to_bf16(acc[h]);
    free(row_acc);
    free(acc);
  }
  free(route);
  return status;
}

/* ------------------------------------------------------------------------- */
/* Array forms of the number-format helpers (used by the tests)               */
/* ------------------------------------------------------------------------- */

ORACLE_API void moe_oracle_f64_to_bf16_array(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = moe_oracle_f64_to_bf16(v[i]);
}
ORACLE_API void moe_oracle_f32_to_e4m3_array(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = moe_oracle_f32_to_e4m3(v[i]);
}
ORACLE_API void moe_oracle_f32_to_e2m1_array(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = moe_oracle_f32_to_e2m1(v[i]);
}
