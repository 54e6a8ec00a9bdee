/*
 * pkv_oracle.c -- plain, slow, float64 CPU oracle for paged-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library: it is written from the statement of the method alone.
 *
 * Sources (blog pages on the paged KV cache, cited by page title and section):
 *   [P2] "Build a Paged KV Cache in Pure Python" -- Step 1 (a block holds
 *        (block_size, num_heads, head_dim) keys and values), Step 3
 *        (PagedKVCache.append: block index = pos // block_size, offset =
 *        pos % block_size; retrieve walks the block list in order and keeps
 *        min(block_size, n - start) rows per block), Step 4
 *        (scaled_dot_product_attention: scores = q.K * scale, max-subtracted
 *        softmax over the sequence axis, weighted sum of V; an empty cache
 *        gives zeros), Step 5 (append the new token first, then attend).
 *   [P3] "Building a Streaming Sliding-Window Attention Engine in Pure
 *        Python" -- Step 2 (contiguous KVCache) and Step 3
 *        (sliding_window_attention: start = max(0, T - window), attend over
 *        [start, T)).
 *
 * Readings of the pages that this file takes:
 *   - The physical pool is stored head-major, [num_blocks][num_kv_heads]
 *     [block_size][head_dim]; this is a storage order only, indexed
 *     explicitly below.  Token t of a sequence lives in physical block
 *     block_table[t / block_size], row t % block_size.
 *   - Grouped-query attention: query head h reads kv head h / (Hq / Hkv).
 *   - window <= 0 means no window; otherwise attend over the last `window`
 *     tokens, current token included.
 *   - Attention sinks ([P3] "Extending" list, the StreamingLLM item: keep
 *     the first 4 tokens regardless of the window): with a window and
 *     num_sinks > 0, positions [0, num_sinks) are attended as well as the
 *     window; num_sinks = 0 is the plain window.
 *   - Inputs of type fp16 / bf16 are widened exactly to double; all
 *     arithmetic is in double with libm exp().
 *   - Quantised cache ("Building a Memory-Compressed Attention Engine with
 *     KV Caching", Extending, item 2: INT8 or FP8 quantisation of the cached
 *     keys and values): FP8 E4M3 codes with one float32 scale per (token, kv
 *     head) row, stored value = code * scale.  A row is quantised when it is
 *     appended: scale = absmax / 448 (448 = largest E4M3 value), code =
 *     E4M3(x * (448 / absmax)) rounded to nearest, ties to even, saturating;
 *     an all-zero row gets scale 1.  The divisions and the product are single
 *     IEEE float32 operations.  Decoding over such a cache attends over the
 *     stored values code * scale, widened to double.
 *   - INT8 codes (same page and item): two's complement int8 with one float32
 *     scale per row, stored value = code * scale; scale = absmax / 127, code =
 *     x * (127 / absmax) rounded to the nearest integer, ties to even, and
 *     clamped to [-127, 127] (the symmetric range: -128 is never produced);
 *     an all-zero row gets scale 1; a NaN element gets code 0.  Single IEEE
 *     float32 divisions and products, as for FP8.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC pkv_oracle.c -o liboracle.so -lm
 * (no fast-math: the reference arithmetic must stay IEEE double).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2, ORACLE_FP8 = 3, ORACLE_I8 = 4 };

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_ARG = -1,       /* null pointer or bad size */
  ORACLE_ERR_BLOCK_ID = -2,  /* block table entry outside [0, num_blocks) */
  ORACLE_ERR_LENGTH = -3,    /* context length outside [0, max_blocks*bs] */
  ORACLE_ERR_NOMEM = -4
};

/* ---- element decoding ---------------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int expo = (bits >> 10) & 0x1f;
  int frac = bits & 0x3ff;
  double mag;
  if (expo == 0) {
    mag = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
  } else if (expo == 31) {
    mag = frac ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) * 2^(e-15) */
  }
  return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE 754 binary32. */
double oracle_bf16_to_double(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* FP8 E4M3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 fraction
 * bits; exponent 0 is subnormal (frac * 2^-9); S.1111.111 is NaN; there is no
 * infinity.  Largest finite magnitude: 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t code) {
  int sign = (code >> 7) & 1;
  int expo = (code >> 3) & 0xf;
  int frac = code & 0x7;
  double mag;
  if (expo == 15 && frac == 7) return NAN;
  if (expo == 0) mag = ldexp((double)frac, -9);
  else mag = ldexp((double)(8 + frac), expo - 10); /* (1 + frac/8) * 2^(e-7) */
  return sign ? -mag : mag;
}

/* Nearest E4M3 code to a float32, ties to the even code, saturating to +-448:
 * a brute-force search over the 127 finite non-negative codes. */
uint8_t oracle_float_to_e4m3(float x) {
  if (x != x) return 0x7f;
  uint8_t sign = (x < 0.0f || (x == 0.0f && 1.0f / x < 0.0f)) ? 0x80 : 0x00;
  double a = fabs((double)x);
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 126; ++c) {
    double err = fabs(oracle_e4m3_to_double((uint8_t)c) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(sign | best);
}

/* Quantise one row of n float32 values: writes n codes, returns the scale. */
float oracle_quantize_row(const float* x, int32_t n, uint8_t* codes) {
  float absmax = 0.0f;
  for (int32_t i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > absmax) absmax = a;
  }
  float scale = 1.0f, inv = 1.0f;
  if (absmax > 0.0f) {
    volatile float num = 448.0f; /* single float32 divisions, as the reading states */
    scale = absmax / num;
    inv = num / absmax;
  }
  for (int32_t i = 0; i < n; ++i) {
    volatile float prod = x[i] * inv;
    codes[i] = oracle_float_to_e4m3(prod);
  }
  return scale;
}

/* INT8 row quantiser (see the reading at the top): writes n codes, returns
 * the scale. */
float oracle_quantize_row_int8(const float* x, int32_t n, int8_t* codes) {
  float absmax = 0.0f;
  for (int32_t i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > absmax) absmax = a;
  }
  float scale = 1.0f, inv = 1.0f;
  if (absmax > 0.0f) {
    volatile float top = 127.0f; /* single float32 divisions */
    scale = absmax / top;
    inv = top / absmax;
  }
  for (int32_t i = 0; i < n; ++i) {
    volatile float prod = x[i] * inv;
    if (prod != prod) {
      codes[i] = 0;
      continue;
    }
    double r = nearbyint((double)prod); /* default rounding: to nearest, ties to even */
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    codes[i] = (int8_t)r;
  }
  return scale;
}

static double load_elem(const void* base, int64_t idx, int dtype) {
  switch (dtype) {
    case ORACLE_F32: return (double)((const float*)base)[idx];
    case ORACLE_F16: return oracle_f16_to_double(((const uint16_t*)base)[idx]);
    default: return oracle_bf16_to_double(((const uint16_t*)base)[idx]);
  }
}

/* Vector forms, used by the tests to pin the decoders. */
void oracle_decode_elements(const void* src, int64_t n, int32_t dtype, double* dst) {
  for (int64_t i = 0; i < n; ++i)
    dst[i] = dtype == ORACLE_FP8 ? oracle_e4m3_to_double(((const uint8_t*)src)[i])
                                 : load_elem(src, i, dtype);
}

void oracle_encode_e4m3(const float* src, int64_t n, uint8_t* dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = oracle_float_to_e4m3(src[i]);
}

/* ---- slot mapping and append ([P2] Step 3, PagedKVCache.append) ---------- */

/* The cache slot of logical position `pos` of a sequence whose block list is
 * `block_table_row`: the block is pos // block_size in the sequence's list,
 * the row inside it is pos % block_size.  Returns -1 when the position is
 * negative or beyond the table. */
int64_t oracle_slot_for_position(const int32_t* block_table_row, int32_t max_blocks,
                                 int32_t block_size, int64_t pos) {
  if (pos < 0 || block_size <= 0) return -1;
  int64_t logical_block = pos / block_size;
  int64_t offset = pos % block_size;
  if (logical_block >= max_blocks) return -1;
  int64_t physical = block_table_row[logical_block];
  return physical * block_size + offset;
}

/* Write token i's key and value rows (all kv heads) into the slot
 * slot_mapping[i]; a negative slot means "no write".  Byte copy: the cache
 * holds exactly the bits it was given. */
int oracle_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                  void* k_cache, void* v_cache, int64_t num_blocks, int32_t num_kv_heads,
                  int32_t block_size, int32_t head_dim, int32_t elem_bytes) {
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return ORACLE_ERR_ARG;
  if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || head_dim <= 0 || elem_bytes <= 0)
    return ORACLE_ERR_ARG;
  const size_t row_bytes = (size_t)head_dim * (size_t)elem_bytes;
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    int64_t block = slot / block_size;
    int64_t row = slot % block_size;
    if (block >= num_blocks) return ORACLE_ERR_BLOCK_ID;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      /* destination: [block][h][row][:] in the head-major pool */
      size_t dst_row = (((size_t)block * num_kv_heads + h) * block_size + row);
      /* source: [i][h][:] */
      size_t src_row = (size_t)i * num_kv_heads + h;
      memcpy((char*)k_cache + dst_row * row_bytes, (const char*)k + src_row * row_bytes, row_bytes);
      memcpy((char*)v_cache + dst_row * row_bytes, (const char*)v + src_row * row_bytes, row_bytes);
    }
  }
  return ORACLE_OK;
}

/* Append into a quantised pool (kind ORACLE_FP8 or ORACLE_I8): each (token,
 * kv head) row of k / v (fp16 / bf16 / fp32, `dtype`) is quantised on its own
 * (see the readings at the top) and its codes and scale written to the slot;
 * negative slots are skipped. */
static int append_quantised(const void* k, const void* v, int32_t dtype,
                            const int64_t* slot_mapping, int64_t num_tokens, uint8_t* k_codes,
                            uint8_t* v_codes, float* k_scale, float* v_scale, int64_t num_blocks,
                            int32_t num_kv_heads, int32_t block_size, int32_t head_dim,
                            int kind) {
  if (!k || !v || !slot_mapping || !k_codes || !v_codes || !k_scale || !v_scale)
    return ORACLE_ERR_ARG;
  float* row = (float*)malloc((size_t)head_dim * sizeof(float));
  if (!row) return ORACLE_ERR_NOMEM;
  int rc = ORACLE_OK;
  for (int64_t i = 0; i < num_tokens && rc == ORACLE_OK; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    int64_t block = slot / block_size, r = slot % block_size;
    if (block >= num_blocks) {
      rc = ORACLE_ERR_BLOCK_ID;
      break;
    }
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      int64_t dst_row = ((block * num_kv_heads + h) * block_size + r);
      int64_t src = ((int64_t)i * num_kv_heads + h) * head_dim;
      for (int pass = 0; pass < 2; ++pass) {
        const void* x = pass ? v : k;
        for (int32_t d = 0; d < head_dim; ++d) row[d] = (float)load_elem(x, src + d, dtype);
        uint8_t* codes = (pass ? v_codes : k_codes) + dst_row * head_dim;
        float sc = kind == ORACLE_I8 ? oracle_quantize_row_int8(row, head_dim, (int8_t*)codes)
                                     : oracle_quantize_row(row, head_dim, codes);
        (pass ? v_scale : k_scale)[dst_row] = sc;
      }
    }
  }
  free(row);
  return rc;
}

int oracle_append_fp8(const void* k, const void* v, int32_t dtype, const int64_t* slot_mapping,
                      int64_t num_tokens, uint8_t* k_codes, uint8_t* v_codes, float* k_scale,
                      float* v_scale, int64_t num_blocks, int32_t num_kv_heads,
                      int32_t block_size, int32_t head_dim) {
  return append_quantised(k, v, dtype, slot_mapping, num_tokens, k_codes, v_codes, k_scale,
                          v_scale, num_blocks, num_kv_heads, block_size, head_dim, ORACLE_FP8);
}

int oracle_append_int8(const void* k, const void* v, int32_t dtype, const int64_t* slot_mapping,
                       int64_t num_tokens, int8_t* k_codes, int8_t* v_codes, float* k_scale,
                       float* v_scale, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t block_size, int32_t head_dim) {
  return append_quantised(k, v, dtype, slot_mapping, num_tokens, (uint8_t*)k_codes,
                          (uint8_t*)v_codes, k_scale, v_scale, num_blocks, num_kv_heads,
                          block_size, head_dim, ORACLE_I8);
}

/* ---- attention over a contiguous cache ([P2] Step 4, [P3] Step 3) -------- */

/* out[d] = sum_t softmax_t(scale * q.K[t]) * V[t][d] for t in [0, T).
 * q: [D]; K, V: [T][D] contiguous, row-major; out: [D].  T == 0 gives zeros. */
void oracle_attend(const double* q, const double* K, const double* V, int64_t T, int32_t D,
                   double scale, double* out) {
  for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
  if (T <= 0) return;
  double* s = (double*)malloc((size_t)T * sizeof(double));
  if (!s) {
    for (int32_t d = 0; d < D; ++d) out[d] = NAN;
    return;
  }
  double m = -INFINITY;
  for (int64_t t = 0; t < T; ++t) {
    double dot = 0.0;
    for (int32_t d = 0; d < D; ++d) dot += q[d] * K[t * D + d];
    s[t] = scale * dot;
    if (s[t] > m) m = s[t];
  }
  double z = 0.0;
  for (int64_t t = 0; t < T; ++t) {
    s[t] = exp(s[t] - m); /* un-normalised softmax weight */
    z += s[t];
  }
  for (int64_t t = 0; t < T; ++t) {
    double w = s[t] / z;
    for (int32_t d = 0; d < D; ++d) out[d] += w * V[t * D + d];
  }
  free(s);
}

/* ---- paged decode ---------------------------------------------------------- */

typedef struct {
  const void* q;
  int32_t num_seqs, num_q_heads;
  const void* k_cache;
  const void* v_cache;
  const float* k_scale; /* FP8 / INT8 pools: per-row scales, else NULL */
  const float* v_scale;
  int64_t num_blocks;
  int32_t num_kv_heads, block_size, head_dim, dtype, kv_dtype;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* context_lens;
  int32_t window;
  int32_t num_sinks;
  double scale;
} decode_problem;

/* First position attended by a sequence of length L ([P3] Step 3). */
static int64_t window_start(int64_t L, int32_t window) {
  if (window <= 0) return 0;
  int64_t lo = L - window;
  return lo > 0 ? lo : 0;
}

/* One (sequence b, query head h): retrieve the sequence's tokens [lo, L) of
 * kv head h/G from its blocks in logical order ([P2] retrieve), then attend. */
static int decode_one(const decode_problem* p, int32_t b, int32_t h, double* out) {
  const int32_t D = p->head_dim;
  const int32_t G = p->num_q_heads / p->num_kv_heads;
  const int32_t hk = h / G;
  const int64_t L = p->context_lens[b];
  if (L < 0 || L > (int64_t)p->max_blocks * p->block_size) {
    for (int32_t d = 0; d < D; ++d) out[d] = NAN;
    return ORACLE_ERR_LENGTH;
  }
  const int64_t lo = window_start(L, p->window);
  /* sink positions before the window: [0, min(num_sinks, lo)) */
  int64_t n_sink = 0;
  if (p->window > 0 && p->num_sinks > 0) n_sink = p->num_sinks < lo ? p->num_sinks : lo;
  const int64_t T = n_sink + (L - lo);

  double* q = (double*)malloc((size_t)D * sizeof(double));
  double* K = (double*)malloc((size_t)(T > 0 ? T : 1) * D * sizeof(double));
  double* V = (double*)malloc((size_t)(T > 0 ? T : 1) * D * sizeof(double));
  if (!q || !K || !V) {
    free(q); free(K); free(V);
    return ORACLE_ERR_NOMEM;
  }
  for (int32_t d = 0; d < D; ++d)
    q[d] = load_elem(p->q, ((int64_t)b * p->num_q_heads + h) * D + d, p->dtype);

  const int32_t* table = p->block_tables + (int64_t)b * p->max_blocks;
  int rc = ORACLE_OK;
  /* the attended positions, in order: the sinks, then the window */
  int64_t i = 0;
  for (int64_t t = 0; t < L && rc == ORACLE_OK; ++t) {
    if (!(t < n_sink || t >= lo)) continue;
    int64_t physical = table[t / p->block_size];
    int64_t row = t % p->block_size;
    if (physical < 0 || physical >= p->num_blocks) {
      rc = ORACLE_ERR_BLOCK_ID;
      break;
    }
    int64_t prow = (physical * p->num_kv_heads + hk) * p->block_size + row;
    int64_t base = prow * D;
    if (p->kv_dtype == ORACLE_FP8 || p->kv_dtype == ORACLE_I8) {
      /* stored value = code * scale of its row */
      double ks = (double)p->k_scale[prow], vs = (double)p->v_scale[prow];
      for (int32_t d = 0; d < D; ++d) {
        double kc, vc;
        if (p->kv_dtype == ORACLE_FP8) {
          kc = oracle_e4m3_to_double(((const uint8_t*)p->k_cache)[base + d]);
          vc = oracle_e4m3_to_double(((const uint8_t*)p->v_cache)[base + d]);
        } else {
          kc = (double)((const int8_t*)p->k_cache)[base + d];
          vc = (double)((const int8_t*)p->v_cache)[base + d];
        }
        K[i * D + d] = kc * ks;
        V[i * D + d] = vc * vs;
      }
    } else {
      for (int32_t d = 0; d < D; ++d) {
        K[i * D + d] = load_elem(p->k_cache, base + d, p->kv_dtype);
        V[i * D + d] = load_elem(p->v_cache, base + d, p->kv_dtype);
      }
    }
    ++i;
  }
  if (rc == ORACLE_OK) {
    oracle_attend(q, K, V, T, D, p->scale, out);
  } else {
    for (int32_t d = 0; d < D; ++d) out[d] = NAN;
  }
  free(q); free(K); free(V);
  return rc;
}

static int decode_pairs(const decode_problem* p, const int32_t* pairs, int64_t n_pairs,
                        double* out, int32_t num_threads);

/* Decode attention for a list of (sequence, query head) pairs.
 *   q            [num_seqs][num_q_heads][head_dim]        dtype
 *   k/v_cache    [num_blocks][num_kv_heads][block_size][head_dim] dtype
 *   block_tables [num_seqs][max_blocks] int32
 *   context_lens [num_seqs] int32 (length after the step's append)
 *   window, num_sinks: see the readings at the top of this file
 *   pairs        [n_pairs][2] = (b, h); NULL means every pair in (b, h) order
 *   out          [n_pairs][head_dim] double
 * Returns ORACLE_OK or the first error met (the affected rows hold NaN). */
int oracle_decode(const void* q, int32_t num_seqs, int32_t num_q_heads,
                  const void* k_cache, const void* v_cache, int64_t num_blocks,
                  int32_t num_kv_heads, int32_t block_size, int32_t head_dim, int32_t dtype,
                  const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                  int32_t window, int32_t num_sinks, double scale, const int32_t* pairs,
                  int64_t n_pairs, double* out, int32_t num_threads) {
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return ORACLE_ERR_ARG;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks < 0 || num_q_heads % num_kv_heads != 0 || dtype < 0 || dtype > 2)
    return ORACLE_ERR_ARG;
  decode_problem p = {q, num_seqs, num_q_heads, k_cache, v_cache, NULL, NULL, num_blocks,
                      num_kv_heads, block_size, head_dim, dtype, dtype, block_tables,
                      max_blocks, context_lens, window, num_sinks, scale};
  return decode_pairs(&p, pairs, n_pairs, out, num_threads);
}

/* Decode over FP8 pools: k_codes / v_codes [NB][Hkv][bs][D] E4M3 codes,
 * k_scale / v_scale [NB][Hkv][bs] float32; q has dtype q_dtype (fp16 / bf16 /
 * fp32).  Otherwise as oracle_decode. */
int oracle_decode_fp8(const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads,
                      const uint8_t* k_codes, const uint8_t* v_codes, const float* k_scale,
                      const float* v_scale, int64_t num_blocks, int32_t num_kv_heads,
                      int32_t block_size, int32_t head_dim, const int32_t* block_tables,
                      int32_t max_blocks, const int32_t* context_lens, int32_t window,
                      int32_t num_sinks, double scale, const int32_t* pairs, int64_t n_pairs,
                      double* out, int32_t num_threads) {
  if (!q || !k_codes || !v_codes || !k_scale || !v_scale || !block_tables || !context_lens ||
      !out)
    return ORACLE_ERR_ARG;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks < 0 || num_q_heads % num_kv_heads != 0 || q_dtype < 0 || q_dtype > 2)
    return ORACLE_ERR_ARG;
  decode_problem p = {q, num_seqs, num_q_heads, k_codes, v_codes, k_scale, v_scale, num_blocks,
                      num_kv_heads, block_size, head_dim, q_dtype, ORACLE_FP8, block_tables,
                      max_blocks, context_lens, window, num_sinks, scale};
  return decode_pairs(&p, pairs, n_pairs, out, num_threads);
}

/* Decode over INT8 pools: as oracle_decode_fp8 with int8 codes. */
int oracle_decode_int8(const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads,
                       const int8_t* k_codes, const int8_t* v_codes, const float* k_scale,
                       const float* v_scale, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t block_size, int32_t head_dim, const int32_t* block_tables,
                       int32_t max_blocks, const int32_t* context_lens, int32_t window,
                       int32_t num_sinks, double scale, const int32_t* pairs, int64_t n_pairs,
                       double* out, int32_t num_threads) {
  if (!q || !k_codes || !v_codes || !k_scale || !v_scale || !block_tables || !context_lens ||
      !out)
    return ORACLE_ERR_ARG;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks < 0 || num_q_heads % num_kv_heads != 0 || q_dtype < 0 || q_dtype > 2)
    return ORACLE_ERR_ARG;
  decode_problem p = {q, num_seqs, num_q_heads, k_codes, v_codes, k_scale, v_scale, num_blocks,
                      num_kv_heads, block_size, head_dim, q_dtype, ORACLE_I8, block_tables,
                      max_blocks, context_lens, window, num_sinks, scale};
  return decode_pairs(&p, pairs, n_pairs, out, num_threads);
}

static int decode_pairs(const decode_problem* pp, const int32_t* pairs, int64_t n_pairs,
                        double* out, int32_t num_threads) {
  const decode_problem p = *pp;
  const int32_t num_seqs = p.num_seqs, num_q_heads = p.num_q_heads, head_dim = p.head_dim;
  const int64_t total = pairs ? n_pairs : (int64_t)num_seqs * num_q_heads;
  int rc = ORACLE_OK;
#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
  for (int64_t i = 0; i < total; ++i) {
    int32_t b = pairs ? pairs[2 * i] : (int32_t)(i / num_q_heads);
    int32_t h = pairs ? pairs[2 * i + 1] : (int32_t)(i % num_q_heads);
    int r;
    if (b < 0 || b >= num_seqs || h < 0 || h >= num_q_heads) {
      for (int32_t d = 0; d < head_dim; ++d) out[i * head_dim + d] = NAN;
      r = ORACLE_ERR_ARG;
    } else {
      r = decode_one(&p, b, h, out + i * head_dim);
    }
    if (r != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
      if (rc == ORACLE_OK) rc = r;
    }
  }
  return rc;
}

/* ---- paged (chunked) prefill ([P3] Step 3, prefill_attention) ------------- */

/* Prefill of a chunk of new tokens per sequence over a paged cache that holds
 * the sequence's earlier tokens and the chunk itself (appended beforehand).
 * Sequence b's chunk is tokens cu_q[b] .. cu_q[b+1]-1 of the packed q / out,
 * at positions L_b - n_b .. L_b - 1 (L_b = context_lens[b], n_b the chunk
 * size).  Query token at position p attends the positions j with j <= p and,
 * when window > 0, p - j < window: the mask of prefill_attention, with the
 * softmax taken per query row.  With a window and num_sinks > 0 the positions
 * j < num_sinks (j <= p) are attended as well (the attention-sink policy, as
 * in decode).  That is a decode of length p + 1 with the same window and
 * sinks, which is how it is computed here.
 *   q   [T][Hq][D] (dtype), out [T][Hq][D] double, T = cu_q[num_seqs]. */
int oracle_prefill(const void* q, int32_t dtype, const int32_t* cu_q, int32_t num_seqs,
                   int32_t num_q_heads, const void* k_cache, const void* v_cache,
                   int64_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                   int32_t head_dim, const int32_t* block_tables, int32_t max_blocks,
                   const int32_t* context_lens, int32_t window, int32_t num_sinks,
                   double scale, double* out,
                   int32_t num_threads) {
  if (!q || !cu_q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return ORACLE_ERR_ARG;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
      dtype < 0 || dtype > 2)
    return ORACLE_ERR_ARG;
  const int64_t T = cu_q[num_seqs];
  int rc = ORACLE_OK;
#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
  for (int64_t t = 0; t < T; ++t) {
    int32_t b = 0;
    while (b + 1 < num_seqs && cu_q[b + 1] <= t) ++b; /* the sequence holding token t */
    const int64_t n = cu_q[b + 1] - cu_q[b];
    const int64_t p = context_lens[b] - n + (t - cu_q[b]); /* its position */
    /* one query row: a decode problem of a single sequence with length p + 1 */
    int32_t len = (int32_t)(p + 1);
    decode_problem dp = {(const char*)q + t * (int64_t)num_q_heads * head_dim *
                                              (dtype == ORACLE_F32 ? 4 : 2),
                         1, num_q_heads, k_cache, v_cache, NULL, NULL, num_blocks,
                         num_kv_heads, block_size, head_dim, dtype, dtype,
                         block_tables + (int64_t)b * max_blocks, max_blocks, &len, window,
                         num_sinks, scale};
    for (int32_t h = 0; h < num_q_heads; ++h) {
      int r = p < 0 ? ORACLE_ERR_LENGTH : decode_one(&dp, 0, h, out + (t * num_q_heads + h) * head_dim);
      if (r != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
        if (rc == ORACLE_OK) rc = r;
      }
    }
  }
  return rc;
}

/* Number of threads the OpenMP runtime would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
