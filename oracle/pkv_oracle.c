/*
 * pkv_oracle.c -- plain, slow CPU oracle for paged KV cache attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The product
 * (libpkv.so and its Python binding) never calls it and shares no code,
 * header, table or helper with it.
 *
 * What it computes, each function citing the passage it follows:
 *
 *   orc_slot_mapping  -- the cache slot of every new token, from the
 *                        sequence's block table.
 *                        nanoserve, "Architecture" (one engine step, step 2
 *                        "Prepare": each token's cache slot is computed from
 *                        its block table); "How to design an LLM serving
 *                        system (a vLLM deep dive)", "PagedAttention (vLLM
 *                        KV manager)": the block table maps logical positions
 *                        to physical blocks of block_size tokens, and
 *                        slot_mapping names each token's physical slot.
 *   orc_append        -- writes each new K/V row into its slot.
 *                        nanoserve, "Architecture" step 3 "Forward": each
 *                        layer first writes this step's K/V into the paged
 *                        cache.
 *   orc_attention     -- causal GQA softmax attention of every packed query
 *   (orc_attention_v, orc_attention_rows_v: the same with a logits soft cap
 *    and a sliding window, "How Easy Is It to Start Serving LLMs?", "2. JIT
 *    compilation: one template, a kernel per variant")
 *                        row over its sequence's pages, gathered through the
 *                        block table in logical order.
 *                        nanoserve, "Architecture" step 3 (attend over the
 *                        full context through the block table) and the
 *                        "Paged KV cache" / "Chunked prefill" /
 *                        "Triton paged-attention decode kernel" bullets;
 *                        "PageServe", "What is implemented" (GQA attention).
 *   orc_e4m3_encode / orc_e4m3_decode / orc_bf16_decode
 *                     -- the 8-bit and 16-bit value formats of the caches.
 *                        "How Easy Is It to Start Serving LLMs?", "What each
 *                        setting does to performance" (FP8 KV cache: every
 *                        value is converted back to 16-bit as it is read).
 *
 * The attention is the plain definition, in fp64:
 *     s_j = scale * sum_d q[d] * K_j[d]          for keys j = 0 .. p
 *     m   = max_j s_j,  w_j = exp(s_j - m)
 *     o   = (sum_j w_j * V_j) / (sum_j w_j)
 * summed over j in increasing logical order.  The online softmax, the
 * split-KV chunks and the log-sum-exp merge that the pages describe reach
 * this same value (up to rounding order); the oracle does none of them.
 *
 * Readings of points the pages leave open:
 *   - slot = block_table[p / block_size] * block_size + p % block_size.
 *   - seq_lens counts this step's appended tokens; query i of a sequence with
 *     q_s new tokens and N keys sits at position p = N - q_s + i and sees
 *     keys 0 .. p (decode is the q_s = 1 case).
 *   - query head h reads KV head h / (Hq / Hkv).
 *   - slot < 0 means "no write".
 *   - fp8 is OCP e4m3: bias 7, largest finite 448, no infinity; encoding
 *     is round-to-nearest-even on x * (1/scale) taken as an fp32 product,
 *     magnitudes at or above 448 saturate to 448, NaN stays NaN.  Decoded
 *     values are multiplied by the per-tensor scale in fp64.
 *
 * Parity pins (tests/test_oracle_pins.py): every function above is pinned
 * by brute force, a library routine, closed forms or invariants; none is
 * "parity unpinned".
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread.
 * -ffp-contract=off keeps the fp32 product of the fp8 encoder a single
 * rounded multiply on every host architecture.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Value formats, numbered like the library's dtype enum only by accident of
 * both following the same list; nothing is shared. */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };

/* ------------------------------------------------------------------ */
/* Value formats                                                        */
/* ------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32. */
double orc_bf16_decode(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3: sign, 4 exponent bits (bias 7), 3
 * mantissa bits.  Exponent field 0 holds the subnormals m/8 * 2^-6; the
 * single pattern S.1111.111 is NaN; there is no infinity. */
double orc_e4m3_decode(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* Nearest e4m3 code to the fp32 value x, ties to the even code, magnitudes
 * at or above 448 saturated to 448, NaN to NaN. */
uint8_t orc_e4m3_encode(float x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* 1.75 * 2^8 */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: step 2^-9; a count of 8 steps is the smallest
     * normal (exponent field 1, mantissa 0), whose code is also 8. */
    double steps = nearbyint(a / ldexp(1.0, -9)); /* ties to even */
    return (uint8_t)(sign | (uint8_t)steps);
  }
  int e2;
  (void)frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
  int e = e2 - 1;      /* a in [2^e, 2^(e+1)) */
  double q = nearbyint(a / ldexp(1.0, e - 3)); /* in [8, 16] */
  if (q == 16.0) {
    q = 8.0;
    e += 1;
  }
  /* a < 448 keeps the result at or below 1.75 * 2^8 */
  return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | ((int)q - 8)));
}

void orc_bf16_decode_n(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_decode(in[i]);
}
void orc_e4m3_decode_n(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(in[i]);
}
void orc_e4m3_encode_n(const float* in, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(in[i]);
}

/* One element of an input of the given format, as fp64.  Source inputs are
 * fp32 or bf16. */
static double load_src(const void* base, int dtype, int64_t idx) {
  if (dtype == ORC_F32) return (double)((const float*)base)[idx];
  return orc_bf16_decode(((const uint16_t*)base)[idx]);
}

/* ------------------------------------------------------------------ */
/* Slot computation                                                     */
/* ------------------------------------------------------------------ */

/* For every sequence s with q_s = cu_seqlens_q[s+1] - cu_seqlens_q[s] new
 * tokens and N_s = seq_lens[s] tokens in all, new token i sits at logical
 * position p = N_s - q_s + i; its slot is
 *     block_tables[s][p / block_size] * block_size + p % block_size.   */
int orc_slot_mapping(int32_t B, const int32_t* cu_seqlens_q,
                     const int32_t* seq_lens, const int32_t* block_tables,
                     int32_t max_blocks, int32_t block_size, int64_t* slot) {
  for (int32_t s = 0; s < B; ++s) {
    int32_t q_s = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
    int32_t n_s = seq_lens[s];
    if (q_s < 0 || q_s > n_s || n_s > (int64_t)max_blocks * block_size)
      return -1;
    for (int32_t i = 0; i < q_s; ++i) {
      int64_t p = (int64_t)n_s - q_s + i;
      int64_t logical_block = p / block_size;
      int64_t offset = p % block_size;
      int64_t physical_block =
          block_tables[(int64_t)s * max_blocks + logical_block];
      slot[cu_seqlens_q[s] + i] = physical_block * block_size + offset;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* KV append                                                            */
/* ------------------------------------------------------------------ */

/* Writes one tensor x[T][H][D] into cache[num_blocks][block_size][H][D]:
 * the row of token t goes to block slot/block_size, offset slot%block_size.
 * Same-format copies are bit copies; an e4m3 cache stores
 * encode(fl32(x) * inv_scale) with inv_scale = 1.0f / scale in fp32. */
static int append_one(const void* x, int src_dtype, const int64_t* slot,
                      int64_t T, int32_t H, int32_t D, void* cache,
                      int cache_dtype, int32_t block_size,
                      int64_t num_blocks, float scale) {
  float inv_scale = 1.0f / scale;
  for (int64_t t = 0; t < T; ++t) {
    if (slot[t] < 0) continue;
    int64_t block = slot[t] / block_size;
    int64_t offset = slot[t] % block_size;
    if (block >= num_blocks) return -1;
    for (int32_t h = 0; h < H; ++h) {
      for (int32_t d = 0; d < D; ++d) {
        int64_t src = (t * H + h) * (int64_t)D + d;
        int64_t dst = ((block * block_size + offset) * H + h) * (int64_t)D + d;
        if (cache_dtype == ORC_E4M3) {
          float v = (float)load_src(x, src_dtype, src); /* exact */
          float prod = v * inv_scale;                    /* fp32 multiply */
          ((uint8_t*)cache)[dst] = orc_e4m3_encode(prod);
        } else if (cache_dtype == ORC_F32 && src_dtype == ORC_F32) {
          ((float*)cache)[dst] = ((const float*)x)[src];
        } else if (cache_dtype == ORC_BF16 && src_dtype == ORC_BF16) {
          ((uint16_t*)cache)[dst] = ((const uint16_t*)x)[src];
        } else {
          return -2;
        }
      }
    }
  }
  return 0;
}

int orc_append(const void* k, const void* v, int src_dtype,
               const int64_t* slot, int64_t T, int32_t Hkv, int32_t D,
               void* k_cache, void* v_cache, int cache_dtype,
               int32_t block_size, int64_t num_blocks, float k_scale,
               float v_scale) {
  int rc = append_one(k, src_dtype, slot, T, Hkv, D, k_cache, cache_dtype,
                      block_size, num_blocks, k_scale);
  if (rc) return rc;
  return append_one(v, src_dtype, slot, T, Hkv, D, v_cache, cache_dtype,
                    block_size, num_blocks, v_scale);
}

/* ------------------------------------------------------------------ */
/* Attention                                                            */
/* ------------------------------------------------------------------ */

typedef struct {
  /* inputs */
  const void* q;
  int q_dtype;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  int32_t B, max_blocks, block_size;
  const void* k_cache;
  const void* v_cache;
  int cache_dtype;
  int64_t num_blocks;
  int32_t Hq, Hkv, D;
  double scale, k_scale, v_scale;
  /* rows to compute: (token t, query head h); NULL = all rows */
  int64_t n_rows;
  const int64_t* rows_t;
  const int32_t* rows_h;
  double* out; /* [T][Hq][D] when all rows, else [n_rows][D] */
  int32_t nthreads;
  int status;
  double soft_cap;     /* > 0: scores s become soft_cap * tanh(s / soft_cap) */
  int64_t window_left; /* >= 0: the query at p sees keys p - window_left .. p */
} attn_job;

/* One element of a cache, decoded to fp64 and multiplied by the per-tensor
 * scale when the cache is e4m3. */
static double load_cache(const void* cache, int dtype, int64_t idx,
                         double scale) {
  if (dtype == ORC_F32) return (double)((const float*)cache)[idx];
  if (dtype == ORC_BF16) return orc_bf16_decode(((const uint16_t*)cache)[idx]);
  return orc_e4m3_decode(((const uint8_t*)cache)[idx]) * scale;
}

/* Flat index of element d of KV head g of logical token j of sequence s,
 * reached through the sequence's block table. */
static int64_t kv_index(const attn_job* J, int32_t s, int64_t j, int32_t g,
                        int32_t d) {
  int64_t physical_block =
      J->block_tables[(int64_t)s * J->max_blocks + j / J->block_size];
  int64_t offset = j % J->block_size;
  return ((physical_block * J->block_size + offset) * J->Hkv + g) *
             (int64_t)J->D + d;
}

/* Output row of query token t (of sequence s, query index i) and head h. */
static int attend_row(const attn_job* J, int32_t s, int32_t i, int64_t t,
                      int32_t h, double* o, double* scores) {
  int32_t q_s = J->cu_seqlens_q[s + 1] - J->cu_seqlens_q[s];
  int64_t n_s = J->seq_lens[s];
  int64_t p = n_s - q_s + i;          /* absolute position of the query */
  int32_t g = h / (J->Hq / J->Hkv);   /* KV head of this query head */
  int64_t qbase = (t * J->Hq + h) * (int64_t)J->D;
  /* visible keys: 0 .. p, or p - window_left .. p with a sliding window */
  int64_t lo = 0;
  if (J->window_left >= 0 && p - J->window_left > 0) lo = p - J->window_left;
  for (int64_t j = lo; j <= p; ++j) {
    int64_t pb = J->block_tables[(int64_t)s * J->max_blocks + j / J->block_size];
    if (pb < 0 || pb >= J->num_blocks) return -1;
  }
  /* scores, in logical key order; a soft cap bends each one through tanh */
  double m = -INFINITY;
  for (int64_t j = lo; j <= p; ++j) {
    double dot = 0.0;
    for (int32_t d = 0; d < J->D; ++d)
      dot += load_src(J->q, J->q_dtype, qbase + d) *
             load_cache(J->k_cache, J->cache_dtype, kv_index(J, s, j, g, d),
                        J->k_scale);
    scores[j] = J->scale * dot;
    if (J->soft_cap > 0.0) scores[j] = J->soft_cap * tanh(scores[j] / J->soft_cap);
    if (scores[j] > m) m = scores[j];
  }
  /* softmax weights and the weighted sum of values */
  double l = 0.0;
  for (int32_t d = 0; d < J->D; ++d) o[d] = 0.0;
  for (int64_t j = lo; j <= p; ++j) {
    double w = exp(scores[j] - m);
    l += w;
    for (int32_t d = 0; d < J->D; ++d)
      o[d] += w * load_cache(J->v_cache, J->cache_dtype,
                             kv_index(J, s, j, g, d), J->v_scale);
  }
  for (int32_t d = 0; d < J->D; ++d) o[d] /= l;
  return 0;
}

/* Sequence owning packed token t. */
static int32_t seq_of_token(const attn_job* J, int64_t t) {
  for (int32_t s = 0; s < J->B; ++s)
    if (t >= J->cu_seqlens_q[s] && t < J->cu_seqlens_q[s + 1]) return s;
  return -1;
}

typedef struct {
  attn_job* J;
  int32_t worker;
  int status;
} worker_arg;

static int64_t max_seq_len(const attn_job* J) {
  int64_t mx = 1;
  for (int32_t s = 0; s < J->B; ++s)
    if (J->seq_lens[s] > mx) mx = J->seq_lens[s];
  return mx;
}

/* All rows: work items are (sequence, KV head) pairs, dealt round-robin to
 * the workers.  Selected rows: dealt round-robin by row.  Every output
 * element is computed by one worker in the same order whatever the worker
 * count, so the result does not depend on it. */
static void* worker_main(void* p) {
  worker_arg* W = (worker_arg*)p;
  attn_job* J = W->J;
  double* scores = (double*)malloc(sizeof(double) * (size_t)max_seq_len(J));
  if (!scores) {
    W->status = -3;
    return NULL;
  }
  W->status = 0;
  if (J->rows_t == NULL) {
    int32_t G = J->Hq / J->Hkv;
    int64_t n_items = (int64_t)J->B * J->Hkv;
    for (int64_t item = W->worker; item < n_items; item += J->nthreads) {
      int32_t s = (int32_t)(item / J->Hkv);
      int32_t g = (int32_t)(item % J->Hkv);
      int32_t q_s = J->cu_seqlens_q[s + 1] - J->cu_seqlens_q[s];
      for (int32_t i = 0; i < q_s; ++i) {
        int64_t t = J->cu_seqlens_q[s] + i;
        for (int32_t h = g * G; h < (g + 1) * G; ++h) {
          double* o = J->out + (t * J->Hq + h) * (int64_t)J->D;
          if (attend_row(J, s, i, t, h, o, scores)) W->status = -1;
        }
      }
    }
  } else {
    for (int64_t r = W->worker; r < J->n_rows; r += J->nthreads) {
      int64_t t = J->rows_t[r];
      int32_t s = seq_of_token(J, t);
      if (s < 0) {
        W->status = -1;
        continue;
      }
      int32_t i = (int32_t)(t - J->cu_seqlens_q[s]);
      if (attend_row(J, s, i, t, J->rows_h[r], J->out + r * (int64_t)J->D,
                     scores))
        W->status = -1;
    }
  }
  free(scores);
  return NULL;
}

static int run_job(attn_job* J) {
  if (J->Hkv <= 0 || J->Hq % J->Hkv != 0 || J->D <= 0 || J->block_size <= 0)
    return -2;
  for (int32_t s = 0; s < J->B; ++s) {
    int32_t q_s = J->cu_seqlens_q[s + 1] - J->cu_seqlens_q[s];
    if (q_s < 0 || q_s > J->seq_lens[s] ||
        J->seq_lens[s] > (int64_t)J->max_blocks * J->block_size)
      return -2;
  }
  if (J->nthreads < 1) J->nthreads = 1;
  worker_arg* args = (worker_arg*)calloc((size_t)J->nthreads, sizeof(worker_arg));
  pthread_t* tids = (pthread_t*)calloc((size_t)J->nthreads, sizeof(pthread_t));
  if (!args || !tids) {
    free(args);
    free(tids);
    return -3;
  }
  int rc = 0;
  int32_t started = 0;
  for (int32_t w = 0; w < J->nthreads; ++w) {
    args[w].J = J;
    args[w].worker = w;
    if (w == 0) continue;
    if (pthread_create(&tids[w], NULL, worker_main, &args[w]) != 0) break;
    started = w;
  }
  /* threads that failed to start leave their items to a second pass below */
  worker_main(&args[0]);
  for (int32_t w = 1; w <= started; ++w) pthread_join(tids[w], NULL);
  if (started + 1 < J->nthreads) {
    for (int32_t w = started + 1; w < J->nthreads; ++w) worker_main(&args[w]);
  }
  for (int32_t w = 0; w < J->nthreads; ++w)
    if (args[w].status) rc = args[w].status;
  free(args);
  free(tids);
  return rc;
}

/* Attention with the two variants ("How Easy Is It to Start Serving LLMs?",
 * "2. JIT compilation: one template, a kernel per variant": a logits soft cap
 * and a sliding window are among the variants a kernel is built for).
 * soft_cap <= 0 and window_left < 0 turn them off. */
int orc_attention_v(const void* q, int q_dtype, const int32_t* cu_seqlens_q,
                    const int32_t* seq_lens, const int32_t* block_tables,
                    int32_t B, int32_t max_blocks, const void* k_cache,
                    const void* v_cache, int cache_dtype, int32_t block_size,
                    int64_t num_blocks, int32_t Hq, int32_t Hkv, int32_t D,
                    double scale, double k_scale, double v_scale,
                    double soft_cap, int64_t window_left, double* out,
                    int32_t nthreads) {
  attn_job J = {q, q_dtype, cu_seqlens_q, seq_lens, block_tables, B,
                max_blocks, block_size, k_cache, v_cache, cache_dtype,
                num_blocks, Hq, Hkv, D, scale, k_scale, v_scale, 0, NULL,
                NULL, out, nthreads, 0, soft_cap, window_left};
  return run_job(&J);
}

int orc_attention_rows_v(const void* q, int q_dtype,
                         const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                         const int32_t* block_tables, int32_t B,
                         int32_t max_blocks, const void* k_cache,
                         const void* v_cache, int cache_dtype,
                         int32_t block_size, int64_t num_blocks, int32_t Hq,
                         int32_t Hkv, int32_t D, double scale, double k_scale,
                         double v_scale, double soft_cap, int64_t window_left,
                         int64_t n_rows, const int64_t* rows_t,
                         const int32_t* rows_h, double* out, int32_t nthreads) {
  attn_job J = {q, q_dtype, cu_seqlens_q, seq_lens, block_tables, B,
                max_blocks, block_size, k_cache, v_cache, cache_dtype,
                num_blocks, Hq, Hkv, D, scale, k_scale, v_scale, n_rows,
                rows_t, rows_h, out, nthreads, 0, soft_cap, window_left};
  if (n_rows > 0 && (rows_t == NULL || rows_h == NULL)) return -2;
  if (n_rows == 0) return 0;
  return run_job(&J);
}

int orc_attention(const void* q, int q_dtype, const int32_t* cu_seqlens_q,
                  const int32_t* seq_lens, const int32_t* block_tables,
                  int32_t B, int32_t max_blocks, const void* k_cache,
                  const void* v_cache, int cache_dtype, int32_t block_size,
                  int64_t num_blocks, int32_t Hq, int32_t Hkv, int32_t D,
                  double scale, double k_scale, double v_scale, double* out,
                  int32_t nthreads) {
  attn_job J = {q, q_dtype, cu_seqlens_q, seq_lens, block_tables, B,
                max_blocks, block_size, k_cache, v_cache, cache_dtype,
                num_blocks, Hq, Hkv, D, scale, k_scale, v_scale, 0, NULL,
                NULL, out, nthreads, 0, 0.0, -1};
  return run_job(&J);
}

int orc_attention_rows(const void* q, int q_dtype,
                       const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                       const int32_t* block_tables, int32_t B,
                       int32_t max_blocks, const void* k_cache,
                       const void* v_cache, int cache_dtype,
                       int32_t block_size, int64_t num_blocks, int32_t Hq,
                       int32_t Hkv, int32_t D, double scale, double k_scale,
                       double v_scale, int64_t n_rows, const int64_t* rows_t,
                       const int32_t* rows_h, double* out, int32_t nthreads) {
  attn_job J = {q, q_dtype, cu_seqlens_q, seq_lens, block_tables, B,
                max_blocks, block_size, k_cache, v_cache, cache_dtype,
                num_blocks, Hq, Hkv, D, scale, k_scale, v_scale, n_rows,
                rows_t, rows_h, out, nthreads, 0, 0.0, -1};
  if (n_rows > 0 && (rows_t == NULL || rows_h == NULL)) return -2;
  if (n_rows == 0) return 0;
  return run_job(&J);
}
