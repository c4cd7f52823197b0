/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged decode attention over an
 * FP8 (e4m3) or BF16 paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this
 * file; only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
 * shares no code, header, table or constant with the CUDA library: it is written
 * from the definitions below, in double precision, with no blocking or fusion.
 *
 * What it computes (one output row per query token, per query head):
 *
 *   Row map.  Request r owns query rows [cu_q[r], cu_q[r+1]); row tok of it is
 *     cu_q[r] + tok.  Requests are recovered from cu_seqlens_q, never by dividing a
 *     flat row index by a maximum query length (ROCm/ATOM PR 2122, "fix(minimax-m3):
 *     unblock fp8 KV cache and EAGLE3 spec decode on the vLLM plugin", section 2,
 *     "A decode segment must be uniform before a decode kernel may have it").
 *
 *   Causal cutoff.  Row tok of a request with context length L and q_len query
 *     tokens attends positions p < L - q_len + tok + 1 (same page, section 2, the
 *     index-topk cutoff "seq_len - max_query_len + tok + 1", read with the request's
 *     own q_len).  context_lens[r] counts the request's own new tokens.
 *
 *   Key set.  Dense: every position p < min(L, cutoff).  Sparse: the positions of
 *     the request's selected logical pages (entries < 0 are padding), restricted to
 *     p < L and p < cutoff (ROCm/ATOM PR 2614, "Change": sparse decode reuses the
 *     dense paged-decode contract).
 *
 *   Gather.  phys = block_table[r][p / page_size], slot o = p % page_size; the code
 *     sits at k_cache[((phys * Hkv + h) * page_size + o) * D + d].
 *
 *   Explicit dequantisation (vLLM PR 52060, "[ROCm][Perf] Fold scalar KV scales in
 *     MiniMax-M3 sparse attention", "Test Plan": outputs are compared against a
 *     dequantised reference):
 *       K^[p][d] = dec(code) * ks, ks = per-token k_scale[phys][h][o], or the scalar,
 *       or 1 for a BF16 cache whose values are read exactly.  Same for V^.
 *
 *   Attention.  s_p = sm_scale * sum_d q[d] * K^[p][d] (q read exactly from bf16),
 *     w_p = exp(s_p - max s) / sum exp(s - max s), out[d] = sum_p w_p V^[p][d],
 *     lse = max s + log(sum exp(s - max s)).  An empty key set gives out = 0 and
 *     lse = -inf.
 *
 * dec() is the OCP e4m3fn decoding (bias 7, subnormals 2^-6 * m/8, no infinities,
 * S.1111.111 is NaN, largest finite 448); bf16 is decoded from its bit fields.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_KV_E4M3 0
#define ORACLE_KV_BF16 1
#define ORACLE_SCALE_NONE 0
#define ORACLE_SCALE_SCALAR 1
#define ORACLE_SCALE_PER_TOKEN 2

typedef struct oracle_problem {
  int32_t num_seqs, num_kv_heads, group_size, head_dim, page_size;
  int32_t kv_dtype, scale_mode;
  int64_t num_pages;
  const uint16_t *q;            /* [rows, Hkv*group, D] bf16 bit patterns */
  const void *k_cache;          /* [num_pages, Hkv, page_size, D] e4m3 codes or bf16 bits */
  const void *v_cache;
  const float *k_scale;         /* per-token: [num_pages, Hkv, page_size] */
  const float *v_scale;
  double k_scale_scalar, v_scale_scalar;
  const int32_t *block_table;   /* [num_seqs, bt_stride] */
  int32_t bt_stride;
  const int32_t *context_lens;  /* [num_seqs] */
  const int32_t *cu_seqlens_q;  /* [num_seqs + 1] */
  const int32_t *selected;      /* [num_seqs, sel_stride] logical pages, -1 = padding; NULL = dense */
  int32_t sel_stride;
  const int32_t *num_selected;  /* [num_seqs] */
  double sm_scale;
} oracle_problem;

/* OCP e4m3fn: s eeee mmm. */
double oracle_dec_e4m3(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* bfloat16: s eeeeeeee mmmmmmm (bias 127). */
double oracle_dec_bf16(uint16_t bits) {
  int s = (bits >> 15) & 1;
  int e = (bits >> 7) & 0xFF;
  int m = bits & 0x7F;
  double v;
  if (e == 0xFF) return m ? NAN : (s ? -INFINITY : INFINITY);
  if (e == 0)
    v = ldexp((double)m / 128.0, -126);
  else
    v = ldexp(1.0 + (double)m / 128.0, e - 127);
  return s ? -v : v;
}

/* The set of attended positions for (request r, query token tok): written into keys[],
 * returns the count.  Order: ascending position for dense, selected-list order for
 * sparse.  keys must hold max(context_len, num_selected * page_size) entries. */
static int64_t key_set(const oracle_problem *pb, int r, int tok, int64_t *keys) {
  int64_t L = pb->context_lens[r];
  int64_t qlen = (int64_t)pb->cu_seqlens_q[r + 1] - pb->cu_seqlens_q[r];
  int64_t cut = L - qlen + tok + 1;
  int64_t lim = cut < L ? cut : L;
  int64_t n = 0;
  if (pb->selected == NULL) {
    for (int64_t p = 0; p < lim; ++p) keys[n++] = p;
  } else {
    int64_t ns = pb->num_selected[r];
    for (int64_t i = 0; i < ns; ++i) {
      int64_t sp = pb->selected[(int64_t)r * pb->sel_stride + i];
      if (sp < 0) continue;
      for (int64_t o = 0; o < pb->page_size; ++o) {
        int64_t p = sp * pb->page_size + o;
        if (p < lim) keys[n++] = p;
      }
    }
  }
  return n;
}

/* e4m3 values of all 256 codes, each filled by oracle_dec_e4m3 itself. */
static double e4m3_value[256];
static pthread_once_t e4m3_once = PTHREAD_ONCE_INIT;
static void fill_e4m3_values(void) {
  for (int c = 0; c < 256; ++c) e4m3_value[c] = oracle_dec_e4m3((uint8_t)c);
}

static double dequant(const oracle_problem *pb, const void *cache, const float *scale_pt,
                      double scale_scalar, int64_t phys, int h, int64_t o, int d) {
  int64_t tok_index = (phys * pb->num_kv_heads + h) * pb->page_size + o;
  int64_t idx = tok_index * pb->head_dim + d;
  double x;
  if (pb->kv_dtype == ORACLE_KV_E4M3)
    x = e4m3_value[((const uint8_t *)cache)[idx]];
  else
    x = oracle_dec_bf16(((const uint16_t *)cache)[idx]);
  if (pb->scale_mode == ORACLE_SCALE_PER_TOKEN) return x * (double)scale_pt[tok_index];
  if (pb->scale_mode == ORACLE_SCALE_SCALAR) return x * scale_scalar;
  return x;
}

/* One (request, kv head) pair: all of its rows and query heads. */
static void decode_one(const oracle_problem *pb, int r, int h, double *out, double *lse,
                       int64_t *keys, double *scores, double *qd) {
  const int D = pb->head_dim, g = pb->group_size;
  const int Hq = pb->num_kv_heads * g;
  const int64_t row0 = pb->cu_seqlens_q[r];
  const int qlen = pb->cu_seqlens_q[r + 1] - pb->cu_seqlens_q[r];
  for (int tok = 0; tok < qlen; ++tok) {
    const int64_t row = row0 + tok;
    const int64_t n = key_set(pb, r, tok, keys);
    for (int i = 0; i < g; ++i) {
      const int head = h * g + i;
      const uint16_t *qv = pb->q + (row * Hq + head) * D;
      for (int d = 0; d < D; ++d) qd[d] = oracle_dec_bf16(qv[d]);
      double *o = out + (row * Hq + head) * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (n == 0) {
        if (lse) lse[row * Hq + head] = -INFINITY;
        continue;
      }
      double smax = -INFINITY;
      for (int64_t j = 0; j < n; ++j) {
        const int64_t p = keys[j];
        const int64_t phys = pb->block_table[(int64_t)r * pb->bt_stride + p / pb->page_size];
        const int64_t slot = p % pb->page_size;
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
          acc += qd[d] *
                 dequant(pb, pb->k_cache, pb->k_scale, pb->k_scale_scalar, phys, h, slot, d);
        scores[j] = pb->sm_scale * acc;
        if (scores[j] > smax) smax = scores[j];
      }
      double z = 0.0;
      for (int64_t j = 0; j < n; ++j) z += exp(scores[j] - smax);
      for (int64_t j = 0; j < n; ++j) {
        const int64_t p = keys[j];
        const int64_t phys = pb->block_table[(int64_t)r * pb->bt_stride + p / pb->page_size];
        const int64_t slot = p % pb->page_size;
        const double w = exp(scores[j] - smax) / z;
        for (int d = 0; d < D; ++d)
          o[d] += w * dequant(pb, pb->v_cache, pb->v_scale, pb->v_scale_scalar, phys, h, slot, d);
      }
      if (lse) lse[row * Hq + head] = smax + log(z);
    }
  }
}

typedef struct {
  const oracle_problem *pb;
  double *out, *lse;
  int64_t max_keys;
  int next;
  pthread_mutex_t mu;
  int failed;
} pool_t;

static void *worker(void *arg) {
  pool_t *P = (pool_t *)arg;
  int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(P->max_keys + 1));
  double *scores = (double *)malloc(sizeof(double) * (size_t)(P->max_keys + 1));
  double *qd = (double *)malloc(sizeof(double) * (size_t)P->pb->head_dim);
  if (!keys || !scores || !qd) {
    pthread_mutex_lock(&P->mu);
    P->failed = 1;
    pthread_mutex_unlock(&P->mu);
    free(keys);
    free(scores);
    free(qd);
    return NULL;
  }
  const int items = P->pb->num_seqs * P->pb->num_kv_heads;
  for (;;) {
    pthread_mutex_lock(&P->mu);
    int it = P->next++;
    pthread_mutex_unlock(&P->mu);
    if (it >= items) break;
    decode_one(P->pb, it / P->pb->num_kv_heads, it % P->pb->num_kv_heads, P->out, P->lse, keys,
               scores, qd);
  }
  free(keys);
  free(scores);
  free(qd);
  return NULL;
}

/* Runs the oracle with up to nthreads worker threads over (request, kv head) pairs.
 * out: [rows, Hq, D] fp64; lse: [rows, Hq] fp64 natural-log LSE (may be NULL).
 * Returns 0 on success, -1 on a bad argument or allocation failure. */
int oracle_decode(const oracle_problem *pb, double *out, double *lse, int nthreads) {
  if (!pb || !out || pb->num_seqs < 0 || pb->head_dim <= 0 || pb->group_size <= 0 ||
      pb->num_kv_heads <= 0 || pb->page_size <= 0)
    return -1;
  pthread_once(&e4m3_once, fill_e4m3_values);
  int64_t max_keys = 1;
  for (int r = 0; r < pb->num_seqs; ++r) {
    int64_t n = pb->context_lens[r];
    if (pb->selected) {
      int64_t m = (int64_t)pb->num_selected[r] * pb->page_size;
      if (m > n) n = m;
    }
    if (n > max_keys) max_keys = n;
  }
  pool_t P;
  P.pb = pb;
  P.out = out;
  P.lse = lse;
  P.max_keys = max_keys;
  P.next = 0;
  P.failed = 0;
  pthread_mutex_init(&P.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  pthread_t th[512];
  int started = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, worker, &P) != 0) break;
    ++started;
  }
  if (started == 0) worker(&P);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&P.mu);
  return P.failed ? -1 : 0;
}

/* The attended positions of one (request, query token), in key-set order, for the
 * gather and row-map checks.  Returns the count, or -1 if cap is too small. */
int64_t oracle_key_positions(const oracle_problem *pb, int r, int tok, int64_t *keys,
                             int64_t cap) {
  int64_t need = pb->context_lens[r];
  if (pb->selected) {
    int64_t m = (int64_t)pb->num_selected[r] * pb->page_size;
    if (m > need) need = m;
  }
  if (need > cap) return -1;
  return key_set(pb, r, tok, keys);
}

/* ------------------------------------------------------------------------------------
 * KV quantise-and-write: the producer of the per-token FP8 cache that the decode reads
 * (ROCm/ATOM PR 2614: MiniMax-M3 writes FP8 KV plus per-token K/V scales, and the
 * "Validation" section runs a producer-to-consumer operator test; the cache-write branch
 * of ATOM PR 2710, "Smaller").
 *
 * For every new token t whose slot s = slot_mapping[t] is >= 0 and every KV head h:
 *   page = s / page_size, o = s % page_size, row = (page * Hkv + h) * page_size + o;
 *   x = the token's head_dim values (bf16, read exactly);
 *   amax = max |x| and scale = amax / 448 (448: largest finite e4m3fn value), rounded
 *   once to fp32: the scale that is stored, and the one the decode multiplies by;
 *   code[d] = the e4m3fn value nearest to the exact real quotient x[d] / scale (ties to
 *   an even mantissa), saturated to +-448; all zero when scale is 0;
 *   k_scale[row] = scale, k_cache[row * D + d] = code[d] (V the same).
 * The quotient is taken in double: x (8 significant bits) and scale (24) are exact
 * there, and a quotient that is not exactly an e4m3 rounding midpoint lies at least
 * 2^-29 (relative) away from it, far beyond the 2^-53 rounding of the double division,
 * so the double quotient falls on the same side of every midpoint as the real one, and
 * on the midpoint itself exactly when the real one does.  (An fp32 product with
 * 448 / amax, or an fp32 quotient rounded before the e4m3 rounding, can differ from it
 * where x / scale is within an fp32 ulp of a midpoint.)
 * Slots >= num_pages * page_size are skipped and counted in the return value.
 * ------------------------------------------------------------------------------------ */

/* Nearest e4m3fn code to the real value x (ties to even mantissa), saturating to +-448.
 * NaN gives the NaN code 0x7F. */
uint8_t oracle_enc_e4m3(double x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: multiples of 2^-9; m = 8 is the smallest normal, code 0x08 */
    double m = nearbyint(ldexp(a, 9));  /* current rounding mode: to nearest, ties even */
    return sign | (uint8_t)m;
  }
  int e;
  (void)frexp(a, &e);  /* a = f * 2^e, f in [0.5, 1) -> a in [2^(e-1), 2^e) */
  int ex = e - 1;      /* unbiased exponent, -6 .. 8 */
  double m = nearbyint((ldexp(a, -ex) - 1.0) * 8.0);  /* the shift and the -1 are exact */
  if (m == 8.0) {
    m = 0.0;
    ++ex;
  }
  if (ex > 8 || (ex == 8 && m > 6.0)) return sign | 0x7E;  /* above 448: saturate */
  return sign | (uint8_t)(((ex + 7) << 3) | (int)m);
}

static float bf16_to_f32(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static void quantize_row(const uint16_t *x, int D, uint8_t *code, float *scale) {
  float amax = 0.0f;
  for (int d = 0; d < D; ++d) {
    float a = fabsf(bf16_to_f32(x[d]));
    if (a > amax) amax = a;
  }
  volatile float s = amax / 448.0f;  /* one fp32 division, stored as fp32 */
  *scale = s;
  for (int d = 0; d < D; ++d) {
    if (s == 0.0f) {  /* amax = 0 (or amax / 448 below the fp32 range): nothing to encode */
      code[d] = 0;
      continue;
    }
    const double q = (double)bf16_to_f32(x[d]) / (double)s;  /* the real quotient's side */
    code[d] = oracle_enc_e4m3(q);
  }
}

int64_t oracle_kv_quantize_write(const uint16_t *k_new, const uint16_t *v_new,
                                 const int64_t *slot_mapping, int64_t num_tokens,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                 int64_t num_pages, uint8_t *k_cache, uint8_t *v_cache,
                                 float *k_scale, float *v_scale) {
  int64_t bad = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;
    if (s >= num_pages * page_size) {
      ++bad;
      continue;
    }
    const int64_t page = s / page_size, o = s % page_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      const int64_t row = (page * num_kv_heads + h) * page_size + o;
      const int64_t src = (t * num_kv_heads + h) * head_dim;
      quantize_row(k_new + src, head_dim, k_cache + row * head_dim, k_scale + row);
      quantize_row(v_new + src, head_dim, v_cache + row * head_dim, v_scale + row);
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------------------
 * Indexer block score and top-k page selection: the step that produces the selected
 * pages of the sparse decode (ROCm/ATOM PR 2122, section 1: the index cache holds
 * (num_blocks, 128, 128) e4m3 codes and the block-score kernel takes q . k scaled by
 * sm_scale * log2(e); section 2: the index top-k maps rows to requests through
 * cu_seqlens_q with the cutoff seq_len - q_len + tok + 1).
 *
 * For query row tok of request r (cutoff c = L - q_len + tok + 1, limit = min(L, c)):
 *   s[h][p] = sm_scale * log2(e) * sum_d q[row][h][d] * K^[p][d], K^ = dec(code) * scale
 *     (per-token index scale, or 1), for attended positions p < limit;
 *   S[b] = log2( sum_h sum_{p in page b, p < limit} 2^s[h][p] ) for every page b holding
 *     an attended position (the candidates);
 *   selected[row] = the page holding position limit - 1 first, then the other candidates
 *     by descending S (equal scores: lower page first), topk entries at most, -1 after;
 *   num_selected[row] = their count.  S itself is returned too.
 * ------------------------------------------------------------------------------------ */
typedef struct oracle_index_problem {
  int32_t num_seqs, index_heads, head_dim, page_size, topk;
  int64_t num_pages;
  const uint16_t *q;            /* [rows, index_heads, D] bf16 bits */
  const uint8_t *k_cache;       /* [num_pages, page_size, D] e4m3 codes */
  const float *k_scale;         /* [num_pages, page_size] or NULL */
  const int32_t *block_table;   /* [num_seqs, bt_stride] */
  int32_t bt_stride;
  const int32_t *context_lens;
  const int32_t *cu_seqlens_q;
  double sm_scale;
} oracle_index_problem;

int oracle_index_topk(const oracle_index_problem *pb, int32_t *selected, int32_t *num_selected,
                      double *scores, int32_t scores_stride) {
  const int D = pb->head_dim, ps = pb->page_size, H = pb->index_heads;
  const double log2e = 1.4426950408889634074;
  for (int r = 0; r < pb->num_seqs; ++r) {
    const int64_t L = pb->context_lens[r];
    const int64_t row0 = pb->cu_seqlens_q[r], qlen = pb->cu_seqlens_q[r + 1] - row0;
    for (int64_t tok = 0; tok < qlen; ++tok) {
      const int64_t row = row0 + tok;
      int64_t lim = L - qlen + tok + 1;
      if (lim > L) lim = L;
      if (lim < 0) lim = 0;
      const int64_t nb = (lim + ps - 1) / ps;
      if (nb > scores_stride) return -1;
      double *S = scores + row * scores_stride;
      for (int64_t b = 0; b < scores_stride; ++b) S[b] = -INFINITY;
      for (int64_t b = 0; b < nb; ++b) {
        const int64_t phys = pb->block_table[(int64_t)r * pb->bt_stride + b];
        double m = -INFINITY;
        int64_t n = (b + 1) * ps <= lim ? ps : lim - b * ps;
        double *s = (double *)malloc(sizeof(double) * (size_t)(n * H));
        if (!s) return -1;
        for (int h = 0; h < H; ++h) {
          const uint16_t *q = pb->q + (row * H + h) * D;
          for (int64_t o = 0; o < n; ++o) {
            const uint8_t *k = pb->k_cache + ((int64_t)phys * ps + o) * D;
            const double ks = pb->k_scale ? (double)pb->k_scale[(int64_t)phys * ps + o] : 1.0;
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += oracle_dec_bf16(q[d]) * (oracle_dec_e4m3(k[d]) * ks);
            const double v = pb->sm_scale * log2e * acc;
            s[h * n + o] = v;
            if (v > m) m = v;
          }
        }
        double z = 0.0;
        for (int64_t i = 0; i < n * H; ++i) z += exp2(s[i] - m);
        free(s);
        S[b] = m + log2(z);
      }
      /* selection: the last attended page first, then by descending score */
      int32_t *sel = selected + row * pb->topk;
      for (int i = 0; i < pb->topk; ++i) sel[i] = -1;
      int cnt = 0;
      if (nb > 0 && pb->topk > 0) sel[cnt++] = (int32_t)(nb - 1);
      while (cnt < pb->topk) {
        int64_t best = -1;
        for (int64_t b = 0; b < nb; ++b) {
          int taken = 0;
          for (int i = 0; i < cnt; ++i)
            if (sel[i] == b) taken = 1;
          if (taken) continue;
          if (best < 0 || S[b] > S[best]) best = b;  /* strict: equal scores keep the lower page */
        }
        if (best < 0) break;
        sel[cnt++] = (int32_t)best;
      }
      num_selected[row] = cnt;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------------------
 * Log-sum-exp merge of attention partials: the combine step of a context split across
 * GPUs, where each GPU attends a disjoint part of a request's positions and the parts'
 * (normalised output, lse) are gathered and merged (the partition scratch of ROCm/ATOM
 * PR 2710, "Smaller": max logits, exp sums and partial outputs per partition, merged into
 * one output; one step further out, across GPUs).
 *
 * For every (row, head) v, over the parts i = 0 .. num_parts - 1 with lse_i > -inf:
 *   M = max_i lse_i,  w_i = exp(lse_i - M),
 *   out[v][d] = sum_i w_i * o_i[v][d] / sum_i w_i,   lse[v] = M + log(sum_i w_i).
 * With every lse_i = -inf (no part attended anything): out = 0 and lse = -inf.
 * Attention over a union of disjoint key sets is exactly this merge of the parts'
 * attentions, since lse_i = log sum_{p in part i} exp(s_p) and o_i is the part's
 * exp(s_p - lse_i)-weighted mean of V.
 * ------------------------------------------------------------------------------------ */
void oracle_lse_merge(const double *part_out, const double *part_lse, int32_t num_parts,
                      int64_t num_vecs, int32_t dim, double *out, double *lse) {
  for (int64_t v = 0; v < num_vecs; ++v) {
    double M = -INFINITY;
    for (int32_t i = 0; i < num_parts; ++i) {
      const double l = part_lse[(int64_t)i * num_vecs + v];
      if (l > M) M = l;
    }
    double *o = out + v * dim;
    for (int32_t d = 0; d < dim; ++d) o[d] = 0.0;
    if (M == -INFINITY) {
      lse[v] = -INFINITY;
      continue;
    }
    double z = 0.0;
    for (int32_t i = 0; i < num_parts; ++i) {
      const double l = part_lse[(int64_t)i * num_vecs + v];
      if (l == -INFINITY) continue;
      const double w = exp(l - M);
      z += w;
      const double *oi = part_out + ((int64_t)i * num_vecs + v) * dim;
      for (int32_t d = 0; d < dim; ++d) o[d] += w * oi[d];
    }
    for (int32_t d = 0; d < dim; ++d) o[d] /= z;
    lse[v] = M + log(z);
  }
}
