/*
 * Ragged paged attention: plain CPU oracle (TEST INFRASTRUCTURE ONLY).
 *
 * This file is the slow, obviously-correct definition that the CUDA library
 * is checked against.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load it; the product path never does.  It shares no code,
 * header or constant with the CUDA library.
 *
 * Everything is computed in double precision with plain loops, in the order
 * the definitions are stated:
 *
 *   - oracle_e4m3_decode / oracle_e4m3_encode: the OCP FP8 E4M3 ("fn") format
 *     (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 *     S.1111.111 is NaN, largest finite 448).  Encoding rounds to nearest,
 *     ties to even, and saturates to +-448 (the "satfinite" reading).
 *     Used by the fp8 KV-cache path: new keys/values are quantised as
 *     x / k_scale before they enter the cache, and read back as code * scale
 *     (tpu-inference 0.11.1rc3, layers/vllm/attention.py,
 *     PallasAttentionBackendImpl.forward: quantize_kv with k_scale/v_scale).
 *
 *   - oracle_update_cache: the new-KV page write.  Token i of sequence s sits
 *     at absolute position ctx + i with ctx = kv_len - q_len (vLLM 0.10.2
 *     differential_flash_attn.py, metadata: seq_len = context_len +
 *     query_len); its page is block_tables[s * pages_per_seq + pos / P] and
 *     its row in the page is pos % P (tpu-inference 0.12.0 RPA v3 kernel.py,
 *     _update_kv_cache).  Key head h goes to channel 2h, value head h to
 *     channel 2h+1 ("k and v are packed together", same kernel, kv-head loop).
 *
 *   - oracle_attention_rows: exact softmax attention per (token, q-head):
 *     GQA head map h = hq / (Hq/Hkv); score s_j = softmax_scale * (q . k_j)
 *     (k_j dequantised with k_scale for fp8 -- or, when per-head scales
 *     are given, with the scale of kv head h; likewise v_scale); optional
 *     soft cap
 *     s = cap * tanh(s / cap); causal mask j <= pos; sliding window keeps
 *     pos - j < W (vLLM's window_size = (W-1, 0)); an optional per-q-head
 *     sink logit joins the softmax denominator with no value vector
 *     (ejkernel ragged_page_attention_v3 interface: attention_sink
 *     [num_q_heads]); output = sum_j softmax_j * v_j (v dequantised with
 *     v_scale).  The online-softmax recurrence of the RPA v3 kernel
 *     (flash_attention_step1_qk_softmax / step2_pv) reaches this same value
 *     up to rounding, so the oracle writes the two-pass definition out.
 *
 *   - q_scale (fp8 caches, optional: w8a8 attention, the ejkernel
 *     interface's q_scale, left disabled by tpu-inference 0.11.1rc3
 *     layers/vllm/attention.py): when q_scale > 0 every query element is
 *     quantised exactly as keys are (x / q_scale in fp32, E4M3 round to
 *     nearest even, saturating) and read back as code * q_scale, so the
 *     logit is softmax_scale * q_scale * k_scale * (q_codes . k_codes).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Parameters as the oracle sees them (its own struct, not the library's). */
typedef struct {
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t num_pages;
  int32_t pages_per_seq;
  int32_t max_num_seqs;
  int32_t total_tokens;
  int32_t kv_fp8;          /* 0: bf16 cache, 1: fp8 e4m3 cache            */
  int32_t sliding_window;  /* 0: none                                     */
  double softmax_scale;
  double logits_soft_cap;  /* 0: none                                     */
  double k_scale;          /* fp8 only; the values are fp32 numbers       */
  double v_scale;
  const double* k_scale_heads;  /* fp8 only, optional: [num_kv_heads] scales  */
  const double* v_scale_heads;  /* that replace k_scale / v_scale per head   */
  double q_scale;               /* fp8 only: > 0 quantises the queries; 0 = off */
} oracle_params;

/* The key / value scale of kv head h. */
static double key_scale(const oracle_params* p, int h) {
  return p->k_scale_heads ? p->k_scale_heads[h] : p->k_scale;
}
static double value_scale(const oracle_params* p, int h) {
  return p->v_scale_heads ? p->v_scale_heads[h] : p->v_scale;
}

enum {
  ORACLE_OK = 0,
  ORACLE_BAD_ARG = 1,        /* shapes / options                          */
  ORACLE_BAD_METADATA = 2,   /* query_start_loc, kv_lens, distribution    */
  ORACLE_BAD_PAGE = 3,       /* block_tables entry outside the pool       */
};

/* ---------------------------------------------------------------- formats */

/* bf16 is the top half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* E4M3 (fn) code -> value. */
double oracle_e4m3_decode(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);          /* subnormal: 0.m * 2^(1-7) */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: 1.m * 2^(e-7)     */
  return sign ? -v : v;
}

/* Value (an fp32 number) -> E4M3 code, round to nearest even, saturating. */
uint8_t oracle_e4m3_encode(float xf) {
  double x = (double)xf;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);  /* satfinite             */
  /* Binade [2^E, 2^(E+1)); below the smallest normal 2^-6 the spacing stays
   * that of the subnormals, 2^-9. */
  int e2;
  frexp(a, &e2);
  int E = e2 - 1;
  if (E < -6) E = -6;
  double quantum = ldexp(1.0, E - 3);
  double r = nearbyint(a / quantum);  /* exact quotient; default mode = RNE */
  double v = r * quantum;             /* a < 448 never rounds above 448    */
  if (v < ldexp(1.0, -6)) {
    int m = (int)(v / ldexp(1.0, -9));  /* 0..8; 8 is never reached here   */
    return (uint8_t)(sign | m);
  }
  frexp(v, &e2);
  E = e2 - 1;
  int m = (int)((v / ldexp(1.0, E) - 1.0) * 8.0);
  return (uint8_t)(sign | ((E + 7) << 3) | m);
}

/* fp8 quantisation of one new key/value element: the bf16 input divided by
 * the fp32 scale in fp32 (a double divide rounded once to float gives the
 * correctly rounded fp32 quotient), then E4M3 encoding. */
uint8_t oracle_quantize(uint16_t bf16_bits, double scale) {
  double q = oracle_bf16_to_double(bf16_bits) / (double)(float)scale;
  return oracle_e4m3_encode((float)q);
}

/* ------------------------------------------------------------- validation */

static int check_params(const oracle_params* p) {
  if (p->num_q_heads <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0 ||
      p->page_size <= 0 || p->num_pages <= 0 || p->pages_per_seq <= 0 ||
      p->max_num_seqs <= 0 || p->total_tokens < 0)
    return ORACLE_BAD_ARG;
  if (p->num_q_heads % p->num_kv_heads != 0) return ORACLE_BAD_ARG;
  if (p->sliding_window < 0 || p->logits_soft_cap < 0.0) return ORACLE_BAD_ARG;
  if (p->kv_fp8 && (!(p->k_scale > 0.0) || !(p->v_scale > 0.0)))
    return ORACLE_BAD_ARG;
  if (!p->kv_fp8 && (p->k_scale_heads || p->v_scale_heads)) return ORACLE_BAD_ARG;
  if (!(p->q_scale >= 0.0) || (p->q_scale > 0.0 && !p->kv_fp8)) return ORACLE_BAD_ARG;
  for (int h = 0; h < p->num_kv_heads; ++h)
    if (!(key_scale(p, h) > 0.0) || !(value_scale(p, h) > 0.0)) return ORACLE_BAD_ARG;
  return ORACLE_OK;
}

/* Checks the ragged metadata of num_seqs sequences and every block-table
 * entry that the call reads or writes. */
static int check_metadata(const oracle_params* p, const int32_t* kv_lens,
                          const int32_t* block_tables,
                          const int32_t* query_start_loc, int32_t num_seqs) {
  if (num_seqs < 0 || num_seqs > p->max_num_seqs) return ORACLE_BAD_METADATA;
  if (query_start_loc[0] != 0) return ORACLE_BAD_METADATA;
  for (int s = 0; s < num_seqs; ++s) {
    int32_t q_len = query_start_loc[s + 1] - query_start_loc[s];
    if (q_len < 0) return ORACLE_BAD_METADATA;
    if (kv_lens[s] < q_len) return ORACLE_BAD_METADATA;
    if ((int64_t)kv_lens[s] > (int64_t)p->pages_per_seq * p->page_size)
      return ORACLE_BAD_METADATA;
  }
  if (query_start_loc[num_seqs] > p->total_tokens) return ORACLE_BAD_METADATA;
  for (int s = 0; s < num_seqs; ++s) {
    int32_t used = (kv_lens[s] + p->page_size - 1) / p->page_size;
    for (int k = 0; k < used; ++k) {
      int32_t page = block_tables[(int64_t)s * p->pages_per_seq + k];
      if (page < 0 || page >= p->num_pages) return ORACLE_BAD_PAGE;
    }
  }
  return ORACLE_OK;
}

/* distribution = cumulative ends of the decode-only, chunked-prefill and
 * mixed classes; the oracle only checks it (results never depend on it). */
int oracle_check_distribution(const oracle_params* p, const int32_t* dist,
                              const int32_t* query_start_loc) {
  if (!(0 <= dist[0] && dist[0] <= dist[1] && dist[1] <= dist[2] &&
        dist[2] <= p->max_num_seqs))
    return ORACLE_BAD_METADATA;
  for (int s = 0; s < dist[0]; ++s)
    if (query_start_loc[s + 1] - query_start_loc[s] != 1)
      return ORACLE_BAD_METADATA;
  return ORACLE_OK;
}

/* --------------------------------------------------------------- indexing */

/* Byte offset of (page, row, channel, 0) in the pool
 * [num_pages, page_size, 2*num_kv_heads, head_dim]. */
static int64_t cache_offset(const oracle_params* p, int64_t page, int64_t row,
                            int64_t channel) {
  int64_t elem = p->kv_fp8 ? 1 : 2;
  int64_t channels = 2 * (int64_t)p->num_kv_heads;
  return (((page * p->page_size + row) * channels + channel) * p->head_dim) *
         elem;
}

static int64_t page_of(const oracle_params* p, const int32_t* block_tables,
                       int s, int64_t pos) {
  return block_tables[(int64_t)s * p->pages_per_seq + pos / p->page_size];
}

/* One element of the pool, as the real number it stands for. */
static double cache_value(const oracle_params* p, const uint8_t* cache,
                          int64_t off_bytes, int d, double fp8_scale) {
  if (p->kv_fp8) return oracle_e4m3_decode(cache[off_bytes + d]) * fp8_scale;
  uint16_t bits;
  memcpy(&bits, cache + off_bytes + 2 * (int64_t)d, 2);
  return oracle_bf16_to_double(bits);
}

/* ------------------------------------------------------------ cache write */

int oracle_update_cache(const oracle_params* p, const uint16_t* keys,
                        const uint16_t* values, uint8_t* kv_cache,
                        const int32_t* kv_lens, const int32_t* block_tables,
                        const int32_t* query_start_loc, int32_t num_seqs) {
  int rc = check_params(p);
  if (rc) return rc;
  rc = check_metadata(p, kv_lens, block_tables, query_start_loc, num_seqs);
  if (rc) return rc;
  const int Hkv = p->num_kv_heads, D = p->head_dim;
  for (int s = 0; s < num_seqs; ++s) {
    int32_t q0 = query_start_loc[s];
    int32_t q_len = query_start_loc[s + 1] - q0;
    int32_t ctx = kv_lens[s] - q_len;
    for (int i = 0; i < q_len; ++i) {
      int64_t pos = (int64_t)ctx + i;
      int64_t page = page_of(p, block_tables, s, pos);
      int64_t row = pos % p->page_size;
      for (int h = 0; h < Hkv; ++h) {
        const uint16_t* k = keys + ((int64_t)(q0 + i) * Hkv + h) * D;
        const uint16_t* v = values + ((int64_t)(q0 + i) * Hkv + h) * D;
        int64_t ok = cache_offset(p, page, row, 2 * h);
        int64_t ov = cache_offset(p, page, row, 2 * h + 1);
        for (int d = 0; d < D; ++d) {
          if (p->kv_fp8) {
            kv_cache[ok + d] = oracle_quantize(k[d], key_scale(p, h));
            kv_cache[ov + d] = oracle_quantize(v[d], value_scale(p, h));
          } else {
            memcpy(kv_cache + ok + 2 * (int64_t)d, &k[d], 2);
            memcpy(kv_cache + ov + 2 * (int64_t)d, &v[d], 2);
          }
        }
      }
    }
  }
  return ORACLE_OK;
}

/* -------------------------------------------------------------- attention */

/* Attention for the listed query tokens (all q-heads of each), reading keys
 * and values from an already-updated pool.  out is [num_rows, Hq, D]. */
int oracle_attention_rows(const oracle_params* p, const uint16_t* queries,
                          const uint8_t* kv_cache, const int32_t* kv_lens,
                          const int32_t* block_tables,
                          const int32_t* query_start_loc, int32_t num_seqs,
                          const float* attention_sink, const int32_t* tokens,
                          int32_t num_rows, double* out, int32_t nthreads) {
  int rc = check_params(p);
  if (rc) return rc;
  rc = check_metadata(p, kv_lens, block_tables, query_start_loc, num_seqs);
  if (rc) return rc;
  const int Hq = p->num_q_heads, Hkv = p->num_kv_heads, D = p->head_dim;
  const int group = Hq / Hkv;
  const int32_t n_tok = query_start_loc[num_seqs];
  for (int r = 0; r < num_rows; ++r)
    if (tokens[r] < 0 || tokens[r] >= n_tok) return ORACLE_BAD_ARG;

  int64_t max_kv = 1;
  for (int s = 0; s < num_seqs; ++s)
    if (kv_lens[s] > max_kv) max_kv = kv_lens[s];

#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int failed = 0;
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)max_kv);
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);  /* the query's values */
    if (!scores || !qv) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t w = 0; w < (int64_t)num_rows * Hq; ++w) {
      if (!scores || !qv) continue;
      int r = (int)(w / Hq), hq = (int)(w % Hq);
      int32_t t = tokens[r];
      int s = 0;  /* the sequence whose query range holds token t */
      while (query_start_loc[s + 1] <= t) ++s;
      int32_t q_len = query_start_loc[s + 1] - query_start_loc[s];
      int64_t ctx = (int64_t)kv_lens[s] - q_len;
      int64_t pos = ctx + (t - query_start_loc[s]);
      int h = hq / group;
      int64_t lo = 0;
      if (p->sliding_window > 0 && pos - p->sliding_window + 1 > 0)
        lo = pos - p->sliding_window + 1;
      const uint16_t* q = queries + ((int64_t)t * Hq + hq) * D;
      /* the query as the scores see it: bf16 values, or with q_scale the
       * e4m3 codes of q / q_scale read back as code * q_scale */
      for (int d = 0; d < D; ++d)
        qv[d] = p->q_scale > 0.0
                    ? oracle_e4m3_decode(oracle_quantize(q[d], p->q_scale)) *
                          (double)(float)p->q_scale
                    : oracle_bf16_to_double(q[d]);

      /* pass 1: logits and their maximum */
      double m = -INFINITY;
      for (int64_t j = lo; j <= pos; ++j) {
        int64_t off = cache_offset(p, page_of(p, block_tables, s, j),
                                   j % p->page_size, 2 * h);
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
          dot += qv[d] * cache_value(p, kv_cache, off, d, key_scale(p, h));
        double sc = p->softmax_scale * dot;
        if (p->logits_soft_cap > 0.0)
          sc = p->logits_soft_cap * tanh(sc / p->logits_soft_cap);
        scores[j - lo] = sc;
        if (sc > m) m = sc;
      }
      double sink = 0.0;
      if (attention_sink) {
        sink = (double)attention_sink[hq];
        if (sink > m) m = sink;
      }
      /* pass 2: normaliser and weighted sum of values */
      double den = attention_sink ? exp(sink - m) : 0.0;
      double* o = out + ((int64_t)r * Hq + hq) * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (int64_t j = lo; j <= pos; ++j) {
        double e = exp(scores[j - lo] - m);
        den += e;
        int64_t off = cache_offset(p, page_of(p, block_tables, s, j),
                                   j % p->page_size, 2 * h + 1);
        for (int d = 0; d < D; ++d)
          o[d] += e * cache_value(p, kv_cache, off, d, value_scale(p, h));
      }
      for (int d = 0; d < D; ++d) o[d] /= den;
    }
    free(scores);
    free(qv);
  }
  return failed ? ORACLE_BAD_ARG : ORACLE_OK;
}

/* The whole call: write the new KV into the pool, then attend every query
 * token of the num_seqs sequences.  out is [query_start_loc[num_seqs], Hq, D]. */
int oracle_forward(const oracle_params* p, const uint16_t* queries,
                   const uint16_t* keys, const uint16_t* values,
                   uint8_t* kv_cache, const int32_t* kv_lens,
                   const int32_t* block_tables, const int32_t* query_start_loc,
                   int32_t num_seqs, const float* attention_sink, double* out,
                   int32_t nthreads) {
  int rc = oracle_update_cache(p, keys, values, kv_cache, kv_lens,
                               block_tables, query_start_loc, num_seqs);
  if (rc) return rc;
  int32_t n = query_start_loc[num_seqs];
  int32_t* tokens = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  if (!tokens) return ORACLE_BAD_ARG;
  for (int32_t t = 0; t < n; ++t) tokens[t] = t;
  rc = oracle_attention_rows(p, queries, kv_cache, kv_lens, block_tables,
                             query_start_loc, num_seqs, attention_sink, tokens,
                             n, out, nthreads);
  free(tokens);
  return rc;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
