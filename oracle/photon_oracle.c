/*
 * photon_oracle.c -- plain, slow, fp64 CPU oracle for one decode step of
 * batched paged attention over a block-level KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * What it follows (PhotonInfer README, the zh-CN / fr / ja pages of the same
 * project):
 *   - "Technical details > Paged attention": a block-level KV cache, per-
 *     sequence cache offsets, one batched operation that writes K/V for many
 *     sequences.
 *   - "Key features > GPU-optimised kernels": batched RoPE, numerically stable
 *     softmax for attention.
 * Readings where the pages are silent (stated in full in the design notes):
 *   - cache layout [num_blocks, num_kv_heads, block_size, head_dim], K and V
 *     in separate pools; element (b,h,o,e) at ((b*H_kv+h)*bs+o)*d+e;
 *   - a token's physical slot is block_tables[s][p / bs] * bs + p % bs;
 *     slot -1 means "do not write";
 *   - RoPE "NEOX" pairs (i, i+d/2), "GPTJ" pairs (2i, 2i+1), angle
 *     position * theta^(-2i/d); K is rotated, V is copied unchanged;
 *   - GQA: query head g reads KV head g / (H_q / H_kv);
 *   - context_lens counts the token written in this step; ctx <= 0 gives a
 *     zero output row.
 *
 * Arithmetic: every value is widened exactly to double, the softmax is the
 * two-pass textbook form (max, exp, sum, normalise), and results are rounded
 * once, to nearest-even, into the storage type.  No blocking, fusion or
 * reordering beyond those definitions.  OpenMP spreads independent
 * (sequence, query-head) rows over host cores; each row is computed
 * sequentially, so the result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F64 3

#define ORC_ROPE_NEOX 0
#define ORC_ROPE_GPTJ 1
#define ORC_ROPE_NONE 2

/* ---- storage types ---------------------------------------------------- */

static double orc_load(const void *base, int64_t idx, int dtype) {
  if (dtype == ORC_F64) return ((const double *)base)[idx];
  if (dtype == ORC_F32) return (double)((const float *)base)[idx];
  uint32_t u = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Nearest bf16 to x, ties to even, in a single rounding step (no detour
 * through float, which would round twice).  bf16 keeps 8 significant bits
 * and float's exponent range; below 2^-126 the spacing is fixed at 2^-133. */
uint16_t orc_round_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double ax = fabs(x);
  if (ax == 0.0) return sign;
  int ex;
  frexp(ax, &ex);                  /* ax = m * 2^ex, m in [0.5, 1) */
  int qexp = ex - 8;               /* spacing of 8-significant-bit numbers */
  if (qexp < -133) qexp = -133;
  double q = ldexp(1.0, qexp);
  double r = nearbyint(ax / q) * q;  /* default rounding mode: to even */
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  float f = (float)r;              /* exact: r has <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (u >> 16));
}

static void orc_store(void *base, int64_t idx, int dtype, double x) {
  if (dtype == ORC_F64)
    ((double *)base)[idx] = x;
  else if (dtype == ORC_F32)
    ((float *)base)[idx] = (float)x; /* C conversion: round to nearest even */
  else
    ((uint16_t *)base)[idx] = orc_round_bf16(x);
}

static size_t orc_size(int dtype) { return dtype == ORC_F64 ? 8 : (dtype == ORC_F32 ? 4 : 2); }

/* ---- FP8 E4M3 (sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; 0x7F / 0xFF are NaN; largest finite 448; subnormal spacing
 * 2^-9) ---------------------------------------------------------------------- */

double orc_fp8_decode(uint8_t b) {
  int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return NAN;
  double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
  return sign ? -v : v;
}

/* Nearest E4M3 to x, ties to even; magnitudes beyond the largest finite
 * value (448) saturate to it; NaN stays NaN. */
uint8_t orc_fp8_encode(double x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double ax = fabs(x);
  if (ax >= 448.0) return (uint8_t)(sign | 0x7E);
  int ex;
  frexp(ax, &ex);                      /* ax = f * 2^ex, f in [0.5, 1) */
  int qexp = ex - 4;                   /* spacing of 4-significant-bit numbers */
  if (qexp < -9) qexp = -9;            /* subnormal spacing */
  double q = ldexp(1.0, qexp);
  double r = nearbyint(ax / q) * q;    /* <= 448: ax < 448 rounds to at most 448 */
  if (r == 0.0) return sign;
  if (r < ldexp(1.0, -6)) return (uint8_t)(sign | (int)(r / ldexp(1.0, -9)));
  int re;
  double f = frexp(r, &re);            /* r = f * 2^re, f in [0.5, 1) */
  int e = re - 1 + 7;
  int m = (int)(f * 16.0) - 8;
  return (uint8_t)(sign | (e << 3) | m);
}

/* ---- slot mapping ------------------------------------------------------ */

/* Physical slot of token position p of sequence s:
 * block_tables[s][p / bs] * bs + p % bs; -1 when p < 0, when p lies past the
 * row, or when the row entry is -1 (no block). */
void orc_slot_mapping(const int32_t *block_tables, int32_t max_blocks_per_seq,
                      const int32_t *token_seq, const int32_t *positions,
                      int32_t num_tokens, int32_t block_size, int64_t *slots) {
  for (int32_t t = 0; t < num_tokens; ++t) {
    int32_t s = token_seq[t], p = positions[t];
    int64_t slot = -1;
    if (s >= 0 && p >= 0 && p / block_size < max_blocks_per_seq) {
      int32_t blk = block_tables[(int64_t)s * max_blocks_per_seq + p / block_size];
      if (blk >= 0) slot = (int64_t)blk * block_size + p % block_size;
    }
    slots[t] = slot;
  }
}

/* ---- RoPE -------------------------------------------------------------- */

/* Rotates one head vector x[0..d) in place, at integer position pos. */
void orc_rope(double *x, int32_t d, int32_t pos, double theta, int style) {
  if (style == ORC_ROPE_NONE) return;
  for (int32_t i = 0; i < d / 2; ++i) {
    double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
    double a = (double)pos * inv_freq;
    double c = cos(a), s = sin(a);
    int32_t i0 = style == ORC_ROPE_NEOX ? i : 2 * i;
    int32_t i1 = style == ORC_ROPE_NEOX ? i + d / 2 : 2 * i + 1;
    double x0 = x[i0], x1 = x[i1];
    x[i0] = x0 * c - x1 * s;
    x[i1] = x1 * c + x0 * s;
  }
}

/* ---- batched cache write ----------------------------------------------- */

/* For every token t with slot_mapping[t] >= 0 and every KV head h:
 *   k_cache[slot/bs, h, slot%bs, :] = round(RoPE(k[t,h,:], positions[t]))
 *   v_cache[slot/bs, h, slot%bs, :] = v[t,h,:]   (bit copy)
 * k, v: [T, H_kv, d]; caches: [num_blocks, H_kv, bs, d]; all in `dtype`.
 * Returns 0, or -1 if a slot falls outside the pool. */
int orc_kv_cache_write(const void *k, const void *v, const int32_t *positions,
                       const int64_t *slot_mapping, void *k_cache, void *v_cache,
                       int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size, int64_t num_blocks, int dtype,
                       double rope_theta, int rope_style) {
  size_t es = orc_size(dtype);
  double *x = (double *)malloc(sizeof(double) * (size_t)head_dim);
  int rc = 0;
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t blk = slot / block_size, off = slot % block_size;
    if (blk >= num_blocks) { rc = -1; continue; }
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
      int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim;
      for (int32_t e = 0; e < head_dim; ++e) x[e] = orc_load(k, src + e, dtype);
      orc_rope(x, head_dim, positions[t], rope_theta, rope_style);
      for (int32_t e = 0; e < head_dim; ++e) orc_store(k_cache, dst + e, dtype, x[e]);
      memcpy((char *)v_cache + dst * es, (const char *)v + src * es, es * (size_t)head_dim);
    }
  }
  free(x);
  return rc;
}

/* Query rows rotated in place: x[r][h][:] = round(RoPE(x[r][h][:], positions[r]))
 * for r < n_rows, h < heads; x in `dtype` storage. */
void orc_rope_rows(void *x, const int32_t *positions, int32_t n_rows, int32_t heads,
                   int32_t head_dim, int dtype, double rope_theta, int rope_style) {
  double *t = (double *)malloc(sizeof(double) * (size_t)head_dim);
  for (int32_t r = 0; r < n_rows; ++r)
    for (int32_t h = 0; h < heads; ++h) {
      int64_t base = ((int64_t)r * heads + h) * head_dim;
      for (int32_t e = 0; e < head_dim; ++e) t[e] = orc_load(x, base + e, dtype);
      orc_rope(t, head_dim, positions[r], rope_theta, rope_style);
      for (int32_t e = 0; e < head_dim; ++e) orc_store(x, base + e, dtype, t[e]);
    }
  free(t);
}

/* ---- FP8 cache (per-KV-head scales) ------------------------------------
 * K pool: [num_blocks][H_kv][bs][d] E4M3 codes, value = decode(code) * k_scale[h].
 * V pool: [num_blocks][H_kv][d][bs] E4M3 codes (dims outer, the block's bs
 *         tokens inner), value = decode(code) * v_scale[h].
 * The write divides by the scale and rounds once: code = orc_fp8_encode(x / scale)
 * with x = RoPE(k) (K) or v (V) and the quotient taken in fp64.  For float x
 * and scale the fp64 quotient is the correctly rounded quotient, and an exact
 * quotient that is not itself an E4M3 rounding boundary lies at least ~2^-30
 * (relative) from one, far beyond fp64's 2^-53: the code is the nearest E4M3
 * to the exact quotient, ties (exact midpoints) to even. */
int orc_kv_cache_write_fp8(const void *k, const void *v, const int32_t *positions,
                           const int64_t *slot_mapping, uint8_t *k_cache, uint8_t *v_cache,
                           const float *k_scale, const float *v_scale, int32_t num_tokens,
                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                           int64_t num_blocks, int in_dtype, double rope_theta, int rope_style) {
  double *x = (double *)malloc(sizeof(double) * (size_t)head_dim);
  int rc = 0;
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t blk = slot / block_size, off = slot % block_size;
    if (blk >= num_blocks) { rc = -1; continue; }
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
      for (int32_t e = 0; e < head_dim; ++e) x[e] = orc_load(k, src + e, in_dtype);
      orc_rope(x, head_dim, positions[t], rope_theta, rope_style);
      for (int32_t e = 0; e < head_dim; ++e) {
        k_cache[((blk * num_kv_heads + h) * block_size + off) * head_dim + e] =
            orc_fp8_encode(x[e] / (double)k_scale[h]);
        v_cache[((blk * num_kv_heads + h) * (int64_t)head_dim + e) * block_size + off] =
            orc_fp8_encode(orc_load(v, src + e, in_dtype) / (double)v_scale[h]);
      }
    }
  }
  free(x);
  return rc;
}

/* Dequantised fp64 copies of FP8 pools in the plain [num_blocks][H_kv][bs][d]
 * layout (for the attention definition below). */
void orc_fp8_dequant(const uint8_t *k_cache, const uint8_t *v_cache, const float *k_scale,
                     const float *v_scale, int64_t num_blocks, int32_t num_kv_heads,
                     int32_t head_dim, int32_t block_size, double *k_out, double *v_out) {
  for (int64_t b = 0; b < num_blocks; ++b)
    for (int32_t h = 0; h < num_kv_heads; ++h)
      for (int32_t o = 0; o < block_size; ++o)
        for (int32_t e = 0; e < head_dim; ++e) {
          int64_t plain = ((b * num_kv_heads + h) * block_size + o) * head_dim + e;
          k_out[plain] = orc_fp8_decode(k_cache[plain]) * (double)k_scale[h];
          v_out[plain] = orc_fp8_decode(v_cache[((b * num_kv_heads + h) * (int64_t)head_dim + e) *
                                                    block_size + o]) * (double)v_scale[h];
        }
}

/* ---- paged attention, one query token per sequence --------------------- */

/* Reads K or V element e of context token j of sequence s, KV head h,
 * through the block table. */
static double orc_kv(const void *cache, const int32_t *block_tables, int32_t mbps,
                     int32_t s, int32_t h, int32_t j, int32_t e, int32_t H_kv,
                     int32_t bs, int32_t d, int dtype) {
  int64_t blk = block_tables[(int64_t)s * mbps + j / bs];
  int64_t idx = ((blk * H_kv + h) * bs + j % bs) * (int64_t)d + e;
  return orc_load(cache, idx, dtype);
}

/* out[s, g, :] = sum_j softmax_j(scale * <q[s,g,:], K_s[h, j, :]>) V_s[h, j, :]
 * over j < context_lens[s], h = g / (H_q / H_kv), K_s / V_s gathered through
 * block_tables.  q: [B, H_q, d] in `dtype`; out: [B, H_q, d] doubles.
 * If weights != NULL it receives the softmax weights, [B, H_q, max_ctx]
 * (zero beyond each row's context). */
void orc_paged_attention(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens,
                         double scale, double *out, int32_t num_seqs,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int32_t max_blocks_per_seq, int dtype,
                         double *weights, int32_t max_ctx) {
  int32_t G = num_q_heads / num_kv_heads;
  int64_t rows = (int64_t)num_seqs * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < rows; ++r) {
    int32_t s = (int32_t)(r / num_q_heads), g = (int32_t)(r % num_q_heads);
    int32_t h = g / G, ctx = context_lens[s], d = head_dim;
    double *o = out + r * d;
    for (int32_t e = 0; e < d; ++e) o[e] = 0.0;
    if (weights)
      for (int32_t j = 0; j < max_ctx; ++j) weights[r * max_ctx + j] = 0.0;
    if (ctx <= 0) continue;
    double *qv = (double *)malloc(sizeof(double) * (size_t)d);
    double *w = (double *)malloc(sizeof(double) * (size_t)ctx);
    for (int32_t e = 0; e < d; ++e) qv[e] = orc_load(q, r * d + e, dtype);
    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int32_t j = 0; j < ctx; ++j) {
      double acc = 0.0;
      for (int32_t e = 0; e < d; ++e)
        acc += qv[e] * orc_kv(k_cache, block_tables, max_blocks_per_seq, s, h, j, e,
                              num_kv_heads, block_size, d, dtype);
      w[j] = scale * acc;
      if (w[j] > m) m = w[j];
    }
    /* pass 2: exponentials, their sum, normalised weights */
    double l = 0.0;
    for (int32_t j = 0; j < ctx; ++j) { w[j] = exp(w[j] - m); l += w[j]; }
    for (int32_t j = 0; j < ctx; ++j) w[j] /= l;
    for (int32_t j = 0; j < ctx; ++j)
      for (int32_t e = 0; e < d; ++e)
        o[e] += w[j] * orc_kv(v_cache, block_tables, max_blocks_per_seq, s, h, j, e,
                              num_kv_heads, block_size, d, dtype);
    if (weights)
      for (int32_t j = 0; j < ctx && j < max_ctx; ++j) weights[r * max_ctx + j] = w[j];
    free(qv);
    free(w);
  }
}

/* Split-K form of the same attention: the context is cut into partitions of
 * `partition_size` tokens; each partition p yields its own maximum score
 * m_p, exponential sum l_p = sum exp(s_j - m_p) and unnormalised output
 * o_p = sum exp(s_j - m_p) V_j; the partitions are then merged by
 * log-sum-exp: M = max_p m_p, L = sum_p l_p exp(m_p - M),
 * out = sum_p o_p exp(m_p - M) / L.  Mathematically equal to
 * orc_paged_attention; kept as a second formulation so that the merge rule
 * itself can be checked against the unpartitioned definition. */
void orc_paged_attention_split(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens,
                               double scale, double *out, int32_t num_seqs,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int32_t max_blocks_per_seq, int dtype,
                               int32_t partition_size) {
  int32_t G = num_q_heads / num_kv_heads;
  int64_t rows = (int64_t)num_seqs * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < rows; ++r) {
    int32_t s = (int32_t)(r / num_q_heads), g = (int32_t)(r % num_q_heads);
    int32_t h = g / G, ctx = context_lens[s], d = head_dim;
    double *o = out + r * d;
    for (int32_t e = 0; e < d; ++e) o[e] = 0.0;
    if (ctx <= 0) continue;
    int32_t P = (ctx + partition_size - 1) / partition_size;
    double *qv = (double *)malloc(sizeof(double) * (size_t)d);
    double *mp = (double *)malloc(sizeof(double) * (size_t)P);
    double *lp = (double *)malloc(sizeof(double) * (size_t)P);
    double *op = (double *)calloc((size_t)P * d, sizeof(double));
    double *sc = (double *)malloc(sizeof(double) * (size_t)partition_size);
    for (int32_t e = 0; e < d; ++e) qv[e] = orc_load(q, r * d + e, dtype);
    for (int32_t p = 0; p < P; ++p) {
      int32_t j0 = p * partition_size;
      int32_t j1 = j0 + partition_size < ctx ? j0 + partition_size : ctx;
      double m = -INFINITY;
      for (int32_t j = j0; j < j1; ++j) {
        double acc = 0.0;
        for (int32_t e = 0; e < d; ++e)
          acc += qv[e] * orc_kv(k_cache, block_tables, max_blocks_per_seq, s, h, j, e,
                                num_kv_heads, block_size, d, dtype);
        sc[j - j0] = scale * acc;
        if (sc[j - j0] > m) m = sc[j - j0];
      }
      double l = 0.0;
      for (int32_t j = j0; j < j1; ++j) {
        double wj = exp(sc[j - j0] - m);
        l += wj;
        for (int32_t e = 0; e < d; ++e)
          op[(int64_t)p * d + e] += wj * orc_kv(v_cache, block_tables, max_blocks_per_seq,
                                                s, h, j, e, num_kv_heads, block_size, d, dtype);
      }
      mp[p] = m;
      lp[p] = l;
    }
    double M = -INFINITY;
    for (int32_t p = 0; p < P; ++p) if (mp[p] > M) M = mp[p];
    double L = 0.0;
    for (int32_t p = 0; p < P; ++p) L += lp[p] * exp(mp[p] - M);
    for (int32_t p = 0; p < P; ++p) {
      double f = exp(mp[p] - M) / L;
      for (int32_t e = 0; e < d; ++e) o[e] += op[(int64_t)p * d + e] * f;
    }
    free(qv); free(mp); free(lp); free(op); free(sc);
  }
}

/* Sets the number of host threads the OpenMP loops above use (n >= 1). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Number of host threads the OpenMP loops above use. */
int orc_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
