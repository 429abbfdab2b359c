/*
 * Paged-attention oracle: a plain, slow, fp64 CPU statement of what the paged-attention path
 * computes.  TEST INFRASTRUCTURE ONLY.  The parity tests, the smoke check and the CPU-baseline
 * leg of the benchmark call it; the CUDA library never does, and it shares no code, header or
 * table with the library.
 *
 * What it follows:
 *  - "Local_LLM_03_vLLM_Architecture", paged-KV slide: the KV cache is cut into fixed-size
 *    blocks (16 tokens by default), each sequence has a block table from logical positions to
 *    physical blocks, and the attention kernel gathers K/V from the scattered blocks.  The
 *    result is therefore ordinary attention over the de-paged K/V: de-paging is written out
 *    below as its own step, followed by the textbook softmax attention.
 *  - "vLLM: LLM Inference That Doesn't Waste Your GPU", section "KV cache, in one picture":
 *    every processed token's K/V is stored once and reused by later tokens; the scatter of new
 *    tokens into their cache slots is pa_oracle_reshape_and_cache.
 *  - Same deck, chunked-prefill slide: a long prompt is processed in chunks interleaved with
 *    decodes.  Reading used here: row i of a chunk of q_len rows sits at absolute position
 *    seq_len - q_len + i and sees keys 0 .. seq_len - q_len + i (bottom-right causal).
 *  - Same deck, KV-sizing slide (GQA-8): query head h reads KV head h / (Hq / Hkv).
 *
 * Layouts (the pages fix none; these are the conventions of the library's C ABI):
 *   q        fp16 [T, Hq, d]          k_cache/v_cache  fp16 [NB, Hkv, bs, d]
 *   block_tables int32 [N, MB]        seq_lens int32 [N]   query_start_loc int32 [N+1]
 *   slot_mapping int64 [T_new], slot = block * bs + offset, negative = skip
 * fp16 values arrive as raw IEEE binary16 bit patterns (uint16) and are widened to double
 * exactly by half_to_double.  A bfloat16 cache (fmt = 1 in the attention entry points) arrives
 * the same way as raw bfloat16 patterns and is widened exactly by bf16_to_double.  Arithmetic
 * is fp64 throughout; exp is the C library's exp().
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = -1, ORACLE_BAD_SLOT = -2, ORACLE_BAD_BLOCK = -3,
       ORACLE_NO_MEMORY = -4 };

/* IEEE 754 binary16 -> double, from the format's definition: 1 sign bit, 5 exponent bits
 * (bias 15), 10 fraction bits; exponent 0 = subnormal (fraction * 2^-24), 31 = inf/NaN. */
double pa_oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int f = h & 1023;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(f + 1024), e - 25);
  }
  return sign ? -v : v;
}

/* bfloat16 -> double, from the format's definition: the upper half of an IEEE binary32, i.e.
 * 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits; exponent 0 = subnormal
 * (fraction * 2^-133), 255 = inf/NaN. */
double pa_oracle_bf16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 255;
  int f = h & 127;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -133);
  } else if (e == 255) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(f + 128), e - 134);
  }
  return sign ? -v : v;
}

typedef double (*widen_fn)(uint16_t);

/* fmt 0: binary16 values, fmt 1: bfloat16 values; NULL for anything else. */
static widen_fn widen_for(int64_t fmt) {
  return fmt == 0 ? pa_oracle_half_to_double : fmt == 1 ? pa_oracle_bf16_to_double : NULL;
}

void pa_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int pa_oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* KV scatter-write: for each new token t with slot_mapping[t] >= 0, copy its K and V rows of
 * every kv head into block slot/bs, offset slot%bs of the pools.  A pure copy of the bit
 * patterns, so a comparison with the GPU result is bytewise. */
int pa_oracle_reshape_and_cache(const uint16_t *k, const uint16_t *v, uint16_t *k_cache,
                                uint16_t *v_cache, const int64_t *slot_mapping,
                                int64_t num_tokens, int64_t num_kv_heads, int64_t head_dim,
                                int64_t num_blocks, int64_t block_size) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return ORACLE_BAD_ARG;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * block_size) return ORACLE_BAD_SLOT;
  }
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t blk = slot / block_size;
    int64_t off = slot % block_size;
    for (int64_t h = 0; h < num_kv_heads; ++h) {
      int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim;
      int64_t src = (t * num_kv_heads + h) * head_dim;
      memcpy(k_cache + dst, k + src, (size_t)head_dim * sizeof(uint16_t));
      memcpy(v_cache + dst, v + src, (size_t)head_dim * sizeof(uint16_t));
    }
  }
  return ORACLE_OK;
}

/* Textbook softmax attention of one query row over keys 0 .. n_visible-1:
 *   s_p = scale * <q, K_p>,  m = max_p s_p,  w_p = exp(s_p - m),  out = sum_p w_p V_p / sum_p w_p.
 * K and V are contiguous [n, d] arrays of one kv head. */
static void attend_one(const double *qrow, const double *K, const double *V, int64_t n_visible,
                       int64_t d, double scale, double *s, double *out) {
  double m = -INFINITY;
  for (int64_t p = 0; p < n_visible; ++p) {
    double dot = 0.0;
    for (int64_t j = 0; j < d; ++j) dot += qrow[j] * K[p * d + j];
    s[p] = scale * dot;
    if (s[p] > m) m = s[p];
  }
  double l = 0.0;
  for (int64_t p = 0; p < n_visible; ++p) {
    s[p] = exp(s[p] - m);
    l += s[p];
  }
  for (int64_t j = 0; j < d; ++j) {
    double acc = 0.0;
    for (int64_t p = 0; p < n_visible; ++p) acc += s[p] * V[p * d + j];
    out[j] = acc / l;
  }
}

/* The same attention done split-context: keys are cut into partitions of `part` positions;
 * each partition keeps its own max m_i, sum l_i and normalised output o_i, and the
 * partitions are combined with the log-sum-exp rule
 *   M = max_i m_i,  w_i = exp(m_i - M) * l_i,  out = sum_i w_i o_i / sum_i w_i.
 * Softmax algebra makes this equal to attend_one up to rounding. */
static void attend_one_split(const double *qrow, const double *K, const double *V,
                             int64_t n_visible, int64_t d, double scale, int64_t part,
                             double *s, double *o_parts, double *m_parts, double *l_parts,
                             double *out) {
  int64_t np = (n_visible + part - 1) / part;
  for (int64_t i = 0; i < np; ++i) {
    int64_t lo = i * part;
    int64_t hi = lo + part < n_visible ? lo + part : n_visible;
    double m = -INFINITY;
    for (int64_t p = lo; p < hi; ++p) {
      double dot = 0.0;
      for (int64_t j = 0; j < d; ++j) dot += qrow[j] * K[p * d + j];
      s[p] = scale * dot;
      if (s[p] > m) m = s[p];
    }
    double l = 0.0;
    for (int64_t p = lo; p < hi; ++p) {
      s[p] = exp(s[p] - m);
      l += s[p];
    }
    for (int64_t j = 0; j < d; ++j) {
      double acc = 0.0;
      for (int64_t p = lo; p < hi; ++p) acc += s[p] * V[p * d + j];
      o_parts[i * d + j] = acc / l;
    }
    m_parts[i] = m;
    l_parts[i] = l;
  }
  double M = -INFINITY;
  for (int64_t i = 0; i < np; ++i)
    if (m_parts[i] > M) M = m_parts[i];
  double wsum = 0.0;
  for (int64_t i = 0; i < np; ++i) wsum += exp(m_parts[i] - M) * l_parts[i];
  for (int64_t j = 0; j < d; ++j) {
    double acc = 0.0;
    for (int64_t i = 0; i < np; ++i) acc += exp(m_parts[i] - M) * l_parts[i] * o_parts[i * d + j];
    out[j] = acc / wsum;
  }
}

/* Shared by the paged and the contiguous entry points: checks of the batch descriptor. */
static int check_descriptor(const int32_t *seq_lens, const int32_t *qsl, int64_t num_seqs,
                            int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return ORACLE_BAD_ARG;
  if (num_q_heads % num_kv_heads) return ORACLE_BAD_ARG;
  if (num_seqs > 0 && qsl[0] != 0) return ORACLE_BAD_ARG;
  for (int64_t s = 0; s < num_seqs; ++s) {
    int64_t q_len = (int64_t)qsl[s + 1] - qsl[s];
    if (q_len < 0 || seq_lens[s] < 0 || q_len > seq_lens[s]) return ORACLE_BAD_ARG;
  }
  return ORACLE_OK;
}

/* One (sequence, kv head) task: K and V of that head as contiguous fp64 [L, d] arrays,
 * then every query row of the sequence and every query head of the group attends.
 * part == 0: textbook attention; part > 0: split-context + log-sum-exp merge. */
static int run_group(const uint16_t *q, const double *K, const double *V, int64_t L,
                     int64_t row0, int64_t q_len, int64_t g, int64_t num_q_heads,
                     int64_t group, int64_t d, double scale, int64_t part,
                     const uint8_t *row_mask, widen_fn widen, double *out) {
  double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
  double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  int64_t np = part > 0 ? (L + part - 1) / part : 1;
  if (np < 1) np = 1;
  double *o_parts = (double *)malloc(sizeof(double) * (size_t)(np * d));
  double *m_parts = (double *)malloc(sizeof(double) * (size_t)np);
  double *l_parts = (double *)malloc(sizeof(double) * (size_t)np);
  if (!qrow || !s || !o_parts || !m_parts || !l_parts) {
    free(qrow); free(s); free(o_parts); free(m_parts); free(l_parts);
    return ORACLE_NO_MEMORY;
  }
  for (int64_t i = 0; i < q_len; ++i) {
    int64_t t = row0 + i;
    if (row_mask && !row_mask[t]) continue;
    int64_t n_visible = L - q_len + i + 1;
    for (int64_t h = g * group; h < (g + 1) * group; ++h) {
      const uint16_t *qh = q + (t * num_q_heads + h) * d;
      for (int64_t j = 0; j < d; ++j) qrow[j] = widen(qh[j]);
      double *o = out + (t * num_q_heads + h) * d;
      if (part > 0)
        attend_one_split(qrow, K, V, n_visible, d, scale, part, s, o_parts, m_parts, l_parts, o);
      else
        attend_one(qrow, K, V, n_visible, d, scale, s, o);
    }
  }
  free(qrow); free(s); free(o_parts); free(m_parts); free(l_parts);
  return ORACLE_OK;
}

/* De-paging: logical position p of sequence s lives in physical block
 * block_tables[s][p / bs] at offset p % bs; kv head g of that token is the row
 * k_cache[blk][g][p % bs][:]. */
static void depage(const uint16_t *cache, const int32_t *table_row, int64_t L, int64_t g,
                   int64_t num_kv_heads, int64_t bs, int64_t d, widen_fn widen, double *dst) {
  for (int64_t p = 0; p < L; ++p) {
    int64_t blk = table_row[p / bs];
    const uint16_t *src = cache + ((blk * num_kv_heads + g) * bs + p % bs) * d;
    for (int64_t j = 0; j < d; ++j) dst[p * d + j] = widen(src[j]);
  }
}

static int attention_paged(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *block_tables, int64_t max_blocks,
                           const int32_t *seq_lens, const int32_t *qsl, int64_t num_seqs,
                           int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim,
                           int64_t block_size, int64_t num_blocks, double scale, int64_t part,
                           const uint8_t *row_mask, int64_t fmt, double *out) {
  int rc = check_descriptor(seq_lens, qsl, num_seqs, num_q_heads, num_kv_heads, head_dim);
  if (rc) return rc;
  widen_fn widen = widen_for(fmt);
  if (block_size <= 0 || part < 0 || !widen) return ORACLE_BAD_ARG;
  for (int64_t s = 0; s < num_seqs; ++s) {
    if (qsl[s + 1] == qsl[s]) continue;
    int64_t nb = (seq_lens[s] + block_size - 1) / block_size;
    if (nb > max_blocks) return ORACLE_BAD_ARG;
    for (int64_t j = 0; j < nb; ++j) {
      int32_t b = block_tables[s * max_blocks + j];
      if (b < 0 || b >= num_blocks) return ORACLE_BAD_BLOCK;
    }
  }
  int64_t group = num_q_heads / num_kv_heads;
  int64_t ntask = num_seqs * num_kv_heads;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t task = 0; task < ntask; ++task) {
    int64_t s = task / num_kv_heads, g = task % num_kv_heads;
    int64_t q_len = (int64_t)qsl[s + 1] - qsl[s];
    int64_t L = seq_lens[s];
    if (q_len == 0) continue;
    double *K = (double *)malloc(sizeof(double) * (size_t)(L * head_dim));
    double *V = (double *)malloc(sizeof(double) * (size_t)(L * head_dim));
    int r = ORACLE_NO_MEMORY;
    if (K && V) {
      depage(k_cache, block_tables + s * max_blocks, L, g, num_kv_heads, block_size, head_dim,
             widen, K);
      depage(v_cache, block_tables + s * max_blocks, L, g, num_kv_heads, block_size, head_dim,
             widen, V);
      r = run_group(q, K, V, L, qsl[s], q_len, g, num_q_heads, group, head_dim, scale, part,
                    row_mask, widen, out);
    }
    free(K);
    free(V);
    if (r) {
#pragma omp atomic write
      err = r;
    }
  }
  return err;
}

/* Attention over the paged cache (textbook, unsplit).  Output fp64 [T, Hq, d]; rows with
 * row_mask[t] == 0 (row_mask may be NULL = all rows) are left untouched.  q and the pools hold
 * binary16 (fmt 0) or bfloat16 (fmt 1) patterns. */
int pa_oracle_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int64_t max_blocks, const int32_t *seq_lens,
                        const int32_t *qsl, int64_t num_seqs, int64_t num_q_heads,
                        int64_t num_kv_heads, int64_t head_dim, int64_t block_size,
                        int64_t num_blocks, double scale, int64_t fmt, const uint8_t *row_mask,
                        double *out) {
  return attention_paged(q, k_cache, v_cache, block_tables, max_blocks, seq_lens, qsl, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, 0,
                         row_mask, fmt, out);
}

/* The same attention computed split-context (partitions of `partition_size` key positions,
 * log-sum-exp merge), in fp64.  Pins the merge algebra the split-context GPU path uses. */
int pa_oracle_attention_split(const uint16_t *q, const uint16_t *k_cache,
                              const uint16_t *v_cache, const int32_t *block_tables,
                              int64_t max_blocks, const int32_t *seq_lens, const int32_t *qsl,
                              int64_t num_seqs, int64_t num_q_heads, int64_t num_kv_heads,
                              int64_t head_dim, int64_t block_size, int64_t num_blocks,
                              double scale, int64_t fmt, int64_t partition_size,
                              const uint8_t *row_mask, double *out) {
  if (partition_size <= 0) return ORACLE_BAD_ARG;
  return attention_paged(q, k_cache, v_cache, block_tables, max_blocks, seq_lens, qsl, num_seqs,
                         num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                         partition_size, row_mask, fmt, out);
}

/* Attention over contiguous per-sequence K/V (the "one region per request" layout the pages
 * contrast paging with): sequence s's K is k[kv_start[s] .. kv_start[s]+L-1][Hkv][d].
 * Uses the same per-head routine as the paged entry point, so paged and contiguous inputs
 * holding the same values give bit-identical outputs. */
int pa_oracle_attention_contiguous(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                   const int64_t *kv_start, const int32_t *seq_lens,
                                   const int32_t *qsl, int64_t num_seqs, int64_t num_q_heads,
                                   int64_t num_kv_heads, int64_t head_dim, double scale,
                                   int64_t fmt, const uint8_t *row_mask, double *out) {
  int rc = check_descriptor(seq_lens, qsl, num_seqs, num_q_heads, num_kv_heads, head_dim);
  if (rc) return rc;
  widen_fn widen = widen_for(fmt);
  if (!widen) return ORACLE_BAD_ARG;
  int64_t group = num_q_heads / num_kv_heads;
  int64_t ntask = num_seqs * num_kv_heads;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t task = 0; task < ntask; ++task) {
    int64_t s = task / num_kv_heads, g = task % num_kv_heads;
    int64_t q_len = (int64_t)qsl[s + 1] - qsl[s];
    int64_t L = seq_lens[s];
    if (q_len == 0) continue;
    double *K = (double *)malloc(sizeof(double) * (size_t)(L * head_dim));
    double *V = (double *)malloc(sizeof(double) * (size_t)(L * head_dim));
    int r = ORACLE_NO_MEMORY;
    if (K && V) {
      for (int64_t p = 0; p < L; ++p) {
        const uint16_t *ks = k + ((kv_start[s] + p) * num_kv_heads + g) * head_dim;
        const uint16_t *vs = v + ((kv_start[s] + p) * num_kv_heads + g) * head_dim;
        for (int64_t j = 0; j < head_dim; ++j) {
          K[p * head_dim + j] = widen(ks[j]);
          V[p * head_dim + j] = widen(vs[j]);
        }
      }
      r = run_group(q, K, V, L, qsl[s], q_len, g, num_q_heads, group, head_dim, scale, 0,
                    row_mask, widen, out);
    }
    free(K);
    free(V);
    if (r) {
#pragma omp atomic write
      err = r;
    }
  }
  return err;
}
