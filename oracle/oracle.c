/*
 * oracle.c -- plain CPU oracle for the paged-attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  It shares
 * no code, header, table or helper with the CUDA library; the two meet only in
 * the seeded input arrays.
 *
 * Everything here is the textbook definition written out, in double
 * precision, with no blocking, fusion or reordering:
 *   - the KV write is an array assignment of whole rows
 *     [tiny-vllm README, curriculum "Paged KV cache", "Why KV cache exists"];
 *   - attention gathers each sequence's K/V rows through its block table into
 *     contiguous arrays [tiny-vllm README, curriculum "Paged Attention";
 *     nano-vLLM guide ch. 4 "PagedAttention": the KV cache as virtual memory
 *     made of fixed-size blocks], then runs two-pass softmax attention:
 *     scores, their maximum, exponentials, their sum, the weighted sum of V
 *     [tiny-vllm README, curriculum "Attention", "Softmax"], with query head h
 *     reading KV head h / G [curriculum "GQA"], and for prefill a causal mask
 *     that lets a query see keys up to its own position [curriculum "Causal
 *     mask", "Prefill vs decode"].
 * The online (running max / running sum) form and the split-K merge are NOT
 * used here: the GPU results of those forms are compared with this direct
 * definition.
 *
 * Element conventions: bf16 values arrive as their 16-bit patterns (uint16);
 * widening bf16 -> float -> double is exact.  Cache layout [NB, bs, Hkv, D].
 *
 * Parity pins (tests check this file against): float64 brute force on tiny
 * inputs, torch scaled_dot_product_attention special cases (contiguous block
 * table), closed forms (two keys, equal keys, scale 0, one key), invariants
 * (physical block permutation, causal independence) and numpy row assignment
 * for the KV write.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Return codes. */
#define ORC_OK 0
#define ORC_BAD_ARG -1
#define ORC_BAD_SLOT -2
#define ORC_BAD_BLOCK -3
#define ORC_BAD_CTX -4
#define ORC_BAD_QLEN -5
#define ORC_NOMEM -6

static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * KV write: for every t with slot_mapping[t] >= 0, row slot_mapping[t] of each
 * cache becomes row t of the new K / V.  A row is row_elems bf16 values.
 * Returns the number of rows written, or ORC_BAD_SLOT if a slot is out of
 * range (nothing is written in that case).
 */
long long oracle_kv_write(uint16_t* k_cache, uint16_t* v_cache,
                          const uint16_t* k_new, const uint16_t* v_new,
                          const int32_t* slot_mapping, long long num_tokens,
                          long long row_elems, long long num_slots) {
  long long written = 0;
  for (long long t = 0; t < num_tokens; ++t) {
    if (slot_mapping[t] >= num_slots) return ORC_BAD_SLOT;
  }
  for (long long t = 0; t < num_tokens; ++t) {
    long long slot = slot_mapping[t];
    if (slot < 0) continue;
    memcpy(k_cache + slot * row_elems, k_new + t * row_elems,
           (size_t)row_elems * sizeof(uint16_t));
    memcpy(v_cache + slot * row_elems, v_new + t * row_elems,
           (size_t)row_elems * sizeof(uint16_t));
    ++written;
  }
  return written;
}

/*
 * Rotary position embedding of one head vector, in double precision
 * [tiny-vllm README, curriculum "RoPE"; Tiny-vLLM digest, "Core Mechanics"]:
 * for i < D/2 the pair (x_i, x_{i+D/2}) is rotated by the angle
 * pos * theta^(-2i/D):
 *   y_i       = x_i cos a - x_{i+D/2} sin a
 *   y_{i+D/2} = x_{i+D/2} cos a + x_i sin a.
 */
void oracle_rope_double(double* y, const double* x, int d, long long pos, double theta) {
  const int half = d / 2;
  for (int i = 0; i < half; ++i) {
    const double inv_freq = pow(theta, -2.0 * i / d);
    const double a = (double)pos * inv_freq;
    const double c = cos(a), s = sin(a);
    y[i] = x[i] * c - x[i + half] * s;
    y[i + half] = x[i + half] * c + x[i] * s;
  }
}

/* double -> bf16 bit pattern, rounded to nearest, ties to even (finite
 * inputs).  The magnitude is bracketed by its two bf16 neighbours and the
 * nearer one is taken, so the double is rounded once. */
static uint16_t double_to_bf16_bits(double v) {
  const uint32_t sign = v < 0 ? 0x80000000u : 0u;
  const double a = fabs(v);
  float f = (float)a;
  uint32_t lo;
  memcpy(&lo, &f, 4);
  lo &= 0xffff0000u;                       /* bf16 at or below f */
  float flo;
  memcpy(&flo, &lo, 4);
  if ((double)flo > a) {                   /* f was rounded up past a */
    lo -= 0x10000u;
    memcpy(&flo, &lo, 4);
  }
  const uint32_t hi = lo + 0x10000u;
  float fhi;
  memcpy(&fhi, &hi, 4);
  const double dl = a - (double)flo, dh = (double)fhi - a;
  uint32_t pick;
  if (dl < dh) pick = lo;
  else if (dh < dl) pick = hi;
  else pick = ((lo >> 16) & 1u) ? hi : lo;
  return (uint16_t)((pick | sign) >> 16);
}

/* Rounds n doubles to bf16 bit patterns (exported for the rounding pin). */
void oracle_round_bf16(uint16_t* out, const double* in, long long n) {
  for (long long i = 0; i < n; ++i) out[i] = double_to_bf16_bits(in[i]);
}

/*
 * RoPE + paged KV write: for every token t, q[t] (if q is not NULL) and k_new[t]
 * are rotated at position positions[t] (each head separately), rounded to
 * bf16; then, for slot_mapping[t] >= 0, the rotated K row and the V row are
 * stored at that slot.  q is rotated in place for every token.
 */
long long oracle_rope_kv_write(uint16_t* q, uint16_t* k_cache, uint16_t* v_cache,
                               const uint16_t* k_new, const uint16_t* v_new,
                               const int32_t* slot_mapping, const int32_t* positions,
                               long long num_tokens, int hq, int hkv, int d,
                               long long num_slots, double theta) {
  if (d <= 0 || d % 2) return -1;
  double x[512], y[512];
  if (d > 512) return -1;
  long long written = 0;
  for (long long t = 0; t < num_tokens; ++t)
    if (slot_mapping[t] >= num_slots) return -2;
  for (long long t = 0; t < num_tokens; ++t) {
    const long long pos = positions[t];
    if (q) {
      for (int h = 0; h < hq; ++h) {
        uint16_t* row = q + (t * hq + h) * d;
        for (int e = 0; e < d; ++e) x[e] = bf16_bits_to_double(row[e]);
        oracle_rope_double(y, x, d, pos, theta);
        for (int e = 0; e < d; ++e) row[e] = double_to_bf16_bits(y[e]);
      }
    }
    const long long slot = slot_mapping[t];
    if (slot < 0) continue;
    for (int h = 0; h < hkv; ++h) {
      const uint16_t* src = k_new + (t * hkv + h) * d;
      uint16_t* dst = k_cache + (slot * hkv + h) * d;
      for (int e = 0; e < d; ++e) x[e] = bf16_bits_to_double(src[e]);
      oracle_rope_double(y, x, d, pos, theta);
      for (int e = 0; e < d; ++e) dst[e] = double_to_bf16_bits(y[e]);
    }
    memcpy(v_cache + slot * hkv * d, v_new + t * hkv * d, (size_t)hkv * d * sizeof(uint16_t));
    ++written;
  }
  return written;
}

/* Checks a sequence's context length and the block ids it will read. */
static int check_sequence(const int32_t* table_row, long long ctx, int bs,
                          int num_blocks, int max_blocks) {
  if (ctx < 0 || ctx > (long long)max_blocks * bs) return ORC_BAD_CTX;
  long long nblk = (ctx + bs - 1) / bs;
  for (long long b = 0; b < nblk; ++b) {
    if (table_row[b] < 0 || table_row[b] >= num_blocks) return ORC_BAD_BLOCK;
  }
  return ORC_OK;
}

/*
 * Gather: logical token j of the sequence is physical block
 * table_row[j / bs], offset j % bs.  Copies KV head g of tokens [0, n) into
 * dst[n][D] as double.
 */
static void gather_head(double* dst, const uint16_t* cache,
                        const int32_t* table_row, long long n, int bs, int hkv,
                        int d, int g) {
  for (long long j = 0; j < n; ++j) {
    long long block = table_row[j / bs];
    long long offset = j % bs;
    const uint16_t* src =
        cache + ((block * bs + offset) * (long long)hkv + g) * (long long)d;
    for (int e = 0; e < d; ++e) dst[j * d + e] = bf16_bits_to_double(src[e]);
  }
}

/*
 * Softmax attention of one query vector over n keys (two passes):
 *   s_j = scale * sum_e q[e] k[j][e];  m = max_j s_j;  w_j = exp(s_j - m);
 *   l = sum_j w_j;  out[e] = (sum_j w_j v[j][e]) / l.
 * n == 0 gives zeros.
 */
static void attend(double* out, const double* qv, const double* kc,
                   const double* vc, long long n, int d, double scale,
                   double* scores) {
  for (int e = 0; e < d; ++e) out[e] = 0.0;
  if (n == 0) return;
  for (long long j = 0; j < n; ++j) {
    double dot = 0.0;
    for (int e = 0; e < d; ++e) dot += qv[e] * kc[j * d + e];
    scores[j] = scale * dot;
  }
  double m = scores[0];
  for (long long j = 1; j < n; ++j)
    if (scores[j] > m) m = scores[j];
  double l = 0.0;
  for (long long j = 0; j < n; ++j) {
    scores[j] = exp(scores[j] - m);
    l += scores[j];
  }
  for (long long j = 0; j < n; ++j)
    for (int e = 0; e < d; ++e) out[e] += scores[j] * vc[j * d + e];
  for (int e = 0; e < d; ++e) out[e] /= l;
}

/*
 * Decode: out[s, h, :] = attention of q[s, h, :] over tokens
 * [0, context_lens[s]) of KV head h / G.  Only sequences with
 * seq_mask[s] != 0 are computed when seq_mask is not NULL (the other rows of
 * out are left as they are).
 */
int oracle_decode(double* out, const uint16_t* q, const uint16_t* k_cache,
                  const uint16_t* v_cache, const int32_t* block_tables,
                  const int32_t* context_lens, int num_seqs, int hq, int hkv,
                  int d, int bs, int num_blocks, int max_blocks, double scale,
                  const uint8_t* seq_mask) {
  if (num_seqs < 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 ||
      bs <= 0 || max_blocks < 0)
    return ORC_BAD_ARG;
  const int group = hq / hkv;
  for (int s = 0; s < num_seqs; ++s) {
    if (seq_mask && !seq_mask[s]) continue;
    int rc = check_sequence(block_tables + (long long)s * max_blocks,
                            context_lens[s], bs, num_blocks, max_blocks);
    if (rc != ORC_OK) return rc;
  }
  int failed = 0;
  const long long tasks = (long long)num_seqs * hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long task = 0; task < tasks; ++task) {
    const int s = (int)(task / hkv);
    const int g = (int)(task % hkv);
    if (seq_mask && !seq_mask[s]) continue;
    const long long n = context_lens[s];
    const int32_t* row = block_tables + (long long)s * max_blocks;
    double* kc = (double*)malloc(sizeof(double) * (size_t)(n * d + 1));
    double* vc = (double*)malloc(sizeof(double) * (size_t)(n * d + 1));
    double* scores = (double*)malloc(sizeof(double) * (size_t)(n + 1));
    double* qv = (double*)malloc(sizeof(double) * (size_t)d);
    if (!kc || !vc || !scores || !qv) {
#pragma omp atomic write
      failed = 1;
    } else {
      gather_head(kc, k_cache, row, n, bs, hkv, d, g);
      gather_head(vc, v_cache, row, n, bs, hkv, d, g);
      for (int h = g * group; h < (g + 1) * group; ++h) {
        const uint16_t* qsrc = q + ((long long)s * hq + h) * d;
        for (int e = 0; e < d; ++e) qv[e] = bf16_bits_to_double(qsrc[e]);
        attend(out + ((long long)s * hq + h) * d, qv, kc, vc, n, d, scale,
               scores);
      }
    }
    free(kc);
    free(vc);
    free(scores);
    free(qv);
  }
  return failed ? ORC_NOMEM : ORC_OK;
}

/*
 * Prefill: sequence s owns query tokens [qsl[s], qsl[s+1]); with
 * Lq = qsl[s+1] - qsl[s], row i sits at absolute position
 * p = context_lens[s] - Lq + i and attends to tokens [0, p] (causal,
 * inclusive) of KV head h / G.  Only tokens with row_mask[t] != 0 are
 * computed when row_mask is not NULL.
 */
int oracle_prefill(double* out, const uint16_t* q, const int32_t* qsl,
                   const uint16_t* k_cache, const uint16_t* v_cache,
                   const int32_t* block_tables, const int32_t* context_lens,
                   int num_seqs, int total_q, int hq, int hkv, int d, int bs,
                   int num_blocks, int max_blocks, double scale,
                   const uint8_t* row_mask) {
  if (num_seqs < 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 ||
      bs <= 0 || max_blocks < 0)
    return ORC_BAD_ARG;
  if (qsl[0] != 0 || qsl[num_seqs] != total_q) return ORC_BAD_ARG;
  const int group = hq / hkv;
  for (int s = 0; s < num_seqs; ++s) {
    const long long lq = (long long)qsl[s + 1] - qsl[s];
    if (lq < 0) return ORC_BAD_ARG;
    if (lq > context_lens[s]) return ORC_BAD_QLEN;
    int rc = check_sequence(block_tables + (long long)s * max_blocks,
                            context_lens[s], bs, num_blocks, max_blocks);
    if (rc != ORC_OK) return rc;
  }
  int failed = 0;
  const long long tasks = (long long)num_seqs * hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long task = 0; task < tasks; ++task) {
    const int s = (int)(task / hkv);
    const int g = (int)(task % hkv);
    const long long first = qsl[s];
    const long long lq = (long long)qsl[s + 1] - first;
    const long long n = context_lens[s];
    int any = 0;
    for (long long i = 0; i < lq; ++i)
      if (!row_mask || row_mask[first + i]) any = 1;
    if (!any) continue;
    const int32_t* row = block_tables + (long long)s * max_blocks;
    double* kc = (double*)malloc(sizeof(double) * (size_t)(n * d + 1));
    double* vc = (double*)malloc(sizeof(double) * (size_t)(n * d + 1));
    double* scores = (double*)malloc(sizeof(double) * (size_t)(n + 1));
    double* qv = (double*)malloc(sizeof(double) * (size_t)d);
    if (!kc || !vc || !scores || !qv) {
#pragma omp atomic write
      failed = 1;
    } else {
      gather_head(kc, k_cache, row, n, bs, hkv, d, g);
      gather_head(vc, v_cache, row, n, bs, hkv, d, g);
      for (long long i = 0; i < lq; ++i) {
        const long long t = first + i;
        if (row_mask && !row_mask[t]) continue;
        const long long pos = n - lq + i;
        for (int h = g * group; h < (g + 1) * group; ++h) {
          const uint16_t* qsrc = q + (t * hq + h) * d;
          for (int e = 0; e < d; ++e) qv[e] = bf16_bits_to_double(qsrc[e]);
          attend(out + (t * hq + h) * d, qv, kc, vc, pos + 1, d, scale,
                 scores);
        }
      }
    }
    free(kc);
    free(vc);
    free(scores);
    free(qv);
  }
  return failed ? ORC_NOMEM : ORC_OK;
}
