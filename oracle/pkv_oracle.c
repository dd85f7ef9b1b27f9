/*
 * pkv_oracle.c -- float64 CPU oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * bench's CPU-baseline leg, never by the CUDA library.  Each function follows
 * the definition stated in pkv_oracle.h step by step, with no blocking,
 * fusion or reordering: one (token, head) row at a time, keys in order.
 * OpenMP only distributes independent rows over host threads.
 */
#include "pkv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: bf16 is the top half of a binary32. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

int orc_strided_page_table(const int32_t *req_to_token, int64_t rtt_stride,
                           int64_t rtt_cols, const int64_t *req_pool_indices,
                           int batch, int page_size, int n_cols, int32_t *out,
                           int64_t out_stride) {
  if (batch < 0 || page_size < 1 || n_cols < 0) return -1;
  if ((int64_t)(n_cols - 1) * page_size >= rtt_cols && n_cols > 0) return -1;
  for (int b = 0; b < batch; ++b) {
    const int32_t *row = req_to_token + req_pool_indices[b] * rtt_stride;
    for (int c = 0; c < n_cols; ++c) {
      /* slots are non-negative, so C division equals the floor division
         that the page applies (`// page_size`). */
      out[(int64_t)b * out_stride + c] = row[(int64_t)c * page_size] / page_size;
    }
  }
  return 0;
}

int orc_swa_page_table(const int32_t *req_to_token, int64_t rtt_stride,
                       int64_t rtt_cols, int64_t rtt_rows,
                       const int64_t *req_pool_indices,
                       const int32_t *seq_lens, const int32_t *prefill_lens,
                       int batch, int window, int32_t *dst, int64_t dst_stride,
                       int dst_cols, int32_t *kv_lens) {
  if (batch < 0 || window < 0 || dst_cols < 0) return -1;
  int too_long = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t req = req_pool_indices[b];
    if (req < 0 || req >= rtt_rows) {
      kv_lens[b] = -1;
      ++too_long;
      continue;
    }
    int32_t sl = seq_lens[b];
    int32_t pf = prefill_lens[req];
    /* the whole prompt, then the last `window` tokens that follow it */
    int32_t decode_start = pf > sl - window ? pf : sl - window;
    int32_t gap = decode_start > pf ? decode_start - pf : 0;
    int32_t kv_len = sl - gap;
    /* last source column read: kv_len-1, shifted by the gap if past pf */
    int64_t last_src = kv_len - 1 < pf ? kv_len - 1 : (int64_t)kv_len - 1 + gap;
    if (kv_len > dst_cols || (kv_len > 0 && last_src >= rtt_cols)) {
      kv_lens[b] = -1;
      ++too_long;
      continue;
    }
    kv_lens[b] = kv_len;
    const int32_t *src = req_to_token + req * rtt_stride;
    for (int32_t i = 0; i < kv_len; ++i) {
      int32_t pos = i < pf ? i : i + gap;
      dst[(int64_t)b * dst_stride + i] = src[pos];
    }
  }
  return too_long;
}

int orc_topk_to_slots(const int32_t *topk, int64_t topk_stride, int n_rows,
                      int topk_len, const int32_t *row_req,
                      const int32_t *page_table, int64_t pt_stride,
                      int pt_cols, int page_size,
                      const int32_t *cache_seqlens, int32_t *out,
                      int64_t out_stride) {
  if (n_rows < 0 || topk_len < 0 || page_size < 1 || pt_cols < 0) return -1;
  int bad = 0;
  for (int r = 0; r < n_rows; ++r) {
    int b = row_req[r];
    int64_t limit = cache_seqlens ? (int64_t)cache_seqlens[b]
                                  : (int64_t)pt_cols * page_size;
    if (limit > (int64_t)pt_cols * page_size) limit = (int64_t)pt_cols * page_size;
    for (int k = 0; k < topk_len; ++k) {
      int32_t idx = topk[(int64_t)r * topk_stride + k];
      int32_t slot;
      if (idx == -1) {
        slot = -1;
      } else if (idx < -1 || idx >= limit) {
        slot = -1;
        ++bad;
      } else {
        slot = page_table[(int64_t)b * pt_stride + idx / page_size] * page_size +
               idx % page_size;
      }
      out[(int64_t)r * out_stride + k] = slot;
    }
  }
  return bad;
}

int orc_set_kv_buffer(const uint16_t *rows, int64_t r_st, int64_t r_sh, int n_tokens,
                      int heads, int d, const int64_t *loc, uint16_t *cache,
                      int64_t c_sp, int64_t c_spos, int64_t c_sh, int64_t num_pages,
                      int page_size) {
  if (n_tokens < 0 || heads < 1 || d < 1 || page_size < 1 || num_pages < 0) return -1;
  int skipped = 0;
  for (int t = 0; t < n_tokens; ++t) {
    int64_t slot = loc[t];
    if (slot < 0 || slot >= num_pages * page_size) { ++skipped; continue; }
    int64_t page = slot / page_size, pos = slot % page_size;
    for (int h = 0; h < heads; ++h)
      for (int c = 0; c < d; ++c)
        cache[page * c_sp + pos * c_spos + h * c_sh + c] =
            rows[(int64_t)t * r_st + (int64_t)h * r_sh + c];
  }
  return skipped;
}

int orc_local_virtual_batches(int attn_chunk_size, int page_size,
                              const int32_t *cu_seqlens_q,
                              const int32_t *seq_lens, int batch,
                              const int32_t *page_table, int64_t pt_stride,
                              int pt_cols, int capacity,
                              int32_t *seqlens_q_local,
                              int32_t *cu_seqlens_q_local,
                              int32_t *seqlens_k_local,
                              int32_t *block_table_local, int64_t bt_stride,
                              int bt_cols, int32_t *info) {
  if (attn_chunk_size < 1 || page_size < 1 || pt_cols < 1 || batch < 0 ||
      capacity < 0)
    return -1;
  /* 1. the effective chunk: no longer than the longest sequence, a whole
        number of pages, at least one page */
  int32_t max_seq_len = 0;
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] > max_seq_len) max_seq_len = seq_lens[b];
  int32_t C = attn_chunk_size < max_seq_len ? attn_chunk_size : max_seq_len;
  C = (C / page_size) * page_size;
  if (C < page_size) C = page_size;
  const int pages_per_local_batch = C / page_size;
  if (bt_cols < pages_per_local_batch) return -1;

  int bad = 0;
  int64_t v = 0;            /* virtual batches so far */
  int32_t cu = cu_seqlens_q[0];
  int32_t max_q_local = 0, max_k_local = 0;
  cu_seqlens_q_local[0] = cu;
  for (int b = 0; b < batch; ++b) {
    int32_t q = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    int32_t kv = seq_lens[b];
    if (q == 0) continue;
    if (q < 0) { ++bad; continue; }
    /* more new tokens than keys: counted; its tokens are cut into chunks
       from the first one and given no keys */
    const int malformed = kv < q;
    if (malformed) ++bad;
    /* 2. new tokens in the chunk of the first new token; keys in the chunk
          of the last key; number of chunks the new tokens touch */
    int32_t first = malformed ? C : C - (kv - q) % C;
    if (first > q) first = q;
    int32_t last_k = malformed ? 0 : kv - C * ((kv - 1) / C);
    int32_t blocks = 1 + (q - first + C - 1) / C;
    /* 3. one virtual batch per chunk */
    for (int32_t a = 0; a < blocks; ++a, ++v) {
      int32_t r = blocks - 1 - a;
      int32_t q_local;
      if (a == 0) {
        q_local = first;
      } else {
        q_local = q - first - C * (a - 1);
        if (q_local > C) q_local = C;
      }
      int32_t k_local = malformed ? 0 : (r == 0 ? last_k : C);
      int64_t k_start = (int64_t)kv - last_k - (int64_t)r * C;
      if (q_local > max_q_local) max_q_local = q_local;
      if (k_local > max_k_local) max_k_local = k_local;
      cu += q_local;
      if (v >= capacity) continue;
      seqlens_q_local[v] = q_local;
      cu_seqlens_q_local[v + 1] = cu; /* 4. running sum */
      seqlens_k_local[v] = k_local;
      /* 5. the pages that hold the chunk's keys */
      int32_t *row = block_table_local + v * bt_stride;
      for (int j = 0; j < bt_cols; ++j) {
        if (j < pages_per_local_batch && !malformed) {
          int64_t col = k_start / page_size + j;
          if (col > pt_cols - 1) col = pt_cols - 1;
          row[j] = page_table[(int64_t)b * pt_stride + col];
        } else {
          row[j] = 0;
        }
      }
    }
  }
  int64_t n_virtual = v;
  for (; v < capacity; ++v) { /* padding rows */
    seqlens_q_local[v] = 0;
    cu_seqlens_q_local[v + 1] = cu;
    seqlens_k_local[v] = 0;
    for (int j = 0; j < bt_cols; ++j) block_table_local[v * bt_stride + j] = 0;
  }
  info[0] = (int32_t)n_virtual;
  info[1] = C;
  info[2] = max_q_local;
  info[3] = max_k_local;
  return bad;
}

/* One (token, head) row of paged attention, straight from the definition. */
static int attend_row(const uint16_t *q, int64_t q_st, int64_t q_sh, int d_qk,
                      const uint16_t *k_cache, int64_t k_sp, int64_t k_spos,
                      int64_t k_sh, const uint16_t *v_cache, int64_t v_sp,
                      int64_t v_spos, int64_t v_sh, int d_v, int h_q, int h_kv,
                      int page_size, int64_t num_pages,
                      const int32_t *page_table, int64_t pt_stride, int pt_cols,
                      const int32_t *cache_seqlens, const int32_t *cu_seqlens_q,
                      int batch, double scale, int causal, int window_left,
                      int attn_chunk, const int32_t *topk,
                      int64_t topk_stride, int topk_len,
                      int t, int h, double *o, double *lse_out, double *s_buf,
                      int64_t *slot_buf) {
  /* request of token t: cu[b] <= t < cu[b+1] */
  int b = 0;
  while (b < batch && !(cu_seqlens_q[b] <= t && t < cu_seqlens_q[b + 1])) ++b;
  int skipped = 0;
  for (int d = 0; d < d_v; ++d) o[d] = 0.0;
  if (b == batch) { /* token not covered by any request: no keys */
    if (lse_out) *lse_out = -INFINITY;
    return 0;
  }
  int64_t kv_len = cache_seqlens[b];
  int64_t q_len = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
  int64_t i = kv_len - q_len + (t - cu_seqlens_q[b]); /* bottom-right */
  int kvh = h / (h_q / h_kv);

  /* 1. the candidate logical key list */
  int64_t n_cand = topk ? topk_len : kv_len;
  int64_t n = 0;
  for (int64_t c = 0; c < n_cand; ++c) {
    int64_t j;
    if (topk) {
      j = topk[(int64_t)t * topk_stride + c];
      if (j == -1) continue;
      if (j < -1 || j >= kv_len) { ++skipped; continue; }
    } else {
      j = c;
    }
    if (causal && j > i) continue;
    if (window_left >= 0 && (j > i || j < i - window_left)) continue;
    /* local chunked attention: keys of the query's own chunk only (j and i
       are non-negative, so C division is floor division) */
    if (attn_chunk > 0 && j / attn_chunk != i / attn_chunk) continue;
    /* 2. logical position -> physical slot through the page table */
    if (j / page_size >= pt_cols) { ++skipped; continue; }
    int64_t page = page_table[(int64_t)b * pt_stride + j / page_size];
    if (page < 0 || page >= num_pages) { ++skipped; continue; }
    slot_buf[n++] = page * page_size + j % page_size;
  }

  if (n == 0) {
    if (lse_out) *lse_out = -INFINITY;
    return skipped;
  }

  /* 3. scores s_j = scale * <q, K_j> in float64 */
  const uint16_t *qrow = q + (int64_t)t * q_st + (int64_t)h * q_sh;
  double m = -INFINITY;
  for (int64_t c = 0; c < n; ++c) {
    int64_t slot = slot_buf[c];
    const uint16_t *krow = k_cache + (slot / page_size) * k_sp +
                           (slot % page_size) * k_spos + (int64_t)kvh * k_sh;
    double dot = 0.0;
    for (int d = 0; d < d_qk; ++d)
      dot += bf16_bits_to_double(qrow[d]) * bf16_bits_to_double(krow[d]);
    s_buf[c] = scale * dot;
    if (s_buf[c] > m) m = s_buf[c];
  }

  /* 4. lse = m + log sum exp(s - m);  o = sum exp(s - lse) V */
  double sum = 0.0;
  for (int64_t c = 0; c < n; ++c) sum += exp(s_buf[c] - m);
  double lse = m + log(sum);
  for (int64_t c = 0; c < n; ++c) {
    int64_t slot = slot_buf[c];
    const uint16_t *vrow = v_cache + (slot / page_size) * v_sp +
                           (slot % page_size) * v_spos + (int64_t)kvh * v_sh;
    double w = exp(s_buf[c] - lse);
    for (int d = 0; d < d_v; ++d) o[d] += w * bf16_bits_to_double(vrow[d]);
  }
  if (lse_out) *lse_out = lse;
  return skipped;
}

int orc_attention(const uint16_t *q, int64_t q_st, int64_t q_sh, int total_q,
                  int h_q, int d_qk, const uint16_t *k_cache, int64_t k_sp,
                  int64_t k_spos, int64_t k_sh, const uint16_t *v_cache,
                  int64_t v_sp, int64_t v_spos, int64_t v_sh, int d_v,
                  int h_kv, int page_size, int64_t num_pages,
                  const int32_t *page_table, int64_t pt_stride, int pt_cols,
                  const int32_t *cache_seqlens, const int32_t *cu_seqlens_q,
                  int batch, double scale, int causal, int window_left,
                  int attn_chunk, const int32_t *topk, int64_t topk_stride,
                  int topk_len, const int32_t *rows, int n_rows, double *out,
                  double *lse, int num_threads) {
  if (total_q < 0 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0 || d_qk < 1 ||
      d_v < 1 || page_size < 1 || batch < 0 || window_left < -1 ||
      attn_chunk < 0)
    return -1;
  int64_t n_work = rows ? (int64_t)n_rows : (int64_t)total_q * h_q;
  /* longest candidate list any row can have */
  int64_t max_keys = 0;
  if (topk) {
    max_keys = topk_len;
  } else {
    for (int b = 0; b < batch; ++b)
      if (cache_seqlens[b] > max_keys) max_keys = cache_seqlens[b];
  }
  if (max_keys < 1) max_keys = 1;
  int skipped_total = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#endif
#pragma omp parallel reduction(+ : skipped_total)
  {
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)max_keys);
    int64_t *slot_buf = (int64_t *)malloc(sizeof(int64_t) * (size_t)max_keys);
#pragma omp for schedule(dynamic, 1)
    for (int64_t w = 0; w < n_work; ++w) {
      int t = rows ? rows[2 * w] : (int)(w / h_q);
      int h = rows ? rows[2 * w + 1] : (int)(w % h_q);
      int sk = attend_row(q, q_st, q_sh, d_qk, k_cache, k_sp, k_spos, k_sh,
                          v_cache, v_sp, v_spos, v_sh, d_v, h_q, h_kv,
                          page_size, num_pages, page_table, pt_stride, pt_cols,
                          cache_seqlens, cu_seqlens_q, batch, scale, causal,
                          window_left, attn_chunk, topk, topk_stride,
                          topk_len, t, h,
                          out + w * d_v, lse ? lse + w : NULL, s_buf, slot_buf);
      /* a token's skipped entries are the same for every head: count them
         on its head-0 row only */
      if (h == 0) skipped_total += sk;
    }
    free(s_buf);
    free(slot_buf);
  }
  return skipped_total;
}

double orc_e4m3_value(uint8_t code) {
  const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -mag : mag;
}

uint8_t orc_e4m3_round(double x) {
  if (isnan(x)) return 0x7f;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;  /* -0.0 keeps its sign */
  const double a = fabs(x);
  /* past the midpoint between the largest value (448) and the next step
     the format would have (480) there is no code but NaN; this also covers
     +-inf and magnitudes so large that both distances below round alike */
  if (a > 464.0) return (uint8_t)(sign | 0x7f);
  /* nearest of the non-negative codes 0..127, code 127 standing for the
     value 480 the format does not have (choosing it means "NaN") */
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c < 128; ++c) {
    const double v = c == 127 ? 480.0 : orc_e4m3_value((uint8_t)c);
    const double dist = fabs(a - v);
    if (dist < best_d || (dist == best_d && (c & 1) == 0)) {
      best = c;
      best_d = dist;
    }
  }
  if (best == 127) return (uint8_t)(sign | 0x7f);
  return (uint8_t)(sign | best);
}

int orc_set_kv_buffer_fp8(const uint16_t *rows, int64_t r_st, int64_t r_sh, int n_tokens,
                          int heads, int d, const int64_t *loc, float scale, uint8_t *cache,
                          int64_t c_sp, int64_t c_spos, int64_t c_sh, int64_t num_pages,
                          int page_size) {
  if (n_tokens < 0 || heads < 1 || d < 1 || page_size < 1 || num_pages < 0) return -1;
  if (!(scale > 0.0f) || isinf(scale)) return -1;
  int skipped = 0;
  for (int t = 0; t < n_tokens; ++t) {
    int64_t slot = loc[t];
    if (slot < 0 || slot >= num_pages * page_size) { ++skipped; continue; }
    int64_t page = slot / page_size, pos = slot % page_size;
    for (int h = 0; h < heads; ++h)
      for (int c = 0; c < d; ++c) {
        /* the bf16 value is exact in binary32; one binary32 division */
        const float x = (float)bf16_bits_to_double(rows[(int64_t)t * r_st + (int64_t)h * r_sh + c]);
        const float quotient = x / scale;
        cache[page * c_sp + pos * c_spos + h * c_sh + c] = orc_e4m3_round((double)quotient);
      }
  }
  return skipped;
}

int orc_attention_fp8(const uint16_t *q, int64_t q_st, int64_t q_sh, int total_q,
                      int h_q, int d_qk, const uint8_t *k_cache, int64_t k_sp,
                      int64_t k_spos, int64_t k_sh, const uint8_t *v_cache,
                      int64_t v_sp, int64_t v_spos, int64_t v_sh, int d_v,
                      int h_kv, int page_size, int64_t num_pages,
                      const int32_t *page_table, int64_t pt_stride, int pt_cols,
                      const int32_t *cache_seqlens, const int32_t *cu_seqlens_q,
                      int batch, double scale, int causal, int window_left,
                      const float *k_descale, const float *v_descale,
                      const int32_t *topk, int64_t topk_stride, int topk_len,
                      double *out, double *lse, int num_threads) {
  if (total_q < 0 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0 || d_qk < 1 ||
      d_v < 1 || page_size < 1 || batch < 0 || window_left < -1 || (topk && topk_len < 0))
    return -1;
  int64_t max_keys = 1;
  if (topk) {
    if (topk_len > max_keys) max_keys = topk_len;
  } else {
    for (int b = 0; b < batch; ++b)
      if (cache_seqlens[b] > max_keys) max_keys = cache_seqlens[b];
  }
  int skipped_total = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#endif
#pragma omp parallel reduction(+ : skipped_total)
  {
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)max_keys);
    int64_t *slot_buf = (int64_t *)malloc(sizeof(int64_t) * (size_t)max_keys);
    double *qv = (double *)malloc(sizeof(double) * (size_t)d_qk);
#pragma omp for schedule(dynamic, 1)
    for (int64_t w = 0; w < (int64_t)total_q * h_q; ++w) {
      const int t = (int)(w / h_q), h = (int)(w % h_q);
      double *o = out + w * d_v;
      for (int dd = 0; dd < d_v; ++dd) o[dd] = 0.0;
      if (lse) lse[w] = -INFINITY;
      int b = 0; /* request of token t */
      while (b < batch && !(cu_seqlens_q[b] <= t && t < cu_seqlens_q[b + 1])) ++b;
      if (b == batch) continue;
      const int64_t kv_len = cache_seqlens[b];
      const int64_t q_len = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
      const int64_t i = kv_len - q_len + (t - cu_seqlens_q[b]); /* bottom-right */
      const int kvh = h / (h_q / h_kv);
      const double kd = k_descale ? (double)k_descale[(int64_t)b * h_kv + kvh] : 1.0;
      const double vd = v_descale ? (double)v_descale[(int64_t)b * h_kv + kvh] : 1.0;
      /* 1. q cast to the cache's e4m3 */
      const uint16_t *qrow = q + (int64_t)t * q_st + (int64_t)h * q_sh;
      for (int dd = 0; dd < d_qk; ++dd)
        qv[dd] = orc_e4m3_value(orc_e4m3_round(bf16_bits_to_double(qrow[dd])));
      /* 2. the visible keys and their slots: every position, or the token's
         top-k list (nsa_backend.py: -1 pads the list, other positions
         outside [0, kv_len) are skipped and counted, a repeated position
         counts each time, and the causal bound applies to the listed
         positions) */
      int64_t n = 0;
      const int64_t n_cand = topk ? topk_len : kv_len;
      for (int64_t cnd = 0; cnd < n_cand; ++cnd) {
        int64_t j = cnd;
        if (topk) {
          j = topk[(int64_t)t * topk_stride + cnd];
          if (j == -1) continue;
          if (j < -1 || j >= kv_len) { ++skipped_total; continue; }
        }
        if (causal && j > i) continue;
        if (window_left >= 0 && (j > i || j < i - window_left)) continue;
        if (j / page_size >= pt_cols) { ++skipped_total; continue; }
        const int64_t page = page_table[(int64_t)b * pt_stride + j / page_size];
        if (page < 0 || page >= num_pages) { ++skipped_total; continue; }
        slot_buf[n++] = page * page_size + j % page_size;
      }
      if (n == 0) continue;
      /* 3. s_j = scale * <q', K'_j>, K'_j = value(code) * k_descale */
      double m = -INFINITY;
      for (int64_t c = 0; c < n; ++c) {
        const int64_t slot = slot_buf[c];
        const uint8_t *krow = k_cache + (slot / page_size) * k_sp +
                              (slot % page_size) * k_spos + (int64_t)kvh * k_sh;
        double dot = 0.0;
        for (int dd = 0; dd < d_qk; ++dd) dot += qv[dd] * (orc_e4m3_value(krow[dd]) * kd);
        s_buf[c] = scale * dot;
        if (s_buf[c] > m) m = s_buf[c];
      }
      /* 4. lse and o = sum exp(s - lse) V'_j, V'_j = value(code) * v_descale */
      double sum = 0.0;
      for (int64_t c = 0; c < n; ++c) sum += exp(s_buf[c] - m);
      const double l = m + log(sum);
      for (int64_t c = 0; c < n; ++c) {
        const int64_t slot = slot_buf[c];
        const uint8_t *vrow = v_cache + (slot / page_size) * v_sp +
                              (slot % page_size) * v_spos + (int64_t)kvh * v_sh;
        const double wgt = exp(s_buf[c] - l);
        for (int dd = 0; dd < d_v; ++dd) o[dd] += wgt * (orc_e4m3_value(vrow[dd]) * vd);
      }
      if (lse) lse[w] = l;
    }
    free(s_buf);
    free(slot_buf);
    free(qv);
  }
  return skipped_total;
}

int orc_merge_state(const double *v_a, const double *lse_a, const double *v_b,
                    const double *lse_b, int64_t n, int d, double *v_out,
                    double *lse_out) {
  if (n < 0 || d < 1) return -1;
  for (int64_t r = 0; r < n; ++r) {
    double la = lse_a[r], lb = lse_b[r];
    double m = la > lb ? la : lb;
    if (m == -INFINITY) { /* both states empty */
      for (int c = 0; c < d; ++c) v_out[r * d + c] = 0.0;
      if (lse_out) lse_out[r] = -INFINITY;
      continue;
    }
    double lse = m + log(exp(la - m) + exp(lb - m));
    double wa = exp(la - lse), wb = exp(lb - lse);
    for (int c = 0; c < d; ++c)
      v_out[r * d + c] = wa * v_a[r * d + c] + wb * v_b[r * d + c];
    if (lse_out) lse_out[r] = lse;
  }
  return 0;
}
