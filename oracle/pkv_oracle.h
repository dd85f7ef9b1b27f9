/*
 * pkv_oracle.h -- float64 CPU oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously-correct
 * restatement of what the paged-KV attention path computes, used to check the
 * CUDA library.  Only the test suite, the smoke check and the bench's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper
 * with the CUDA library, and the CUDA library never calls it.
 *
 * Sources (SGLang attention-backend source pages):
 *   - flashattention_backend.py, `init_forward_metadata` (strided page table,
 *     decode/extend metadata), `_build_pa_page_table_kernel` (prefill-aware
 *     sliding-window page table), `forward_extend` / `forward_decode`
 *     (`flash_attn_with_kvcache` calls, window_size convention, absorbed MLA
 *     call with q_rope/k_rope and q_nope/c_kv).
 *   - dual_chunk_flashattention_backend.py, `_merge_attn_outputs` and the
 *     three-way decode merge (log-sum-exp state merge), and
 *     `_dual_chunk_flash_attn_decoding_with_exp_sums` (empty-KV convention:
 *     out = 0, lse = -inf).
 *   - nsa_backend.py, `TopkTransformMethod.PAGED`, `forward_decode`,
 *     `_pad_topk_indices` (top-k logical index -> KV slot, -1 = skip),
 *     `init_forward_metadata` (`seqlens_expanded`: bottom-right causal).
 *
 * Conventions.  All bf16 arrays are passed as their raw 16-bit patterns and
 * widened exactly to double.  Every function returns 0 on success, a
 * negative value on a malformed argument, or a positive count of skipped
 * out-of-range entries where stated.
 */
#ifndef PKV_ORACLE_H
#define PKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Strided page table (flashattention_backend.py, `init_forward_metadata`,
 * "Convert the page table to a strided format"):
 *   out[b][c] = req_to_token[req_pool_indices[b]][c * page_size] / page_size
 * for c in [0, n_cols).  Returns 0, or -1 on bad arguments. */
int orc_strided_page_table(const int32_t *req_to_token, int64_t rtt_stride,
                           int64_t rtt_cols, const int64_t *req_pool_indices,
                           int batch, int page_size, int n_cols,
                           int32_t *out, int64_t out_stride);

/* Prefill-aware sliding-window page table
 * (flashattention_backend.py, `_build_pa_page_table_kernel`):
 *   decode_start = max(pf, sl - window); gap = max(decode_start - pf, 0);
 *   kv_len = sl - gap; dst[i] = req_to_token[req][i < pf ? i : i + gap]
 * for i < kv_len.  Entries of dst at or past kv_len are left untouched.
 * A malformed row -- req outside [0, rtt_rows), a kv_len that does not fit
 * in dst_cols, or a source column past rtt_cols -- is skipped as a whole:
 * left untouched, with kv_lens -1 (the data-dependent faults of the ABI are
 * skipped and flagged, never partly applied).  Returns -1 on bad arguments,
 * else the number of skipped rows. */
int orc_swa_page_table(const int32_t *req_to_token, int64_t rtt_stride,
                       int64_t rtt_cols, int64_t rtt_rows,
                       const int64_t *req_pool_indices,
                       const int32_t *seq_lens, const int32_t *prefill_lens,
                       int batch, int window, int32_t *dst, int64_t dst_stride,
                       int dst_cols, int32_t *kv_lens);

/* Top-k logical index -> physical KV slot (nsa_backend.py,
 * `TopkTransformMethod.PAGED`):
 *   slot = page_table[b][idx / page_size] * page_size + idx % page_size,
 * -1 stays -1.  Row r of `topk` belongs to request row_req[r].  An index
 * < -1 or >= limit[b] (limit = cache_seqlens when given, else
 * pt_cols * page_size) is written as -1 and counted.
 * Returns the number of such out-of-range entries, or -1 on bad arguments. */
int orc_topk_to_slots(const int32_t *topk, int64_t topk_stride, int n_rows,
                      int topk_len, const int32_t *row_req,
                      const int32_t *page_table, int64_t pt_stride,
                      int pt_cols, int page_size,
                      const int32_t *cache_seqlens, int32_t *out,
                      int64_t out_stride);

/* KV write before attention (flashattention_backend.py `forward_extend` /
 * `forward_decode`: `token_to_kv_pool.set_kv_buffer(layer, cache_loc, k, v)`
 * and, for MLA, `set_mla_kv_buffer(layer, cache_loc, k, k_rope)`): new row t
 * (all heads) goes to slot loc[t] of the pool, slot s = page * page_size +
 * position, i.e. cache[s / page_size][s % page_size][h][d] = rows[t][h][d].
 * Called once for K and once for V.  rows: bf16 bits, element (t, h, d) at
 * rows[t*r_st + h*r_sh + d]; cache: bf16 bits, (page, pos, h, d) at
 * cache[page*c_sp + pos*c_spos + h*c_sh + d].  Tokens are written in order
 * (a repeated slot keeps the last row).  A slot outside
 * [0, num_pages * page_size) is skipped and counted.  Returns that count, or
 * -1 on bad arguments. */
int orc_set_kv_buffer(const uint16_t *rows, int64_t r_st, int64_t r_sh, int n_tokens,
                      int heads, int d, const int64_t *loc, uint16_t *cache,
                      int64_t c_sp, int64_t c_spos, int64_t c_sh, int64_t num_pages,
                      int page_size);

/* Local (chunked) attention as virtual batches (flashattention_backend.py,
 * `make_local_attention_virtual_batches` and its worked example):
 *   1. effective chunk C = min(attn_chunk_size, max_b seq_lens[b]), rounded
 *      down to a multiple of page_size, and at least page_size;
 *   2. per request b with q = cu[b+1] - cu[b] new tokens and kv = seq_lens[b]
 *      keys: first = min(C - (kv - q) % C, q) new tokens fall in the chunk
 *      that holds the first new token; the chunk holding the last key has
 *      last_k = kv - C * ((kv - 1) / C) keys; blocks = 1 + ceil((q - first) / C);
 *   3. virtual batch a of request b (a = 0 .. blocks-1, reverse index
 *      r = blocks - 1 - a): q_local = first for a = 0, else
 *      min(q - first - C * (a - 1), C); k_local = last_k for r = 0, else C;
 *      its keys start at kv - last_k - r * C;
 *   4. cu_seqlens_q_local = cu[0] followed by the running sum of q_local;
 *   5. block_table_local row = the C / page_size page ids that cover the
 *      virtual batch's keys, page_table[b][min(start / page_size + j,
 *      pt_cols - 1)] (a column past the row repeats its last entry).
 * Virtual batches are numbered request by request.  A request with q = 0
 * makes none; one with q < 0 makes none and is counted; one with kv < q is
 * counted and its tokens are cut into chunks from the first one (first =
 * min(C, q)) with k_local = 0 and a table row of 0 (attention then gives
 * those tokens the empty-key result).  Rows at
 * or past the count, up to `capacity`, are padding: q_local = k_local = 0,
 * cu repeats the total, table row all 0; table columns at or past
 * C / page_size are 0.  info = {virtual batches, C, max q_local,
 * max k_local} (the count may exceed capacity: only capacity rows exist).
 * Returns the number of requests counted as malformed, or -1 on bad
 * arguments (attn_chunk_size < 1, page_size < 1, pt_cols < 1,
 * bt_cols < C / page_size). */
int orc_local_virtual_batches(int attn_chunk_size, int page_size,
                              const int32_t *cu_seqlens_q,
                              const int32_t *seq_lens, int batch,
                              const int32_t *page_table, int64_t pt_stride,
                              int pt_cols, int capacity,
                              int32_t *seqlens_q_local,
                              int32_t *cu_seqlens_q_local,
                              int32_t *seqlens_k_local,
                              int32_t *block_table_local, int64_t bt_stride,
                              int bt_cols, int32_t *info);

/* Paged attention of new query tokens against a paged KV cache
 * (flashattention_backend.py `forward_decode` / `forward_extend`,
 * nsa_backend.py `forward_decode` for the top-k variant).
 *
 * q:        bf16 bits, element (t, h, d) at q[t*q_st + h*q_sh + d], d < d_qk.
 * k_cache:  bf16 bits, element (page, pos, head, d) at
 *           k[page*k_sp + pos*k_spos + head*k_sh + d], d < d_qk.
 * v_cache:  same with v_* strides, d < d_v.  For absorbed MLA pass the
 *           k buffer again: the value row is the first d_v entries of the
 *           576-wide latent row.
 * page_table: int32 [batch][pt_cols] page ids (row stride pt_stride).
 * cache_seqlens: int32 [batch], total KV length including the new tokens.
 * cu_seqlens_q:  int32 [batch+1], query token offsets.
 * Query token t of request b at local index u = t - cu[b] sits at absolute
 * position i = cache_seqlens[b] - (cu[b+1]-cu[b]) + u (bottom-right causal).
 * Dense key set: j in [0, kv_len); causal => j <= i;
 * window_left >= 0 => i - window_left <= j <= i (window (left, 0), both ends
 * inclusive); attn_chunk > 0 => j / attn_chunk == i / attn_chunk (local
 * chunked attention: a query sees only keys of its own chunk, the mask that
 * flashattention_backend.py draws for `make_local_attention_virtual_batches`).  Top-k (topk != NULL): the keys are the entries of
 * topk[t*topk_stride + 0 .. topk_len), -1 skipped, each occurrence counted,
 * then the same masks; an index < -1 or >= kv_len is skipped and counted.
 * q head h reads kv head h / (h_q / h_kv).
 * s_j = scale * <q, K_j>;  lse = log sum_j exp(s_j);  o = sum_j exp(s_j-lse) V_j.
 * Empty key set: o = 0, lse = -inf.
 *
 * rows: optional list of n_rows (token, head) pairs (int32 pairs) to compute;
 *       NULL computes every (token, head), n_rows ignored.
 * out:  double, [n][d_v] in row order (all rows: n = total_q*h_q, ordered
 *       token-major then head).  lse: double [n] (may be NULL).
 * Returns the number of skipped out-of-range top-k entries or page ids, or
 * a negative value on bad arguments. */
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
                  double *lse, int num_threads);

/* FP8 KV cache (flashattention_backend.py `forward_extend` / `forward_decode`
 * with an fp8 `kv_cache_dtype`: `k_descale` / `v_descale` = the layer's
 * k_scale / v_scale expanded to (batch, KV heads), and q cast to the cache
 * dtype).  Format e4m3 ("fn"): sign, 4 exponent bits (bias 7), 3 mantissa
 * bits, exponent 0 subnormal, codes 0x7f / 0xff NaN, no infinities; largest
 * finite 448. */

/* Value of an e4m3 code (NaN for 0x7f / 0xff). */
double orc_e4m3_value(uint8_t code);

/* Nearest e4m3 code to x, ties to the even code; a magnitude that rounds
 * past 448 (above 464) gives the NaN code, as does NaN. */
uint8_t orc_e4m3_round(double x);

/* The KV write into a pool of fp8 codes (flashattention_backend.py: the
 * layer's k_scale / v_scale passed to set_kv_buffer when kv_cache_dtype is
 * fp8): as orc_set_kv_buffer, except that element (t, h, d) is stored as
 * orc_e4m3_round(x / scale), where x is the bf16 value and the quotient is
 * taken in binary32 (the precision the pool's writer divides in), so that
 * reading the code back as value(code) * scale recovers x to e4m3 precision.
 * cache: uint8 codes at cache[page*c_sp + pos*c_spos + h*c_sh + d].  Returns
 * the skipped-slot count, or -1 on bad arguments (scale not finite and > 0). */
int orc_set_kv_buffer_fp8(const uint16_t *rows, int64_t r_st, int64_t r_sh, int n_tokens,
                          int heads, int d, const int64_t *loc, float scale, uint8_t *cache,
                          int64_t c_sp, int64_t c_spos, int64_t c_sh, int64_t num_pages,
                          int page_size);

/* Attention over an fp8 cache: q rounded to e4m3 (orc_e4m3_round) and widened;
 * K_j = value(k code) * k_descale[b * n_kv_heads + kvh], V_j likewise with
 * v_descale (NULL descales = 1); then the definition of orc_attention (same
 * layouts, masks, bottom-right alignment, top-k lists and empty-key result;
 * the skipped count is per (token, head) row here).
 * k / v: uint8 codes, (page, pos, head, d) at page*sp + pos*spos + head*sh + d. */
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
                      double *out, double *lse, int num_threads);

/* Log-sum-exp state merge (dual_chunk_flashattention_backend.py,
 * `_merge_attn_outputs`; merge_state_v2 in flashattention_backend.py):
 *   m = max(lse_a, lse_b); lse = m + log(exp(lse_a-m) + exp(lse_b-m));
 *   o = exp(lse_a-lse) o_a + exp(lse_b-lse) o_b.
 * Both -inf gives (0, -inf).  Arrays are contiguous [n][d] / [n]. */
int orc_merge_state(const double *v_a, const double *lse_a, const double *v_b,
                    const double *lse_b, int64_t n, int d, double *v_out,
                    double *lse_out);

#ifdef __cplusplus
}
#endif
#endif
