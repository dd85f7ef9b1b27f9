/*
 * pkv.h -- C ABI of libpkv, paged-KV attention for GB300 (sm_103a).
 *
 * The operations are those of the SGLang attention-backend pages
 * (flashattention_backend.py, dual_chunk_flashattention_backend.py,
 * nsa_backend.py): attention of new query tokens against a paged KV cache,
 * the log-sum-exp state merge, and the integer page-table builders.
 *
 * General rules for every entry point
 * -----------------------------------
 * - Tensors are passed as `pkv_tensor` descriptors: a pointer, a dtype, a
 *   rank and per-dimension sizes and strides counted in ELEMENTS.  All data
 *   pointers are DEVICE pointers on the current CUDA device, owned by the
 *   caller; the library never allocates, frees or retains them.  An optional
 *   tensor is "absent" when its `data` is NULL.
 * - Every call is asynchronous on `stream` (0 = the legacy default stream)
 *   and returns an `int` status: PKV_OK (0) or a negative PKV_ERR_* code.  A
 *   negative status means nothing was launched.  No C++ exception crosses
 *   this boundary.
 * - Stream order is kept.  The short kernels (the strided page table, short
 *   decode) are launched with programmatic stream serialization: they may be
 *   scheduled while the previous kernel on the stream is still running, but
 *   wait for it to complete (griddepcontrol.wait) before their first access
 *   to global memory, so they see everything it wrote.
 * - Data-dependent faults that can only be seen on the device (a page id
 *   outside the KV pool, a top-k index outside [-1, kv_len), a page-table row
 *   too short for its sequence) never trap: the offending entry is skipped
 *   (treated as masked / written as -1) and a sticky bit is set in a device
 *   error word, read with pkv_get_error_flags() after synchronising.
 * - The library keeps no state between calls apart from that error word,
 *   per-device lookups made once, and the fixed scratch array of
 *   pkv_attn_with_kvcache_noalloc (PKV_NOALLOC_SCRATCH_BYTES per device that
 *   loads the library; it keeps the last call's contents and calls of that
 *   entry point that overlap on the GPU race on it: see its comment).  Entry
 *   points may be called from several host threads at once; each call must
 *   own its workspace and outputs, and the error word is shared by all calls
 *   on a device.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ types */

enum pkv_dtype {
  PKV_BF16 = 1, /* bfloat16 */
  PKV_F32 = 2,  /* float32 */
  PKV_I32 = 3,  /* int32 */
  PKV_I64 = 4,  /* int64 */
  PKV_FP8_E4M3 = 5 /* fp8 e4m3 ("fn": bias 7, no infinities, largest 448) codes */
};

enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = -1, /* shape / dtype / stride / value mismatch */
  PKV_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. head dim) */
  PKV_ERR_CUDA = -3,        /* a CUDA runtime call failed */
  PKV_ERR_WORKSPACE = -4    /* workspace missing or too small */
};

/* Bits of the device error word (sticky until pkv_clear_error_flags). */
enum pkv_error_bits {
  PKV_EFLAG_PAGE_OOB = 1,    /* page id outside [0, num_pages): key skipped */
  PKV_EFLAG_TOPK_OOB = 2,    /* top-k index < -1 or >= kv_len: entry skipped */
  PKV_EFLAG_ROW_TOO_SHORT = 4, /* page-table / dst row narrower than needed */
  PKV_EFLAG_SRC_OOB = 8,     /* req_to_token column or pool row out of range */
  PKV_EFLAG_TIMEOUT = 16,    /* a bounded in-kernel wait expired (work dropped) */
  PKV_EFLAG_LAYOUT = 32,     /* shared memory not aligned as a kernel needs (work dropped) */
  PKV_EFLAG_BAD_LENGTHS = 64, /* a request with q_len < 0 or kv_len < q_len */
  PKV_EFLAG_CAPACITY = 128   /* an output with fewer rows than the result needs */
};

typedef struct pkv_tensor {
  void *data;        /* device pointer; NULL = absent (optional tensors) */
  int32_t dtype;     /* enum pkv_dtype */
  int32_t ndim;      /* 1..4 */
  int64_t shape[4];  /* sizes; unused trailing entries ignored */
  int64_t stride[4]; /* strides in elements */
} pkv_tensor;

/* ------------------------------------------------------------- attention */

/*
 * pkv_attn_with_kvcache -- paged attention of new query tokens.
 *
 * Defined by the `flash_attn_with_kvcache` calls of
 * flashattention_backend.py (`forward_decode`, `forward_extend`, the
 * absorbed-MLA call that passes q_rope/k_rope plus q_nope/c_kv) and by the
 * NSA sparse decode of nsa_backend.py (`forward_decode`: top-k lists mapped
 * through the page table, `TopkTransformMethod.PAGED`).
 *
 * For request b (B = cache_seqlens.shape[0]) with q_len_b =
 * cu_seqlens_q[b+1] - cu_seqlens_q[b] new tokens and kv_len_b =
 * cache_seqlens[b] keys (the new tokens included), new token u sits at
 * absolute position i = kv_len_b - q_len_b + u (bottom-right alignment,
 * `seqlens_expanded` in nsa_backend.py).  Query head h reads KV head
 * h / (H_q / H_kv).  Logical key j lives in slot
 *   page_table[b][j / P] * P + j % P,   P = k_cache.shape[1].
 * Visible keys: j < kv_len_b; j <= i if causal; i - window_left <= j <= i
 * if window_left >= 0 (the (window_left, 0) window, both ends inclusive).
 * With topk_indices the keys are instead the entries of that token's row
 * (logical positions; -1 = skip; each occurrence counts), under the same
 * masks.
 *   s_j = scale * <q, K_j>,  lse = ln sum_j exp(s_j),
 *   out = sum_j exp(s_j - lse) V_j;  no visible key: out = 0, lse = -inf.
 *
 * q            bf16 [total_q, H_q, Dq], last dim contiguous.
 * k_cache      bf16 [num_pages, P, H_kv, Dq], last dim contiguous.
 * v_cache      bf16 [num_pages, P, H_kv, Dv], last dim contiguous.  For
 *              absorbed MLA (Dq = 576, Dv = 512, H_kv = 1) pass a view of
 *              the k_cache rows (same pointer and strides, shape[3] = 512).
 * page_table   int32 [B, max_pages] page ids.
 * cache_seqlens int32 [B].
 * cu_seqlens_q int32 [B + 1], non-decreasing, cu[B] <= total_q.
 * max_seqlen_q host int, >= every q_len_b.
 * topk_indices optional int32 [total_q, topk] logical key positions.
 * num_splits   0 = chosen by the library, 1 = no split, k = at most k
 *              contiguous key chunks per (request, KV head), combined by the
 *              log-sum-exp state merge inside the library.
 * out          bf16 [total_q, H_q, Dv] (written).
 * lse          optional fp32 [total_q, H_q], natural log (written).
 * workspace    device scratch of at least pkv_attn_workspace_size(...) bytes
 *              for the same arguments (may be NULL when that size is 0).
 *              Its contents need no initialisation and are clobbered.
 *
 * Supported: Dq = Dv in {64, 128} with H_q % H_kv == 0; and absorbed MLA
 * Dq = 576, Dv = 512, H_kv = 1.  Other shapes return PKV_ERR_UNSUPPORTED.
 * k_cache / v_cache may also be fp8 codes (PKV_FP8_E4M3, both): see
 * pkv_attn_with_kvcache_fp8 (this entry point uses descales of 1).
 * Concurrent calls that share one workspace race.
 */
int pkv_attn_with_kvcache(pkv_tensor q, pkv_tensor k_cache, pkv_tensor v_cache,
                          pkv_tensor page_table, pkv_tensor cache_seqlens,
                          pkv_tensor cu_seqlens_q, int max_seqlen_q,
                          float scale, int causal, int window_left,
                          pkv_tensor topk_indices, int num_splits,
                          pkv_tensor out, pkv_tensor lse, void *workspace,
                          size_t workspace_bytes, cudaStream_t stream);

/*
 * pkv_attn_with_kvcache_fp8 -- paged attention over an fp8 (e4m3) KV cache.
 *
 * Defined by flashattention_backend.py with an fp8 `kv_cache_dtype`
 * (`forward_extend` / `forward_decode`): `k_descale` / `v_descale` are the
 * layer's k_scale / v_scale expanded to (batch, KV heads), and q is cast to
 * the cache dtype before the call.  With K'_j = code_j * k_descale[b][kvh],
 * V'_j = code_j * v_descale[b][kvh] and q' = q rounded to e4m3 (nearest,
 * ties to even): the attention of pkv_attn_with_kvcache over q', K', V'.
 * q must lie within the e4m3 range (|q| <= 448; larger values saturate).
 *
 * k_cache / v_cache  PKV_FP8_E4M3 [num_pages, P, H_kv, 128] codes, last dim
 *                    contiguous, 16-byte aligned rows.
 * k_descale / v_descale device pointers to fp32 [B][H_kv] (row-major,
 *                    contiguous), or NULL for 1.
 * Other arguments, outputs and workspace as pkv_attn_with_kvcache
 * (pkv_attn_workspace_size takes the fp8 tensors as they are).
 * topk_indices (optional, absorbed MLA only) as pkv_attn_with_kvcache.
 * Supported:
 *  - head dim 128, no top-k lists, extend (max_seqlen_q >= 64): page size a
 *    multiple of 8 that divides 128 or is a multiple of 128, strides that
 *    nest (head inside position inside page), any num_splits (no split is
 *    made, no workspace), any sign of scale * k_descale;
 *  - head dim 128, no top-k lists, decode: H_kv <= 8, at most 16 query rows
 *    per KV head (max_seqlen_q * H_q / H_kv), page size < 8 or a multiple of
 *    16, num_splits = 0, B <= 2048;
 *  - absorbed MLA over top-k lists (576 / 512 dims, 128 heads, one latent
 *    head, v_cache the first 512 columns of k_cache): as pkv_attn_with_kvcache,
 *    k_descale / v_descale per request;
 * otherwise PKV_ERR_UNSUPPORTED.
 */
int pkv_attn_with_kvcache_fp8(pkv_tensor q, pkv_tensor k_cache,
                              pkv_tensor v_cache, pkv_tensor page_table,
                              pkv_tensor cache_seqlens, pkv_tensor cu_seqlens_q,
                              int max_seqlen_q, float scale, int causal,
                              int window_left, pkv_tensor topk_indices,
                              const float *k_descale, const float *v_descale,
                              int num_splits, pkv_tensor out, pkv_tensor lse,
                              void *workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/* Bytes of workspace pkv_attn_with_kvcache needs for these sizes (0 if
 * none).  Arguments mirror the attention call's; returns 0 and sets
 * *bytes, or a negative status. */
int pkv_attn_workspace_size(pkv_tensor q, pkv_tensor k_cache,
                            pkv_tensor v_cache, pkv_tensor page_table,
                            pkv_tensor cache_seqlens, int max_seqlen_q,
                            pkv_tensor topk_indices, int num_splits,
                            size_t *bytes);

/* Size of the library-owned scratch array used by
 * pkv_attn_with_kvcache_noalloc (32 MiB per device that loads the library,
 * held until the process exits). */
#define PKV_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * pkv_attn_with_kvcache_noalloc -- pkv_attn_with_kvcache without workspace.
 *
 * The source pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory on this path.  Such callers
 * are handed only their input and output buffers (a plugin interface with
 * no workspace hook), or run under a memory plan that forbids allocating
 * after start-up, or must not call cudaMalloc / cudaFree here because those
 * calls can synchronise the device or fail while another allocator holds
 * the memory.
 *
 * Same arguments, computation, outputs and status codes as
 * pkv_attn_with_kvcache, minus the workspace.  The caller still passes all
 * inputs and outputs.  The split-KV scratch is a fixed array inside the
 * library (PKV_NOALLOC_SCRATCH_BYTES per device); this entry point never
 * allocates or frees device memory.
 * - If the call would need more scratch than PKV_NOALLOC_SCRATCH_BYTES
 *   (pkv_attn_workspace_size for the same arguments), it returns
 *   PKV_ERR_WORKSPACE and launches nothing; ask for fewer splits
 *   (num_splits = 1 needs no scratch).
 * - The first call on a device, with that device current, looks up the
 *   array's device address (cudaGetSymbolAddress) and caches it; make that
 *   first call before any stream capture.
 * - All calls on a device share the array and it keeps the last call's
 *   contents; what must start at zero is cleared by every call.  Calls whose
 *   work overlaps on the GPU (e.g. on two unordered streams) race on it.
 */
int pkv_attn_with_kvcache_noalloc(pkv_tensor q, pkv_tensor k_cache,
                                  pkv_tensor v_cache, pkv_tensor page_table,
                                  pkv_tensor cache_seqlens,
                                  pkv_tensor cu_seqlens_q, int max_seqlen_q,
                                  float scale, int causal, int window_left,
                                  pkv_tensor topk_indices, int num_splits,
                                  pkv_tensor out, pkv_tensor lse,
                                  cudaStream_t stream);

/*
 * pkv_merge_state -- log-sum-exp merge of two attention states.
 *
 * Defined by `_merge_attn_outputs` and the three-way decode merge of
 * dual_chunk_flashattention_backend.py and by the merge_state_v2 call of
 * flashattention_backend.py (cascade decode), per row (n, h):
 *   m = max(lse_a, lse_b);  lse = m + ln(exp(lse_a - m) + exp(lse_b - m));
 *   v = exp(lse_a - lse) v_a + exp(lse_b - lse) v_b;
 * both lse = -inf gives v = 0, lse = -inf.
 *
 * v_a, v_b   bf16 or fp32 [N, H, D], last dim contiguous (same dtype).
 * lse_a/b    fp32 [N, H] (natural log; the transposed FA layout).
 * v_out      bf16 or fp32 [N, H, D].
 * lse_out    optional fp32 [N, H].
 * v_out may alias v_a or v_b (in-place merge); lse_out must not alias
 * lse_a or lse_b (PKV_ERR_INVALID_ARG).  D must be a multiple of 8 with
 * 16-byte aligned rows (PKV_ERR_UNSUPPORTED otherwise).
 */
int pkv_merge_state(pkv_tensor v_a, pkv_tensor lse_a, pkv_tensor v_b,
                    pkv_tensor lse_b, pkv_tensor v_out, pkv_tensor lse_out,
                    cudaStream_t stream);

/* ---------------------------------------------------------- page tables */

/*
 * pkv_build_swa_page_table -- prefill-aware sliding-window page table.
 *
 * Defined by `_build_pa_page_table_kernel` / `_build_pa_page_table` in
 * flashattention_backend.py.  For row b with req = req_pool_indices[b],
 * sl = seq_lens[b], pf = prefill_lens[req]:
 *   decode_start = max(pf, sl - window);  gap = max(decode_start - pf, 0);
 *   kv_len = sl - gap;
 *   dst_page_table[b][i] = req_to_token[req][i < pf ? i : i + gap], i < kv_len;
 *   dst_kv_lens[b] = kv_len.
 * Entries at or past kv_len are not written (in-place refill of caller
 * buffers, as in CUDA-graph replay).
 *
 * req_to_token     int32 [pool_rows, max_ctx].
 * req_pool_indices int32 or int64 [B].
 * seq_lens         int32 [B].
 * prefill_lens     int32 [pool_rows] (indexed through req_pool_indices).
 * window           >= 0 (the model's sliding window, as passed by the page).
 * dst_page_table   int32 [B, W]; a row whose kv_len exceeds W is not
 *                  written, gets dst_kv_lens = -1 and sets
 *                  PKV_EFLAG_ROW_TOO_SHORT.
 * dst_kv_lens      int32 [B].
 * A row whose pool index lies outside [0, pool_rows), or which would read a
 * req_to_token column at or past max_ctx, is likewise not written at all:
 * dst_kv_lens = -1 and PKV_EFLAG_SRC_OOB.
 */
int pkv_build_swa_page_table(pkv_tensor req_to_token,
                             pkv_tensor req_pool_indices, pkv_tensor seq_lens,
                             pkv_tensor prefill_lens, int window,
                             pkv_tensor dst_page_table, pkv_tensor dst_kv_lens,
                             cudaStream_t stream);

/*
 * pkv_strided_page_table -- token-level table to page-level table.
 *
 * Defined in flashattention_backend.py `init_forward_metadata` ("Convert
 * the page table to a strided format"):
 *   out[b][c] = req_to_token[req_pool_indices[b]][c * page_size] / page_size,
 * for c < out.shape[1].  Columns whose source lies past req_to_token's width
 * are written as -1 and set PKV_EFLAG_SRC_OOB.
 *
 * req_to_token int32 [pool_rows, max_ctx]; req_pool_indices int32|int64 [B];
 * out int32 [B, n_cols].
 */
int pkv_strided_page_table(pkv_tensor req_to_token,
                           pkv_tensor req_pool_indices, int page_size,
                           pkv_tensor out, cudaStream_t stream);

/*
 * pkv_strided_table_attn_with_kvcache -- build the page table, then attend.
 *
 * flashattention_backend.py forms the page-level table in
 * `init_forward_metadata` ("Convert the page table to a strided format")
 * and passes it to `flash_attn_with_kvcache` (`forward_decode`).  This call
 * has the result of
 *   pkv_strided_page_table(req_to_token, req_pool_indices, P, page_table)
 *   pkv_attn_with_kvcache(q, k_cache, v_cache, page_table, ...)
 * on one stream, P = k_cache.shape[1]: page_table (int32 [B, n_cols], rows
 * contiguous) is written, the attention reads the pages it names, and the
 * error bits are those of the two calls.  When the short decode kernels
 * serve the attention (head dim 128, at most 16 query rows per KV head, no
 * split, n_cols * P <= 256 keys, a bf16 cache, no top-k lists) both happen
 * in one launch: each CTA forms the page ids it needs from the token pool
 * and the CTAs of KV head 0 store the request's table row; otherwise the
 * builder runs first, then the attention.
 *
 * req_to_token, req_pool_indices  (descriptors passed by host pointer, read
 *          during the call) as pkv_strided_page_table, B entries; NULL is
 *          PKV_ERR_INVALID_ARG.
 * All other arguments as pkv_attn_with_kvcache (page_table is written, not
 * read); the workspace size is pkv_attn_workspace_size of the same
 * attention arguments.
 */
int pkv_strided_table_attn_with_kvcache(pkv_tensor q, pkv_tensor k_cache, pkv_tensor v_cache,
                                        pkv_tensor page_table, pkv_tensor cache_seqlens,
                                        pkv_tensor cu_seqlens_q, int max_seqlen_q, float scale,
                                        int causal, int window_left, pkv_tensor topk_indices,
                                        int num_splits, pkv_tensor out, pkv_tensor lse,
                                        const pkv_tensor *req_to_token,
                                        const pkv_tensor *req_pool_indices, void *workspace,
                                        size_t workspace_bytes, cudaStream_t stream);

/*
 * pkv_topk_to_slots -- top-k logical positions to physical KV slots.
 *
 * Defined by nsa_backend.py `TopkTransformMethod.PAGED` (the page-table
 * transform of `forward_decode`):
 *   out[t][k] = page_table[b][idx / P] * P + idx % P,  idx = topk[t][k],
 * where b is the request of token t (cu_seqlens_q[b] <= t < cu[b+1]);
 * idx = -1 stays -1; idx < -1 or idx >= cache_seqlens[b] is written as -1
 * and sets PKV_EFLAG_TOPK_OOB.
 *
 * topk int32 [total_q, K]; cu_seqlens_q int32 [B+1]; page_table int32
 * [B, max_pages]; cache_seqlens int32 [B]; out int32 [total_q, K].
 */
int pkv_topk_to_slots(pkv_tensor topk, pkv_tensor cu_seqlens_q,
                      pkv_tensor page_table, pkv_tensor cache_seqlens,
                      int page_size, pkv_tensor out, cudaStream_t stream);

/*
 * pkv_set_kv_buffer -- store the new tokens' K/V rows into the paged pool.
 *
 * Defined by the KV write that precedes attention in
 * flashattention_backend.py (`forward_extend` / `forward_decode`:
 * `token_to_kv_pool.set_kv_buffer(layer, cache_loc, k, v, ...)` with
 * `cache_loc = forward_batch.out_cache_loc`; for MLA
 * `set_mla_kv_buffer(layer, cache_loc, k, k_rope)`).  For every new token t
 * and head h, with slot s = loc[t] = page * P + position (P =
 * k_cache.shape[1]):
 *   k_cache[s / P][s % P][h][:] = k[t][h][:],
 *   v_cache[s / P][s % P][h][:] = v[t][h][:]   (when v is given).
 * For absorbed MLA pass k = the nope part [T, 1, 512], v = the rope part
 * [T, 1, 64], k_cache = the first 512 columns of the 576-wide latent pool and
 * v_cache = its last 64 columns (two views of one buffer).
 *
 * loc      int32 or int64 [T] slot ids, distinct (with a repeated slot the
 *          stored row is one of the candidates, unspecified which).
 * k        bf16 [T, H, dk];  v optional bf16 [T, H, dv] (absent: K only).
 * k_cache  bf16 [num_pages, P, H, dk];  v_cache bf16 [num_pages, P, H, dv]
 *          (same num_pages and P), present iff v is.
 * Last dimensions contiguous, rows 16-byte aligned, dk and dv multiples of 8
 * (PKV_ERR_UNSUPPORTED otherwise).  A slot outside [0, num_pages * P) is
 * skipped and sets PKV_EFLAG_PAGE_OOB.  No value is converted: the rows are
 * copied bit for bit.  Pools of fp8 codes (both PKV_FP8_E4M3) are stored as
 * by pkv_set_kv_buffer_fp8 with scales of 1.
 */
int pkv_set_kv_buffer(pkv_tensor loc, pkv_tensor k, pkv_tensor v,
                      pkv_tensor k_cache, pkv_tensor v_cache,
                      cudaStream_t stream);

/*
 * pkv_set_kv_buffer_fp8 -- store the new tokens' rows into a pool of fp8
 * (e4m3) codes.
 *
 * The same write for a pool whose `kv_cache_dtype` is fp8, where the
 * backend passes the layer's `k_scale` / `v_scale` to `set_kv_buffer`
 * (flashattention_backend.py `forward_extend` / `forward_decode`).  Every
 * element is divided by its tensor's scale in fp32 (IEEE division) and
 * rounded to the nearest e4m3 code, ties to even:
 *   k_cache[s / P][s % P][h][c] = e4m3(float(k[t][h][c]) / k_scale),
 * v likewise with v_scale, so that pkv_attn_with_kvcache_fp8 with
 * k_descale = k_scale (and v_descale = v_scale) reads back code * scale.
 * A quotient whose magnitude is 464 or more, which the format cannot hold
 * (torch's conversion gives NaN there), is stored as +-448: such inputs are
 * outside the contract.
 *
 * k_cache / v_cache  PKV_FP8_E4M3 [num_pages, P, H, dk] / [.., dv], else as
 *          pkv_set_kv_buffer (PKV_ERR_INVALID_ARG for any other dtype);
 *          dk and dv multiples of 16.
 * k_scale, v_scale  DEVICE pointers to one fp32 each (finite, > 0), read by
 *          the kernel; NULL means 1.
 */
int pkv_set_kv_buffer_fp8(pkv_tensor loc, pkv_tensor k, pkv_tensor v,
                          pkv_tensor k_cache, pkv_tensor v_cache,
                          const float *k_scale, const float *v_scale,
                          cudaStream_t stream);

/*
 * pkv_append_attn_with_kvcache -- the KV write and the attention in one launch.
 *
 * flashattention_backend.py `forward_decode` (and `forward_extend`) stores the
 * new tokens' K/V with `set_kv_buffer(layer, cache_loc, k, v)` and then runs
 * `flash_attn_with_kvcache` over the cache that holds them.  This call has
 * the same result as pkv_set_kv_buffer(cache_loc, k_new, v_new, k_cache,
 * v_cache) followed by pkv_attn_with_kvcache(... num_splits ...) on one
 * stream, in one kernel: the attention takes the rows of the request's new
 * positions (the last q_len_b of its cache_seqlens[b] keys) from k_new /
 * v_new, and the CTA that covers the request's last key tile stores them
 * into the cache, so that no part of the launch reads a slot while it is
 * being written.
 *
 * k_new, v_new  (descriptors passed by host pointer, read during the call)
 *          bf16 [total_q, H_kv, D] / [total_q, H_kv, Dv]: the rows of
 *          query token t (row t) for the key position
 *          cache_seqlens[b] - q_len_b + (t - cu_seqlens_q[b]); last dimension
 *          contiguous, a token's heads adjacent (stride D / Dv), rows
 *          16-byte aligned.
 * cache_loc (descriptor by host pointer) int32 or int64 [total_q] slots
 *          (page * P + position) of those
 *          positions: they must be the slots the page table maps the
 *          positions to (the kernel reads the new rows' values from k_new /
 *          v_new, not from the slots).  A slot outside [0, num_pages * P) is
 *          skipped and sets PKV_EFLAG_PAGE_OOB.
 * All other arguments as pkv_attn_with_kvcache (the workspace size is
 * pkv_attn_workspace_size of the same call), with bf16 caches only.
 * Served by the all-heads decode kernel (head dim 128, at most 8 KV heads,
 * at most 16 query rows per KV head; page size below 8 with each slot one
 * contiguous H_kv x 128 row, or page size a multiple of 16); other shapes
 * and fp8 caches return PKV_ERR_UNSUPPORTED (use pkv_set_kv_buffer then
 * pkv_attn_with_kvcache).
 */
int pkv_append_attn_with_kvcache(pkv_tensor q, pkv_tensor k_cache, pkv_tensor v_cache,
                                 pkv_tensor page_table, pkv_tensor cache_seqlens,
                                 pkv_tensor cu_seqlens_q, int max_seqlen_q, float scale,
                                 int causal, int window_left, const pkv_tensor *k_new,
                                 const pkv_tensor *v_new, const pkv_tensor *cache_loc,
                                 int num_splits, pkv_tensor out, pkv_tensor lse,
                                 void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * pkv_make_local_attention_virtual_batches -- local (chunked) attention as
 * virtual batches.
 *
 * Defined by `make_local_attention_virtual_batches` in
 * flashattention_backend.py (its docstring, steps and worked example), where
 * local attention lets a query token see only the keys of its own
 * attn_chunk_size-long chunk, up to itself.  Each request's new tokens are
 * cut at chunk boundaries; every piece becomes one "virtual" request whose
 * keys are its chunk's keys up to its last token, so that a plain causal
 * pkv_attn_with_kvcache call over the virtual requests computes local
 * attention.  With B requests, q = cu_seqlens_q[b+1] - cu_seqlens_q[b] and
 * kv = seq_lens[b]:
 *   C      = min(attn_chunk_size, max_b kv) rounded down to a multiple of
 *            page_size, and at least page_size (the effective chunk);
 *   first  = min(C - (kv - q) % C, q) new tokens in the first chunk;
 *   last_k = kv - C * ((kv - 1) / C) keys in the chunk of the last key;
 *   blocks = 1 + ceil((q - first) / C) virtual requests, a = 0 .. blocks-1,
 *            r = blocks - 1 - a:
 *   seqlens_q_local = first (a = 0), else min(q - first - C (a - 1), C);
 *   seqlens_k_local = last_k (r = 0), else C;
 *   block_table_local row = page_table[b][min(s / page_size + j, W - 1)] for
 *            j < C / page_size, s = kv - last_k - r C the chunk's first key
 *            (W = page_table.shape[1]; columns past the row repeat its last
 *            entry, they lie past the virtual request's keys);
 *   cu_seqlens_q_local = cu_seqlens_q[0], then the running sum of
 *            seqlens_q_local.
 * Virtual requests are numbered request by request, so the query rows keep
 * their order and the attention output needs no reordering.  A request with
 * q = 0 makes none.  A request with q < 0 makes none; one with kv < q has its
 * tokens cut from its first token into pieces of at most C with
 * seqlens_k_local = 0 and table rows of 0 (attention gives them out = 0,
 * lse = -inf); both set PKV_EFLAG_BAD_LENGTHS.
 *
 * cu_seqlens_q  int32 [B + 1].   seq_lens int32 [B] (B <= 16384).
 * page_table    int32 [B, W], W >= 1, last dim contiguous.
 * attn_chunk_size >= 1, page_size >= 1.
 * Outputs, sized for a capacity V chosen by the caller (no more than
 * min(total_q, B * (1 + ceil((max_q - 1) / page_size))) rows are needed):
 * seqlens_q_local int32 [V]; cu_seqlens_q_local int32 [V + 1];
 * seqlens_k_local int32 [V]; block_table_local int32 [V, Wl] with
 * Wl >= max(attn_chunk_size / page_size, 1), last dim contiguous;
 * info int32 [4] = {virtual requests, C, max seqlens_q_local,
 * max seqlens_k_local}.
 * Rows past the count are padding: lengths 0, cu repeats the total, table
 * row 0; table columns at or past C / page_size are 0.  If the count
 * exceeds V only V rows are written, info[0] still holds the count and
 * PKV_EFLAG_CAPACITY is set.  Every output entry is written, on the device;
 * the host reads nothing back.
 */
int pkv_make_local_attention_virtual_batches(
    int attn_chunk_size, int page_size, pkv_tensor cu_seqlens_q,
    pkv_tensor seq_lens, pkv_tensor page_table, pkv_tensor seqlens_q_local,
    pkv_tensor cu_seqlens_q_local, pkv_tensor seqlens_k_local,
    pkv_tensor block_table_local, pkv_tensor info, cudaStream_t stream);

/* ------------------------------------------------------------ errors */

/* Reads the current device's error word (synchronous copy; call after the
 * work of interest has completed).  Returns PKV_OK and sets *flags. */
int pkv_get_error_flags(uint32_t *flags);

/* Clears the current device's error word (synchronous). */
int pkv_clear_error_flags(void);

/* Library version, for the bindings' sanity check. */
int pkv_version(void);

/*
 * pkv_check_bounded_wait -- exercises the expiry path of the library's
 * bounded in-kernel waits (no construct of the pages: every pipeline wait
 * of these kernels gives up after about 2^31 SM cycles, about a second at
 * full clock, sets PKV_EFLAG_TIMEOUT and lets the kernel return instead of
 * hanging).  Launches one CTA whose two waiters (the sleeping wait and its
 * cluster-scope variant) wait on a barrier that nothing arrives on; both
 * expire, the flag is set and the kernel ends, leaving the context usable.
 * Asynchronous on `stream`; read the flag after synchronising.  Returns
 * PKV_OK or PKV_ERR_CUDA (launch failure).
 */
int pkv_check_bounded_wait(cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
