// pkv_internal.h -- parameter blocks and launchers shared by libpkv's
// translation units.  Nothing here is part of the public C ABI (include/pkv.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"  // include/ is on the include path

namespace pkv {

using bf16 = __nv_bfloat16;

constexpr int kNumSMs = 152;        // GB300: 2 dies x 76 SMs
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

#ifdef __CUDACC__
// Launches `kernel` with programmatic stream serialization: it may be
// scheduled while the previous kernel of the stream still runs, and must call
// griddepcontrol.wait (ptx::griddep_wait) before its first global access.
// Used for the short kernels of a decode step, where the launch latency of
// the next kernel is a large part of the step.
template <typename... Params, typename... Args>
cudaError_t launch_programmatic(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// (lo, hi) rounded to e4m3 (nearest, ties to even; magnitudes past 448
// saturate to 448): lo in the low byte of the result.
__device__ __forceinline__ uint32_t round_e4m3x2(float lo, float hi) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(c) : "f"(hi), "f"(lo));
  return c;
}
#endif

// Everything a paged-attention kernel needs, with strides in elements.
struct AttnParams {
  const bf16 *q;
  int64_t q_st, q_sh;                 // token, head strides
  const bf16 *k;
  int64_t k_sp, k_spos, k_sh;         // page, in-page position, head strides
  const bf16 *v;
  int64_t v_sp, v_spos, v_sh;
  int64_t num_pages;
  int page_size;
  const int32_t *page_table;
  int64_t pt_stride;
  int pt_cols;
  const int32_t *cache_seqlens;       // [batch]
  const int32_t *cu_seqlens_q;        // [batch + 1]
  int batch, total_q, h_q, h_kv, group, d, dv;
  int max_seqlen_q;
  float scale;                        // softmax scale
  float scale_log2;                   // scale * log2(e)
  int causal, window_left;
  const int32_t *topk;                // optional [total_q, topk_len]
  int64_t topk_stride;
  int topk_len;
  bf16 *out;
  int64_t o_st, o_sh;
  float *lse;                         // optional
  int64_t lse_st, lse_sh;
  // split-KV
  int num_splits;
  int n_row_tiles;                    // row tiles per (request, kv head)
  float *ws_o;                        // [splits][total_q][h_q][dv] partial O
  float *ws_lse;                      // [splits][total_q][h_q] partial lse
  int32_t *ws_counter;                // [batch][h_kv][n_row_tiles]
  uint32_t *err;                      // device error word
  // fp8 (e4m3) cache: k / v point at byte codes, strides still in elements
  int kv_fp8;
  const float *k_descale;             // optional [batch][h_kv]
  const float *v_descale;             // optional [batch][h_kv]
  // fused KV append (all-heads decode kernel): the new tokens' rows k_new /
  // v_new [total_q][h_kv][d] stand in for the cache rows of their positions
  // and are stored into their slots new_loc[t] by the kernel
  int append;
  const bf16 *k_new;
  int64_t kn_st, kn_sh;
  const bf16 *v_new;
  int64_t vn_st, vn_sh;
  const void *new_loc;
  int new_loc_is64;
  // page table built in the same launch (short decode kernels): page ids are
  // formed from the token pool as the strided table builder forms them,
  // req_to_token[req_pool_indices[b]][c * page_size] / page_size, and the
  // request's row of the table is stored into pt_out (the page_table
  // memory, pt_stride / pt_cols as above)
  const int32_t *rtt;                 // req_to_token [rtt_rows][rtt_cols]
  int64_t rtt_stride, rtt_rows, rtt_cols;
  const void *rpi;                    // req_pool_indices [batch]
  int rpi_is64;
  int32_t *pt_out;
};

// Error word of the current device (static __device__ in pkv_abi.cu).
uint32_t *device_error_word();

// ---- launchers (return a pkv_status) ----
// GQA decode / small-q paged attention on mma.sync tiles.
int launch_decode_gqa(const AttnParams &p, cudaStream_t stream);
// Rows per (request, kv head) tile used by the decode kernel.
constexpr int kDecodeRowTile = 16;
// All-heads decode (head dim 128, <= 8 KV heads, <= 16 query rows per KV
// head; page size < 8 with each slot one contiguous H_kv x 128 row in K and
// in V, or page size a multiple of 16): one CTA covers every KV head of a
// request.  num_splits == 0 selects its balanced persistent schedule:
// the batch's 16-key tiles, laid end to end, are cut into
// kDecodeBalancedShares equal shares, which kDecodeBalancedCtas persistent
// CTAs claim from a counter (batches up to kDecodeBalancedMaxBatch
// requests); fixed splits serve slot rows (all heads per CTA) and page boxes
// (kDecodeFixedSplitHeads heads per CTA).
constexpr int kDecodeBalancedCtas = kNumSMs;
// Shares per CTA of the balanced schedule: finer shares would absorb the
// SMs' different memory service rates, but each split adds a partial state
// and a merge.  Measured with the merges in a background warp: 1 share per
// CTA 0.718 / 0.891 of HBM (sliding-window / GQA decode batches), 2 shares
// 0.600 / 0.843, 4 shares 0.448 / 0.762: the merges cost more than the
// finer balance recovers.
constexpr int kDecodeSharesPerCta = 1;
constexpr int kDecodeBalancedShares = kDecodeBalancedCtas * kDecodeSharesPerCta;
// Page boxes (page size a multiple of 16) with a fixed split count also run on
// the all-heads kernel, kDecodeFixedSplitHeads KV heads per CTA (0: they stay
// on the per-KV-head kernel).  Measured on the GQA decode batch with 4 key
// chunks (64 requests, 8 KV heads): 2 heads 0.849, 4 heads 0.890, 8 heads
// 0.875 of HBM, against 0.782 on the per-KV-head kernel.
constexpr int kDecodeFixedSplitHeads = 4;
constexpr int kDecodeBalancedMaxBatch = 2048;
bool decode_allheads_eligible(const AttnParams &p);
int launch_decode_allheads(const AttnParams &p, cudaStream_t stream);
// Short decode (head dim 128, <= 16 query rows per KV head, bf16 cache, a
// page table of at most kDecodeShortMaxKeys keys, no split): one CTA per
// (request, KV head) with every row loaded up front and the warps' states
// merged in shared memory; no workspace.  Batches of at most
// kDecodeShortClusterMaxPairs (request, KV head) pairs run a 4-CTA cluster
// per pair instead, the keys and value columns split over its CTAs.
constexpr int kDecodeShortMaxKeys = 256;
constexpr int kDecodeShortClusterMaxPairs = 2 * kNumSMs / 4;
bool decode_short_eligible(const AttnParams &p);
int launch_decode_short(const AttnParams &p, cudaStream_t stream);
// tcgen05 varlen extend kernel (head dim 128, whole-page TMA boxes).
bool extend_eligible(const AttnParams &p);
int launch_extend_tc(const AttnParams &p, cudaStream_t stream);
// Query-run length from which the extend kernel serves a call.
constexpr int kExtendMinSeqlenQ = 64;
// tcgen05 absorbed-MLA top-k kernel (128 heads, 576 / 512 dims, one latent
// head; grid = splits x 2 value halves x tokens).
int launch_mla_topk(const AttnParams &p, cudaStream_t stream);
constexpr int kMlaMaxSplits = 64;

int launch_merge_state(const void *va, const void *vb, void *vo, int v_dtype,
                       int o_dtype, int64_t n, int h, int d, int64_t va_sn,
                       int64_t va_sh, int64_t vb_sn, int64_t vb_sh,
                       int64_t vo_sn, int64_t vo_sh, const float *la,
                       int64_t la_sn, int64_t la_sh, const float *lb,
                       int64_t lb_sn, int64_t lb_sh, float *lo, int64_t lo_sn,
                       int64_t lo_sh, cudaStream_t stream);

int launch_swa_page_table(const int32_t *rtt, int64_t rtt_stride,
                          int64_t rtt_rows, int64_t rtt_cols, const void *rpi,
                          int rpi_is_64, const int32_t *seq_lens,
                          const int32_t *prefill_lens, int batch, int window,
                          int32_t *dst, int64_t dst_stride, int dst_cols,
                          int32_t *kv_lens, uint32_t *err,
                          cudaStream_t stream);

int launch_strided_page_table(const int32_t *rtt, int64_t rtt_stride,
                              int64_t rtt_rows, int64_t rtt_cols,
                              const void *rpi, int rpi_is_64, int batch,
                              int page_size, int32_t *out, int64_t out_stride,
                              int n_cols, uint32_t *err, cudaStream_t stream);

// The KV write before attention: rows of k [T, H, dk] / v [T, H, dv] go to
// slot loc[t] = page * page_size + pos of k_cache / v_cache (element strides;
// last dimension contiguous, 16-byte aligned rows, dk and dv multiples of 8).
struct SetKvParams {
  const void *loc;
  int loc_is64;
  int n_tokens, heads, dk, dv;
  const bf16 *k;
  int64_t k_st, k_sh;
  const bf16 *v;
  int64_t v_st, v_sh;
  void *k_cache;  // bf16, or e4m3 codes when fp8
  int64_t kc_sp, kc_spos, kc_sh;
  void *v_cache;
  int64_t vc_sp, vc_spos, vc_sh;
  int64_t num_pages;
  int page_size;
  int fp8;                             // caches hold e4m3 codes
  const float *k_scale, *v_scale;      // fp8: one device float each, or null (1)
  uint32_t *err;
};

int launch_set_kv_buffer(const SetKvParams &p, cudaStream_t stream);

// Largest batch the local-attention virtual batch builder takes (two
// [batch + 1] int32 arrays in shared memory).
constexpr int kLocalBatchesMaxBatch = 16384;

int launch_local_virtual_batches(int attn_chunk_size, int page_size,
                                 const int32_t *cu, const int32_t *seq_lens,
                                 int batch, const int32_t *pt,
                                 int64_t pt_stride, int pt_cols, int capacity,
                                 int32_t *q_local, int32_t *cu_local,
                                 int32_t *k_local, int32_t *bt,
                                 int64_t bt_stride, int bt_cols, int32_t *info,
                                 uint32_t *err, cudaStream_t stream);

int launch_topk_to_slots(const int32_t *topk, int64_t topk_stride,
                         int total_q, int topk_len, const int32_t *cu,
                         int batch, const int32_t *pt, int64_t pt_stride,
                         int pt_cols, const int32_t *cache_seqlens,
                         int page_size, int32_t *out, int64_t out_stride,
                         uint32_t *err, cudaStream_t stream);

}  // namespace pkv
