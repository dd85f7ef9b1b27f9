// pkv_abi.cu -- the C entry points of libpkv (include/pkv.h): argument
// validation, split-KV planning, workspace carving and kernel dispatch.
// Every step of the computation runs in this library's CUDA kernels.
#include <math.h>

#include <algorithm>

#include <cuda.h>

#include <atomic>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {

bool encode_tensor_map(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims,
                       const cuuint64_t *strides_bytes, const cuuint32_t *box, bool bytes) {
  using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                     const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                     const cuuint32_t *, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);
  // looked up once; a function-local static is initialised thread-safely
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return nullptr;
  }();
  if (fn == nullptr) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
            const_cast<void *>(base), dims,
            strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Sticky device error word (one per device that loads the library).
static __device__ uint32_t g_error_word;

uint32_t *device_error_word() {
  static std::atomic<uint32_t *> cache[64] = {};  // per device; calls may race
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev >= 64) return nullptr;
  uint32_t *word = cache[dev].load(std::memory_order_acquire);
  if (word == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return nullptr;
    word = static_cast<uint32_t *>(ptr);
    cache[dev].store(word, std::memory_order_release);
  }
  return word;
}

namespace {

bool present(const pkv_tensor &t) { return t.data != nullptr; }

bool has(const pkv_tensor &t, int dtype, int ndim) {
  return t.data != nullptr && t.dtype == dtype && t.ndim == ndim;
}

// dimension `dim` steps by one element (any stride when it has <= 1 entry)
bool unit_stride(const pkv_tensor &t, int dim) {
  return t.shape[dim] <= 1 || t.stride[dim] == 1;
}

bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// vector (16-byte) access along the last dimension of a bf16/fp32 tensor
bool vec_ok(const pkv_tensor &t, int elem_bytes) {
  if (!aligned16(t.data)) return false;
  if (t.stride[t.ndim - 1] != 1) return false;
  const int per16 = 16 / elem_bytes;
  for (int i = 0; i < t.ndim - 1; ++i)
    if (t.stride[i] % per16 != 0) return false;
  return true;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct AttnPlan {
  int kind;          // 0 = decode-gqa, 1 = tcgen05 extend, 2 = tcgen05 MLA top-k,
                     // 3 = all-heads small-page decode, 4 = short decode
  int num_splits;    // 0 with kind 3: balanced persistent schedule
  int n_row_tiles;
  size_t ws_o_bytes, ws_lse_bytes, ws_ctr_bytes;
  bool split() const { return num_splits > 1 || (kind == 3 && num_splits == 0); }
  size_t total() const { return split() ? ws_o_bytes + ws_lse_bytes + ws_ctr_bytes : 0; }
};

// Validates the attention arguments (everything but the outputs) and plans
// the launch.  Returns a pkv_status.
int plan_attention(const pkv_tensor &q, const pkv_tensor &k,
                   const pkv_tensor &v, const pkv_tensor &pt,
                   const pkv_tensor &cs, int max_seqlen_q,
                   const pkv_tensor &topk, int num_splits, AttnPlan *plan) {
  // the cache is bf16, or fp8 e4m3 codes (both tensors the same)
  const bool fp8 = k.data != nullptr && k.dtype == PKV_FP8_E4M3;
  const int kv_dtype = fp8 ? PKV_FP8_E4M3 : PKV_BF16;
  if (!has(q, PKV_BF16, 3) || !has(k, kv_dtype, 4) || !has(v, kv_dtype, 4) ||
      !has(pt, PKV_I32, 2) || !has(cs, PKV_I32, 1))
    return PKV_ERR_INVALID_ARG;
  const int64_t total_q = q.shape[0], h_q = q.shape[1], d = q.shape[2];
  const int64_t num_pages = k.shape[0], page = k.shape[1], h_kv = k.shape[2];
  const int64_t dv = v.shape[3];
  const int64_t batch = cs.shape[0];
  if (total_q < 0 || h_q < 1 || d < 1 || num_pages < 1 || page < 1 || h_kv < 1)
    return PKV_ERR_INVALID_ARG;
  if (k.shape[3] != d || v.shape[0] != num_pages || v.shape[1] != page ||
      v.shape[2] != h_kv || h_q % h_kv != 0)
    return PKV_ERR_INVALID_ARG;
  if (pt.shape[0] != batch || pt.stride[1] != 1 || cs.stride[0] != 1)
    return PKV_ERR_INVALID_ARG;
  if (max_seqlen_q < 0 || num_splits < 0) return PKV_ERR_INVALID_ARG;
  if (!vec_ok(q, 2) || !vec_ok(k, fp8 ? 1 : 2) || !vec_ok(v, fp8 ? 1 : 2))
    return PKV_ERR_INVALID_ARG;
  if (present(topk)) {
    if (!has(topk, PKV_I32, 2) || topk.shape[0] != total_q || topk.stride[1] != 1)
      return PKV_ERR_INVALID_ARG;
  }
  if (total_q > 0x7fffffffLL || batch > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;

  const int group = static_cast<int>(h_q / h_kv);
  const bool mla = d == 576 && dv == 512;
  if (fp8 && !mla) {
    // fp8 caches: runs of >= kExtendMinSeqlenQ new tokens on the tcgen05
    // extend kernel (e4m3 QK^T, f16 PV; no split, no workspace); decode on
    // the all-heads kernel with page boxes and its balanced schedule (head
    // dim 128, <= 8 KV heads, <= 16 query rows per KV head, page size a
    // multiple of 16), the library's split choice
    if (present(topk) || d != 128 || dv != 128) return PKV_ERR_UNSUPPORTED;
    AttnParams lx{};
    lx.d = 128;
    lx.dv = 128;
    lx.h_q = static_cast<int>(h_q);
    lx.h_kv = static_cast<int>(h_kv);
    lx.page_size = static_cast<int>(page);
    lx.num_pages = num_pages;
    lx.q_st = q.stride[0];
    lx.q_sh = q.stride[1];
    lx.k_sp = k.stride[0];
    lx.k_spos = k.stride[1];
    lx.k_sh = k.stride[2];
    lx.v_sp = v.stride[0];
    lx.v_spos = v.stride[1];
    lx.v_sh = v.stride[2];
    lx.kv_fp8 = 1;
    if (max_seqlen_q >= kExtendMinSeqlenQ && extend_eligible(lx)) {
      plan->kind = 1;
      plan->num_splits = 1;
      plan->n_row_tiles = 0;
      plan->ws_o_bytes = plan->ws_lse_bytes = plan->ws_ctr_bytes = 0;
      return PKV_OK;
    }
    if (num_splits != 0 || batch > kDecodeBalancedMaxBatch) return PKV_ERR_UNSUPPORTED;
    AttnParams lp{};
    lp.d = 128;
    lp.dv = 128;
    lp.h_q = static_cast<int>(h_q);
    lp.h_kv = static_cast<int>(h_kv);
    lp.group = group;
    lp.max_seqlen_q = max_seqlen_q;
    lp.page_size = static_cast<int>(page);
    lp.num_pages = num_pages;
    lp.k = static_cast<const bf16 *>(k.data);
    lp.v = static_cast<const bf16 *>(v.data);
    lp.k_sp = k.stride[0];
    lp.k_spos = k.stride[1];
    lp.k_sh = k.stride[2];
    lp.v_sp = v.stride[0];
    lp.v_spos = v.stride[1];
    lp.v_sh = v.stride[2];
    lp.kv_fp8 = 1;
    if (max_seqlen_q < 1 || !decode_allheads_eligible(lp)) return PKV_ERR_UNSUPPORTED;
    plan->kind = 3;
    plan->num_splits = 0;
    plan->n_row_tiles = 1;
    const size_t slots = 2ull * kDecodeBalancedShares * max_seqlen_q * h_q;
    plan->ws_o_bytes = align256(slots * dv * 4);
    plan->ws_lse_bytes = align256(slots * 4);
    // merge tickets [batch][h_kv], then the share counter
    plan->ws_ctr_bytes = align256((static_cast<size_t>(batch) * h_kv + 1) * 4);
    return PKV_OK;
  }
  if (mla) {
    // absorbed MLA over top-k lists: 128 heads, one latent head, V = the
    // first 512 columns of the K rows (same buffer and row strides)
    if (!present(topk) || h_q != 128 || h_kv != 1 || v.data != k.data ||
        v.stride[0] != k.stride[0] || v.stride[1] != k.stride[1])
      return PKV_ERR_UNSUPPORTED;
    plan->kind = 2;
    plan->n_row_tiles = 0;
    int splits = num_splits;
    if (splits == 0) {
      // One 2-CTA cluster per (token, split).  Each cluster pays a fixed
      // start (Q into TMEM, the pipeline fill) and a split adds a 256 KB
      // partial and a merge, so lists are split only as far as needed to
      // give every SM pair a cluster, and never below 512 keys a split.
      const int64_t base = std::max<int64_t>(1, total_q);
      splits = static_cast<int>((kNumSMs / 2 + base - 1) / base);
      splits = std::max(1, std::min<int>(splits, static_cast<int>(topk.shape[1] / 512)));
    }
    splits = std::min(splits, kMlaMaxSplits);
    plan->num_splits = splits;
    const size_t rows_total = static_cast<size_t>(total_q) * h_q;
    plan->ws_o_bytes = align256(static_cast<size_t>(splits) * rows_total * dv * 4);
    plan->ws_lse_bytes = align256(static_cast<size_t>(splits) * rows_total * 4);
    plan->ws_ctr_bytes = align256(static_cast<size_t>(total_q) * 4);
    return PKV_OK;
  }
  if (!((d == 128 && dv == 128) || (d == 64 && dv == 64)))
    return PKV_ERR_UNSUPPORTED;

  plan->kind = 0;
  if (!present(topk) && d == 128 && dv == 128) {
    AttnParams lp{};
    lp.d = 128;
    lp.dv = 128;
    lp.h_q = static_cast<int>(h_q);
    lp.h_kv = static_cast<int>(h_kv);
    lp.group = group;
    lp.max_seqlen_q = max_seqlen_q;
    lp.page_size = static_cast<int>(page);
    lp.num_pages = num_pages;
    lp.k = static_cast<const bf16 *>(k.data);
    lp.v = static_cast<const bf16 *>(v.data);
    lp.q_st = q.stride[0];
    lp.q_sh = q.stride[1];
    lp.k_sp = k.stride[0];
    lp.k_spos = k.stride[1];
    lp.k_sh = k.stride[2];
    lp.v_sp = v.stride[0];
    lp.v_spos = v.stride[1];
    lp.v_sh = v.stride[2];
    lp.pt_cols = static_cast<int>(std::min<int64_t>(pt.shape[1], 0x7fffffff));
    if (max_seqlen_q >= kExtendMinSeqlenQ && extend_eligible(lp))
      plan->kind = 1;  // tcgen05 extend, no workspace
    else if (num_splits <= 1 && decode_short_eligible(lp))
      plan->kind = 4;  // short requests: one CTA per (request, KV head), no workspace
    else if (decode_allheads_eligible(lp) &&
             (page < 8 || (num_splits == 0 && batch <= kDecodeBalancedMaxBatch) ||
              (num_splits > 0 && kDecodeFixedSplitHeads > 0 && page % 16 == 0)))
      plan->kind = 3;  // one CTA covers several (or every) KV heads of a request
  }
  if (present(topk)) {
    plan->n_row_tiles = max_seqlen_q * ((group + kDecodeRowTile - 1) / kDecodeRowTile);
  } else {
    const int64_t rows = static_cast<int64_t>(max_seqlen_q) * group;
    plan->n_row_tiles = static_cast<int>((rows + kDecodeRowTile - 1) / kDecodeRowTile);
  }
  int splits = num_splits;
  if (splits == 0) {
    // Enough CTAs for ~4 waves at two resident CTAs per SM (three waves at one
    // per SM for the all-heads kernel), but never chunks shorter than 256 keys.
    const int64_t base = std::max<int64_t>(
        1, plan->kind == 3 ? batch : batch * h_kv * plan->n_row_tiles);
    const int64_t max_keys = present(topk) ? topk.shape[1] : pt.shape[1] * page;
    const int64_t target = plan->kind == 3 ? 3LL * kNumSMs : 4LL * kNumSMs * 2;
    int64_t s = (target + base - 1) / base;
    s = std::min<int64_t>(s, std::max<int64_t>(1, max_keys / 256));
    splits = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(s, 64)));
  }
  splits = std::min(splits, 1024);
  if (plan->kind == 1 || plan->kind == 4) splits = 1;
  plan->num_splits = splits;
  const size_t rows_total = static_cast<size_t>(total_q) * h_q;
  plan->ws_o_bytes = align256(static_cast<size_t>(splits) * rows_total * dv * 4);
  plan->ws_lse_bytes = align256(static_cast<size_t>(splits) * rows_total * 4);
  plan->ws_ctr_bytes =
      align256(static_cast<size_t>(batch) * h_kv * plan->n_row_tiles * 4);
  if (plan->kind == 3 && num_splits == 0 && batch <= kDecodeBalancedMaxBatch) {
    // balanced persistent schedule: per share two partial slots (its first
    // and last request) of one request's rows; the share counter follows the
    // merge tickets
    plan->num_splits = 0;
    const size_t slots = 2ull * kDecodeBalancedShares * max_seqlen_q * h_q;
    plan->ws_o_bytes = align256(slots * dv * 4);
    plan->ws_lse_bytes = align256(slots * 4);
    plan->ws_ctr_bytes = align256((static_cast<size_t>(batch) * h_kv + 1) * 4);
  }
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

namespace pkv {
namespace {
// One CTA whose warps wait on a barrier that nothing arrives on: thread 0
// through the bounded sleeping wait every pipeline wait of the library
// uses, thread 32 through its cluster-scope variant.  Each gives up after
// its bound, records the expiry in the error word and returns.
__global__ void bounded_wait_check_kernel(uint32_t *err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = ptx::smem_addr(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    ptx::mbar_init_fence();
  }
  __syncthreads();
  bool ok = true;
  if (threadIdx.x == 0) ok = ptx::mbar_wait_sleep(b, 0);
  else if (threadIdx.x == 32) ok = ptx::mbar_wait_cluster_sleep(b, 0);
  if (!ok) atomicOr(err, PKV_EFLAG_TIMEOUT);
}
}  // namespace
}  // namespace pkv

extern "C" {

int pkv_version(void) { return 1; }

int pkv_check_bounded_wait(cudaStream_t stream) {
  uint32_t *err = device_error_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  pkv::bounded_wait_check_kernel<<<1, 64, 0, stream>>>(err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_get_error_flags(uint32_t *flags) {
  if (flags == nullptr) return PKV_ERR_INVALID_ARG;
  return cudaMemcpyFromSymbol(flags, g_error_word, sizeof(uint32_t)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

int pkv_clear_error_flags(void) {
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(uint32_t)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

int pkv_attn_workspace_size(pkv_tensor q, pkv_tensor k_cache,
                            pkv_tensor v_cache, pkv_tensor page_table,
                            pkv_tensor cache_seqlens, int max_seqlen_q,
                            pkv_tensor topk_indices, int num_splits,
                            size_t *bytes) {
  if (bytes == nullptr) return PKV_ERR_INVALID_ARG;
  AttnPlan plan;
  const int rc = plan_attention(q, k_cache, v_cache, page_table, cache_seqlens,
                                max_seqlen_q, topk_indices, num_splits, &plan);
  if (rc != PKV_OK) return rc;
  *bytes = plan.total();
  return PKV_OK;
}

}  // extern "C"

namespace pkv {
namespace {

// The new tokens' rows for the fused KV append (pkv_append_attn_with_kvcache).
struct AppendArgs {
  pkv_tensor k_new, v_new, loc;
};
// The token pool of a page table built by the same call
// (pkv_strided_table_attn_with_kvcache).
struct TableArgs {
  pkv_tensor req_to_token, req_pool_indices;
};

int attn_impl(pkv_tensor q, pkv_tensor k_cache, pkv_tensor v_cache, pkv_tensor page_table,
              pkv_tensor cache_seqlens, pkv_tensor cu_seqlens_q, int max_seqlen_q,
              float scale, int causal, int window_left, pkv_tensor topk_indices,
              int num_splits, pkv_tensor k_descale, pkv_tensor v_descale, pkv_tensor out,
              pkv_tensor lse, void *workspace, size_t workspace_bytes, cudaStream_t stream,
              const AppendArgs *app = nullptr, const TableArgs *tab = nullptr) {
  AttnPlan plan;
  int rc = plan_attention(q, k_cache, v_cache, page_table, cache_seqlens,
                          max_seqlen_q, topk_indices, num_splits, &plan);
  if (rc != PKV_OK) return rc;
  const int64_t batch = cache_seqlens.shape[0];
  if (!has(cu_seqlens_q, PKV_I32, 1) || cu_seqlens_q.shape[0] != batch + 1 ||
      cu_seqlens_q.stride[0] != 1)
    return PKV_ERR_INVALID_ARG;
  if (!has(out, PKV_BF16, 3) || out.shape[0] != q.shape[0] ||
      out.shape[1] != q.shape[1] || out.shape[2] != v_cache.shape[3] ||
      !vec_ok(out, 2))
    return PKV_ERR_INVALID_ARG;
  if (present(lse) && (!has(lse, PKV_F32, 2) || lse.shape[0] != q.shape[0] ||
                       lse.shape[1] != q.shape[1]))
    return PKV_ERR_INVALID_ARG;
  if (window_left < -1 || !isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (tab != nullptr) {  // the token pool of a table built by this call
    const pkv_tensor &rtt = tab->req_to_token, &rpi = tab->req_pool_indices;
    if (!has(rtt, PKV_I32, 2) || rtt.stride[1] != 1) return PKV_ERR_INVALID_ARG;
    if (rpi.data == nullptr || rpi.ndim != 1 || (rpi.dtype != PKV_I32 && rpi.dtype != PKV_I64) ||
        rpi.stride[0] != 1 || rpi.shape[0] != batch)
      return PKV_ERR_INVALID_ARG;
  }
  const bool fp8 = k_cache.dtype == PKV_FP8_E4M3;
  for (const pkv_tensor *ds : {&k_descale, &v_descale}) {
    if (!present(*ds)) continue;
    if (!fp8 || !has(*ds, PKV_F32, 2) || ds->shape[0] != batch ||
        ds->shape[1] != k_cache.shape[2] || ds->stride[1] != 1 ||
        ds->stride[0] != k_cache.shape[2])
      return PKV_ERR_INVALID_ARG;
  }
  if (plan.total() > 0 && (workspace == nullptr || workspace_bytes < plan.total() ||
                           (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return PKV_ERR_WORKSPACE;
  uint32_t *err = device_error_word();
  if (err == nullptr) return PKV_ERR_CUDA;

  AttnParams p{};
  p.q = static_cast<const bf16 *>(q.data);
  p.q_st = q.stride[0];
  p.q_sh = q.stride[1];
  p.k = static_cast<const bf16 *>(k_cache.data);
  p.k_sp = k_cache.stride[0];
  p.k_spos = k_cache.stride[1];
  p.k_sh = k_cache.stride[2];
  p.v = static_cast<const bf16 *>(v_cache.data);
  p.v_sp = v_cache.stride[0];
  p.v_spos = v_cache.stride[1];
  p.v_sh = v_cache.stride[2];
  p.num_pages = k_cache.shape[0];
  p.page_size = static_cast<int>(k_cache.shape[1]);
  p.page_table = static_cast<const int32_t *>(page_table.data);
  p.pt_stride = page_table.stride[0];
  p.pt_cols = static_cast<int>(page_table.shape[1]);
  p.cache_seqlens = static_cast<const int32_t *>(cache_seqlens.data);
  p.cu_seqlens_q = static_cast<const int32_t *>(cu_seqlens_q.data);
  p.batch = static_cast<int>(batch);
  p.total_q = static_cast<int>(q.shape[0]);
  p.h_q = static_cast<int>(q.shape[1]);
  p.h_kv = static_cast<int>(k_cache.shape[2]);
  p.group = p.h_q / p.h_kv;
  p.d = static_cast<int>(q.shape[2]);
  p.dv = static_cast<int>(v_cache.shape[3]);
  p.max_seqlen_q = max_seqlen_q;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.causal = causal ? 1 : 0;
  p.window_left = window_left;
  if (present(topk_indices)) {
    p.topk = static_cast<const int32_t *>(topk_indices.data);
    p.topk_stride = topk_indices.stride[0];
    p.topk_len = static_cast<int>(topk_indices.shape[1]);
  }
  p.out = static_cast<bf16 *>(out.data);
  p.o_st = out.stride[0];
  p.o_sh = out.stride[1];
  if (present(lse)) {
    p.lse = static_cast<float *>(lse.data);
    p.lse_st = lse.stride[0];
    p.lse_sh = lse.stride[1];
  }
  p.num_splits = plan.num_splits;
  p.n_row_tiles = plan.n_row_tiles;
  p.err = err;
  p.kv_fp8 = fp8 ? 1 : 0;
  p.k_descale = static_cast<const float *>(k_descale.data);
  p.v_descale = static_cast<const float *>(v_descale.data);
  if (app != nullptr) {
    // fused KV append: bf16 caches on the all-heads decode kernel (short
    // batches too, unsplit: no workspace, as planned)
    const int64_t T = q.shape[0], hkv = k_cache.shape[2];
    const int64_t dk = k_cache.shape[3], dvv = v_cache.shape[3];
    if (plan.kind == 4 && decode_allheads_eligible(p)) {
      plan.kind = 3;
      plan.num_splits = 1;
      p.num_splits = 1;
    }
    if (fp8 || plan.kind != 3) return PKV_ERR_UNSUPPORTED;
    if (!has(app->k_new, PKV_BF16, 3) || !has(app->v_new, PKV_BF16, 3) ||
        app->k_new.shape[0] != T || app->k_new.shape[1] != hkv || app->k_new.shape[2] != dk ||
        app->v_new.shape[0] != T || app->v_new.shape[1] != hkv || app->v_new.shape[2] != dvv ||
        !vec_ok(app->k_new, 2) || !vec_ok(app->v_new, 2))
      return PKV_ERR_INVALID_ARG;
    if (app->loc.data == nullptr || app->loc.ndim != 1 || app->loc.shape[0] != T ||
        (app->loc.dtype != PKV_I32 && app->loc.dtype != PKV_I64) || !unit_stride(app->loc, 0))
      return PKV_ERR_INVALID_ARG;
    // a token's heads contiguous (slot rows copy a new row with one bulk copy)
    if (app->k_new.stride[1] != dk || app->v_new.stride[1] != dvv) return PKV_ERR_UNSUPPORTED;
    p.append = 1;
    p.k_new = static_cast<const bf16 *>(app->k_new.data);
    p.kn_st = app->k_new.stride[0];
    p.kn_sh = app->k_new.stride[1];
    p.v_new = static_cast<const bf16 *>(app->v_new.data);
    p.vn_st = app->v_new.stride[0];
    p.vn_sh = app->v_new.stride[1];
    p.new_loc = app->loc.data;
    p.new_loc_is64 = app->loc.dtype == PKV_I64 ? 1 : 0;
  }
  if (tab != nullptr) {
    // the page table is built from the token pool first: by the short
    // kernels inside the attention launch, else by the strided builder
    const pkv_tensor &rtt = tab->req_to_token, &rpi = tab->req_pool_indices;
    if (plan.kind == 4 && p.total_q > 0) {
      p.rtt = static_cast<const int32_t *>(rtt.data);
      p.rtt_stride = rtt.stride[0];
      p.rtt_rows = rtt.shape[0];
      p.rtt_cols = rtt.shape[1];
      p.rpi = rpi.data;
      p.rpi_is64 = rpi.dtype == PKV_I64 ? 1 : 0;
      p.pt_out = static_cast<int32_t *>(page_table.data);
    } else {
      if (batch > 65535) return PKV_ERR_UNSUPPORTED;
      rc = launch_strided_page_table(
          static_cast<const int32_t *>(rtt.data), rtt.stride[0], rtt.shape[0], rtt.shape[1],
          rpi.data, rpi.dtype == PKV_I64, static_cast<int>(batch), p.page_size,
          static_cast<int32_t *>(page_table.data), page_table.stride[0], p.pt_cols, err, stream);
      if (rc != PKV_OK) return rc;
    }
  }
  if (plan.split()) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.ws_o = reinterpret_cast<float *>(ws);
    p.ws_lse = reinterpret_cast<float *>(ws + plan.ws_o_bytes);
    p.ws_counter = reinterpret_cast<int32_t *>(ws + plan.ws_o_bytes + plan.ws_lse_bytes);
    if (cudaMemsetAsync(p.ws_counter, 0, plan.ws_ctr_bytes, stream) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  if (p.total_q == 0) return PKV_OK;
  if (plan.kind == 2) return launch_mla_topk(p, stream);
  if (plan.kind == 3) return launch_decode_allheads(p, stream);
  if (plan.kind == 4) return launch_decode_short(p, stream);
  if (plan.kind == 1 && fp8) return launch_extend_tc(p, stream);  // any scale sign
  if (plan.kind == 1) {
    // the bf16 extend kernel takes row maxima of raw scores: positive scale
    // only (the decode kernel serves the others)
    rc = scale > 0.f ? launch_extend_tc(p, stream) : PKV_ERR_UNSUPPORTED;
    if (rc != PKV_ERR_UNSUPPORTED) return rc;
    p.num_splits = 1;  // otherwise the unsplit decode kernel (no workspace)
  }
  return launch_decode_gqa(p, stream);
}

}  // namespace
}  // namespace pkv

extern "C" {

int pkv_attn_with_kvcache(pkv_tensor q, pkv_tensor k_cache, pkv_tensor v_cache,
                          pkv_tensor page_table, pkv_tensor cache_seqlens,
                          pkv_tensor cu_seqlens_q, int max_seqlen_q,
                          float scale, int causal, int window_left,
                          pkv_tensor topk_indices, int num_splits,
                          pkv_tensor out, pkv_tensor lse, void *workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  const pkv_tensor none{};
  return pkv::attn_impl(q, k_cache, v_cache, page_table, cache_seqlens, cu_seqlens_q,
                        max_seqlen_q, scale, causal, window_left, topk_indices, num_splits,
                        none, none, out, lse, workspace, workspace_bytes, stream);
}

int pkv_append_attn_with_kvcache(pkv_tensor q, pkv_tensor k_cache, pkv_tensor v_cache,
                                 pkv_tensor page_table, pkv_tensor cache_seqlens,
                                 pkv_tensor cu_seqlens_q, int max_seqlen_q, float scale,
                                 int causal, int window_left, const pkv_tensor *k_new,
                                 const pkv_tensor *v_new, const pkv_tensor *cache_loc,
                                 int num_splits, pkv_tensor out, pkv_tensor lse,
                                 void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (k_new == nullptr || v_new == nullptr || cache_loc == nullptr) return PKV_ERR_INVALID_ARG;
  const pkv_tensor none{};
  const pkv::AppendArgs app{*k_new, *v_new, *cache_loc};
  return pkv::attn_impl(q, k_cache, v_cache, page_table, cache_seqlens, cu_seqlens_q,
                        max_seqlen_q, scale, causal, window_left, none, num_splits, none, none,
                        out, lse, workspace, workspace_bytes, stream, &app);
}

int pkv_attn_with_kvcache_fp8(pkv_tensor q, pkv_tensor k_cache, pkv_tensor v_cache,
                              pkv_tensor page_table, pkv_tensor cache_seqlens,
                              pkv_tensor cu_seqlens_q, int max_seqlen_q, float scale,
                              int causal, int window_left, pkv_tensor topk_indices,
                              const float *k_descale, const float *v_descale, int num_splits,
                              pkv_tensor out, pkv_tensor lse, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  if (k_cache.data == nullptr || k_cache.dtype != PKV_FP8_E4M3 || k_cache.ndim != 4 ||
      cache_seqlens.data == nullptr || cache_seqlens.ndim != 1)
    return PKV_ERR_INVALID_ARG;
  // the descales as [B][H_kv] fp32 descriptors (contiguous rows)
  pkv_tensor kd{}, vd{};
  for (int i = 0; i < 2; ++i) {
    pkv_tensor &t = i == 0 ? kd : vd;
    t.data = const_cast<float *>(i == 0 ? k_descale : v_descale);
    t.dtype = PKV_F32;
    t.ndim = 2;
    t.shape[0] = cache_seqlens.shape[0];
    t.shape[1] = k_cache.shape[2];
    t.stride[0] = k_cache.shape[2];
    t.stride[1] = 1;
  }
  return pkv::attn_impl(q, k_cache, v_cache, page_table, cache_seqlens, cu_seqlens_q,
                        max_seqlen_q, scale, causal, window_left, topk_indices, num_splits, kd,
                        vd, out, lse, workspace, workspace_bytes, stream);
}

int pkv_merge_state(pkv_tensor v_a, pkv_tensor lse_a, pkv_tensor v_b,
                    pkv_tensor lse_b, pkv_tensor v_out, pkv_tensor lse_out,
                    cudaStream_t stream) {
  if (v_a.data == nullptr || v_b.data == nullptr || v_out.data == nullptr)
    return PKV_ERR_INVALID_ARG;
  if (v_a.ndim != 3 || v_b.ndim != 3 || v_out.ndim != 3) return PKV_ERR_INVALID_ARG;
  if (v_a.dtype != v_b.dtype || (v_a.dtype != PKV_BF16 && v_a.dtype != PKV_F32) ||
      (v_out.dtype != PKV_BF16 && v_out.dtype != PKV_F32))
    return PKV_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i)
    if (v_b.shape[i] != v_a.shape[i] || v_out.shape[i] != v_a.shape[i])
      return PKV_ERR_INVALID_ARG;
  const int64_t n = v_a.shape[0], h = v_a.shape[1], d = v_a.shape[2];
  if (!has(lse_a, PKV_F32, 2) || !has(lse_b, PKV_F32, 2) || lse_a.shape[0] != n ||
      lse_a.shape[1] != h || lse_b.shape[0] != n || lse_b.shape[1] != h)
    return PKV_ERR_INVALID_ARG;
  if (present(lse_out) && (!has(lse_out, PKV_F32, 2) || lse_out.shape[0] != n ||
                           lse_out.shape[1] != h))
    return PKV_ERR_INVALID_ARG;
  if (present(lse_out) && (lse_out.data == lse_a.data || lse_out.data == lse_b.data))
    return PKV_ERR_INVALID_ARG;
  const int eb_in = v_a.dtype == PKV_BF16 ? 2 : 4;
  const int eb_out = v_out.dtype == PKV_BF16 ? 2 : 4;
  if (d % 8 != 0 || !vec_ok(v_a, eb_in) || !vec_ok(v_b, eb_in) || !vec_ok(v_out, eb_out))
    return PKV_ERR_UNSUPPORTED;
  if (h > 0x7fffffffLL || d > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  return launch_merge_state(
      v_a.data, v_b.data, v_out.data, v_a.dtype, v_out.dtype, n,
      static_cast<int>(h), static_cast<int>(d), v_a.stride[0], v_a.stride[1],
      v_b.stride[0], v_b.stride[1], v_out.stride[0], v_out.stride[1],
      static_cast<const float *>(lse_a.data), lse_a.stride[0], lse_a.stride[1],
      static_cast<const float *>(lse_b.data), lse_b.stride[0], lse_b.stride[1],
      static_cast<float *>(lse_out.data), present(lse_out) ? lse_out.stride[0] : 0,
      present(lse_out) ? lse_out.stride[1] : 0, stream);
}

int pkv_build_swa_page_table(pkv_tensor req_to_token,
                             pkv_tensor req_pool_indices, pkv_tensor seq_lens,
                             pkv_tensor prefill_lens, int window,
                             pkv_tensor dst_page_table, pkv_tensor dst_kv_lens,
                             cudaStream_t stream) {
  if (!has(req_to_token, PKV_I32, 2) || req_to_token.stride[1] != 1)
    return PKV_ERR_INVALID_ARG;
  if (req_pool_indices.data == nullptr || req_pool_indices.ndim != 1 ||
      (req_pool_indices.dtype != PKV_I32 && req_pool_indices.dtype != PKV_I64) ||
      req_pool_indices.stride[0] != 1)
    return PKV_ERR_INVALID_ARG;
  const int64_t batch = req_pool_indices.shape[0];
  if (!has(seq_lens, PKV_I32, 1) || seq_lens.shape[0] != batch || seq_lens.stride[0] != 1)
    return PKV_ERR_INVALID_ARG;
  if (!has(prefill_lens, PKV_I32, 1) || prefill_lens.shape[0] != req_to_token.shape[0] ||
      prefill_lens.stride[0] != 1)
    return PKV_ERR_INVALID_ARG;
  if (!has(dst_page_table, PKV_I32, 2) || dst_page_table.shape[0] != batch ||
      dst_page_table.stride[1] != 1)
    return PKV_ERR_INVALID_ARG;
  if (!has(dst_kv_lens, PKV_I32, 1) || dst_kv_lens.shape[0] != batch ||
      dst_kv_lens.stride[0] != 1)
    return PKV_ERR_INVALID_ARG;
  if (window < 0) return PKV_ERR_INVALID_ARG;
  if (batch > 0x7fffffffLL || dst_page_table.shape[1] > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;
  uint32_t *err = device_error_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  return launch_swa_page_table(
      static_cast<const int32_t *>(req_to_token.data), req_to_token.stride[0],
      req_to_token.shape[0], req_to_token.shape[1], req_pool_indices.data,
      req_pool_indices.dtype == PKV_I64, static_cast<const int32_t *>(seq_lens.data),
      static_cast<const int32_t *>(prefill_lens.data), static_cast<int>(batch), window,
      static_cast<int32_t *>(dst_page_table.data), dst_page_table.stride[0],
      static_cast<int>(dst_page_table.shape[1]),
      static_cast<int32_t *>(dst_kv_lens.data), err, stream);
}

int pkv_strided_table_attn_with_kvcache(pkv_tensor q, pkv_tensor k_cache, pkv_tensor v_cache,
                                        pkv_tensor page_table, pkv_tensor cache_seqlens,
                                        pkv_tensor cu_seqlens_q, int max_seqlen_q, float scale,
                                        int causal, int window_left, pkv_tensor topk_indices,
                                        int num_splits, pkv_tensor out, pkv_tensor lse,
                                        const pkv_tensor *req_to_token,
                                        const pkv_tensor *req_pool_indices, void *workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
  if (req_to_token == nullptr || req_pool_indices == nullptr) return PKV_ERR_INVALID_ARG;
  const pkv_tensor none{};
  const pkv::TableArgs tab{*req_to_token, *req_pool_indices};
  return pkv::attn_impl(q, k_cache, v_cache, page_table, cache_seqlens, cu_seqlens_q,
                        max_seqlen_q, scale, causal, window_left, topk_indices, num_splits,
                        none, none, out, lse, workspace, workspace_bytes, stream, nullptr, &tab);
}

int pkv_strided_page_table(pkv_tensor req_to_token,
                           pkv_tensor req_pool_indices, int page_size,
                           pkv_tensor out, cudaStream_t stream) {
  if (!has(req_to_token, PKV_I32, 2) || req_to_token.stride[1] != 1)
    return PKV_ERR_INVALID_ARG;
  if (req_pool_indices.data == nullptr || req_pool_indices.ndim != 1 ||
      (req_pool_indices.dtype != PKV_I32 && req_pool_indices.dtype != PKV_I64) ||
      req_pool_indices.stride[0] != 1)
    return PKV_ERR_INVALID_ARG;
  const int64_t batch = req_pool_indices.shape[0];
  if (!has(out, PKV_I32, 2) || out.shape[0] != batch || out.stride[1] != 1)
    return PKV_ERR_INVALID_ARG;
  if (page_size < 1) return PKV_ERR_INVALID_ARG;
  if (batch > 65535 || out.shape[1] > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  uint32_t *err = device_error_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  return launch_strided_page_table(
      static_cast<const int32_t *>(req_to_token.data), req_to_token.stride[0],
      req_to_token.shape[0], req_to_token.shape[1], req_pool_indices.data,
      req_pool_indices.dtype == PKV_I64, static_cast<int>(batch), page_size,
      static_cast<int32_t *>(out.data), out.stride[0],
      static_cast<int>(out.shape[1]), err, stream);
}

int pkv_topk_to_slots(pkv_tensor topk, pkv_tensor cu_seqlens_q,
                      pkv_tensor page_table, pkv_tensor cache_seqlens,
                      int page_size, pkv_tensor out, cudaStream_t stream) {
  if (!has(topk, PKV_I32, 2) || topk.stride[1] != 1) return PKV_ERR_INVALID_ARG;
  if (!has(cache_seqlens, PKV_I32, 1) || cache_seqlens.stride[0] != 1)
    return PKV_ERR_INVALID_ARG;
  const int64_t batch = cache_seqlens.shape[0];
  if (!has(cu_seqlens_q, PKV_I32, 1) || cu_seqlens_q.shape[0] != batch + 1 ||
      cu_seqlens_q.stride[0] != 1)
    return PKV_ERR_INVALID_ARG;
  if (!has(page_table, PKV_I32, 2) || page_table.shape[0] != batch ||
      page_table.stride[1] != 1)
    return PKV_ERR_INVALID_ARG;
  if (!has(out, PKV_I32, 2) || out.shape[0] != topk.shape[0] ||
      out.shape[1] != topk.shape[1] || out.stride[1] != 1)
    return PKV_ERR_INVALID_ARG;
  if (page_size < 1) return PKV_ERR_INVALID_ARG;
  if (topk.shape[0] > 0x7fffffffLL || topk.shape[1] > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;
  uint32_t *err = device_error_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  return launch_topk_to_slots(
      static_cast<const int32_t *>(topk.data), topk.stride[0],
      static_cast<int>(topk.shape[0]), static_cast<int>(topk.shape[1]),
      static_cast<const int32_t *>(cu_seqlens_q.data), static_cast<int>(batch),
      static_cast<const int32_t *>(page_table.data), page_table.stride[0],
      static_cast<int>(page_table.shape[1]),
      static_cast<const int32_t *>(cache_seqlens.data), page_size,
      static_cast<int32_t *>(out.data), out.stride[0], err, stream);
}

namespace pkv {
namespace {

int set_kv_impl(pkv_tensor loc, pkv_tensor k, pkv_tensor v, pkv_tensor k_cache,
                pkv_tensor v_cache, const float *k_scale, const float *v_scale,
                bool want_fp8, cudaStream_t stream) {
  if (loc.data == nullptr || loc.ndim != 1 || (loc.dtype != PKV_I32 && loc.dtype != PKV_I64) ||
      !unit_stride(loc, 0))
    return PKV_ERR_INVALID_ARG;
  const int64_t T = loc.shape[0];
  // the pool's type: bf16 rows, or e4m3 codes (both pools alike)
  const bool fp8 = k_cache.data != nullptr && k_cache.dtype == PKV_FP8_E4M3;
  if (want_fp8 && !fp8) return PKV_ERR_INVALID_ARG;
  const int cdt = fp8 ? PKV_FP8_E4M3 : PKV_BF16;
  const int ces = fp8 ? 1 : 2;  // cache bytes per element
  if (!has(k, PKV_BF16, 3) || !has(k_cache, cdt, 4)) return PKV_ERR_INVALID_ARG;
  if (present(v) != present(v_cache)) return PKV_ERR_INVALID_ARG;
  const int64_t H = k.shape[1], dk = k.shape[2];
  if (k.shape[0] != T || k_cache.shape[2] != H || k_cache.shape[3] != dk)
    return PKV_ERR_INVALID_ARG;
  int64_t dv = 0;
  if (present(v)) {
    if (!has(v, PKV_BF16, 3) || !has(v_cache, cdt, 4)) return PKV_ERR_INVALID_ARG;
    dv = v.shape[2];
    if (v.shape[0] != T || v.shape[1] != H || v_cache.shape[0] != k_cache.shape[0] ||
        v_cache.shape[1] != k_cache.shape[1] || v_cache.shape[2] != H ||
        v_cache.shape[3] != dv)
      return PKV_ERR_INVALID_ARG;
  }
  const int64_t epp = fp8 ? 16 : 8;  // elements per 16-byte piece of the pool
  if (dk % epp != 0 || dv % epp != 0 || !vec_ok(k, 2) || !vec_ok(k_cache, ces) ||
      (present(v) && (!vec_ok(v, 2) || !vec_ok(v_cache, ces))))
    return PKV_ERR_UNSUPPORTED;
  if (T > 0x7fffffffLL || H > 0x7fffffffLL || dk > 0x7fffffffLL || dv > 0x7fffffffLL ||
      k_cache.shape[1] > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;
  uint32_t *err = device_error_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  SetKvParams p{};
  p.loc = loc.data;
  p.loc_is64 = loc.dtype == PKV_I64;
  p.n_tokens = static_cast<int>(T);
  p.heads = static_cast<int>(H);
  p.dk = static_cast<int>(dk);
  p.dv = static_cast<int>(dv);
  p.k = static_cast<const bf16 *>(k.data);
  p.k_st = k.stride[0];
  p.k_sh = k.stride[1];
  p.k_cache = k_cache.data;
  p.kc_sp = k_cache.stride[0];
  p.kc_spos = k_cache.stride[1];
  p.kc_sh = k_cache.stride[2];
  if (present(v)) {
    p.v = static_cast<const bf16 *>(v.data);
    p.v_st = v.stride[0];
    p.v_sh = v.stride[1];
    p.v_cache = v_cache.data;
    p.vc_sp = v_cache.stride[0];
    p.vc_spos = v_cache.stride[1];
    p.vc_sh = v_cache.stride[2];
  }
  p.num_pages = k_cache.shape[0];
  p.page_size = static_cast<int>(k_cache.shape[1]);
  p.fp8 = fp8 ? 1 : 0;
  p.k_scale = fp8 ? k_scale : nullptr;
  p.v_scale = fp8 ? v_scale : nullptr;
  p.err = err;
  return launch_set_kv_buffer(p, stream);
}

}  // namespace
}  // namespace pkv

int pkv_set_kv_buffer(pkv_tensor loc, pkv_tensor k, pkv_tensor v,
                      pkv_tensor k_cache, pkv_tensor v_cache,
                      cudaStream_t stream) {
  return set_kv_impl(loc, k, v, k_cache, v_cache, nullptr, nullptr, false, stream);
}

int pkv_set_kv_buffer_fp8(pkv_tensor loc, pkv_tensor k, pkv_tensor v,
                          pkv_tensor k_cache, pkv_tensor v_cache,
                          const float *k_scale, const float *v_scale,
                          cudaStream_t stream) {
  return set_kv_impl(loc, k, v, k_cache, v_cache, k_scale, v_scale, true, stream);
}

int pkv_make_local_attention_virtual_batches(
    int attn_chunk_size, int page_size, pkv_tensor cu_seqlens_q,
    pkv_tensor seq_lens, pkv_tensor page_table, pkv_tensor seqlens_q_local,
    pkv_tensor cu_seqlens_q_local, pkv_tensor seqlens_k_local,
    pkv_tensor block_table_local, pkv_tensor info, cudaStream_t stream) {
  if (attn_chunk_size < 1 || page_size < 1) return PKV_ERR_INVALID_ARG;
  if (!has(seq_lens, PKV_I32, 1) || !unit_stride(seq_lens, 0)) return PKV_ERR_INVALID_ARG;
  const int64_t batch = seq_lens.shape[0];
  if (!has(cu_seqlens_q, PKV_I32, 1) || cu_seqlens_q.shape[0] != batch + 1 ||
      !unit_stride(cu_seqlens_q, 0))
    return PKV_ERR_INVALID_ARG;
  if (!has(page_table, PKV_I32, 2) || page_table.shape[0] != batch ||
      page_table.shape[1] < 1 || !unit_stride(page_table, 1))
    return PKV_ERR_INVALID_ARG;
  if (!has(seqlens_q_local, PKV_I32, 1) || !unit_stride(seqlens_q_local, 0))
    return PKV_ERR_INVALID_ARG;
  const int64_t cap = seqlens_q_local.shape[0];
  if (!has(cu_seqlens_q_local, PKV_I32, 1) || cu_seqlens_q_local.shape[0] != cap + 1 ||
      !unit_stride(cu_seqlens_q_local, 0))
    return PKV_ERR_INVALID_ARG;
  if (!has(seqlens_k_local, PKV_I32, 1) || seqlens_k_local.shape[0] != cap ||
      !unit_stride(seqlens_k_local, 0))
    return PKV_ERR_INVALID_ARG;
  const int64_t min_cols = attn_chunk_size / page_size > 1 ? attn_chunk_size / page_size : 1;
  if (!has(block_table_local, PKV_I32, 2) || block_table_local.shape[0] != cap ||
      block_table_local.shape[1] < min_cols || !unit_stride(block_table_local, 1))
    return PKV_ERR_INVALID_ARG;
  if (!has(info, PKV_I32, 1) || info.shape[0] < 4 || !unit_stride(info, 0))
    return PKV_ERR_INVALID_ARG;
  if (batch > kLocalBatchesMaxBatch || cap > 0x7fffffffLL ||
      page_table.shape[1] > 0x7fffffffLL || block_table_local.shape[1] > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;
  uint32_t *err = device_error_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  return launch_local_virtual_batches(
      attn_chunk_size, page_size, static_cast<const int32_t *>(cu_seqlens_q.data),
      static_cast<const int32_t *>(seq_lens.data), static_cast<int>(batch),
      static_cast<const int32_t *>(page_table.data), page_table.stride[0],
      static_cast<int>(page_table.shape[1]), static_cast<int>(cap),
      static_cast<int32_t *>(seqlens_q_local.data),
      static_cast<int32_t *>(cu_seqlens_q_local.data),
      static_cast<int32_t *>(seqlens_k_local.data),
      static_cast<int32_t *>(block_table_local.data), block_table_local.stride[0],
      static_cast<int>(block_table_local.shape[1]), static_cast<int32_t *>(info.data), err,
      stream);
}

}  // extern "C"
