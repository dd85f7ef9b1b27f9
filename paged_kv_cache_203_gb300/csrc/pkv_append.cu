// pkv_append.cu -- the KV write that precedes attention: each new token's
// K and V rows (all KV heads) are stored into their pool slots
// (flashattention_backend.py `forward_extend` / `forward_decode`:
// `token_to_kv_pool.set_kv_buffer(layer, cache_loc, k, v)`; for MLA
// `set_mla_kv_buffer(layer, cache_loc, k, k_rope)`, the nope and rope parts
// of one 576-wide latent row, written here as two column ranges).
//
// HBM-bound scatter: every thread moves 16-byte pieces of one (token, head)
// row; a token's K pieces and V pieces are contiguous in the thread index, so
// a warp stores whole 256-byte rows.  The slot is loaded once per thread
// (L1 broadcast within the row).
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ int64_t load_slot(const void *p, int is64, int64_t i) {
  return is64 ? static_cast<const int64_t *>(p)[i]
              : static_cast<int64_t>(static_cast<const int32_t *>(p)[i]);
}

__global__ void __launch_bounds__(256)
set_kv_buffer_kernel(SetKvParams p) {
  const int64_t kc = p.dk >> 3, vc = p.dv >> 3;  // 16-byte pieces per head row
  const int64_t per_token = static_cast<int64_t>(p.heads) * (kc + vc);
  const int64_t total = static_cast<int64_t>(p.n_tokens) * per_token;
  const int64_t pool = p.num_pages * p.page_size;
  bool bad = false;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / per_token;
    int64_t r = i - t * per_token;
    const int64_t slot = load_slot(p.loc, p.loc_is64, t);
    if (slot < 0 || slot >= pool) {
      bad = true;
      continue;
    }
    const int64_t page = slot / p.page_size, pos = slot - page * p.page_size;
    const bool is_k = r < p.heads * kc;
    if (!is_k) r -= p.heads * kc;
    const int64_t per_head = is_k ? kc : vc;
    const int64_t h = r / per_head, c = (r - h * per_head) * 8;
    const bf16 *src;
    bf16 *dst;
    if (is_k) {
      src = p.k + t * p.k_st + h * p.k_sh + c;
      dst = p.k_cache + page * p.kc_sp + pos * p.kc_spos + h * p.kc_sh + c;
    } else {
      src = p.v + t * p.v_st + h * p.v_sh + c;
      dst = p.v_cache + page * p.vc_sp + pos * p.vc_spos + h * p.vc_sh + c;
    }
    *reinterpret_cast<uint4 *>(dst) = __ldg(reinterpret_cast<const uint4 *>(src));
  }
  if (bad) atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
}

}  // namespace

int launch_set_kv_buffer(const SetKvParams &p, cudaStream_t stream) {
  const int64_t per_token = static_cast<int64_t>(p.heads) * ((p.dk + p.dv) >> 3);
  const int64_t total = static_cast<int64_t>(p.n_tokens) * per_token;
  if (total == 0) return PKV_OK;
  // enough CTAs to fill every SM several times over; the loop covers the rest
  const int64_t want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 8 * kNumSMs ? want : 8 * kNumSMs);
  set_kv_buffer_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
