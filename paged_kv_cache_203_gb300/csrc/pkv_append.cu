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

constexpr int kSetKvUnroll = 4;  // independent pieces in flight per thread

// One 16-byte piece: the source address depends only on (t, h, c), so its
// load does not wait for the slot; the slot only gates the store.
struct SetKvPiece {
  uint4 val;
  bf16 *dst;
};

__global__ void __launch_bounds__(256)
set_kv_buffer_kernel(SetKvParams p) {
  const uint32_t kc = p.dk >> 3, vc = p.dv >> 3;  // 16-byte pieces per head row
  const uint32_t k_pieces = static_cast<uint32_t>(p.heads) * kc;
  const uint32_t per_token = k_pieces + static_cast<uint32_t>(p.heads) * vc;
  const uint32_t total = static_cast<uint32_t>(p.n_tokens) * per_token;
  const int64_t pool = p.num_pages * p.page_size;
  const uint32_t stride = gridDim.x * blockDim.x;
  bool bad = false;
  for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < total;
       base += kSetKvUnroll * stride) {
    SetKvPiece pc[kSetKvUnroll];
    int64_t slot[kSetKvUnroll];
    bool is_v[kSetKvUnroll];
#pragma unroll
    for (int u = 0; u < kSetKvUnroll; ++u) {
      const uint32_t i = base + u * stride;
      pc[u].dst = nullptr;
      slot[u] = -1;
      is_v[u] = false;
      if (i >= total) continue;
      const uint32_t t = i / per_token;
      uint32_t r = i - t * per_token;
      slot[u] = load_slot(p.loc, p.loc_is64, t);
      const bool is_k = r < k_pieces;
      if (!is_k) r -= k_pieces;
      const uint32_t per_head = is_k ? kc : vc;
      const uint32_t h = r / per_head, c = (r - h * per_head) * 8;
      const bf16 *src = is_k ? p.k + t * p.k_st + h * p.k_sh + c
                             : p.v + t * p.v_st + h * p.v_sh + c;
      pc[u].val = __ldg(reinterpret_cast<const uint4 *>(src));
      // destination relative to the slot's row, completed below
      pc[u].dst = is_k ? p.k_cache + h * p.kc_sh + c : p.v_cache + h * p.vc_sh + c;
      is_v[u] = !is_k;
    }
#pragma unroll
    for (int u = 0; u < kSetKvUnroll; ++u) {
      if (pc[u].dst == nullptr) continue;
      const int64_t s = slot[u];
      if (s < 0 || s >= pool) {
        bad = true;
        continue;
      }
      const int64_t page = s / p.page_size, pos = s - page * p.page_size;
      bf16 *dst = pc[u].dst + (is_v[u] ? page * p.vc_sp + pos * p.vc_spos
                                       : page * p.kc_sp + pos * p.kc_spos);
      *reinterpret_cast<uint4 *>(dst) = pc[u].val;
    }
  }
  if (bad) atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
}

}  // namespace

int launch_set_kv_buffer(const SetKvParams &p, cudaStream_t stream) {
  const int64_t per_token = static_cast<int64_t>(p.heads) * ((p.dk + p.dv) >> 3);
  const int64_t total = static_cast<int64_t>(p.n_tokens) * per_token;
  if (total == 0) return PKV_OK;
  if (total > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;  // 32-bit piece index
  // about kSetKvUnroll pieces per thread, all of them issued before any store
  const int64_t want = (total + 256 * kSetKvUnroll - 1) / (256 * kSetKvUnroll);
  const int grid = static_cast<int>(want < 64 * kNumSMs ? want : 64 * kNumSMs);
  set_kv_buffer_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
