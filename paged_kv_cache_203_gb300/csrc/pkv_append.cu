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
//
// An fp8 pool (the backend's fp8 `kv_cache_dtype`, whose write takes
// `k_scale` / `v_scale`) stores e4m3 codes of row / scale: a 16-byte piece is
// then 16 codes, from 32 bytes of bf16 input, each value divided by the
// scale in fp32 (IEEE division) and rounded to the nearest code, ties to
// even.  Attention reads such a pool back as code * scale (the descale).
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ int64_t load_slot(const void *p, int is64, int64_t i) {
  return is64 ? static_cast<const int64_t *>(p)[i]
              : static_cast<int64_t>(static_cast<const int32_t *>(p)[i]);
}

constexpr int kSetKvUnroll = 4;  // independent pieces in flight per thread

// One 16-byte output piece: its source address depends only on (t, h, c), so
// the loads do not wait for the slot; the slot only gates the store.
template <bool FP8>
struct SetKvPiece {
  uint4 val[FP8 ? 2 : 1];  // bf16 input: 8 values, or 16 for 16 codes
  char *dst;               // byte address, relative to the slot's row
};

template <bool FP8>
__global__ void __launch_bounds__(256)
set_kv_buffer_kernel(SetKvParams p) {
  constexpr uint32_t EPP = FP8 ? 16 : 8;          // elements per 16-byte piece
  constexpr int64_t ES = FP8 ? 1 : 2;             // cache bytes per element
  const uint32_t kc = p.dk / EPP, vc = p.dv / EPP;  // pieces per head row
  const uint32_t k_pieces = static_cast<uint32_t>(p.heads) * kc;
  const uint32_t per_token = k_pieces + static_cast<uint32_t>(p.heads) * vc;
  const uint32_t total = static_cast<uint32_t>(p.n_tokens) * per_token;
  const int64_t pool = p.num_pages * p.page_size;
  const uint32_t stride = gridDim.x * blockDim.x;
  float k_scale = 1.f, v_scale = 1.f;
  if constexpr (FP8) {
    if (p.k_scale != nullptr) k_scale = __ldg(p.k_scale);
    if (p.v_scale != nullptr) v_scale = __ldg(p.v_scale);
  }
  bool bad = false;
  for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < total;
       base += kSetKvUnroll * stride) {
    SetKvPiece<FP8> pc[kSetKvUnroll];
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
      const uint32_t h = r / per_head, c = (r - h * per_head) * EPP;
      const bf16 *src = is_k ? p.k + t * p.k_st + h * p.k_sh + c
                             : p.v + t * p.v_st + h * p.v_sh + c;
      pc[u].val[0] = __ldg(reinterpret_cast<const uint4 *>(src));
      if constexpr (FP8) pc[u].val[1] = __ldg(reinterpret_cast<const uint4 *>(src + 8));
      // destination relative to the slot's row, completed below
      pc[u].dst = is_k ? static_cast<char *>(p.k_cache) + (h * p.kc_sh + c) * ES
                       : static_cast<char *>(p.v_cache) + (h * p.vc_sh + c) * ES;
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
      char *dst = pc[u].dst + (is_v[u] ? page * p.vc_sp + pos * p.vc_spos
                                       : page * p.kc_sp + pos * p.kc_spos) * ES;
      uint4 out = pc[u].val[0];
      if constexpr (FP8) {
        // 16 bf16 values -> 16 codes of value / scale, lowest column first
        const float sc = is_v[u] ? v_scale : k_scale;
        const uint32_t *w = reinterpret_cast<const uint32_t *>(pc[u].val);
        uint32_t codes[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t word = 0;
#pragma unroll
          for (int hw = 0; hw < 2; ++hw) {
            const __nv_bfloat162 two = *reinterpret_cast<const __nv_bfloat162 *>(&w[2 * q + hw]);
            word |= round_e4m3x2(__fdiv_rn(__low2float(two), sc),
                                 __fdiv_rn(__high2float(two), sc)) << (16 * hw);
          }
          codes[q] = word;
        }
        out = make_uint4(codes[0], codes[1], codes[2], codes[3]);
      }
      *reinterpret_cast<uint4 *>(dst) = out;
    }
  }
  if (bad) atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
}

}  // namespace

int launch_set_kv_buffer(const SetKvParams &p, cudaStream_t stream) {
  const int epp = p.fp8 ? 16 : 8;
  const int64_t per_token = static_cast<int64_t>(p.heads) * ((p.dk + p.dv) / epp);
  const int64_t total = static_cast<int64_t>(p.n_tokens) * per_token;
  if (total == 0) return PKV_OK;
  if (total > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;  // 32-bit piece index
  // about kSetKvUnroll pieces per thread, all of them issued before any store
  const int64_t want = (total + 256 * kSetKvUnroll - 1) / (256 * kSetKvUnroll);
  const int grid = static_cast<int>(want < 64 * kNumSMs ? want : 64 * kNumSMs);
  if (p.fp8)
    set_kv_buffer_kernel<true><<<grid, 256, 0, stream>>>(p);
  else
    set_kv_buffer_kernel<false><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
