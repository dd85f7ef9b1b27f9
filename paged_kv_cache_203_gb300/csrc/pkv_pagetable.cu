// pkv_pagetable.cu -- integer metadata kernels: the prefill-aware
// sliding-window page table, the strided (page-level) table, the top-k
// index -> KV slot transform and the local-attention virtual batches.  All
// integer, bit-exact by construction.
#include <atomic>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

using ptx::griddep_launch_dependents;
using ptx::griddep_wait;

__device__ __forceinline__ int64_t load_index(const void *p, int is64, int i) {
  return is64 ? static_cast<const int64_t *>(p)[i]
              : static_cast<int64_t>(static_cast<const int32_t *>(p)[i]);
}

// Prefill-aware SWA row build (flashattention_backend.py,
// `_build_pa_page_table_kernel`).  The kept source positions form two
// contiguous runs, [0, pf) and [decode_start, sl), so the row is two
// coalesced copies: dst[i] = src[i] for i < pf, and dst[i] = src[i + gap] for
// pf <= i < kv_len.  One CTA per (row, 1024-entry chunk of it): each thread
// issues its four loads before any store, so a chunk costs one memory round
// trip after the two dependent index loads.  Every CTA of a row judges the
// row the same way; a malformed row (pool index out of range, kv_len past
// dst's width, a source column past req_to_token's width) is written by none
// of them and gets kv_len -1 from chunk 0, which also sets the flag.
constexpr int kSwaThreads = 256;
constexpr int kSwaPerThread = 4;
constexpr int kSwaChunk = kSwaThreads * kSwaPerThread;

__global__ void __launch_bounds__(kSwaThreads)
swa_page_table_kernel(const int32_t *__restrict__ rtt, int64_t rtt_stride,
                      int64_t rtt_rows, int64_t rtt_cols, const void *rpi,
                      int rpi_is_64, const int32_t *__restrict__ seq_lens,
                      const int32_t *__restrict__ prefill_lens, int window,
                      int32_t *__restrict__ dst, int64_t dst_stride,
                      int dst_cols, int32_t *__restrict__ kv_lens,
                      uint32_t *err) {
  const int b = blockIdx.x;
  const bool lead = blockIdx.y == 0 && threadIdx.x == 0;
  const int64_t req = load_index(rpi, rpi_is_64, b);
  if (req < 0 || req >= rtt_rows) {
    if (lead) {
      kv_lens[b] = -1;
      atomicOr(err, PKV_EFLAG_SRC_OOB);
    }
    return;
  }
  const int sl = seq_lens[b];
  const int pf = prefill_lens[req];
  const int decode_start = max(pf, sl - window);
  const int gap = max(decode_start - pf, 0);
  const int kv_len = sl - gap;
  if (kv_len > dst_cols) {
    if (lead) {
      kv_lens[b] = -1;
      atomicOr(err, PKV_EFLAG_ROW_TOO_SHORT);
    }
    return;
  }
  // positions grow with i, so the last entry reads the largest column
  const int64_t last_src =
      kv_len - 1 < pf ? static_cast<int64_t>(kv_len) - 1 : static_cast<int64_t>(kv_len) - 1 + gap;
  if (kv_len > 0 && last_src >= rtt_cols) {
    if (lead) {
      kv_lens[b] = -1;
      atomicOr(err, PKV_EFLAG_SRC_OOB);
    }
    return;
  }
  if (lead) kv_lens[b] = kv_len;
  const int32_t *src = rtt + req * rtt_stride;
  int32_t *out = dst + static_cast<int64_t>(b) * dst_stride;
  const int i0 = blockIdx.y * kSwaChunk + threadIdx.x;
  int32_t v[kSwaPerThread];
#pragma unroll
  for (int e = 0; e < kSwaPerThread; ++e) {
    const int i = i0 + e * kSwaThreads;
    v[e] = i < kv_len ? src[i < pf ? i : static_cast<int64_t>(i) + gap] : 0;
  }
#pragma unroll
  for (int e = 0; e < kSwaPerThread; ++e) {
    const int i = i0 + e * kSwaThreads;
    if (i < kv_len) out[i] = v[e];
  }
}

// Strided table: out[b][c] = req_to_token[req_b][c * P] / P
// (flashattention_backend.py, `init_forward_metadata`).
__global__ void strided_page_table_kernel(
    const int32_t *__restrict__ rtt, int64_t rtt_stride, int64_t rtt_rows,
    int64_t rtt_cols, const void *rpi, int rpi_is_64, int page_size,
    int32_t *__restrict__ out, int64_t out_stride, int n_cols, uint32_t *err) {
  griddep_wait();  // launched with programmatic serialization
  griddep_launch_dependents();
  const int b = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= n_cols) return;
  const int64_t req = load_index(rpi, rpi_is_64, b);
  const int64_t col = static_cast<int64_t>(c) * page_size;
  int32_t v = -1;
  if (req >= 0 && req < rtt_rows && col < rtt_cols) {
    // slots are non-negative: C division is the page's floor division
    v = rtt[req * rtt_stride + col] / page_size;
  } else {
    atomicOr(err, PKV_EFLAG_SRC_OOB);
  }
  out[static_cast<int64_t>(b) * out_stride + c] = v;
}

// Top-k logical position -> slot (nsa_backend.py, TopkTransformMethod.PAGED).
// One CTA per query token; the token's request is found by binary search of
// cu_seqlens_q.
__global__ void __launch_bounds__(256)
topk_to_slots_kernel(const int32_t *__restrict__ topk, int64_t topk_stride,
                     int topk_len, const int32_t *__restrict__ cu, int batch,
                     const int32_t *__restrict__ pt, int64_t pt_stride,
                     int pt_cols, const int32_t *__restrict__ cache_seqlens,
                     int page_size, int32_t *__restrict__ out,
                     int64_t out_stride, uint32_t *err) {
  const int t = blockIdx.x;
  // largest b with cu[b] <= t
  int lo = 0, hi = batch;  // answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid;
  }
  const int b = lo;
  const bool covered = batch > 0 && cu[b] <= t && t < cu[b + 1];
  int64_t limit = covered ? cache_seqlens[b] : 0;
  const int64_t table_limit = static_cast<int64_t>(pt_cols) * page_size;
  bool bad = false;
  for (int k = threadIdx.x; k < topk_len; k += blockDim.x) {
    const int32_t idx = topk[static_cast<int64_t>(t) * topk_stride + k];
    int32_t slot = -1;
    if (idx != -1) {
      if (idx < -1 || idx >= limit || idx >= table_limit) {
        bad = true;
      } else {
        slot = pt[static_cast<int64_t>(b) * pt_stride + idx / page_size] * page_size +
               idx % page_size;
      }
    }
    out[static_cast<int64_t>(t) * out_stride + k] = slot;
  }
  if (bad) atomicOr(err, PKV_EFLAG_TOPK_OOB);
}


// ---------------------------------------------------------------------------
// Local (chunked) attention as virtual batches (flashattention_backend.py,
// `make_local_attention_virtual_batches`).  The page builds these arrays on
// the host with numpy; here one launch builds them on the device, so the
// forward needs no device-to-host copy.  Every CTA scans the whole batch
// into shared memory (per request: first virtual batch and first query
// token of the local arrays), then each warp owns output rows: a binary
// search finds the row's request, the lane-0 writes the three lengths and
// the warp gathers the row's pages.  Batches are small (<= 16384 requests),
// so the redundant scan costs less than a second launch would.

constexpr int kLvbThreads = 512;
constexpr int kLvbWarps = kLvbThreads / 32;

// Per-request quantities of the routine, for effective chunk C.
struct LvbRequest {
  int32_t q;       // new tokens (0 when none or negative)
  int32_t kv;      // keys
  int32_t first;   // new tokens in the chunk of the first new token
  int32_t last_k;  // keys in the chunk of the last key
  int32_t blocks;  // virtual batches of this request
  bool keyless;    // kv < q: tokens chunked from the first, no keys
  bool bad;        // q < 0 or kv < q
};

__device__ __forceinline__ LvbRequest lvb_request(const int32_t *cu,
                                                  const int32_t *seq_lens,
                                                  int b, int32_t C) {
  LvbRequest r;
  r.q = cu[b + 1] - cu[b];
  r.kv = seq_lens[b];
  r.first = r.last_k = r.blocks = 0;
  r.keyless = false;
  r.bad = r.q < 0;
  if (r.q <= 0) {
    r.q = 0;
    return r;
  }
  r.keyless = r.kv < r.q;
  r.bad = r.keyless;
  // kv - q >= 0 on the regular path, so % is the floor remainder
  r.first = min(r.keyless ? C : C - (r.kv - r.q) % C, r.q);
  r.last_k = r.keyless ? 0 : r.kv - C * ((r.kv - 1) / C);
  r.blocks = 1 + (r.q - r.first + C - 1) / C;
  return r;
}

// Exclusive scan of one int per thread over the CTA; *total gets the sum.
__device__ __forceinline__ int32_t lvb_block_scan(int32_t x, int32_t *warp_tot,
                                                  int32_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t t = lane < kLvbWarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kLvbWarps) warp_tot[lane] = t;  // inclusive warp prefix
  }
  __syncthreads();
  const int32_t before = warp > 0 ? warp_tot[warp - 1] : 0;
  *total = warp_tot[kLvbWarps - 1];
  __syncthreads();  // warp_tot is reused by the next scan
  return before + incl - x;
}

__device__ __forceinline__ int32_t lvb_block_max(int32_t x, int32_t *warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = __reduce_max_sync(0xffffffffu, x);
  if (lane == 0) warp_tot[warp] = x;
  __syncthreads();
  int32_t m = warp_tot[0];
#pragma unroll
  for (int w = 1; w < kLvbWarps; ++w) m = max(m, warp_tot[w]);
  __syncthreads();
  return m;
}

__global__ void __launch_bounds__(kLvbThreads)
local_virtual_batches_kernel(int attn_chunk_size, int page_size,
                             const int32_t *__restrict__ cu,
                             const int32_t *__restrict__ seq_lens, int batch,
                             const int32_t *__restrict__ pt, int64_t pt_stride,
                             int pt_cols, int capacity,
                             int32_t *__restrict__ q_local,
                             int32_t *__restrict__ cu_local,
                             int32_t *__restrict__ k_local,
                             int32_t *__restrict__ bt, int64_t bt_stride,
                             int bt_cols, int32_t *__restrict__ info,
                             uint32_t *err) {
  extern __shared__ int32_t lvb_smem[];
  int32_t *vbase = lvb_smem;              // [batch + 1] first virtual batch
  int32_t *qbase = lvb_smem + batch + 1;  // [batch + 1] first local token
  __shared__ int32_t warp_tot[kLvbWarps];
  const int tid = threadIdx.x;

  // 1. effective chunk: min(chunk, longest sequence), whole pages, >= 1 page
  int32_t longest = 0;
  for (int b = tid; b < batch; b += kLvbThreads) longest = max(longest, seq_lens[b]);
  longest = lvb_block_max(longest, warp_tot);
  int32_t C = min(attn_chunk_size, longest);
  C = (C / page_size) * page_size;
  if (C < page_size) C = page_size;
  const int pages_per_batch = C / page_size;

  // 2. per-request virtual batch and local token offsets
  int32_t carry_v = 0, carry_q = 0, max_q = 0, max_k = 0;
  bool any_bad = false;
  for (int base = 0; base < batch; base += kLvbThreads) {
    const int b = base + tid;
    int32_t nb = 0, nq = 0;
    if (b < batch) {
      const LvbRequest r = lvb_request(cu, seq_lens, b, C);
      nb = r.blocks;
      nq = r.q;
      any_bad |= r.bad;
      if (r.blocks > 0) {
        // the largest local q is the first block or a full later one; the
        // largest local k is a full chunk unless there is one block
        max_q = max(max_q, r.first);
        if (r.blocks > 1) max_q = max(max_q, min(C, r.q - r.first));
        max_k = max(max_k, r.keyless ? 0 : (r.blocks > 1 ? C : r.last_k));
      }
    }
    int32_t tot_v, tot_q;
    const int32_t ev = lvb_block_scan(nb, warp_tot, &tot_v);
    const int32_t eq = lvb_block_scan(nq, warp_tot, &tot_q);
    if (b < batch) {
      vbase[b] = carry_v + ev;
      qbase[b] = carry_q + eq;
    }
    carry_v += tot_v;
    carry_q += tot_q;
  }
  if (tid == 0) {
    vbase[batch] = carry_v;
    qbase[batch] = carry_q;
  }
  const int32_t n_virtual = carry_v;
  const int32_t cu0 = cu[0];
  if (blockIdx.x == 0) {
    max_q = lvb_block_max(max_q, warp_tot);
    max_k = lvb_block_max(max_k, warp_tot);
    const int bad = __syncthreads_or(any_bad);
    if (tid == 0) {
      info[0] = n_virtual;
      info[1] = C;
      info[2] = max_q;
      info[3] = max_k;
      cu_local[0] = cu0;
      if (bad) atomicOr(err, PKV_EFLAG_BAD_LENGTHS);
      if (n_virtual > capacity) atomicOr(err, PKV_EFLAG_CAPACITY);
    }
  }
  __syncthreads();

  // 3. one warp per output row
  const int lane = tid & 31;
  for (int v = blockIdx.x * kLvbWarps + (tid >> 5); v < capacity;
       v += gridDim.x * kLvbWarps) {
    int32_t ql = 0, kl = 0, cul = cu0 + carry_q;
    int b = 0;
    int64_t first_page = 0;
    bool gather = false;
    if (v < n_virtual) {
      int lo = 0, hi = batch;  // largest b with vbase[b] <= v
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (vbase[mid] <= v) lo = mid; else hi = mid;
      }
      b = lo;
      const LvbRequest r = lvb_request(cu, seq_lens, b, C);
      const int32_t a = v - vbase[b];
      const int32_t rev = r.blocks - 1 - a;
      ql = a == 0 ? r.first : min(r.q - r.first - C * (a - 1), C);
      kl = r.keyless ? 0 : (rev == 0 ? r.last_k : C);
      cul = cu0 + qbase[b] + (a == 0 ? 0 : r.first + C * (a - 1)) + ql;
      gather = !r.keyless;
      const int64_t k_start = static_cast<int64_t>(r.kv) - r.last_k -
                              static_cast<int64_t>(rev) * C;
      first_page = k_start / page_size;
    }
    if (lane == 0) {
      q_local[v] = ql;
      cu_local[v + 1] = cul;
      k_local[v] = kl;
    }
    const int32_t *src = pt + static_cast<int64_t>(b) * pt_stride;
    int32_t *row = bt + static_cast<int64_t>(v) * bt_stride;
    for (int j = lane; j < bt_cols; j += 32) {
      int32_t val = 0;
      if (gather && j < pages_per_batch) {
        // a column past the row repeats its last entry (never read: it lies
        // past the batch's keys)
        const int64_t col = min(first_page + j, static_cast<int64_t>(pt_cols - 1));
        val = src[col];
      }
      row[j] = val;
    }
  }
}

}  // namespace

int launch_swa_page_table(const int32_t *rtt, int64_t rtt_stride,
                          int64_t rtt_rows, int64_t rtt_cols, const void *rpi,
                          int rpi_is_64, const int32_t *seq_lens,
                          const int32_t *prefill_lens, int batch, int window,
                          int32_t *dst, int64_t dst_stride, int dst_cols,
                          int32_t *kv_lens, uint32_t *err,
                          cudaStream_t stream) {
  if (batch == 0) return PKV_OK;
  // chunks of each row along y (at least one: chunk 0 writes kv_len)
  const int64_t chunks = (static_cast<int64_t>(dst_cols) + kSwaChunk - 1) / kSwaChunk;
  if (chunks > 65535) return PKV_ERR_UNSUPPORTED;
  const dim3 grid(batch, static_cast<unsigned>(chunks > 0 ? chunks : 1));
  swa_page_table_kernel<<<grid, kSwaThreads, 0, stream>>>(
      rtt, rtt_stride, rtt_rows, rtt_cols, rpi, rpi_is_64, seq_lens,
      prefill_lens, window, dst, dst_stride, dst_cols, kv_lens, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int launch_strided_page_table(const int32_t *rtt, int64_t rtt_stride,
                              int64_t rtt_rows, int64_t rtt_cols,
                              const void *rpi, int rpi_is_64, int batch,
                              int page_size, int32_t *out, int64_t out_stride,
                              int n_cols, uint32_t *err, cudaStream_t stream) {
  if (batch == 0 || n_cols == 0) return PKV_OK;
  const dim3 grid((n_cols + 255) / 256, batch);
  const cudaError_t e = launch_programmatic(strided_page_table_kernel, grid, dim3(256), 0, stream,
                                            rtt, rtt_stride, rtt_rows, rtt_cols, rpi, rpi_is_64,
                                            page_size, out, out_stride, n_cols, err);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int launch_topk_to_slots(const int32_t *topk, int64_t topk_stride,
                         int total_q, int topk_len, const int32_t *cu,
                         int batch, const int32_t *pt, int64_t pt_stride,
                         int pt_cols, const int32_t *cache_seqlens,
                         int page_size, int32_t *out, int64_t out_stride,
                         uint32_t *err, cudaStream_t stream) {
  if (total_q == 0 || topk_len == 0) return PKV_OK;
  topk_to_slots_kernel<<<total_q, 256, 0, stream>>>(
      topk, topk_stride, topk_len, cu, batch, pt, pt_stride, pt_cols,
      cache_seqlens, page_size, out, out_stride, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int launch_local_virtual_batches(int attn_chunk_size, int page_size,
                                 const int32_t *cu, const int32_t *seq_lens,
                                 int batch, const int32_t *pt,
                                 int64_t pt_stride, int pt_cols, int capacity,
                                 int32_t *q_local, int32_t *cu_local,
                                 int32_t *k_local, int32_t *bt,
                                 int64_t bt_stride, int bt_cols, int32_t *info,
                                 uint32_t *err, cudaStream_t stream) {
  if (batch > kLocalBatchesMaxBatch) return PKV_ERR_UNSUPPORTED;
  const size_t smem = 2 * static_cast<size_t>(batch + 1) * sizeof(int32_t);
  static std::atomic<bool> configured[64] = {};  // per device; calls may race
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(local_virtual_batches_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             2 * (kLocalBatchesMaxBatch + 1) * 4) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  // about one row per warp, at most one CTA per SM
  int grid = (capacity + kLvbWarps - 1) / kLvbWarps;
  grid = max(1, min(grid, kNumSMs));
  local_virtual_batches_kernel<<<grid, kLvbThreads, smem, stream>>>(
      attn_chunk_size, page_size, cu, seq_lens, batch, pt, pt_stride, pt_cols,
      capacity, q_local, cu_local, k_local, bt, bt_stride, bt_cols, info, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
