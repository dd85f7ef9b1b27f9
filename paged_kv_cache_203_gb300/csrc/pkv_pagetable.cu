// pkv_pagetable.cu -- integer metadata kernels: the prefill-aware
// sliding-window page table, the strided (page-level) table and the top-k
// index -> KV slot transform.  All integer, bit-exact by construction.
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ int64_t load_index(const void *p, int is64, int i) {
  return is64 ? static_cast<const int64_t *>(p)[i]
              : static_cast<int64_t>(static_cast<const int32_t *>(p)[i]);
}

// Prefill-aware SWA row build (flashattention_backend.py,
// `_build_pa_page_table_kernel`).  One CTA per request row.  The kept source
// positions form two contiguous runs, [0, pf) and [decode_start, sl), so the
// row is two coalesced copies: dst[i] = src[i] for i < pf, and
// dst[i] = src[i + gap] for pf <= i < kv_len.
__global__ void __launch_bounds__(256)
swa_page_table_kernel(const int32_t *__restrict__ rtt, int64_t rtt_stride,
                      int64_t rtt_rows, int64_t rtt_cols, const void *rpi,
                      int rpi_is_64, const int32_t *__restrict__ seq_lens,
                      const int32_t *__restrict__ prefill_lens, int window,
                      int32_t *__restrict__ dst, int64_t dst_stride,
                      int dst_cols, int32_t *__restrict__ kv_lens,
                      uint32_t *err) {
  const int b = blockIdx.x;
  const int64_t req = load_index(rpi, rpi_is_64, b);
  if (req < 0 || req >= rtt_rows) {
    if (threadIdx.x == 0) {
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
    if (threadIdx.x == 0) {
      kv_lens[b] = -1;
      atomicOr(err, PKV_EFLAG_ROW_TOO_SHORT);
    }
    return;
  }
  if (threadIdx.x == 0) kv_lens[b] = kv_len;
  const int32_t *src = rtt + req * rtt_stride;
  int32_t *out = dst + static_cast<int64_t>(b) * dst_stride;
  bool oob = false;
  for (int i = threadIdx.x; i < kv_len; i += blockDim.x) {
    const int64_t pos = i < pf ? i : static_cast<int64_t>(i) + gap;
    int32_t v = -1;
    if (pos < rtt_cols) {
      v = src[pos];
    } else {
      oob = true;
    }
    out[i] = v;
  }
  if (oob) atomicOr(err, PKV_EFLAG_SRC_OOB);
}

// Strided table: out[b][c] = req_to_token[req_b][c * P] / P
// (flashattention_backend.py, `init_forward_metadata`).
__global__ void strided_page_table_kernel(
    const int32_t *__restrict__ rtt, int64_t rtt_stride, int64_t rtt_rows,
    int64_t rtt_cols, const void *rpi, int rpi_is_64, int page_size,
    int32_t *__restrict__ out, int64_t out_stride, int n_cols, uint32_t *err) {
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

}  // namespace

int launch_swa_page_table(const int32_t *rtt, int64_t rtt_stride,
                          int64_t rtt_rows, int64_t rtt_cols, const void *rpi,
                          int rpi_is_64, const int32_t *seq_lens,
                          const int32_t *prefill_lens, int batch, int window,
                          int32_t *dst, int64_t dst_stride, int dst_cols,
                          int32_t *kv_lens, uint32_t *err,
                          cudaStream_t stream) {
  if (batch == 0) return PKV_OK;
  swa_page_table_kernel<<<batch, 256, 0, stream>>>(
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
  dim3 grid((n_cols + 255) / 256, batch);
  strided_page_table_kernel<<<grid, 256, 0, stream>>>(
      rtt, rtt_stride, rtt_rows, rtt_cols, rpi, rpi_is_64, page_size, out,
      out_stride, n_cols, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
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

}  // namespace pkv
