// pkv_noalloc.cu -- paged attention for callers that cannot allocate.
//
// pkv_attn_with_kvcache needs caller-provided workspace whenever it splits
// the keys of a request into chunks.  Some callers cannot obtain one: they
// are handed only their input and output buffers (plugin interfaces with no
// workspace hook), or they run under a memory plan that forbids device
// allocation after start-up, or they must not call cudaMalloc / cudaFree on
// this path because those calls can synchronise the device or fail while
// another allocator holds the memory.  For them this file provides
// pkv_attn_with_kvcache_noalloc: the same computation, with its scratch in a
// fixed array that lives in the library itself.
//
// The scratch is one file-scope device array of PKV_NOALLOC_SCRATCH_BYTES
// bytes.  Every GPU that loads this library holds it until the process
// exits.  All calls on a device share it and it keeps the last call's
// contents; the parts that must start at zero (the split tickets) are
// cleared by every call with an asynchronous memset, and the partial states
// are always written before they are read.  Two calls whose work overlaps on
// the GPU (different streams, no ordering between them) race on the array.
#include <atomic>

#include "pkv_internal.h"

namespace pkv {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch for each device, filled on the first
// call made with that device current.  In host code the array's name is only
// a host-side stand-in, so the address must come from cudaGetSymbolAddress.
// Calls may come from several host threads at once: two first calls on a
// device may both look the address up and store the same value.
std::atomic<void *> g_scratch_addr[64] = {};

int scratch_for_current_device(void **ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= 64) return PKV_ERR_UNSUPPORTED;
  void *addr = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (addr == nullptr) {
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
      return PKV_ERR_CUDA;
    g_scratch_addr[dev].store(addr, std::memory_order_release);
  }
  *ptr = addr;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_attn_with_kvcache_noalloc(
    pkv_tensor q, pkv_tensor k_cache, pkv_tensor v_cache, pkv_tensor page_table,
    pkv_tensor cache_seqlens, pkv_tensor cu_seqlens_q, int max_seqlen_q,
    float scale, int causal, int window_left, pkv_tensor topk_indices,
    int num_splits, pkv_tensor out, pkv_tensor lse, cudaStream_t stream) {
  size_t need = 0;
  int rc = pkv_attn_workspace_size(q, k_cache, v_cache, page_table, cache_seqlens,
                                   max_seqlen_q, topk_indices, num_splits, &need);
  if (rc != PKV_OK) return rc;
  if (need > static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES)) return PKV_ERR_WORKSPACE;
  void *scratch = nullptr;
  rc = pkv::scratch_for_current_device(&scratch);
  if (rc != PKV_OK) return rc;
  return pkv_attn_with_kvcache(q, k_cache, v_cache, page_table, cache_seqlens,
                               cu_seqlens_q, max_seqlen_q, scale, causal,
                               window_left, topk_indices, num_splits, out, lse,
                               scratch, PKV_NOALLOC_SCRATCH_BYTES, stream);
}
