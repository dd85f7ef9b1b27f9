// pkv_decode.cu -- paged attention for decode and short query runs (GQA).
//
// Computes, for the query rows of one (request, KV head, row tile) and one
// contiguous chunk of that request's keys, the state (O, lse) of
// flashattention_backend.py's `flash_attn_with_kvcache` call, and combines
// the chunks of a split request with the log-sum-exp state merge
// (dual_chunk_flashattention_backend.py, `_merge_attn_outputs`).
//
// Design (HBM-bound: every K/V byte is read once per KV head):
//  * One CTA = 4 consumer warps + producer warp(s), one tile of 16 query rows.
//    The rows are the (new token, q head) pairs that share one KV head, so all
//    GQA heads of a KV head are served by a single read of its K/V rows.
//  * Keys stream through an NSTAGE-deep shared-memory ring of 64-key stages,
//    handed over with mbarriers (full: data landed, empty: consumers done).
//    Two loaders fill the same layout:
//      - TMA (page size a multiple of 8): one producer lane per page issues
//        one 4-D tensor-map box per 64-column half of K and of V
//        ([D, H_kv, P, pages] map, 128-byte swizzle), completion counted in
//        bytes on the stage's full barrier;
//      - cp.async (any page size, top-k lists): two producer warps gather
//        16-byte chunks through the page table, each thread's completion
//        tracked by the full barrier (cp.async.mbarrier.arrive).
//    Layout of a [rows][D] bf16 tile: [D/64 halves][rows][128 B], 16-byte
//    chunk c of row r at chunk (c ^ (r & 7)) -- the TMA 128-byte swizzle --
//    so the ldmatrix reads of the consumers are bank-conflict free.
//  * Consumer warp w owns keys [16w, 16w + 16) of every stage: S = Q K^T and
//    O += P V on bf16 mma.sync m16n8k16 tiles with fp32 accumulation and an
//    online softmax in the log2 domain; the four warps' states are merged in
//    shared memory at the end.  Keys outside the chunk, masked by
//    causality / window, or skipped (bad page id, -1 / out-of-range top-k
//    entry) get -inf scores; the V rows of skipped keys are zeroed before use
//    so that stale or garbage rows of a partially used page never reach the
//    output.
//  * Split-KV: the CTA for chunk s writes its normalised partial (O_s, lse_s)
//    to the workspace; the last CTA of the (request, KV head, tile) to finish
//    (atomic ticket, no waiting) merges all partials and writes the output.
//  * Every mbarrier wait is bounded; on expiry the kernel sets
//    PKV_EFLAG_TIMEOUT and leaves the loop instead of hanging.
#include <cuda.h>
#include <cuda_fp16.h>
#include <string.h>

#include <atomic>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

using namespace ptx;

constexpr int BK = 64;          // keys per stage
constexpr int NCW = 4;          // consumer warps
constexpr int NCT = NCW * 32;   // consumer threads
constexpr int ROWS = kDecodeRowTile;  // 16
constexpr int kPrefetchStages = 3;         // cp.async loader: L2 prefetch distance

// ------------------------------------------------------------ PTX helpers
// (mbarriers, cp.async, TMA and L2 prefetch come from pkv_ptx.cuh)

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(NCT) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0,
                                        uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0,
                                          uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0,
                                         uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1,
                                        uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D(16x8, f32) += A(16x32, e4m3, row) * B(32x8, e4m3, col); four codes per
// register, the lowest k in the lowest byte.
__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}

// Byte offset of 16-byte chunk c of row r in a [rows][D] tile stored as
// [D/64 halves][rows][128 B] with the 128-byte swizzle.
template <int NROWS>
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (NROWS * 128) + r * 128 +
                               (((c & 7) ^ (r & 7)) << 4));
}

struct RowInfo {
  int tok;   // query token index, -1 if the row is padding
  int head;  // q head
  int pos;   // absolute position i of the token
};

// Row r (0..15) of tile `tile` of KV head kvh of the current request.
__device__ __forceinline__ RowInfo row_info(const AttnParams &p, int kvh,
                                            int tile, int r, int q_len,
                                            int kv_len, int q_begin) {
  RowInfo ri{-1, 0, 0};
  int u, g;
  if (p.topk != nullptr) {
    const int tpt = (p.group + ROWS - 1) / ROWS;  // tiles per token
    u = tile / tpt;
    g = (tile % tpt) * ROWS + r;
    if (u >= q_len || g >= p.group) return ri;
  } else {
    const int R = tile * ROWS + r;
    if (R >= q_len * p.group) return ri;
    u = R / p.group;
    g = R % p.group;
  }
  ri.tok = q_begin + u;
  if (ri.tok < 0 || ri.tok >= p.total_q) {  // malformed cu_seqlens_q
    ri.tok = -1;
    return ri;
  }
  ri.head = kvh * p.group + g;
  ri.pos = kv_len - q_len + u;
  return ri;
}

struct DecodeMaps {
  CUtensorMap k;
  CUtensorMap v;
};

// Shared-memory plan (offsets from a 1024-byte aligned base).
template <int D, int NSTAGE>
struct Smem {
  static constexpr uint32_t kStage = BK * D * 2;            // one K (or V) stage
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + NSTAGE * kStage;
  static constexpr uint32_t kQ = kV + NSTAGE * kStage;       // [16][D]
  static constexpr uint32_t kPos = kQ + ROWS * D * 2;        // int [NSTAGE][BK]
  static constexpr uint32_t kBar = kPos + NSTAGE * BK * 4;   // full, empty
  static constexpr uint32_t kM = kBar + 2 * NSTAGE * 8;      // float [NCW][16]
  static constexpr uint32_t kL = kM + NCW * ROWS * 4;
  static constexpr uint32_t kFlag = kL + NCW * ROWS * 4;
  static constexpr uint32_t kProdFlag = kFlag + 4;            // producers: stage free
  static constexpr uint32_t kOff = kFlag + 16;                // int64 [NSTAGE][BK][2]
  static constexpr uint32_t kEnd = kOff + NSTAGE * BK * 16;
  static constexpr size_t kDynamic = kEnd + 1024;  // + alignment slack
  static_assert(NCW * ROWS * (D + 4) * 4 <= 2 * NSTAGE * kStage,
                "epilogue buffer must fit in the stage buffers");
  static_assert(kBar % 8 == 0, "mbarriers need 8-byte alignment");
};

// ---------------------------------------------------------------- kernel

template <int D, int NSTAGE, bool TMA>
__global__ void __launch_bounds__(NCT + (TMA ? 32 : 64), 2)
decode_gqa_kernel(const __grid_constant__ AttnParams p,
                  const __grid_constant__ DecodeMaps maps) {
  using S = Smem<D, NSTAGE>;
  constexpr int CPR = D / 8;   // 16-byte chunks per row
  constexpr int KT = D / 16;   // k-steps of QK^T
  constexpr int NT = D / 8;    // n-tiles of PV
  constexpr int NPROD = TMA ? 1 : 2;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  int *sPos = reinterpret_cast<int *>(smem + S::kPos);
  float *sM = reinterpret_cast<float *>(smem + S::kM);
  float *sL = reinterpret_cast<float *>(smem + S::kL);
  int *sFlag = reinterpret_cast<int *>(smem + S::kFlag);
  const uint32_t full0 = sbase + S::kBar;
  const uint32_t empty0 = full0 + NSTAGE * 8;

  const int split = blockIdx.x;
  const int kvh = blockIdx.y / p.n_row_tiles;
  const int tile = blockIdx.y % p.n_row_tiles;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- longest requests first: blockIdx.z is a rank, not a request ----
  // The grid's CTAs start in launch order and their key ranges differ by
  // up to 16x, so request order leaves the longest chunks for the last wave.
  // Every CTA ranks the requests by keys to read (descending, ties by index:
  // a permutation) and serves the one whose rank is its blockIdx.z; the
  // ranks live in the key-position ring, which the producer fills only after
  // the barrier that follows the mbarrier setup.
  int b = blockIdx.z;
  if (p.batch > 1 && p.batch <= static_cast<int>(blockDim.x) && p.batch <= NSTAGE * BK) {
    int *sWork = sPos;
    int *sPick = reinterpret_cast<int *>(smem + S::kFlag + 8);
    if (tid < p.batch) {
      int w = 0;
      if (p.topk == nullptr) {
        w = p.cache_seqlens[tid];
        if (p.window_left >= 0)
          w = min(w, p.window_left + p.cu_seqlens_q[tid + 1] - p.cu_seqlens_q[tid]);
      }
      sWork[tid] = w;
    }
    __syncthreads();
    if (tid < p.batch) {
      const int w = sWork[tid];
      int rank = 0;
      for (int j = 0; j < p.batch; ++j) {
        const int v = sWork[j];
        rank += (v > w) || (v == w && j < tid);
      }
      if (rank == static_cast<int>(blockIdx.z)) *sPick = tid;
    }
    __syncthreads();
    b = *sPick;
  }

  const int q_begin = p.cu_seqlens_q[b];
  const int q_len = p.cu_seqlens_q[b + 1] - q_begin;
  const int kv_len = p.cache_seqlens[b];

  // ---- rows of this tile; CTAs past the request's rows have no work ----
  int n_valid_rows = 0, u_min = 0, u_max = -1;
  if (p.topk != nullptr) {
    const int tpt = (p.group + ROWS - 1) / ROWS;
    const int u = tile / tpt;
    const int g0 = (tile % tpt) * ROWS;
    if (u < q_len && g0 < p.group && q_begin + u >= 0 && q_begin + u < p.total_q) {
      n_valid_rows = min(ROWS, p.group - g0);
      u_min = u_max = u;
    }
  } else {
    const int R0 = tile * ROWS;
    const int R1 = min(R0 + ROWS, q_len * p.group);
    if (R1 > R0) {
      n_valid_rows = R1 - R0;
      u_min = R0 / p.group;
      u_max = (R1 - 1) / p.group;
    }
  }
  if (n_valid_rows == 0) return;  // uniform over the CTA

  // ---- key range [lo, hi) of the tile; this split's 64-key tiles ----
  int lo, hi;
  if (p.topk != nullptr) {
    lo = 0;
    hi = p.topk_len;
  } else {
    const int i_min = kv_len - q_len + u_min;
    const int i_max = kv_len - q_len + u_max;
    hi = kv_len;
    if (p.causal || p.window_left >= 0) hi = min(hi, i_max + 1);
    lo = 0;
    if (p.window_left >= 0) lo = max(0, i_min - p.window_left);
    hi = max(hi, lo);
  }
  const int t_lo = lo / BK;
  const int t_hi = (hi + BK - 1) / BK;
  const int per = (t_hi - t_lo + p.num_splits - 1) / p.num_splits;
  const int t0 = min(t_hi, t_lo + split * per);
  const int t1 = min(t_hi, t0 + per);
  const int n_kt = t1 - t0;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(full0 + 8 * s, TMA ? 1 : NPROD * 32);
      mbar_init(empty0 + 8 * s, NCW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    fence_proxy_async();
  }
  __syncthreads();

  if (warp >= NCW) {
    // ================================ producer ================================
    const int ptid = tid - NCT;
    volatile int *sProdFlag = reinterpret_cast<volatile int *>(smem + S::kProdFlag);
    for (int kt = 0; kt < n_kt; ++kt) {
      const int st = kt % NSTAGE;
      const uint32_t full = full0 + 8 * st;
      if constexpr (TMA) {
        if (kt >= NSTAGE && !mbar_wait_sleep(empty0 + 8 * st, ((kt / NSTAGE) & 1) ^ 1)) {
          if (lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
          break;
        }
      }
      const int base = (t0 + kt) * BK;  // absolute key (or list) index of row 0
      const uint32_t kdst = sbase + S::kK + st * S::kStage;
      const uint32_t vdst = sbase + S::kV + st * S::kStage;
      if constexpr (TMA) {
        // page box: the page, or 64 rows of a longer page
        const int pbox = p.page_size <= BK ? p.page_size : BK;
        const int nbox = BK / pbox;
        bool box_ok = false;
        int page = 0, inpage = 0;
        const int bpos0 = base + lane * pbox;
        if (lane < nbox && bpos0 < hi && bpos0 + pbox > lo) {
          const int pidx = bpos0 / p.page_size;
          inpage = bpos0 - pidx * p.page_size;
          if (pidx < p.pt_cols) {
            const int64_t pg = p.page_table[static_cast<int64_t>(b) * p.pt_stride + pidx];
            if (pg >= 0 && pg < p.num_pages) {
              page = static_cast<int>(pg);
              box_ok = true;
            } else {
              atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
            }
          } else {
            atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
          }
        }
        // positions of rows lane and lane + 32 (-1: skipped)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = lane + 32 * h;
          const int ok = __shfl_sync(0xffffffffu, box_ok ? 1 : 0, r / pbox);
          const int pos = base + r;
          sPos[st * BK + r] = (ok && pos >= lo && pos < hi) ? pos : -1;
        }
        const uint32_t box_bytes = static_cast<uint32_t>(pbox) * 128u;
        uint32_t bytes = box_ok ? box_bytes * (D / 64) * 2 : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(full, bytes);
        __syncwarp();
        if (box_ok) {
          const uint32_t roff = static_cast<uint32_t>(lane * pbox) * 128u;
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            const uint32_t hoff = hf * (BK * 128) + roff;
            tma_load_4d(kdst + hoff, &maps.k, hf * 64, kvh, inpage, page, full);
            tma_load_4d(vdst + hoff, &maps.v, hf * 64, kvh, inpage, page, full);
          }
        }
      } else {
        // cp.async gather.  (1) one thread per row maps the stage's 64 keys
        // (and those kPrefetchStages stages ahead, warming L2); (2) all
        // producer threads copy 16-byte chunks using the mapped offsets.
        int64_t *sOff = reinterpret_cast<int64_t *>(smem + S::kOff);
        const int topk_tok = q_begin + u_min;
        auto map_row = [&](int j, bool flag, int &pos, int64_t &koff, int64_t &voff) {
          pos = -1;
          koff = voff = -1;
          if (j < lo || j >= hi || j >= t1 * BK) return;
          int q = j;
          if (p.topk != nullptr) {
            q = p.topk[static_cast<int64_t>(topk_tok) * p.topk_stride + j];
            if (q < 0 || q >= kv_len) {
              if (flag && q != -1) atomicOr(p.err, PKV_EFLAG_TOPK_OOB);
              return;
            }
          }
          const int pidx = q / p.page_size;
          if (pidx >= p.pt_cols) {
            if (flag) atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
            return;
          }
          const int64_t pg = p.page_table[static_cast<int64_t>(b) * p.pt_stride + pidx];
          if (pg < 0 || pg >= p.num_pages) {
            if (flag) atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
            return;
          }
          const int inpage = q - pidx * p.page_size;
          pos = q;
          koff = pg * p.k_sp + static_cast<int64_t>(inpage) * p.k_spos + kvh * p.k_sh;
          voff = pg * p.v_sp + static_cast<int64_t>(inpage) * p.v_spos + kvh * p.v_sh;
        };
        // mapping loads (this stage, and L2 warming ahead) go out before the
        // wait for the stage, so their latency overlaps it
        int pos = -1;
        int64_t koff = -1, voff = -1;
        if (ptid < BK) {
          int pa;
          int64_t ka, va;
          map_row((t0 + kt + kPrefetchStages) * BK + ptid, false, pa, ka, va);
          if (ka >= 0) {
            prefetch_l2(p.k + ka, D * 2);
            prefetch_l2(p.v + va, D * 2);
          }
          map_row(base + ptid, true, pos, koff, voff);
        }
        // one thread waits for the stage; all producer threads meet at the
        // barrier and leave together on a timeout (no one is left behind at
        // a named barrier)
        if (ptid == 0) {
          const bool free_ok = kt < NSTAGE || mbar_wait_sleep(empty0 + 8 * st, ((kt / NSTAGE) & 1) ^ 1);
          if (!free_ok) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
          *sProdFlag = free_ok ? 1 : 0;
        }
        asm volatile("bar.sync 2, %0;\n" ::"n"(NPROD * 32) : "memory");
        if (*sProdFlag == 0) break;
        if (ptid < BK) {
          sPos[st * BK + ptid] = pos;
          sOff[(st * BK + ptid) * 2] = koff;
          sOff[(st * BK + ptid) * 2 + 1] = voff;
        }
        asm volatile("bar.sync 2, %0;\n" ::"n"(NPROD * 32) : "memory");
        constexpr int RPP = NPROD * 32 / CPR;  // rows per pass
        const int chunk = ptid % CPR;
        const int prow = ptid / CPR;
#pragma unroll 4
        for (int r = prow; r < BK; r += RPP) {
          const int64_t ko = sOff[(st * BK + r) * 2];
          const int64_t vo = sOff[(st * BK + r) * 2 + 1];
          const int nbytes = ko >= 0 ? 16 : 0;
          cp_async16(kdst + tile_off<BK>(r, chunk), ko >= 0 ? p.k + ko + chunk * 8 : p.k, nbytes);
          cp_async16(vdst + tile_off<BK>(r, chunk), ko >= 0 ? p.v + vo + chunk * 8 : p.v, nbytes);
        }
        cp_async_arrive(full);
        mbar_arrive(full);
      }
    }
    return;
  }

  // ================================== consumers ==================================
  // Q rows into shared memory (zero rows for padding)
  for (int e = tid; e < ROWS * CPR; e += NCT) {
    const int r = e / CPR, c = e % CPR;
    const RowInfo ri = row_info(p, kvh, tile, r, q_len, kv_len, q_begin);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (ri.tok >= 0)
      val = *reinterpret_cast<const uint4 *>(p.q + static_cast<int64_t>(ri.tok) * p.q_st +
                                             static_cast<int64_t>(ri.head) * p.q_sh + c * 8);
    *reinterpret_cast<uint4 *>(smem + S::kQ + tile_off<ROWS>(r, c)) = val;
  }
  consumer_sync();

  uint32_t qf[KT][4];
  {
    const int m = lane >> 3;
    const int r = (m & 1) * 8 + (lane & 7);
#pragma unroll
    for (int kk = 0; kk < KT; ++kk)
      ldsm_x4(sbase + S::kQ + tile_off<ROWS>(r, 2 * kk + (m >> 1)), qf[kk][0], qf[kk][1],
              qf[kk][2], qf[kk][3]);
  }

  const int g = lane >> 2;
  const int tq = lane & 3;
  int rpos[2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    rpos[h] = row_info(p, kvh, tile, g + 8 * h, q_len, kv_len, q_begin).pos;
  const bool use_upper = p.causal || p.window_left >= 0;

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  const int key0 = warp * 16;

  for (int kt = 0; kt < n_kt; ++kt) {
    const int st = kt % NSTAGE;
    if (!mbar_wait_sleep(full0 + 8 * st, (kt / NSTAGE) & 1)) {
      if (lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
      break;
    }
    const uint32_t kbase = sbase + S::kK + st * S::kStage;
    const uint32_t vbase = sbase + S::kV + st * S::kStage;
    const int *pos_st = sPos + st * BK + key0;

    // zero the V rows of skipped keys among this warp's 16 (a masked key must
    // contribute exactly 0, whatever its row holds)
    const bool any_skipped = __any_sync(0xffffffffu, pos_st[lane & 15] < 0);
    if (any_skipped) {
#pragma unroll
      for (int i = 0; i < 16 * CPR / 32; ++i) {
        const int idx = i * 32 + lane;
        const int rr = idx / CPR, cc = idx % CPR;
        if (pos_st[rr] < 0)
          *reinterpret_cast<uint4 *>(smem + S::kV + st * S::kStage +
                                     tile_off<BK>(key0 + rr, cc)) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }

    // S = Q K^T for this warp's 16 keys
    float s[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
    {
      const int kr = key0 + (lane >> 4) * 8 + (lane & 7);
      const int kc = (lane >> 3) & 1;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + tile_off<BK>(kr, 2 * kk + kc), b0, b1, b2, b3);
        mma_bf16(s[0], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
        mma_bf16(s[1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
      }
    }

    // masks; scale to the log2 domain
    int kpos[2][2];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      kpos[n][0] = pos_st[n * 8 + 2 * tq];
      kpos[n][1] = pos_st[n * 8 + 2 * tq + 1];
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        const int kp = kpos[n][e & 1];
        bool masked = kp < 0;
        if (use_upper && kp > rpos[h]) masked = true;
        if (p.window_left >= 0 && kp < rpos[h] - p.window_left) masked = true;
        s[n][e] = masked ? -INFINITY : s[n][e] * p.scale_log2;
      }

    // online softmax per row
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = fmaxf(fmaxf(s[0][2 * h], s[0][2 * h + 1]), fmaxf(s[1][2 * h], s[1][2 * h + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[h], mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(m_run[h] - m_use);
      m_run[h] = m_new;
      float sum = 0.f;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        s[n][2 * h] = exp2f(s[n][2 * h] - m_use);
        s[n][2 * h + 1] = exp2f(s[n][2 * h + 1] - m_use);
        sum += s[n][2 * h] + s[n][2 * h + 1];
      }
      l_run[h] = l_run[h] * alpha + sum;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][2 * h] *= alpha;
        o[n][2 * h + 1] *= alpha;
      }
    }

    // O += P V (P as the A operand straight from the S accumulators)
    const uint32_t a0 = pack_bf16(s[0][0], s[0][1]);
    const uint32_t a1 = pack_bf16(s[0][2], s[0][3]);
    const uint32_t a2 = pack_bf16(s[1][0], s[1][1]);
    const uint32_t a3 = pack_bf16(s[1][2], s[1][3]);
    {
      const int m = lane >> 3;
      const int vr = key0 + (m & 1) * 8 + (lane & 7);
      const int vc = m >> 1;
#pragma unroll
      for (int cc = 0; cc < NT / 2; ++cc) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + tile_off<BK>(vr, 2 * cc + vc), b0, b1, b2, b3);
        mma_bf16(o[2 * cc], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[2 * cc + 1], a0, a1, a2, a3, b2, b3);
      }
    }

    // hand the stage back to the producer
    if (TMA && any_skipped) fence_proxy_async();  // generic zeros before TMA rewrites
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
  }
  consumer_sync();  // every consumer is done with the stage buffers

  // ---- merge the four warps' states ----
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  if (tq == 0) {
    sM[warp * ROWS + g] = m_run[0];
    sM[warp * ROWS + g + 8] = m_run[1];
    sL[warp * ROWS + g] = l_run[0];
    sL[warp * ROWS + g + 8] = l_run[1];
  }
  consumer_sync();
  constexpr int OSTRIDE = D + 4;  // padded fp32 row
  float *sO = reinterpret_cast<float *>(smem + S::kK);  // [NCW][16][D + 4]
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = g + 8 * h;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, sM[w * ROWS + r]);
    const float f = M == -INFINITY ? 0.f : exp2f(m_run[h] - M);
    float *dst = sO + (warp * ROWS + r) * OSTRIDE;
#pragma unroll
    for (int n = 0; n < NT; ++n)
      *reinterpret_cast<float2 *>(dst + n * 8 + 2 * tq) =
          make_float2(o[n][2 * h] * f, o[n][2 * h + 1] * f);
  }
  consumer_sync();

  // each consumer thread: one row, D/8 consecutive columns
  constexpr int CPT = D / 8;
  const int fr = tid >> 3;
  const int fc = (tid & 7) * CPT;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NCW; ++w) M = fmaxf(M, sM[w * ROWS + fr]);
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < NCW; ++w)
    L += (M == -INFINITY) ? 0.f : sL[w * ROWS + fr] * exp2f(sM[w * ROWS + fr] - M);
  float acc[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) acc[c] = 0.f;
#pragma unroll
  for (int w = 0; w < NCW; ++w) {
    const float *src = sO + (w * ROWS + fr) * OSTRIDE + fc;
#pragma unroll
    for (int c = 0; c < CPT; c += 4) {
      const float4 v4 = *reinterpret_cast<const float4 *>(src + c);
      acc[c] += v4.x; acc[c + 1] += v4.y; acc[c + 2] += v4.z; acc[c + 3] += v4.w;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const float lse_nat = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  const RowInfo fri = row_info(p, kvh, tile, fr, q_len, kv_len, q_begin);

  if (p.num_splits == 1) {
    if (fri.tok >= 0) {
      bf16 *dst = p.out + static_cast<int64_t>(fri.tok) * p.o_st +
                  static_cast<int64_t>(fri.head) * p.o_sh + fc;
#pragma unroll
      for (int c = 0; c < CPT; c += 8) {
        uint4 u;
        u.x = pack_bf16(acc[c] * inv, acc[c + 1] * inv);
        u.y = pack_bf16(acc[c + 2] * inv, acc[c + 3] * inv);
        u.z = pack_bf16(acc[c + 4] * inv, acc[c + 5] * inv);
        u.w = pack_bf16(acc[c + 6] * inv, acc[c + 7] * inv);
        *reinterpret_cast<uint4 *>(dst + c) = u;
      }
      if (p.lse != nullptr && (tid & 7) == 0)
        p.lse[static_cast<int64_t>(fri.tok) * p.lse_st + fri.head * p.lse_sh] = lse_nat;
    }
    return;
  }

  // ---- split-KV: publish this chunk's normalised state ----
  const int64_t rows_total = static_cast<int64_t>(p.total_q) * p.h_q;
  if (fri.tok >= 0) {
    const int64_t row = static_cast<int64_t>(fri.tok) * p.h_q + fri.head;
    float *dst = p.ws_o + (static_cast<int64_t>(split) * rows_total + row) * p.dv + fc;
#pragma unroll
    for (int c = 0; c < CPT; c += 4)
      __stcg(reinterpret_cast<float4 *>(dst + c),
             make_float4(acc[c] * inv, acc[c + 1] * inv, acc[c + 2] * inv, acc[c + 3] * inv));
    if ((tid & 7) == 0) __stcg(p.ws_lse + split * rows_total + row, lse_nat);
  }
  __threadfence();
  consumer_sync();
  if (tid == 0) {
    int32_t *ctr = p.ws_counter + (static_cast<int64_t>(b) * p.h_kv + kvh) * p.n_row_tiles + tile;
    const int ticket = atomicAdd(ctr, 1);
    *sFlag = (ticket == p.num_splits - 1);
  }
  consumer_sync();
  if (!*sFlag) return;
  __threadfence();  // every other chunk's state is visible from here on

  // ---- last CTA: merge all chunks (the state merge of merge_state) ----
  if (fri.tok < 0) return;
  const int64_t row = static_cast<int64_t>(fri.tok) * p.h_q + fri.head;
  float Ms = -INFINITY;
  for (int sp = 0; sp < p.num_splits; ++sp) Ms = fmaxf(Ms, __ldcg(p.ws_lse + sp * rows_total + row));
  float outv[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) outv[c] = 0.f;
  float wsum = 0.f;
  if (Ms != -INFINITY) {
    for (int sp = 0; sp < p.num_splits; ++sp) {
      const float ls = __ldcg(p.ws_lse + sp * rows_total + row);
      const float w = exp2f((ls - Ms) * kLog2e);
      wsum += w;
      const float *src = p.ws_o + (static_cast<int64_t>(sp) * rows_total + row) * p.dv + fc;
#pragma unroll
      for (int c = 0; c < CPT; c += 4) {
        const float4 v4 = __ldcg(reinterpret_cast<const float4 *>(src + c));
        outv[c] += w * v4.x; outv[c + 1] += w * v4.y;
        outv[c + 2] += w * v4.z; outv[c + 3] += w * v4.w;
      }
    }
  }
  const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
  bf16 *dst = p.out + static_cast<int64_t>(fri.tok) * p.o_st +
              static_cast<int64_t>(fri.head) * p.o_sh + fc;
#pragma unroll
  for (int c = 0; c < CPT; c += 8) {
    uint4 u;
    u.x = pack_bf16(outv[c] * winv, outv[c + 1] * winv);
    u.y = pack_bf16(outv[c + 2] * winv, outv[c + 3] * winv);
    u.z = pack_bf16(outv[c + 4] * winv, outv[c + 5] * winv);
    u.w = pack_bf16(outv[c + 6] * winv, outv[c + 7] * winv);
    *reinterpret_cast<uint4 *>(dst + c) = u;
  }
  if (p.lse != nullptr && (tid & 7) == 0)
    p.lse[static_cast<int64_t>(fri.tok) * p.lse_st + fri.head * p.lse_sh] =
        wsum > 0.f ? Ms + logf(wsum) : -INFINITY;
}

// ============================================================================
// All-heads decode (head dim 128).  A CTA covers `hpc` KV heads of a request
// (every head in the balanced schedule): consumer warp w owns KV head
// head0 + w and its GQA query rows (at most 16), and one producer warp stages
// 16-key tiles of K and V for all of the CTA's heads at once, so each copy is
// large and the copy engine's per-copy cost stays small against its bytes.
//
// Two copy modes:
//  * slot rows (page size < 8, each slot one contiguous H_kv x 128 row): per
//    key one bulk copy of the K row by the producer, and the V row copied by
//    the consumer warps themselves, each its own head's 256-byte slice with
//    16-byte cp.async two tiles ahead (skipped keys zero-filled), into
//    shared memory at a pitch of H_kv * 256 + 16 bytes (the skew keeps
//    ldmatrix reads conflict-free without a swizzle).  At 2 KB per copy the
//    bulk-copy engine's per-copy cost limits it, so it takes half the rows;
//    moving K to cp.async as well measured slower;
//  * page boxes (page size a multiple of 16): per tile one TMA box
//    {64 columns, 16 positions, hpc heads} per 64-column half and tensor, from
//    a tensor map that lists position before head, so the box lands as
//    [head][position][128-byte row] with the 128-byte swizzle: a head's 16
//    rows are consecutive and their ldmatrix reads conflict-free.
// Page ids are fetched AH_LOOKAHEAD tiles ahead of the copies (4-byte cp.async
// into a shared ring), which keeps the page-table latency off the copy path.
//
// Two schedules:
//  * fixed splits (num_splits >= 1): CTA (split, head group, request rank)
//    takes an equal share of the request's 16-key tiles; the requests are
//    ranked by length in the kernel so the longest chunks start first; page
//    boxes use kDecodeFixedSplitHeads heads per CTA (smaller work items that
//    balance over the grid, boxes still 8 KB); partials are merged by the
//    last CTA of each (request, KV head);
//  * balanced (num_splits == 0, persistent, one CTA per SM, all heads): the
//    16-key tiles of the whole batch are laid end to end and CTA c takes the
//    c-th equal share, crossing request boundaries with the copy pipeline
//    still full.  A request covered by one CTA is written directly; a split
//    request leaves one partial per CTA (slot 0 when it is the CTA's first
//    request, slot 1 when its last) and the CTA that finishes last merges.
// ============================================================================

constexpr int AH_BK = 16;        // keys per tile (= per stage)
constexpr int AH_NSTAGE = 3;
// fp8 stages hold half the bytes; twice as many keep as many bytes in flight
constexpr int AH_NSTAGE_FP8 = 6;
constexpr int AH_LOOKAHEAD = 4;  // tiles the page-id fetch runs ahead of the copies
constexpr int AH_RING = AH_LOOKAHEAD + 1;
constexpr int AH_MAXH = 8;       // KV heads per CTA (one consumer warp each)
constexpr int AH_MAXB = kDecodeBalancedMaxBatch;  // requests a balanced launch schedules
constexpr int AH_SMEM_MAX = 232448;
// KV heads per CTA for page boxes with fixed splits (see the launcher)
constexpr int kAhFixedHeads = kDecodeFixedSplitHeads;

// stage flags published by the producer beside each tile's key positions
constexpr int AH_SEG_START = 1;    // first tile of a segment (a share's run of one request)
constexpr int AH_SEG_END = 2;      // last tile of a segment
constexpr int AH_REQ_START = 4;    // the request's first tile
constexpr int AH_REQ_END = 8;      // the request's last tile
constexpr int AH_SHARE_FIRST = 16; // the share's first tile
constexpr int AH_CTA_LAST = 32;    // the CTA's last tile
constexpr int AH_MQ = 64;          // merge-queue slots of a CTA (a ring)
constexpr int AH_CLAIM_RING = 8;   // shares claimed ahead of the copy cursor

// Shared-memory plan from the heads per CTA and the copy mode (the same
// function on host and device).
struct AhLayout {
  uint32_t stage;  // bytes of one K (or V) stage
  uint32_t k, v, pos, newt, meta, ring_pg, ring_j, voff, pre, scan, mq, bar, end;
};
__host__ __device__ inline AhLayout ah_layout(int hpc, bool boxes, bool balanced,
                                              bool fp8 = false) {
  AhLayout L;
  const int ns = fp8 ? AH_NSTAGE_FP8 : AH_NSTAGE;
  // page boxes: [head][16 positions][128 B] per 64-column half (bf16) or for
  // all 128 columns (fp8 codes)
  L.stage = boxes ? static_cast<uint32_t>(hpc) * AH_BK * (fp8 ? 128u : 256u)
                  : AH_BK * (static_cast<uint32_t>(hpc) * (fp8 ? 128u : 256u) + 16u);
  L.k = 0;
  L.v = L.k + ns * L.stage;
  L.pos = L.v + ns * L.stage;  // int [NSTAGE][BK]
  L.newt = L.pos + ns * AH_BK * 4;  // int [NSTAGE][BK]: new token of the key, or -1
  L.meta = L.newt + ns * AH_BK * 4;  // int [NSTAGE][4]: request, flags, share
  L.ring_pg = L.meta + ns * 16;  // int [RING][BK] page ids
  L.ring_j = L.ring_pg + AH_RING * AH_BK * 4;  // int [RING][BK] key or -1
  L.voff = (L.ring_j + AH_RING * AH_BK * 4 + 7) & ~7u;  // int64 [NSTAGE][BK] (slot rows)
  L.pre = L.voff + ns * AH_BK * 8;  // int64 [MAXB + 1]
  L.scan = L.pre + (balanced ? (AH_MAXB + 1) * 8 : 0);  // int64 [16]
  // merge queue: int jobs [AH_MQ], int sequence numbers [AH_MQ], then head,
  // tail, consumers done, first share, and the claimed shares [AH_CLAIM_RING]
  L.mq = L.scan + 16 * 8;
  L.bar = L.mq + (2 * AH_MQ + 4 + AH_CLAIM_RING) * 4;
  L.end = L.bar + 3 * ns * 8;  // full, empty, V offsets published
  return L;
}
static_assert(AH_NSTAGE * 2 * (AH_BK * (AH_MAXH * 256 + 16)) + 19 * 1024 <= AH_SMEM_MAX,
              "all-heads decode smem plan exceeds 227 KB");
static_assert((2 * AH_MQ + 4 + AH_CLAIM_RING) % 2 == 0, "8-byte aligned barriers");

struct AhMaps {
  CUtensorMap k;
  CUtensorMap v;
};

// A request's query run and key range [lo, hi) in 16-key tiles.
struct AhReq {
  int q_begin, q_len, kv_len, lo, hi, t_lo, ntiles;  // ntiles 0: nothing to do
};

__device__ __forceinline__ AhReq ah_request(const AttnParams &p, int b) {
  AhReq r;
  r.q_begin = p.cu_seqlens_q[b];
  r.q_len = p.cu_seqlens_q[b + 1] - r.q_begin;
  r.kv_len = p.cache_seqlens[b];
  r.hi = max(r.kv_len, 0);
  r.lo = p.window_left >= 0 ? max(0, r.kv_len - r.q_len - p.window_left) : 0;
  r.hi = max(r.hi, r.lo);
  r.t_lo = r.lo / AH_BK;
  const int t_hi = (r.hi + AH_BK - 1) / AH_BK;
  // a request with no key still takes one (empty) tile: its rows get 0 / -inf
  r.ntiles = max(1, t_hi - r.t_lo);
  if (r.q_len <= 0 || r.q_begin < 0 || r.q_begin + r.q_len > p.total_q) r.ntiles = 0;
  return r;
}

// The request of rank blockIdx.z when the batch is ordered by tiles to read
// (descending, ties by index: a permutation); every thread of the CTA calls
// it (block barriers inside).  work: an int scratch of batch entries; pick:
// one int.
__device__ __forceinline__ int ah_rank_to_request(const AttnParams &p, int *work, int *pick) {
  const int tid = threadIdx.x;
  if (tid < p.batch) work[tid] = ah_request(p, tid).ntiles;
  __syncthreads();
  if (tid < p.batch) {
    const int wv = work[tid];
    int rank = 0;
    for (int j = 0; j < p.batch; ++j) {
      const int v = work[j];
      rank += (v > wv) || (v == wv && j < tid);
    }
    if (rank == static_cast<int>(blockIdx.z)) *pick = tid;
  }
  __syncthreads();
  const int b = *pick;
  __syncthreads();  // the ranks are read before the scratch is reused
  return b;
}

// CTA of a balanced launch (g CTAs over t tiles) whose share holds tile x.
__device__ __forceinline__ int ah_cta_of(int64_t x, int64_t g, int64_t t) {
  return static_cast<int>(((x + 1) * g - 1) / t);
}

__device__ __forceinline__ float ah_warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float ah_warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Log-sum-exp merge of the np partial states of rows [0, n_rows) of request
// r, KV head h, into the output (one warp; Dv = 128, each lane 4 columns).
// pidx(sp, rloc) is the workspace index of partial sp of the row whose
// offset in the request's rows is rloc = u * h_q + head.  Four rows at a
// time; partials in passes of 32 (lane = partial for the lse; the running
// sums are rescaled between passes) with the value loads of a pass unrolled
// so that 16 of them are in flight.
template <class PIdx>
__device__ void ah_merge_rows(const AttnParams &p, const AhReq &r, int h, int n_rows, int np,
                              PIdx pidx) {
  constexpr int R = 4;
  const int lane = threadIdx.x & 31;
  for (int rr0 = 0; rr0 < n_rows; rr0 += R) {
    const int nr = min(R, n_rows - rr0);
    int64_t rl[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int rr = rr0 + min(i, nr - 1);
      rl[i] = static_cast<int64_t>(rr / p.group) * p.h_q + h * p.group + rr % p.group;
    }
    float Ms[R], ws[R], acc[R][4];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      Ms[i] = -INFINITY;
      ws[i] = 0.f;
      acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    }
    for (int s0 = 0; s0 < np; s0 += 32) {
      const int sp = s0 + lane;
      float l[R], w[R];
#pragma unroll
      for (int i = 0; i < R; ++i)
        l[i] = (sp < np && i < nr) ? __ldcg(p.ws_lse + pidx(sp, rl[i])) : -INFINITY;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const float mx = fmaxf(Ms[i], ah_warp_max(l[i]));
        // rescale what earlier passes added (exactly 1 when the max holds)
        const float sc = mx == -INFINITY ? 1.f : exp2f((Ms[i] - mx) * kLog2e);
        ws[i] *= sc;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] *= sc;
        Ms[i] = mx;
        w[i] = l[i] == -INFINITY ? 0.f : exp2f((l[i] - mx) * kLog2e);
        ws[i] += ah_warp_sum(w[i]);
      }
      const int cnt = min(32, np - s0);
#pragma unroll 4
      for (int j = 0; j < cnt; ++j) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const float wj = __shfl_sync(0xffffffffu, w[i], j);
          if (i < nr) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                        p.ws_o + pidx(s0 + j, rl[i]) * p.dv) + lane);
            acc[i][0] += wj * v.x;
            acc[i][1] += wj * v.y;
            acc[i][2] += wj * v.z;
            acc[i][3] += wj * v.w;
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (i >= nr) break;
      const int rr = rr0 + i;
      const int tok = r.q_begin + rr / p.group;
      const int head = h * p.group + rr % p.group;
      const float winv = ws[i] > 0.f ? 1.f / ws[i] : 0.f;
      bf16 *dst = p.out + static_cast<int64_t>(tok) * p.o_st + static_cast<int64_t>(head) * p.o_sh +
                  lane * 4;
      uint2 w2;
      w2.x = pack_bf16(acc[i][0] * winv, acc[i][1] * winv);
      w2.y = pack_bf16(acc[i][2] * winv, acc[i][3] * winv);
      *reinterpret_cast<uint2 *>(dst) = w2;
      if (p.lse != nullptr && lane == 0)
        p.lse[static_cast<int64_t>(tok) * p.lse_st + static_cast<int64_t>(head) * p.lse_sh] =
            ws[i] > 0.f ? Ms[i] + logf(ws[i]) : -INFINITY;
    }
  }
}

template <bool BOXES, bool FP8, bool APPEND>
__global__ void __launch_bounds__((AH_MAXH + 2) * 32, 1)
decode_allheads_kernel(const __grid_constant__ AttnParams p,
                       const __grid_constant__ AhMaps maps) {
  static_assert(!(FP8 && APPEND), "the fused append serves bf16 caches");
  constexpr int NST = FP8 ? AH_NSTAGE_FP8 : AH_NSTAGE;  // ring stages
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nthreads = blockDim.x;
  const bool balanced = p.num_splits == 0;
  // KV heads of this CTA = consumer warps; then the producer warp and (the
  // balanced schedule) the merge warp
  const int hpc = nthreads / 32 - (balanced ? 2 : 1);
  const int head0 = blockIdx.y * hpc;  // its first KV head
  const AhLayout L = ah_layout(hpc, BOXES, balanced, FP8);
  const uint32_t sbase = smem_addr(smem);
  if (BOXES && (sbase & 1023u) != 0) {  // swizzled boxes need a 1024-byte aligned base
    if (tid == 0) atomicOr(p.err, PKV_EFLAG_LAYOUT);
    return;  // uniform
  }
  int *sPos = reinterpret_cast<int *>(smem + L.pos);
  int *sNew = reinterpret_cast<int *>(smem + L.newt);
  int *sMeta = reinterpret_cast<int *>(smem + L.meta);
  int64_t *sPre = reinterpret_cast<int64_t *>(smem + L.pre);
  int64_t *sScan = reinterpret_cast<int64_t *>(smem + L.scan);
  const uint32_t full0 = sbase + L.bar;
  const uint32_t empty0 = full0 + NST * 8;
  const uint32_t vmeta0 = empty0 + NST * 8;
  int64_t *sVoff = reinterpret_cast<int64_t *>(smem + L.voff);
  // merge queue: jobs, then head / tail / consumer warps done / the first
  // share (balanced), then the ring of claimed shares
  int *sQ = reinterpret_cast<int *>(smem + L.mq);
  int *sQSeq = sQ + AH_MQ;
  int *sQHead = sQ + 2 * AH_MQ, *sQTail = sQHead + 1, *sQDone = sQHead + 2;
  int *sFirstShare = sQHead + 3;
  int *sClaim = sQHead + 4;
  int *share_ctr = p.ws_counter + static_cast<int64_t>(p.batch) * p.h_kv;  // balanced
  // the CTA's heads of one key (bf16, or one byte per fp8 code)
  const uint32_t row_bytes = static_cast<uint32_t>(hpc) * (FP8 ? 128u : 256u);
  const uint32_t pitch = row_bytes + 16u;                         // slot-row mode

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, hpc);
      mbar_init(vmeta0 + 8 * s, 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    fence_proxy_async();
    // the CTA's first share (balanced); its latency overlaps the scan below
    if (balanced) *sFirstShare = atomicAdd(share_ctr, 1);
    *sQHead = 0;
    *sQTail = 0;
    *sQDone = 0;
  }
  for (int i = tid; i < AH_MQ; i += nthreads) sQSeq[i] = i;  // slot i free for job i

  // ---- this CTA's tiles: balanced, the shares it claims (the first one
  // above); fixed splits, n tiles from tile t_first of request b_first ----
  int b_first = 0, t_first = 0, n = 0;
  int64_t T = 0, G = 1;
  if (balanced) {
    // exclusive prefix of tiles over the batch (each thread a contiguous run)
    const int per = (p.batch + nthreads - 1) / nthreads;
    const int e0 = min(p.batch, tid * per), e1 = min(p.batch, e0 + per);
    int64_t sum = 0;
    for (int b = e0; b < e1; ++b) sum += ah_request(p, b).ntiles;
    int64_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sScan[warp] = incl;
    __syncthreads();
    int64_t run = incl - sum;
    for (int w = 0; w < warp; ++w) run += sScan[w];
    for (int b = e0; b < e1; ++b) {
      sPre[b] = run;
      run += ah_request(p, b).ntiles;
    }
    if (tid == nthreads - 1) sPre[p.batch] = run;
    __syncthreads();
    T = sPre[p.batch];
    G = min(static_cast<int64_t>(kDecodeBalancedShares), T);  // shares
    if (*sFirstShare >= G) return;  // uniform: no share left (also T == 0)
  } else {
    __syncthreads();
    // longest requests first: blockIdx.z is a rank, not a request.  The
    // chunks of a request are its tiles / num_splits, so request order would
    // leave the longest chunks for the last wave; every CTA ranks the
    // requests by tiles (descending, ties by index: a permutation) in the
    // K ring, which the producer fills only after the barrier below.
    b_first = blockIdx.z;
    if (p.batch > 1 && p.batch <= nthreads && p.batch * 4 <= static_cast<int>(L.stage))
      b_first = ah_rank_to_request(p, reinterpret_cast<int *>(smem + L.k),
                                   reinterpret_cast<int *>(smem + L.scan));
    const AhReq r = ah_request(p, b_first);
    if (r.ntiles == 0) return;  // uniform
    const int split = blockIdx.x;
    const int per = (r.ntiles + p.num_splits - 1) / p.num_splits;
    const int t0 = min(r.ntiles, split * per);
    const int t1 = min(r.ntiles, t0 + per);
    t_first = t0;
    n = max(1, t1 - t0);  // an empty share still reports (as an empty tile)
  }

  if (warp == hpc) {
    // ================================ producer ================================
    // A fetch cursor runs AH_LOOKAHEAD tiles ahead of the copy cursor: per
    // tile it puts page ids (slot rows: one per key, lanes 0-15; page boxes:
    // one per tile, lane 0) in a shared ring slot with 4-byte cp.async, one
    // commit group per tile, and the key (or -1) beside each; the copy cursor
    // waits for its tile's group and reads the ids back (each lane its own).
    int *ring_pg = reinterpret_cast<int *>(smem + L.ring_pg);
    int *ring_j = reinterpret_cast<int *>(smem + L.ring_j);
    // A cursor walks the CTA's tiles: share k of the CTA (share id c), tile i
    // of the share's len, request b and its tile t.  A fixed split is one
    // share of one request.  Balanced: the shares come from the counter; the
    // fetch cursor claims them (one claim in flight ahead of it) and records
    // them in a ring that the copy cursor reads.
    struct Cur {
      int k, c, i, len, b, t;
      AhReq r;
    };
    auto enter = [&](Cur &u, int k, int c) {
      u.k = k;
      u.c = c;
      u.i = 0;
      if (balanced) {
        const int64_t x0 = c * T / G, x1 = (c + 1) * T / G;
        u.len = static_cast<int>(x1 - x0);
        // request holding tile x0: the last b with sPre[b] <= x0
        int lo_b = 0, hi_b = p.batch;  // sPre[lo_b] <= x0 < sPre[hi_b]
        while (hi_b - lo_b > 1) {
          const int mid = (lo_b + hi_b) >> 1;
          if (sPre[mid] <= x0) lo_b = mid; else hi_b = mid;
        }
        u.b = lo_b;
        u.t = static_cast<int>(x0 - sPre[lo_b]);
      } else {
        u.len = n;
        u.b = b_first;
        u.t = t_first;
      }
      u.r = ah_request(p, u.b);
    };
    // to the next tile of the share (a balanced share moves on to the next
    // request with tiles; a fixed split never leaves its request)
    auto step_in_share = [&](Cur &u) {
      ++u.i;
      if (++u.t >= u.r.ntiles && balanced && u.b < p.batch - 1) {
        do {
          ++u.b;
        } while (u.b < p.batch - 1 && sPre[u.b + 1] == sPre[u.b]);
        u.t = 0;
        u.r = ah_request(p, u.b);
      }
    };
    int pend = 0;  // lane 0: the claim for the share after the fetch cursor's
    if (balanced && lane == 0) pend = atomicAdd(share_ctr, 1);
    // fetch cursor: to the next tile; false at the end of the CTA's tiles
    auto fetch_step = [&](Cur &u) -> bool {
      if (u.i + 1 < u.len) {
        step_in_share(u);
        return true;
      }
      if (!balanced) return false;
      int c = __shfl_sync(0xffffffffu, pend, 0);
      if (c >= G) c = -1;
      if (lane == 0) {
        sClaim[(u.k + 1) % AH_CLAIM_RING] = c;
        if (c >= 0) pend = atomicAdd(share_ctr, 1);
      }
      __syncwarp();
      if (c < 0) return false;
      enter(u, u.k + 1, c);
      return true;
    };
    // copy cursor: the share after share k (or -1), as the fetch cursor
    // claimed it (the fetch cursor passed the end of share k first)
    auto next_share = [&](const Cur &u) -> int {
      return balanced ? sClaim[(u.k + 1) % AH_CLAIM_RING] : -1;
    };
    Cur f, cc;
    enter(f, 0, balanced ? *sFirstShare : 0);
    cc = f;
    auto fetch = [&](int x) {
      const int slot = (x % AH_RING) * AH_BK + lane;
      const int key0 = (f.r.t_lo + f.t) * AH_BK;
      if (BOXES) {
        if (lane == 0) {
          int jj = -1;
          if (max(key0, f.r.lo) < min(key0 + AH_BK, f.r.hi)) {  // a key of the tile is live
            const int pidx = key0 / p.page_size;  // the whole tile lies in this page
            if (pidx < p.pt_cols) {
              cp_async4(sbase + L.ring_pg + slot * 4,
                        p.page_table + static_cast<int64_t>(f.b) * p.pt_stride + pidx);
              jj = key0;
            } else {
              atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
            }
          }
          ring_j[slot] = jj;
        }
      } else if (lane < AH_BK) {
        const int j = key0 + lane;
        int jj = -1;
        if (j >= f.r.lo && j < f.r.hi) {
          const int pidx = j / p.page_size;
          if (pidx < p.pt_cols) {
            cp_async4(sbase + L.ring_pg + slot * 4,
                      p.page_table + static_cast<int64_t>(f.b) * p.pt_stride + pidx);
            jj = j;
          } else {
            atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
          }
        }
        ring_j[slot] = jj;
      }
      cp_async_commit();
    };
    bool f_live = true;  // the fetch cursor points at a tile
    for (int x = 0; x < AH_LOOKAHEAD; ++x) {
      if (f_live) {
        fetch(x);
        f_live = fetch_step(f);
      } else {
        cp_async_commit();
      }
    }
    int kt = 0;
    for (;; ++kt) {
      const int st = kt % NST;
      if (f_live) {
        fetch(kt + AH_LOOKAHEAD);
        f_live = fetch_step(f);
      } else {
        cp_async_commit();
      }
      cp_async_wait_group<AH_LOOKAHEAD>();  // this tile's ids have landed
      const AhReq &r = cc.r;
      const int b = cc.b, t = cc.t;
      const bool cta_last = cc.i + 1 >= cc.len && next_share(cc) < 0;
      const int slot = (kt % AH_RING) * AH_BK + lane;
      const int key0 = (r.t_lo + t) * AH_BK;
      int pos = -1;
      int64_t koff = 0, voff = 0;  // slot-row mode: element offsets of the key's rows
      int page = -1, inpage0 = 0;  // page-box mode: the tile's page
      if (BOXES) {
        if (lane == 0 && ring_j[slot] >= 0) {
          const int64_t pg = ring_pg[slot];
          if (pg < 0 || pg >= p.num_pages) atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
          else page = static_cast<int>(pg);
        }
        page = __shfl_sync(0xffffffffu, page, 0);
        inpage0 = key0 - (key0 / p.page_size) * p.page_size;
        const int j = key0 + lane;
        if (lane < AH_BK && page >= 0 && j >= r.lo && j < r.hi) pos = j;
      } else if (lane < AH_BK) {
        const int j = ring_j[slot];
        if (j >= 0) {
          const int64_t pg = ring_pg[slot];
          if (pg < 0 || pg >= p.num_pages) {
            atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
          } else {
            const int inpage = j - (j / p.page_size) * p.page_size;
            koff = pg * p.k_sp + static_cast<int64_t>(inpage) * p.k_spos;
            voff = pg * p.v_sp + static_cast<int64_t>(inpage) * p.v_spos;
            pos = j;
          }
        }
      }
      int flags = 0;
      if (cc.i == 0 || t == 0) flags |= AH_SEG_START;
      if (cc.i == cc.len - 1 || t == r.ntiles - 1) flags |= AH_SEG_END;
      if (t == 0) flags |= AH_REQ_START;
      if (t == r.ntiles - 1) flags |= AH_REQ_END;
      if (cc.i == 0) flags |= AH_SHARE_FIRST;
      if (cta_last) flags |= AH_CTA_LAST;

      int ok = 1;
      if (lane == 0 && kt >= NST)
        ok = mbar_wait_sleep(empty0 + 8 * st, ((kt / NST) & 1) ^ 1) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
        break;
      }
      const uint32_t full = full0 + 8 * st;
      const uint32_t kdst = sbase + L.k + st * L.stage;
      const uint32_t vdst = sbase + L.v + st * L.stage;
      if (lane < AH_BK) sPos[st * AH_BK + lane] = pos;
      if (APPEND && lane < AH_BK) {
        // fused append: a key at one of the request's new positions is read
        // from the new rows, not from the cache slot the kernel is filling
        const int first_new = r.kv_len - r.q_len;
        sNew[st * AH_BK + lane] = (pos >= 0 && pos >= first_new) ? r.q_begin + (pos - first_new) : -1;
      }
      if (lane == 0) {
        sMeta[4 * st] = b;
        sMeta[4 * st + 1] = flags;
        sMeta[4 * st + 2] = cc.c;
      }
      if (BOXES) {
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(full, page >= 0 ? 2u * L.stage : 0u);
          if (page >= 0) {
            if (FP8) {  // one box of all 128 columns (bytes) per tensor
              tma_load_4d(kdst, &maps.k, 0, inpage0, head0, page, full);
              tma_load_4d(vdst, &maps.v, 0, inpage0, head0, page, full);
            } else {
              const uint32_t half = L.stage / 2;
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                tma_load_4d(kdst + hf * half, &maps.k, hf * 64, inpage0, head0, page, full);
                tma_load_4d(vdst + hf * half, &maps.v, hf * 64, inpage0, head0, page, full);
              }
            }
          }
        }
      } else {
        // K rows by bulk copy (a new key's from the new rows: the kernel is
        // filling its slot); the V rows' offsets are published for the
        // consumer warps, which copy their own head's slices with cp.async
        if (lane < AH_BK) sVoff[st * AH_BK + lane] = pos >= 0 ? voff : -1;
        const int tk_new = (APPEND && lane < AH_BK) ? sNew[st * AH_BK + lane] : -1;
        const uint32_t bytes = __popc(__ballot_sync(0xffffffffu, pos >= 0)) * row_bytes;
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(vmeta0 + 8 * st);
          mbar_arrive_expect_tx(full, bytes);
        }
        __syncwarp();
        if (pos >= 0)
          bulk_g2s(kdst + lane * pitch,
                   tk_new >= 0 ? static_cast<const void *>(p.k_new + tk_new * p.kn_st + head0 * p.kn_sh)
                   : FP8       ? static_cast<const void *>(reinterpret_cast<const uint8_t *>(p.k) + koff)
                               : static_cast<const void *>(p.k + koff),
                   row_bytes, full);
      }
      // fused append: the CTA that takes the request's last tile stores the
      // new rows of its heads into their slots (one writer per (request, KV
      // head group); no CTA reads the new slots of the cache for attention)
      if (APPEND && (flags & AH_REQ_END)) {
        const int64_t slots = p.num_pages * p.page_size;
        const int per_row = hpc * 16;  // 16-byte pieces of one tensor's row
        for (int u = 0; u < r.q_len; ++u) {
          const int tk = r.q_begin + u;
          const int64_t slot = p.new_loc_is64 ? static_cast<const int64_t *>(p.new_loc)[tk]
                                              : static_cast<const int32_t *>(p.new_loc)[tk];
          if (slot < 0 || slot >= slots) {
            if (lane == 0) atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
            continue;
          }
          const int64_t pg = slot / p.page_size, ps = slot - pg * p.page_size;
          for (int i = lane; i < 2 * per_row; i += 32) {
            const bool is_v = i >= per_row;
            const int piece = is_v ? i - per_row : i;
            const int hh = head0 + piece / 16, c = piece % 16;
            const bf16 *src = is_v ? p.v_new + tk * p.vn_st + hh * p.vn_sh + c * 8
                                   : p.k_new + tk * p.kn_st + hh * p.kn_sh + c * 8;
            bf16 *dst = is_v ? const_cast<bf16 *>(p.v) + pg * p.v_sp + ps * p.v_spos + hh * p.v_sh
                             : const_cast<bf16 *>(p.k) + pg * p.k_sp + ps * p.k_spos + hh * p.k_sh;
            *reinterpret_cast<uint4 *>(dst + c * 8) = *reinterpret_cast<const uint4 *>(src);
          }
        }
      }
      if (cta_last) break;
      if (cc.i + 1 < cc.len) step_in_share(cc);
      else enter(cc, cc.k + 1, next_share(cc));
    }
    // Slot rows: the consumer warps copy V two tiles ahead, so the two
    // stages after the CTA's last tile get V offsets too (none: zero fills),
    // published once their previous tiles are released.
    if (!BOXES) {
      for (int x = kt + 1; x <= kt + 2; ++x) {
        const int st = x % NST;
        int ok = 1;
        if (lane == 0 && x >= NST)
          ok = mbar_wait_sleep(empty0 + 8 * st, ((x / NST) & 1) ^ 1) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
          break;
        }
        if (lane < AH_BK) {
          sVoff[st * AH_BK + lane] = -1;
          if (APPEND) sNew[st * AH_BK + lane] = -1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(vmeta0 + 8 * st);
      }
    }
    cp_async_commit();
    cp_async_wait_group<0>();  // no ring write outlives the CTA
    return;
  }
  const int64_t rows_total = static_cast<int64_t>(p.total_q) * p.h_q;
  const int64_t rows_req = static_cast<int64_t>(p.max_seqlen_q) * p.h_q;  // balanced slots
  // Merge of the partial states of request b, KV head hk, by one warp:
  // balanced, one partial per share that holds a tile of the request (the
  // first share's second slot when the request starts inside it); fixed
  // splits, one per split.
  auto merge_job = [&](int b, int hk) {
    const AhReq r = ah_request(p, b);
    const int n_rows = min(r.q_len, p.max_seqlen_q) * p.group;
    if (balanced) {
      const int c0 = ah_cta_of(sPre[b], G, T);
      const int np = ah_cta_of(sPre[b + 1] - 1, G, T) - c0 + 1;
      const bool c0_second = static_cast<int64_t>(c0) * T / G < sPre[b];
      ah_merge_rows(p, r, hk, n_rows, np, [&](int sp, int64_t rl) -> int64_t {
        return (static_cast<int64_t>(c0 + sp) * 2 + (sp == 0 && c0_second ? 1 : 0)) * rows_req + rl;
      });
    } else {
      const int64_t base = static_cast<int64_t>(r.q_begin) * p.h_q;
      ah_merge_rows(p, r, hk, n_rows, p.num_splits, [&](int sp, int64_t rl) -> int64_t {
        return static_cast<int64_t>(sp) * rows_total + base + rl;
      });
    }
  };
  volatile int *vQ = sQ;
  const int n_cons = min(hpc, p.h_kv - head0);  // consumer warps with a KV head
  // Merge queue of the CTA: a ring of AH_MQ jobs (request << 4 | KV head)
  // with a sequence number per slot (job n goes to slot n % AH_MQ; the slot
  // holds n when free for it and n + 1 once it holds it).  Consumer warps
  // append (waiting for a free slot, which the merge warp always makes);
  // the merge warp takes jobs while the consumers stream, and every warp
  // once the consumers' tiles are done.  pop_job returns a job, or -1 when
  // none is queued; lane 0 decides, the warp gets the result.
  volatile int *vSeq = sQSeq;
  auto pop_job = [&]() -> int {
    int job = -1;
    if (lane == 0) {
      volatile int *vh = sQHead, *vt = sQTail;
      int hd = *vh;
      while (hd < *vt) {
        const int got = atomicCAS(sQHead, hd, hd + 1);
        if (got == hd) {
          // job hd is written right after its ticket was taken (or once its
          // slot was freed)
          const int sl = hd % AH_MQ;
          const long long t0 = clock64();
          while (vSeq[sl] != hd + 1 && clock64() - t0 < kSleepWaitCycles) __nanosleep(32);
          if (vSeq[sl] == hd + 1) {
            __threadfence_block();
            job = vQ[sl];
            __threadfence_block();
            vSeq[sl] = hd + AH_MQ;  // free for job hd + AH_MQ
          } else {
            atomicOr(p.err, PKV_EFLAG_TIMEOUT);
          }
          break;
        }
        hd = got;
      }
    }
    return __shfl_sync(0xffffffffu, job, 0);
  };
  // Takes jobs until every consumer warp is done and the queue is empty.
  auto drain_jobs = [&](int sleep_ns) {
    long long idle0 = clock64();
    while (true) {
      int job = pop_job();
      if (job >= 0) {
        __threadfence();  // the other CTAs' partials (their tickets came first)
        merge_job(job >> 4, job & 15);
        idle0 = clock64();
        continue;
      }
      int done = lane == 0 ? *reinterpret_cast<volatile int *>(sQDone) : 0;
      done = __shfl_sync(0xffffffffu, done, 0);
      if (done >= n_cons) {
        __threadfence_block();  // jobs queued before the last count are seen
        job = pop_job();
        if (job < 0) break;
        __threadfence();
        merge_job(job >> 4, job & 15);
        continue;
      }
      if (clock64() - idle0 > kSleepWaitCycles) {
        if (lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
        break;
      }
      __nanosleep(sleep_ns);
    }
  };

  if (balanced && warp == hpc + 1) {
    // =============================== merge warp ===============================
    // Merges split requests from the queue while the consumer warps stream,
    // so that neither they nor the CTA's ring wait on a merge.
    drain_jobs(256);
    return;
  }
  if (warp > hpc || head0 + warp >= p.h_kv) return;  // no KV head for this warp

  // ================================ consumers ================================
  const int w = warp;          // head within the CTA
  const int h = head0 + w;     // KV head
  const int g = lane >> 2, tq = lane & 3;
  const bool use_upper = p.causal || p.window_left >= 0;
  // byte offset of 16-byte chunk c of key `key` of this head within a stage
  // (fp8: chunk c holds the 16 codes of columns 16c..16c+15)
  auto soff = [&](int key, int c) -> uint32_t {
    if (FP8 && !BOXES)  // slot rows of codes: [key][pitch], the head's 128 B at w * 128
      return static_cast<uint32_t>(key) * pitch + static_cast<uint32_t>(w * 128 + c * 16);
    if (FP8)
      return static_cast<uint32_t>(w * 2048 + key * 128 + (((c & 7) ^ (key & 7)) << 4));
    if (BOXES)
      return static_cast<uint32_t>((c >> 3) * (hpc * 2048) + w * 2048 + key * 128 +
                                   (((c & 7) ^ (key & 7)) << 4));
    return static_cast<uint32_t>(key) * pitch + static_cast<uint32_t>(w * 256 + c * 16);
  };

  uint32_t qf[8][4];
  float o[16][4];
  float m_run[2], l_run[2];
  int rpos[2];
  AhReq r{};
  int n_rows = 0;
  float sl2 = p.scale_log2;  // softmax scale (log2 domain), times k_descale
  float vdesc = 1.f;         // v_descale of the current request and head
  bool seg_req_start = false, seg_share_first = false;

  // Slot rows: this warp copies its head's 256-byte V slice of every key of
  // tile x (16 rows x 16 chunks, 8 per lane; skipped keys zero-filled), one
  // cp.async group per tile.  The stage's region of this head was last read
  // by this warp's own PV three tiles earlier.
  auto issue_v = [&](int x) -> bool {
    if (!BOXES) {  // the producer publishes V offsets up to two tiles past the CTA's last
      const int sx = x % NST;
      if (!mbar_wait_sleep(vmeta0 + 8 * sx, (x / NST) & 1)) return false;
      const uint32_t vdst = sbase + L.v + sx * L.stage;
      if (FP8) {  // 128 codes (8 chunks) per key: 16 rows x 8 chunks, 4 per lane
        const int c = lane & 7;
        const uint8_t *vb8 = reinterpret_cast<const uint8_t *>(p.v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = (lane >> 3) + 4 * i;
          const int64_t vo = sVoff[sx * AH_BK + rr];
          cp_async16(vdst + soff(rr, c), vo >= 0 ? vb8 + vo + h * 128 + c * 16 : vb8,
                     vo >= 0 ? 16 : 0);
        }
      } else {
        const int c = lane & 15;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = (lane >> 4) + 2 * i;
          const int64_t vo = sVoff[sx * AH_BK + rr];
          const int tk = APPEND ? sNew[sx * AH_BK + rr] : -1;  // fused append: the new row
          const bf16 *src = tk >= 0   ? p.v_new + tk * p.vn_st + h * p.vn_sh + c * 8
                            : vo >= 0 ? p.v + vo + h * 128 + c * 8
                                      : p.v;
          cp_async16(vdst + soff(rr, c), src, (tk >= 0 || vo >= 0) ? 16 : 0);
        }
      }
    }
    if (!BOXES) cp_async_commit();
    return true;
  };
  bool v_ok = issue_v(0) && issue_v(1);

  bool stop = false;
  for (int kt = 0; v_ok && !stop; ++kt) {
    const int st = kt % NST;
    if (!mbar_wait_sleep(full0 + 8 * st, (kt / NST) & 1) || !issue_v(kt + 2)) {
      if (lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
      break;
    }
    const int b = sMeta[4 * st];
    const int flags = sMeta[4 * st + 1];
    const int share = sMeta[4 * st + 2];
    stop = (flags & AH_CTA_LAST) != 0;
    if (flags & AH_SEG_START) {
      // a new request: its rows for this head, Q fragments from global memory
      r = ah_request(p, b);
      n_rows = min(r.q_len, p.max_seqlen_q) * p.group;  // <= 16 on this path
      seg_req_start = (flags & AH_REQ_START) != 0;
      seg_share_first = (flags & AH_SHARE_FIRST) != 0;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int rr = g + 8 * hh;
        const bool rv = rr < n_rows;
        const int u = rv ? rr / p.group : 0;
        const int gg = rv ? rr % p.group : 0;
        rpos[hh] = r.kv_len - r.q_len + u;
        const bf16 *qrow = p.q + static_cast<int64_t>(r.q_begin + u) * p.q_st +
                           static_cast<int64_t>(h * p.group + gg) * p.q_sh;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if (FP8) {
            // q rounded to e4m3 (the cache's type): the m16n8k32 A fragment,
            // columns 32kk + 4tq .. +3 and 32kk + 16 + 4tq .. +3 (kk < 4)
            if (kk < 4) {
              uint32_t pk[2] = {0u, 0u};
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const int c0 = kk * 32 + half * 16 + 4 * tq;
                if (rv) {
                  const __nv_bfloat162 q01 = *reinterpret_cast<const __nv_bfloat162 *>(qrow + c0);
                  const __nv_bfloat162 q23 =
                      *reinterpret_cast<const __nv_bfloat162 *>(qrow + c0 + 2);
                  pk[half] = round_e4m3x2(__low2float(q01), __high2float(q01)) |
                             (round_e4m3x2(__low2float(q23), __high2float(q23)) << 16);
                }
              }
              qf[kk][hh] = pk[0];
              qf[kk][2 + hh] = pk[1];
            }
          } else {
            const int c0 = kk * 16 + 2 * tq;
            qf[kk][hh] = rv ? *reinterpret_cast<const uint32_t *>(qrow + c0) : 0u;
            qf[kk][2 + hh] = rv ? *reinterpret_cast<const uint32_t *>(qrow + c0 + 8) : 0u;
          }
        }
      }
      sl2 = p.scale_log2;
      vdesc = 1.f;
      if (FP8) {
        const int64_t di = static_cast<int64_t>(b) * p.h_kv + h;
        if (p.k_descale != nullptr) sl2 *= p.k_descale[di];
        if (p.v_descale != nullptr) vdesc = p.v_descale[di];
      }
#pragma unroll
      for (int nn = 0; nn < 16; ++nn) o[nn][0] = o[nn][1] = o[nn][2] = o[nn][3] = 0.f;
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
    }
    const uint32_t kb = sbase + L.k + st * L.stage;
    const uint32_t vb = sbase + L.v + st * L.stage;
    const int *pos_st = sPos + st * AH_BK;
    // page boxes: zero this head's V rows of skipped keys (a masked key must
    // add exactly 0); slot rows arrive zero-filled
    const bool any_skipped = BOXES && __any_sync(0xffffffffu, pos_st[lane & 15] < 0);
    if (any_skipped) {
      constexpr int kChunks = FP8 ? 8 : 16;  // 16-byte chunks per key row of the head
#pragma unroll
      for (int i = 0; i < AH_BK * kChunks / 32; ++i) {
        const int idx = i * 32 + lane;
        const int rr = idx / kChunks, cc = idx % kChunks;
        if (pos_st[rr] < 0)
          *reinterpret_cast<uint4 *>(smem + L.v + st * L.stage + soff(rr, cc)) =
              make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    // fused append, page boxes: the boxes hold the cache rows of the
    // request's new positions as they were before this call (the slots are
    // being filled by this launch); this head's K and V slices of those keys
    // are replaced by the new rows (slot rows get them from the copies)
    bool patched = false;
    if (BOXES && APPEND) {
      const int *new_st = sNew + st * AH_BK;
      uint32_t nm = __ballot_sync(0xffffffffu, lane < AH_BK && new_st[lane & 15] >= 0);
      patched = nm != 0;
      while (nm) {
        const int rr = __ffs(nm) - 1;
        nm &= nm - 1;
        const int tk = new_st[rr];
        if (lane < 16) {
          const uint4 kv = *reinterpret_cast<const uint4 *>(p.k_new + tk * p.kn_st + h * p.kn_sh +
                                                            lane * 8);
          const uint4 vv = *reinterpret_cast<const uint4 *>(p.v_new + tk * p.vn_st + h * p.vn_sh +
                                                            lane * 8);
          *reinterpret_cast<uint4 *>(smem + L.k + st * L.stage + soff(rr, lane)) = kv;
          *reinterpret_cast<uint4 *>(smem + L.v + st * L.stage + soff(rr, lane)) = vv;
        }
      }
      __syncwarp();
    }
    // S = Q K^T for the stage's 16 keys
    float sc[2][4];
#pragma unroll
    for (int nn = 0; nn < 2; ++nn) sc[nn][0] = sc[nn][1] = sc[nn][2] = sc[nn][3] = 0.f;
    if (FP8) {
      // e4m3 MMAs on the codes as they lie: for keys g and g + 8, four codes
      // of columns 32kk + 4tq .. and 32kk + 16 + 4tq .. per 32-bit read
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_e4m3(sc[0], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3],
                 lds32(kb + soff(g, 2 * kk) + 4 * tq), lds32(kb + soff(g, 2 * kk + 1) + 4 * tq));
        mma_e4m3(sc[1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3],
                 lds32(kb + soff(g + 8, 2 * kk) + 4 * tq),
                 lds32(kb + soff(g + 8, 2 * kk + 1) + 4 * tq));
      }
    } else {
      const int key = (lane >> 4) * 8 + (lane & 7);
      const int kc = (lane >> 3) & 1;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + soff(key, 2 * kk + kc), b0, b1, b2, b3);
        mma_bf16(sc[0], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
        mma_bf16(sc[1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
      }
    }
    int kpos[2][2];
#pragma unroll
    for (int nn = 0; nn < 2; ++nn) {
      kpos[nn][0] = pos_st[nn * 8 + 2 * tq];
      kpos[nn][1] = pos_st[nn * 8 + 2 * tq + 1];
    }
#pragma unroll
    for (int nn = 0; nn < 2; ++nn)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hh = e >> 1;
        const int kp = kpos[nn][e & 1];
        bool masked = kp < 0;
        if (use_upper && kp > rpos[hh]) masked = true;
        if (p.window_left >= 0 && kp < rpos[hh] - p.window_left) masked = true;
        sc[nn][e] = masked ? -INFINITY : sc[nn][e] * sl2;
      }
    float alpha[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float mx = fmaxf(fmaxf(sc[0][2 * hh], sc[0][2 * hh + 1]), fmaxf(sc[1][2 * hh], sc[1][2 * hh + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[hh], mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      alpha[hh] = fast_exp2(m_run[hh] - m_use);  // exactly 1 while the max holds
      m_run[hh] = m_new;
      float sum = 0.f;
#pragma unroll
      for (int nn = 0; nn < 2; ++nn) {
        sc[nn][2 * hh] = fast_exp2(sc[nn][2 * hh] - m_use);
        sc[nn][2 * hh + 1] = fast_exp2(sc[nn][2 * hh + 1] - m_use);
        sum += sc[nn][2 * hh] + sc[nn][2 * hh + 1];
      }
      l_run[hh] = l_run[hh] * alpha[hh] + sum;
    }
    // rescale O only when some row's max moved
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int nn = 0; nn < 16; ++nn) {
        o[nn][0] *= alpha[0];
        o[nn][1] *= alpha[0];
        o[nn][2] *= alpha[1];
        o[nn][3] *= alpha[1];
      }
    }
    const uint32_t a0 = FP8 ? pack_f16(sc[0][0], sc[0][1]) : pack_bf16(sc[0][0], sc[0][1]);
    const uint32_t a1 = FP8 ? pack_f16(sc[0][2], sc[0][3]) : pack_bf16(sc[0][2], sc[0][3]);
    const uint32_t a2 = FP8 ? pack_f16(sc[1][0], sc[1][1]) : pack_bf16(sc[1][0], sc[1][1]);
    const uint32_t a3 = FP8 ? pack_f16(sc[1][2], sc[1][3]) : pack_bf16(sc[1][2], sc[1][3]);
    if (!BOXES) {  // this tile's V slices (two later tiles' groups may be pending)
      cp_async_wait_group<2>();
      __syncwarp();
    }
    if (FP8) {
      // transposed 8x8 loads of code pairs: a register holds columns
      // (2g, 2g+1) of keys (2tq, 2tq+1); its even and odd columns are the B
      // operands of two n-blocks: block 2ch covers columns 16ch + 2n, block
      // 2ch + 1 columns 16ch + 2n + 1
      const int m = lane >> 3;
      const int key = (m & 1) * 8 + (lane & 7);
#pragma unroll
      for (int cp = 0; cp < 4; ++cp) {
        uint32_t r0, r1, r2, r3;  // keys 0-7 / 8-15 of chunks 2cp and 2cp + 1
        ldsm_x4_t(vb + soff(key, 2 * cp + (m >> 1)), r0, r1, r2, r3);
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          const uint32_t lo = hc ? r2 : r0, hi = hc ? r3 : r1;
          const int ch = 2 * cp + hc;
          mma_f16(o[2 * ch], a0, a1, a2, a3, e4m3x2_to_f16x2(__byte_perm(lo, 0u, 0x4420)),
                  e4m3x2_to_f16x2(__byte_perm(hi, 0u, 0x4420)));
          mma_f16(o[2 * ch + 1], a0, a1, a2, a3, e4m3x2_to_f16x2(__byte_perm(lo, 0u, 0x4431)),
                  e4m3x2_to_f16x2(__byte_perm(hi, 0u, 0x4431)));
        }
      }
    } else {
      const int m = lane >> 3;
      const int key = (m & 1) * 8 + (lane & 7);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + soff(key, 2 * cc + (m >> 1)), b0, b1, b2, b3);
        mma_bf16(o[2 * cc], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[2 * cc + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    if (any_skipped || patched) fence_proxy_async();  // generic writes before async rewrites
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);

    if (!(flags & AH_SEG_END)) continue;
    // ------------------- end of this CTA's share of request b -------------------
    const bool whole = balanced ? (seg_req_start && (flags & AH_REQ_END) != 0) : p.num_splits == 1;
    // a share's first segment takes its slot 0, its last one slot 1 (every
    // other segment of the share is a whole request)
    const int slot = seg_share_first ? 0 : 1;
    float Lsum[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      Lsum[hh] = l_run[hh];
      Lsum[hh] += __shfl_xor_sync(0xffffffffu, Lsum[hh], 1);
      Lsum[hh] += __shfl_xor_sync(0xffffffffu, Lsum[hh], 2);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int rr = g + 8 * hh;
      if (rr >= n_rows) continue;
      const int u = rr / p.group;
      const int tok = r.q_begin + u;
      const int head = h * p.group + rr % p.group;
      // (v_descale multiplies the output and every partial: merges are linear)
      const float inv = Lsum[hh] > 0.f ? vdesc / Lsum[hh] : 0.f;
      const float lse_nat = Lsum[hh] > 0.f ? (m_run[hh] + log2f(Lsum[hh])) * kLn2 : -INFINITY;
      if (whole) {
        bf16 *dst = p.out + static_cast<int64_t>(tok) * p.o_st + static_cast<int64_t>(head) * p.o_sh;
        if (FP8) {  // blocks 2ch / 2ch+1 hold the even / odd columns of 16ch..
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint2 w2;
            w2.x = pack_bf16(o[2 * ch][2 * hh] * inv, o[2 * ch + 1][2 * hh] * inv);
            w2.y = pack_bf16(o[2 * ch][2 * hh + 1] * inv, o[2 * ch + 1][2 * hh + 1] * inv);
            *reinterpret_cast<uint2 *>(dst + ch * 16 + 4 * tq) = w2;
          }
        } else {
#pragma unroll
          for (int nn = 0; nn < 16; ++nn)
            *reinterpret_cast<uint32_t *>(dst + nn * 8 + 2 * tq) =
                pack_bf16(o[nn][2 * hh] * inv, o[nn][2 * hh + 1] * inv);
        }
        if (p.lse != nullptr && tq == 0)
          p.lse[static_cast<int64_t>(tok) * p.lse_st + static_cast<int64_t>(head) * p.lse_sh] =
              lse_nat;
      } else {
        const int64_t widx =
            balanced ? (static_cast<int64_t>(share) * 2 + slot) * rows_req +
                           static_cast<int64_t>(u) * p.h_q + head
                     : static_cast<int64_t>(blockIdx.x) * rows_total +
                           static_cast<int64_t>(tok) * p.h_q + head;
        float *dst = p.ws_o + widx * p.dv;
        if (FP8) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            __stcg(reinterpret_cast<float4 *>(dst + ch * 16 + 4 * tq),
                   make_float4(o[2 * ch][2 * hh] * inv, o[2 * ch + 1][2 * hh] * inv,
                               o[2 * ch][2 * hh + 1] * inv, o[2 * ch + 1][2 * hh + 1] * inv));
        } else {
#pragma unroll
          for (int nn = 0; nn < 16; ++nn)
            __stcg(reinterpret_cast<float2 *>(dst + nn * 8 + 2 * tq),
                   make_float2(o[nn][2 * hh] * inv, o[nn][2 * hh + 1] * inv));
        }
        if (tq == 0) __stcg(p.ws_lse + widx, lse_nat);
      }
    }
    if (whole) continue;

    // partial written: the last warp to finish this (request, KV head) hands
    // the merge to its CTA's merge warp
    int expected = p.num_splits;
    if (balanced)
      expected = ah_cta_of(sPre[b + 1] - 1, G, T) - ah_cta_of(sPre[b], G, T) + 1;
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0)
      last = atomicAdd(p.ws_counter + static_cast<int64_t>(b) * p.h_kv + h, 1) == expected - 1;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;
    if (lane == 0) {
      const int q = atomicAdd(sQTail, 1);
      const int sl = q % AH_MQ;
      const long long t0 = clock64();
      while (vSeq[sl] != q && clock64() - t0 < kSleepWaitCycles) __nanosleep(64);
      if (vSeq[sl] == q) {
        vQ[sl] = (b << 4) | h;
        __threadfence_block();
        vSeq[sl] = q + 1;
      } else {
        atomicOr(p.err, PKV_EFLAG_TIMEOUT);
      }
    }
  }
  if (!v_ok) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
  if (!BOXES) cp_async_wait_group<0>();  // none of this warp's copies outlives the CTA
  if (lane == 0) {
    __threadfence_block();  // the jobs this warp queued before the count
    atomicAdd(sQDone, 1);
  }
  drain_jobs(64);  // the CTA's remaining merges, shared by all its warps
}

// ============================================================================
// Short decode (head dim 128, <= 16 query rows per KV head, bf16 cache, a
// page table that covers at most kDecodeShortMaxKeys keys): one CTA per
// (request, KV head), SD_WARPS warps of SD_KEYS keys each.  Everything is
// loaded up front: the request's lengths and each lane's page id in one
// step (the ids of the whole table row are read, so they need not wait for
// the lengths), then every K and V row of the warp's keys and the Q
// fragments.  Each warp computes the softmax state of its keys (mma.sync,
// log2 domain) and the CTA merges the warps' states in shared memory: no
// split partials, tickets or second pass, for batches whose whole attention
// is a few microseconds of latency.
// ============================================================================

// Page ids of the short kernels.  With a table built in the launch
// (p.rtt set) a column's page id is formed from the token pool exactly as
// the strided table builder forms it, and the CTAs of the request's KV head
// 0 store the request's table row (one column per thread), so the launch
// has the result of the builder followed by the attention.
// Token-pool row of request b (-1: none; every column is then -1).
__device__ __forceinline__ int64_t short_pool_row(const AttnParams &p, int b) {
  if (p.rtt == nullptr) return -1;
  const int64_t r = p.rpi_is64 ? static_cast<const int64_t *>(p.rpi)[b]
                               : static_cast<const int32_t *>(p.rpi)[b];
  return r >= 0 && r < p.rtt_rows ? r : -1;
}
// Page id of column c of request b's table row (-1 past the row).
__device__ __forceinline__ int short_page_id(const AttnParams &p, int b, int64_t rrow, int c) {
  if (c >= p.pt_cols) return -1;
  if (p.rtt == nullptr) return p.page_table[static_cast<int64_t>(b) * p.pt_stride + c];
  const int64_t col = static_cast<int64_t>(c) * p.page_size;
  // slots are non-negative: C division is the page's floor division
  return rrow >= 0 && col < p.rtt_cols ? p.rtt[rrow * p.rtt_stride + col] / p.page_size : -1;
}
// Store column c of request b's table row (one thread per column, its load
// issued beside the page-id loads); a column whose source lies outside the
// token pool is -1 and flagged.
__device__ __forceinline__ void short_store_table_col(const AttnParams &p, int b, int64_t rrow,
                                                      int c) {
  if (c >= p.pt_cols) return;
  if (rrow < 0 || static_cast<int64_t>(c) * p.page_size >= p.rtt_cols)
    atomicOr(p.err, PKV_EFLAG_SRC_OOB);
  p.pt_out[static_cast<int64_t>(b) * p.pt_stride + c] = short_page_id(p, b, rrow, c);
}

constexpr int SD_WARPS = 8;
constexpr int SD_KEYS = 32;                  // keys per warp
constexpr int SD_PITCH = 128 * 2 + 16;       // bytes per K / V row (skewed: conflict-free ldmatrix)
constexpr int SD_OPITCH = 128 + 4;           // floats per row of a warp's merged O
static_assert(SD_WARPS * SD_KEYS == kDecodeShortMaxKeys, "short decode key budget");
constexpr uint32_t SD_ROWS = 2u * SD_WARPS * SD_KEYS * SD_PITCH;  // K and V rows
// then each key's (K, V) element offsets: int64 [WARPS][KEYS][2]
constexpr uint32_t SD_SMEM = SD_ROWS + SD_WARPS * SD_KEYS * 16;
static_assert(SD_WARPS * (2 * 16 + 16 * SD_OPITCH) * 4 <= SD_ROWS, "merge area fits the rows");

__global__ void __launch_bounds__(SD_WARPS * 32, 1)
decode_short_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;  // KV head
  const int b = blockIdx.y;  // request
  const uint32_t sbase = smem_addr(smem);
  const uint32_t kw = sbase + static_cast<uint32_t>(warp * SD_KEYS * SD_PITCH);
  const uint32_t vw = kw + static_cast<uint32_t>(SD_WARPS * SD_KEYS * SD_PITCH);
  const int g = lane >> 2, tq = lane & 3;
  griddep_wait();  // launched with programmatic serialization
  griddep_launch_dependents();

  // ---- lengths and this lane's page id, loaded together ----
  const int j = warp * SD_KEYS + lane;  // this lane's key
  const int pidx = j / p.page_size;
  const int64_t rrow = short_pool_row(p, b);
  const int pg_raw = short_page_id(p, b, rrow, pidx);
  const int q_begin = p.cu_seqlens_q[b];
  const int q_len = p.cu_seqlens_q[b + 1] - q_begin;
  const int kv_len = p.cache_seqlens[b];
  // the table row (at most 256 columns): column tid
  if (p.rtt != nullptr && h == 0) short_store_table_col(p, b, rrow, tid);
  if (q_len <= 0 || q_begin < 0 || q_begin + q_len > p.total_q) return;  // uniform
  const int n_rows = min(q_len, p.max_seqlen_q) * p.group;  // <= 16
  const int hi = max(kv_len, 0);
  const int lo = p.window_left >= 0 ? max(0, kv_len - q_len - p.window_left) : 0;
  // keys past the kernel's 256 lie past the table (at most 256 keys): the
  // row is too short for them, as for the keys checked one by one below
  if (tid == 0 && hi > max(lo, kDecodeShortMaxKeys)) atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
  bool live = j >= lo && j < hi;
  if (live && pidx >= p.pt_cols) {
    atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
    live = false;
  }
  if (live && (pg_raw < 0 || pg_raw >= p.num_pages)) {
    atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
    live = false;
  }
  const int inpage = j - pidx * p.page_size;
  const int64_t koff = live ? pg_raw * p.k_sp + static_cast<int64_t>(inpage) * p.k_spos + h * p.k_sh : -1;
  const int64_t voff = live ? pg_raw * p.v_sp + static_cast<int64_t>(inpage) * p.v_spos + h * p.v_sh : -1;
  const uint32_t live_mask = __ballot_sync(0xffffffffu, live);

  // ---- the warp's K and V rows (dead keys zero-filled), then Q ----
  // Offsets go through shared memory (one broadcast load per key instead of
  // shuffles); a half of 16 keys with no live key is neither copied nor
  // computed (its scores are masked, so its terms are exactly 0).
  const bool half_live[2] = {(live_mask & 0xffffu) != 0u, (live_mask >> 16) != 0u};
  {
    int64_t *sOff = reinterpret_cast<int64_t *>(smem + SD_ROWS) + warp * SD_KEYS * 2;
    sOff[2 * lane] = koff;
    sOff[2 * lane + 1] = voff;
    __syncwarp();
    const int c = lane & 15;
    const bool is_v = lane >= 16;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      if (!half_live[hf]) continue;
#pragma unroll 8
      for (int i = 16 * hf; i < 16 * hf + 16; ++i) {
        const longlong2 kv = *reinterpret_cast<const longlong2 *>(sOff + 2 * i);
        const int64_t off = is_v ? kv.y : kv.x;
        const bf16 *base = is_v ? p.v : p.k;
        cp_async16((is_v ? vw : kw) + static_cast<uint32_t>(i * SD_PITCH + c * 16),
                   off >= 0 ? base + off + c * 8 : base, off >= 0 ? 16 : 0);
      }
    }
    cp_async_commit();
  }
  uint32_t qf[8][4];
  int rpos[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int rr = g + 8 * hh;
    const bool rv = rr < n_rows;
    const int u = rv ? rr / p.group : 0;
    const int gg = rv ? rr % p.group : 0;
    rpos[hh] = kv_len - q_len + u;
    const bf16 *qrow = p.q + static_cast<int64_t>(q_begin + u) * p.q_st +
                       static_cast<int64_t>(h * p.group + gg) * p.q_sh;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int c0 = kk * 16 + 2 * tq;
      qf[kk][hh] = rv ? *reinterpret_cast<const uint32_t *>(qrow + c0) : 0u;
      qf[kk][2 + hh] = rv ? *reinterpret_cast<const uint32_t *>(qrow + c0 + 8) : 0u;
    }
  }
  cp_async_wait_group<0>();
  __syncwarp();

  // ---- S = Q K^T over the warp's 32 keys (4 blocks of 8), masked ----
  float sc[4][4];
#pragma unroll
  for (int nb = 0; nb < 4; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
  {
    const int key = (lane >> 4) * 8 + (lane & 7);
    const int kc = (lane >> 3) & 1;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      if (!half_live[hf]) continue;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kw + static_cast<uint32_t>((16 * hf + key) * SD_PITCH + (2 * kk + kc) * 16), b0,
                b1, b2, b3);
        mma_bf16(sc[2 * hf], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
        mma_bf16(sc[2 * hf + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
      }
    }
  }
  const bool use_upper = p.causal || p.window_left >= 0;
  float m_row[2], l_row[2];
#pragma unroll
  for (int nb = 0; nb < 4; ++nb)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int kl = nb * 8 + 2 * tq + (e & 1);  // key within the warp
      const int kp = warp * SD_KEYS + kl;
      const int hh = e >> 1;
      bool masked = ((live_mask >> kl) & 1u) == 0u;
      if (use_upper && kp > rpos[hh]) masked = true;
      if (p.window_left >= 0 && kp < rpos[hh] - p.window_left) masked = true;
      sc[nb][e] = masked ? -INFINITY : sc[nb][e] * p.scale_log2;
    }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float mx = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) mx = fmaxf(mx, fmaxf(sc[nb][2 * hh], sc[nb][2 * hh + 1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mu = mx == -INFINITY ? 0.f : mx;
    float sum = 0.f;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      sc[nb][2 * hh] = fast_exp2(sc[nb][2 * hh] - mu);
      sc[nb][2 * hh + 1] = fast_exp2(sc[nb][2 * hh + 1] - mu);
      sum += sc[nb][2 * hh] + sc[nb][2 * hh + 1];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    m_row[hh] = mx;
    l_row[hh] = sum;
  }

  // ---- O = P V (two 16-key steps) ----
  float o[16][4];
#pragma unroll
  for (int nn = 0; nn < 16; ++nn) o[nn][0] = o[nn][1] = o[nn][2] = o[nn][3] = 0.f;
  {
    const int m = lane >> 3;
    const int key = (m & 1) * 8 + (lane & 7);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      if (!half_live[hf]) continue;
      const uint32_t a0 = pack_bf16(sc[2 * hf][0], sc[2 * hf][1]);
      const uint32_t a1 = pack_bf16(sc[2 * hf][2], sc[2 * hf][3]);
      const uint32_t a2 = pack_bf16(sc[2 * hf + 1][0], sc[2 * hf + 1][1]);
      const uint32_t a3 = pack_bf16(sc[2 * hf + 1][2], sc[2 * hf + 1][3]);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vw + static_cast<uint32_t>((16 * hf + key) * SD_PITCH + (2 * cc + (m >> 1)) * 16),
                  b0, b1, b2, b3);
        mma_bf16(o[2 * cc], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[2 * cc + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }

  // ---- the warps' states merged in shared memory (the rows' area reused) ----
  __syncthreads();  // every warp is done with the K / V rows
  float *sM = reinterpret_cast<float *>(smem);               // [WARPS][16]
  float *sL = sM + SD_WARPS * 16;                            // [WARPS][16]
  float *sO = sL + SD_WARPS * 16;                            // [WARPS][16][OPITCH]
  if (tq == 0) {
    sM[warp * 16 + g] = m_row[0];
    sM[warp * 16 + g + 8] = m_row[1];
    sL[warp * 16 + g] = l_row[0];
    sL[warp * 16 + g + 8] = l_row[1];
  }
  float *ow = sO + warp * 16 * SD_OPITCH;
#pragma unroll
  for (int nn = 0; nn < 16; ++nn) {
    if (live_mask == 0u) break;  // no key: m = -inf, the merge skips this warp
    *reinterpret_cast<float2 *>(ow + g * SD_OPITCH + nn * 8 + 2 * tq) = make_float2(o[nn][0], o[nn][1]);
    *reinterpret_cast<float2 *>(ow + (g + 8) * SD_OPITCH + nn * 8 + 2 * tq) =
        make_float2(o[nn][2], o[nn][3]);
  }
  __syncthreads();
  // thread -> (row, 8 columns)
  const int r = tid >> 4, c8 = (tid & 15) * 8;
  if (r < n_rows) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < SD_WARPS; ++w) M = fmaxf(M, sM[w * 16 + r]);
    float L = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < SD_WARPS; ++w) {
        const float mw = sM[w * 16 + r];
        if (mw == -INFINITY) continue;
        const float f = fast_exp2(mw - M);
        L += f * sL[w * 16 + r];
        const float *src = sO + (w * 16 + r) * SD_OPITCH + c8;
        const float4 x0 = *reinterpret_cast<const float4 *>(src);
        const float4 x1 = *reinterpret_cast<const float4 *>(src + 4);
        acc[0] += f * x0.x; acc[1] += f * x0.y; acc[2] += f * x0.z; acc[3] += f * x0.w;
        acc[4] += f * x1.x; acc[5] += f * x1.y; acc[6] += f * x1.z; acc[7] += f * x1.w;
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int tok = q_begin + r / p.group;
    const int head = h * p.group + r % p.group;
    uint4 w4;
    w4.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    w4.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    w4.z = pack_bf16(acc[4] * inv, acc[5] * inv);
    w4.w = pack_bf16(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4 *>(p.out + static_cast<int64_t>(tok) * p.o_st +
                               static_cast<int64_t>(head) * p.o_sh + c8) = w4;
    if (p.lse != nullptr && (tid & 15) == 0)
      p.lse[static_cast<int64_t>(tok) * p.lse_st + static_cast<int64_t>(head) * p.lse_sh] =
          L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
}

// ============================================================================
// Short decode on a cluster (the same calls as decode_short_kernel, for
// batches of few (request, KV head) pairs): the SC_CTAS CTAs of a cluster
// share one pair.  Rank r scores keys [64r, 64r + 64), one 16-key block per
// warp, and computes output columns [32r, 32r + 32) of P V over all the
// pair's keys, so each CTA copies a quarter of the K rows and a quarter of
// every V row (the copies of one SM were the step's longest part).  A warp
// stores its block's P (bf16, as mma A fragments) and each row's block max m
// and sum l into every CTA of the cluster; after one cluster barrier, warp w
// of rank r forms its 8 output columns as sum_b 2^(m_b - M) (P_b V_b) with M
// the row's max over blocks -- the split-softmax identity of the state
// merge, applied per 16-key block -- so no CTA waits for another's max
// before its exponentials, and only P and (m, l) cross the cluster.  The
// stores are asynchronous and complete bytes on an mbarrier of the
// receiving CTA, which expects 640 B per live block: a CTA waits only for
// what it receives (every CTA receives everything addressed to it before it
// leaves, so none is written after it exits).
// ============================================================================

constexpr int SC_CTAS = 4;
constexpr int SC_WARPS = 4;
constexpr int SC_KEYS = kDecodeShortMaxKeys;       // 256: the whole table row
constexpr int SC_BLOCKS = SC_KEYS / 16;            // 16-key blocks
constexpr int SC_KPITCH = 128 * 2 + 16;            // K row, skewed: conflict-free ldmatrix
constexpr int SC_VCOLS = 128 / SC_CTAS;            // value columns per CTA
constexpr int SC_VPITCH = SC_VCOLS * 2 + 16;       // 80 B: conflict-free ldmatrix
static_assert(SC_CTAS * SC_WARPS * 16 == SC_KEYS, "one 16-key block per warp");
static_assert(SC_WARPS * 8 == SC_VCOLS, "8 output columns per warp");
static_assert(SC_WARPS * 32 * 2 == SC_KEYS, "each thread resolves two keys");
struct ScSmem {
  static constexpr uint32_t kK = 0;                               // [64 keys][KPITCH]
  static constexpr uint32_t kV = kK + SC_WARPS * 16 * SC_KPITCH;  // [256 keys][VPITCH]
  static constexpr uint32_t kP = kV + SC_KEYS * SC_VPITCH;        // uint4 [blocks][32 lanes]
  static constexpr uint32_t kML = kP + SC_BLOCKS * 32 * 16;       // float4 [blocks][8]
  static constexpr uint32_t kVoff = kML + SC_BLOCKS * 8 * 16;     // int64 [256]
  static constexpr uint32_t kKoff = kVoff + SC_KEYS * 8;          // int64 [64]
  static constexpr uint32_t kLive = kKoff + SC_WARPS * 16 * 8;    // uint32 [8]: key bits
  static constexpr uint32_t kBar = kLive + 8 * 4;                 // mbarrier: blocks received
  static constexpr uint32_t kEnd = kBar + 8;
};
static_assert(ScSmem::kV % 16 == 0 && ScSmem::kP % 16 == 0 && ScSmem::kML % 16 == 0 &&
                  ScSmem::kVoff % 8 == 0 && ScSmem::kBar % 8 == 0,
              "aligned short-cluster areas");
constexpr uint32_t kScBlockBytes = 32 * 16 + 8 * 16;  // one block's P and (m, l) rows

__global__ void __cluster_dims__(SC_CTAS, 1, 1) __launch_bounds__(SC_WARPS * 32, 1)
decode_short_cluster_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int h = blockIdx.x / SC_CTAS;  // KV head
  const int b = blockIdx.y;            // request
  const uint32_t sbase = smem_addr(smem);
  const int g = lane >> 2, tq = lane & 3;
  griddep_wait();  // launched with programmatic serialization
  griddep_launch_dependents();

  // ---- lengths and page ids, loaded together: keys tid and tid + 128 (V
  // columns of every key), key 64 * rank + tid (K rows of this rank) ----
  const int j0 = tid, j1 = tid + SC_WARPS * 32;
  const int jk = rank * SC_WARPS * 16 + (tid & 63);
  const int pi0 = j0 / p.page_size, pi1 = j1 / p.page_size, pik = jk / p.page_size;
  const int64_t rrow = short_pool_row(p, b);
  const int pg0 = short_page_id(p, b, rrow, pi0);
  const int pg1 = short_page_id(p, b, rrow, pi1);
  const int pgk = tid < 64 ? short_page_id(p, b, rrow, pik) : -1;
  const int q_begin = p.cu_seqlens_q[b];
  const int q_len = p.cu_seqlens_q[b + 1] - q_begin;
  const int kv_len = p.cache_seqlens[b];
  // the table row (at most 256 columns): column 64 rank + tid of KV head 0
  if (p.rtt != nullptr && h == 0 && tid < 64) short_store_table_col(p, b, rrow, rank * 64 + tid);
  if (q_len <= 0 || q_begin < 0 || q_begin + q_len > p.total_q) return;  // the whole cluster
  const uint32_t xbar = sbase + ScSmem::kBar;
  if (tid == 0) {
    mbar_init(xbar, 1);
    mbar_init_fence();
  }
  const int n_rows = min(q_len, p.max_seqlen_q) * p.group;  // <= 16
  const int hi = max(kv_len, 0);
  const int lo = p.window_left >= 0 ? max(0, kv_len - q_len - p.window_left) : 0;
  // keys past the kernel's 256 lie past the table (at most 256 keys): the
  // row is too short for them, as for the keys checked one by one below
  if (tid == 0 && rank == 0 && hi > max(lo, SC_KEYS)) atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
  auto key_live = [&](int j, int pidx, int pg, bool report) {
    bool live = j >= lo && j < hi;
    if (live && pidx >= p.pt_cols) {
      if (report) atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
      live = false;
    }
    if (live && (pg < 0 || pg >= p.num_pages)) {
      if (report) atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
      live = false;
    }
    return live;
  };
  const bool live0 = key_live(j0, pi0, pg0, rank == 0);
  const bool live1 = key_live(j1, pi1, pg1, rank == 0);
  const bool livek = tid < 64 && key_live(jk, pik, pgk, false);
  int64_t *sVoff = reinterpret_cast<int64_t *>(smem + ScSmem::kVoff);
  int64_t *sKoff = reinterpret_cast<int64_t *>(smem + ScSmem::kKoff);
  uint32_t *sLive = reinterpret_cast<uint32_t *>(smem + ScSmem::kLive);
  const int64_t vcol = static_cast<int64_t>(h) * p.v_sh + rank * SC_VCOLS;
  sVoff[j0] = live0 ? pg0 * p.v_sp + static_cast<int64_t>(j0 - pi0 * p.page_size) * p.v_spos + vcol : -1;
  sVoff[j1] = live1 ? pg1 * p.v_sp + static_cast<int64_t>(j1 - pi1 * p.page_size) * p.v_spos + vcol : -1;
  if (tid < 64)
    sKoff[tid] = livek ? pgk * p.k_sp + static_cast<int64_t>(jk - pik * p.page_size) * p.k_spos +
                             static_cast<int64_t>(h) * p.k_sh
                       : -1;
  {
    const uint32_t w0 = __ballot_sync(0xffffffffu, live0), w1 = __ballot_sync(0xffffffffu, live1);
    if (lane == 0) {
      sLive[warp] = w0;             // keys 32 * warp + lane
      sLive[SC_WARPS + warp] = w1;  // keys 128 + 32 * warp + lane
    }
  }
  __syncthreads();
  uint32_t blk = 0;  // bit i: 16-key block i holds a live key
#pragma unroll
  for (int i = 0; i < SC_KEYS / 32; ++i) {
    const uint32_t w = sLive[i];
    blk |= ((w & 0xffffu) != 0u ? 1u : 0u) << (2 * i);
    blk |= ((w >> 16) != 0u ? 1u : 0u) << (2 * i + 1);
  }
  // every live block of the pair arrives here once; the barrier's
  // initialisation and this expectation precede every peer's stores (the
  // cluster barrier below is released here and waited on before they send)
  if (tid == 0) mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(__popc(blk)) * kScBlockBytes);
  cluster_arrive_release();

  // ---- copies: this CTA's value columns of every key of a live block, and
  // the K rows of its own keys (dead keys of a live block read zeros) ----
  const uint32_t sK = sbase + ScSmem::kK, sV = sbase + ScSmem::kV;
#pragma unroll
  for (int it = 0; it < SC_KEYS * 4 / (SC_WARPS * 32); ++it) {  // 4 16-B chunks a key
    const int idx = tid + SC_WARPS * 32 * it;
    const int key = idx >> 2, c = idx & 3;
    if ((blk >> (key >> 4)) & 1u) {
      const int64_t off = sVoff[key];
      cp_async16(sV + static_cast<uint32_t>(key * SC_VPITCH + c * 16),
                 off >= 0 ? p.v + off + c * 8 : p.v, off >= 0 ? 16 : 0);
    }
  }
#pragma unroll
  for (int it = 0; it < SC_WARPS * 16 * 16 / (SC_WARPS * 32); ++it) {  // 16 chunks a row
    const int idx = tid + SC_WARPS * 32 * it;
    const int key = idx >> 4, c = idx & 15;
    if ((blk >> (rank * SC_WARPS + (key >> 4))) & 1u) {
      const int64_t off = sKoff[key];
      cp_async16(sK + static_cast<uint32_t>(key * SC_KPITCH + c * 16),
                 off >= 0 ? p.k + off + c * 8 : p.k, off >= 0 ? 16 : 0);
    }
  }
  cp_async_commit();
  uint32_t qf[8][4];
  int rpos[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int rr = g + 8 * hh;
    const bool rv = rr < n_rows;
    const int u = rv ? rr / p.group : 0;
    const int gg = rv ? rr % p.group : 0;
    rpos[hh] = kv_len - q_len + u;
    const bf16 *qrow = p.q + static_cast<int64_t>(q_begin + u) * p.q_st +
                       static_cast<int64_t>(h * p.group + gg) * p.q_sh;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int c0 = kk * 16 + 2 * tq;
      qf[kk][hh] = rv ? *reinterpret_cast<const uint32_t *>(qrow + c0) : 0u;
      qf[kk][2 + hh] = rv ? *reinterpret_cast<const uint32_t *>(qrow + c0 + 8) : 0u;
    }
  }
  cp_async_wait_group<0>();
  __syncthreads();  // rows copied by other warps

  // ---- this warp's 16-key block: scores, mask, block softmax ----
  const int blk_id = rank * SC_WARPS + warp;
  const bool my_live = ((blk >> blk_id) & 1u) != 0u;
  uint4 pf = make_uint4(0u, 0u, 0u, 0u);
  float m_row[2] = {-INFINITY, -INFINITY}, l_row[2] = {0.f, 0.f};
  if (my_live) {
    float sc[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
    const int key = (lane >> 4) * 8 + (lane & 7);
    const int kc = (lane >> 3) & 1;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(sK + static_cast<uint32_t>((warp * 16 + key) * SC_KPITCH + (2 * kk + kc) * 16), b0, b1,
              b2, b3);
      mma_bf16(sc[0], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
      mma_bf16(sc[1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
    }
    const uint32_t kbits = (sLive[blk_id >> 1] >> ((blk_id & 1) * 16)) & 0xffffu;
    const bool use_upper = p.causal || p.window_left >= 0;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kl = nb * 8 + 2 * tq + (e & 1);
        const int kp = blk_id * 16 + kl;
        const int hh = e >> 1;
        bool masked = ((kbits >> kl) & 1u) == 0u;
        if (use_upper && kp > rpos[hh]) masked = true;
        if (p.window_left >= 0 && kp < rpos[hh] - p.window_left) masked = true;
        sc[nb][e] = masked ? -INFINITY : sc[nb][e] * p.scale_log2;
      }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float mx = fmaxf(fmaxf(sc[0][2 * hh], sc[0][2 * hh + 1]), fmaxf(sc[1][2 * hh], sc[1][2 * hh + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mu = mx == -INFINITY ? 0.f : mx;
      float sum = 0.f;
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        sc[nb][2 * hh] = fast_exp2(sc[nb][2 * hh] - mu);
        sc[nb][2 * hh + 1] = fast_exp2(sc[nb][2 * hh + 1] - mu);
        sum += sc[nb][2 * hh] + sc[nb][2 * hh + 1];
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      m_row[hh] = mx;
      l_row[hh] = sum;
    }
    pf = make_uint4(pack_bf16(sc[0][0], sc[0][1]), pack_bf16(sc[0][2], sc[0][3]),
                    pack_bf16(sc[1][0], sc[1][1]), pack_bf16(sc[1][2], sc[1][3]));
  }

  // ---- the block's P and (m, l) into every CTA of the cluster ----
  cluster_wait();  // every CTA of the cluster runs and expects its bytes
  if (my_live) {
    const uint32_t pl = sbase + ScSmem::kP + static_cast<uint32_t>((blk_id * 32 + lane) * 16);
    const uint32_t ml = sbase + ScSmem::kML + static_cast<uint32_t>((blk_id * 8 + g) * 16);
    const uint4 mlv = make_uint4(__float_as_uint(m_row[0]), __float_as_uint(m_row[1]),
                                 __float_as_uint(l_row[0]), __float_as_uint(l_row[1]));
#pragma unroll
    for (int d = 0; d < SC_CTAS; ++d) {
      const uint32_t rb = map_to_cta(xbar, static_cast<uint32_t>(d));
      st_async_v4(map_to_cta(pl, static_cast<uint32_t>(d)), pf, rb);
      if (tq == 0) st_async_v4(map_to_cta(ml, static_cast<uint32_t>(d)), mlv, rb);
    }
  }
  // every live block's P, m and l are in this CTA
  if (!mbar_wait_sleep(xbar, 0) && tid == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);

  // ---- this warp's 8 output columns over every live block ----
  const float4 *sML = reinterpret_cast<const float4 *>(smem + ScSmem::kML);
  const uint4 *sP = reinterpret_cast<const uint4 *>(smem + ScSmem::kP);
  // every block's row maxima first (all loads in flight together), then
  // each block's P V with its factor, the loop unrolled so that the loads
  // of later blocks are issued ahead; a dead block (its shared memory not
  // written in this launch) issues no MMA and has the factor 0
  float4 mlb[SC_BLOCKS];
  float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
  for (int i = 0; i < SC_BLOCKS; ++i) {
    mlb[i] = sML[i * 8 + g];
    if (!((blk >> i) & 1u)) mlb[i] = make_float4(-INFINITY, -INFINITY, 0.f, 0.f);
    M0 = fmaxf(M0, mlb[i].x);
    M1 = fmaxf(M1, mlb[i].y);
  }
  float o[4] = {0.f, 0.f, 0.f, 0.f}, L0 = 0.f, L1 = 0.f;
#pragma unroll
  for (int i = 0; i < SC_BLOCKS; ++i) {
    const bool lv = ((blk >> i) & 1u) != 0u;
    const uint4 a = sP[i * 32 + lane];
    uint32_t b0, b1;
    ldsm_x2_t(sV + static_cast<uint32_t>((i * 16 + (lane & 15)) * SC_VPITCH + warp * 16), b0, b1);
    float t[4] = {0.f, 0.f, 0.f, 0.f};
    if (lv) mma_bf16(t, a.x, a.y, a.z, a.w, b0, b1);
    const float f0 = mlb[i].x == -INFINITY ? 0.f : fast_exp2(mlb[i].x - M0);
    const float f1 = mlb[i].y == -INFINITY ? 0.f : fast_exp2(mlb[i].y - M1);
    o[0] += f0 * t[0];
    o[1] += f0 * t[1];
    o[2] += f1 * t[2];
    o[3] += f1 * t[3];
    L0 += f0 * mlb[i].z;
    L1 += f1 * mlb[i].w;
  }
  const int col = rank * SC_VCOLS + warp * 8 + 2 * tq;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int r = g + 8 * hh;
    if (r >= n_rows) continue;
    const float L = hh ? L1 : L0;
    const float M = hh ? M1 : M0;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int tok = q_begin + r / p.group;
    const int head = h * p.group + r % p.group;
    *reinterpret_cast<uint32_t *>(p.out + static_cast<int64_t>(tok) * p.o_st +
                                  static_cast<int64_t>(head) * p.o_sh + col) =
        pack_bf16(o[2 * hh] * inv, o[2 * hh + 1] * inv);
    if (p.lse != nullptr && rank == 0 && warp == 0 && tq == 0)
      p.lse[static_cast<int64_t>(tok) * p.lse_st + static_cast<int64_t>(head) * p.lse_sh] =
          L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
}

// ------------------------------------------------------------------- host

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                   void *, const cuuint64_t *, const cuuint64_t *,
                                   const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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
  return fn;
}

// 4-D map over a [pages][P][H_kv][D] cache (dims innermost first); one box =
// one 64-column half of `pbox` rows of one page of one head.
bool encode_kv_map(CUtensorMap *map, const bf16 *base, int d, int h_kv, int page,
                   int64_t num_pages, int64_t s_head, int64_t s_pos, int64_t s_page,
                   int pbox) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h_kv),
                        static_cast<cuuint64_t>(page), static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s_head) * 2,
                           static_cast<cuuint64_t>(s_pos) * 2,
                           static_cast<cuuint64_t>(s_page) * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(pbox), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<bf16 *>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The TMA loader covers dense attention with page boxes of 8 or more rows
// (1024-byte aligned in shared memory) and strides that nest (head inside
// position inside page).
bool tma_eligible(const AttnParams &p) {
  if (p.topk != nullptr) return false;
  const int P = p.page_size;
  if (P % 8 != 0) return false;
  if (P <= BK ? (BK % P != 0) : (P % BK != 0)) return false;
  if (p.num_pages > 0xffffffffLL) return false;
  auto nests = [&](int64_t sh, int64_t spos, int64_t sp, int d) {
    return sh >= d && spos >= sh * p.h_kv && sp >= spos * P;
  };
  return nests(p.k_sh, p.k_spos, p.k_sp, p.d) && nests(p.v_sh, p.v_spos, p.v_sp, p.dv);
}

template <int D, int NSTAGE, bool TMA>
int launch_typed(const AttnParams &p, const DecodeMaps &maps, cudaStream_t stream) {
  constexpr size_t smem = Smem<D, NSTAGE>::kDynamic;
  constexpr int threads = NCT + (TMA ? 32 : 64);
  static std::atomic<bool> configured[64] = {};  // per device; calls may race
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(decode_gqa_kernel<D, NSTAGE, TMA>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  dim3 grid(p.num_splits, p.h_kv * p.n_row_tiles, p.batch);
  decode_gqa_kernel<D, NSTAGE, TMA><<<grid, threads, smem, stream>>>(p, maps);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

namespace {

// 4-D map over a paged cache listing position before head (dims innermost
// first: D, position, head, page), whatever the strides' order; one box =
// one 64-column half (bf16) or all 128 columns (fp8 codes, one byte each) of
// 16 positions of `hpc` heads of one page: 128-byte rows either way.
bool encode_allheads_map(CUtensorMap *map, const void *base, int h_kv, int page,
                         int64_t num_pages, int64_t s_head, int64_t s_pos, int64_t s_page,
                         int hpc, bool fp8) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t eb = fp8 ? 1 : 2;
  cuuint64_t dims[4] = {128, static_cast<cuuint64_t>(page), static_cast<cuuint64_t>(h_kv),
                        static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s_pos) * eb,
                           static_cast<cuuint64_t>(s_head) * eb,
                           static_cast<cuuint64_t>(s_page) * eb};
  cuuint32_t box[4] = {fp8 ? 128u : 64u, AH_BK, static_cast<cuuint32_t>(hpc), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
            const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_allheads_maps(AhMaps *m, const AttnParams &p, int hpc) {
  const bool fp8 = p.kv_fp8 != 0;
  return encode_allheads_map(&m->k, p.k, p.h_kv, p.page_size, p.num_pages, p.k_sh, p.k_spos,
                             p.k_sp, hpc, fp8) &&
         encode_allheads_map(&m->v, p.v, p.h_kv, p.page_size, p.num_pages, p.v_sh, p.v_spos,
                             p.v_sp, hpc, fp8);
}

}  // namespace

bool decode_allheads_eligible(const AttnParams &p) {
  if (p.topk != nullptr || p.d != 128 || p.dv != 128) return false;
  if (p.h_kv > AH_MAXH || p.max_seqlen_q < 1 || p.max_seqlen_q * p.group > 16) return false;
  // fp8: page boxes (multiples of 16) or slot rows (page size < 8)
  if (p.kv_fp8 && p.page_size >= 8 && p.page_size % AH_BK != 0) return false;
  if (p.page_size < 8) {
    // slot rows: every slot's heads form one contiguous H_kv x 128 row
    return p.k_sh == 128 && p.k_spos == static_cast<int64_t>(p.h_kv) * 128 &&
           p.v_sh == 128 && p.v_spos == static_cast<int64_t>(p.h_kv) * 128;
  }
  if (p.page_size % AH_BK != 0 || p.num_pages > 0x7fffffffLL) return false;
  // page boxes: the driver must accept the maps (strides, alignment)
  AhMaps m;
  return encode_allheads_maps(&m, p, p.h_kv);
}

int launch_decode_allheads(const AttnParams &p, cudaStream_t stream) {
  if (p.batch == 0) return PKV_OK;
  if (!decode_allheads_eligible(p)) return PKV_ERR_UNSUPPORTED;
  if (p.batch > 65535 || p.num_splits > 65535) return PKV_ERR_UNSUPPORTED;
  const bool balanced = p.num_splits == 0;
  if (balanced && p.batch > AH_MAXB) return PKV_ERR_UNSUPPORTED;
  const bool boxes = p.page_size >= 8;
  const bool fp8 = p.kv_fp8 != 0;
  if (fp8 && !balanced) return PKV_ERR_UNSUPPORTED;
  // Page boxes with fixed splits: kAhFixedHeads KV heads per CTA, so a
  // request's chunk is kAhFixedHeads / h_kv of a work item that covers every
  // head, and the items balance over the grid (longest requests first).
  int hpc = p.h_kv;
  if (boxes && !balanced && p.h_kv % kAhFixedHeads == 0) hpc = kAhFixedHeads;
  const AhLayout L = ah_layout(hpc, boxes, balanced, fp8);
  if (L.end > AH_SMEM_MAX) return PKV_ERR_UNSUPPORTED;
  if (p.append && fp8) return PKV_ERR_UNSUPPORTED;
  static std::atomic<bool> configured[64] = {};  // per device; calls may race
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    const void *fns[] = {reinterpret_cast<const void *>(decode_allheads_kernel<true, false, false>),
                         reinterpret_cast<const void *>(decode_allheads_kernel<false, false, false>),
                         reinterpret_cast<const void *>(decode_allheads_kernel<true, true, false>),
                         reinterpret_cast<const void *>(decode_allheads_kernel<true, false, true>),
                         reinterpret_cast<const void *>(decode_allheads_kernel<false, false, true>),
                         reinterpret_cast<const void *>(decode_allheads_kernel<false, true, false>)};
    for (const void *fn : fns)
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, AH_SMEM_MAX) !=
          cudaSuccess)
        return PKV_ERR_CUDA;
    if (dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  AhMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (boxes && !encode_allheads_maps(&maps, p, hpc)) return PKV_ERR_UNSUPPORTED;
  // balanced: one persistent CTA per SM, claiming shares; fixed splits:
  // (split, head group, request rank)
  const dim3 grid = balanced ? dim3(kDecodeBalancedCtas, 1, 1)
                             : dim3(p.num_splits, p.h_kv / hpc, p.batch);
  const dim3 block((hpc + (balanced ? 2 : 1)) * 32);  // + producer (+ merge warp)
  if (fp8 && boxes)
    decode_allheads_kernel<true, true, false><<<grid, block, L.end, stream>>>(p, maps);
  else if (fp8)
    decode_allheads_kernel<false, true, false><<<grid, block, L.end, stream>>>(p, maps);
  else if (boxes && p.append)
    decode_allheads_kernel<true, false, true><<<grid, block, L.end, stream>>>(p, maps);
  else if (boxes)
    decode_allheads_kernel<true, false, false><<<grid, block, L.end, stream>>>(p, maps);
  else if (p.append)
    decode_allheads_kernel<false, false, true><<<grid, block, L.end, stream>>>(p, maps);
  else
    decode_allheads_kernel<false, false, false><<<grid, block, L.end, stream>>>(p, maps);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

bool decode_short_eligible(const AttnParams &p) {
  return p.topk == nullptr && !p.kv_fp8 && p.d == 128 && p.dv == 128 && p.max_seqlen_q >= 1 &&
         p.max_seqlen_q * p.group <= 16 && p.page_size >= 1 &&
         static_cast<int64_t>(p.pt_cols) * p.page_size <= kDecodeShortMaxKeys;
}

int launch_decode_short(const AttnParams &p, cudaStream_t stream) {
  if (p.batch == 0) return PKV_OK;
  if (!decode_short_eligible(p)) return PKV_ERR_UNSUPPORTED;
  if (p.batch > 65535 || p.h_kv > 65535) return PKV_ERR_UNSUPPORTED;
  static std::atomic<bool> configured[64] = {};  // per device; calls may race
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(decode_short_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SD_SMEM)) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  if (static_cast<int64_t>(p.batch) * p.h_kv <= kDecodeShortClusterMaxPairs) {
    if (p.h_kv * SC_CTAS > 65535) return PKV_ERR_UNSUPPORTED;
    static std::atomic<bool> configured_c[64] = {};
    if (dev >= 64 || !configured_c[dev].load(std::memory_order_acquire)) {
      if (cudaFuncSetAttribute(decode_short_cluster_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(ScSmem::kEnd)) != cudaSuccess)
        return PKV_ERR_CUDA;
      if (dev < 64) configured_c[dev].store(true, std::memory_order_release);
    }
    const cudaError_t e = launch_programmatic(decode_short_cluster_kernel,
                                              dim3(p.h_kv * SC_CTAS, p.batch), dim3(SC_WARPS * 32),
                                              ScSmem::kEnd, stream, p);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  }
  const cudaError_t e = launch_programmatic(decode_short_kernel, dim3(p.h_kv, p.batch),
                                            dim3(SD_WARPS * 32), SD_SMEM, stream, p);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int launch_decode_gqa(const AttnParams &p, cudaStream_t stream) {
  if (p.batch == 0 || p.n_row_tiles == 0) return PKV_OK;
  if (p.h_kv * p.n_row_tiles > 65535 || p.batch > 65535 || p.num_splits > 65535)
    return PKV_ERR_UNSUPPORTED;
  if (!((p.d == 128 && p.dv == 128) || (p.d == 64 && p.dv == 64)))
    return PKV_ERR_UNSUPPORTED;
  DecodeMaps maps;
  memset(&maps, 0, sizeof(maps));
  bool tma = tma_eligible(p);
  if (tma) {
    const int pbox = p.page_size <= BK ? p.page_size : BK;
    tma = encode_kv_map(&maps.k, p.k, p.d, p.h_kv, p.page_size, p.num_pages, p.k_sh,
                        p.k_spos, p.k_sp, pbox) &&
          encode_kv_map(&maps.v, p.v, p.dv, p.h_kv, p.page_size, p.num_pages, p.v_sh,
                        p.v_spos, p.v_sp, pbox);
  }
  if (p.d == 128) {
    return tma ? launch_typed<128, 3, true>(p, maps, stream)
               : launch_typed<128, 3, false>(p, maps, stream);
  }
  return tma ? launch_typed<64, 4, true>(p, maps, stream)
             : launch_typed<64, 4, false>(p, maps, stream);
}

}  // namespace pkv
