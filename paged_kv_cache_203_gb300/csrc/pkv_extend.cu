// pkv_extend.cu -- varlen causal extend (chunked prefill) against a paged KV
// cache on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Computes the same attention as the decode kernel (flashattention_backend.py
// `forward_extend`: `flash_attn_with_kvcache` with cu_seqlens_q, causal, the
// (W, 0) window, bottom-right alignment) for long runs of new tokens, where
// it is a dense contraction.
//
// One CTA = one tile of 128 consecutive new tokens of one request for one q
// head; its keys stream in 128-key tiles (whole page boxes).
//   warp 8  producer: TMA loads of the Q tile once, then K and V tiles into
//           two 3-stage rings (4-D tensor-map boxes per page and 64-column
//           half, 128-byte swizzle), plus a per-tile key-validity bitmask;
//   warp 9  MMA issuer (one thread): S_j = Q K_j^T into TMEM buffer j%2,
//           then O += P_{j-1} V_{j-1} into the TMEM accumulator, each a chain
//           of eight 128x128x16 bf16 MMAs with fp32 accumulation; completion
//           signalled with tcgen05.commit on mbarriers (a K stage is released
//           when its QK^T is done, a V stage and the S/P buffer when its PV
//           is done);
//   warps 0-7 softmax: warps w and w+4 share TMEM lane quadrant w (query
//           rows 32w..32w+31) and split each key tile's 128 columns in two
//           halves.  Each half is an independent online softmax with its own
//           accumulator (keys 0-63 of every tile go to O_A, keys 64-127 to
//           O_B), so the halves never synchronise inside the loop; their
//           states are combined once in the epilogue (log-sum-exp merge).
//           Log2 domain, lazy reference max (O_hf and l rescaled in place only
//           when the max grows by more than 2^8); P_j (bf16, two per 32-bit
//           column) is stored back into TMEM over the half's own S_j columns
//           and is the A operand of the PV MMA straight from TMEM, so no
//           shared-memory store or proxy fence sits in the softmax loop; V
//           rows of keys past the sequence or in skipped pages are zeroed.
// TMEM: S0 | S1 | O_A | O_B (128 columns each, 512 in all; 1 CTA per SM);
// P_j occupies columns 0-31 and 64-95 of S_j's buffer until its PV is done.
// Every mbarrier wait is bounded (PKV_EFLAG_TIMEOUT on expiry).
#include <cuda.h>
#include <limits.h>
#include <string.h>

#include <atomic>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

using namespace ptx;

constexpr int BM = 128;           // query rows per CTA
constexpr int BN = 128;           // keys per tile
constexpr int D = 128;            // head dim (q/k and v)
constexpr int NSM_WARPS = 8;      // softmax warps: 2 per TMEM lane quadrant
constexpr int NTHREADS = NSM_WARPS * 32 + 64;  // + producer warp, MMA warp
constexpr int kProducerWarp = NSM_WARPS;
constexpr int kMmaWarp = NSM_WARPS + 1;
constexpr int HALF = BN / 2;      // S / P / O columns per softmax thread
constexpr uint32_t kTileBytes = BM * D * 2;  // 32 KB, any 128x128 bf16 tile
constexpr int NKV = 3;            // K and V ring stages

// Shared-memory plan; FP8 (a cache of e4m3 codes) adds the e4m3 Q tile, keeps
// K and V as codes (16 KB stages) and two f16 V tiles widened from them.
template <bool FP8>
struct Smem {
  static constexpr uint32_t kKStage = FP8 ? BN * 128u : kTileBytes;  // one K / V stage
  static constexpr uint32_t kQ = 0;                                   // Q, bf16 (TMA)
  static constexpr uint32_t kQ8 = kQ + kTileBytes;                    // Q rounded to e4m3
  static constexpr uint32_t kK = kQ8 + (FP8 ? BM * 128u : 0u);        // NKV stages
  static constexpr uint32_t kV = kK + NKV * kKStage;                  // NKV stages
  static constexpr uint32_t kV16 = kV + NKV * kKStage;                // [2] f16 V (FP8)
  static constexpr uint32_t kMask = kV16 + (FP8 ? 2 * kTileBytes : 0u);  // uint32 [4][4]
  static constexpr uint32_t kXchg = kMask + 64;  // float [m, l][2 halves][128 rows]
  static constexpr uint32_t kBar = kXchg + 2 * 2 * BM * 4;
  // barriers: q_full, k_full[NKV], v_full[NKV], k_empty[NKV], v_empty[NKV],
  //           s_full[2], s_free[2], p_full[2], o_done[2], xchg[2], mask_full[4],
  //           q8_ready
  static constexpr int kNumBars = 1 + 4 * NKV + 10 + 4 + 1;
  static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
  static constexpr uint32_t kEnd = kTmemSlot + 16;
  // The dynamic shared memory base must be 1024-byte aligned (128-byte
  // swizzle atoms); the kernel checks it and does no work otherwise.
  static constexpr size_t kDynamic = kEnd;
};
static_assert(Smem<false>::kDynamic <= 232448 && Smem<true>::kDynamic <= 232448,
              "shared memory plan exceeds 227 KB");
static_assert(Smem<true>::kK % 1024 == 0 && Smem<true>::kV % 1024 == 0 &&
                  Smem<true>::kV16 % 1024 == 0,
              "swizzled tiles start on 1024-byte boundaries");

enum BarId {
  Q_FULL = 0, K_FULL = 1, V_FULL = K_FULL + NKV, K_EMPTY = V_FULL + NKV,
  V_EMPTY = K_EMPTY + NKV, S_FULL = V_EMPTY + NKV, S_FREE = S_FULL + 2,
  P_FULL = S_FREE + 2, O_DONE = P_FULL + 2, XCHG = O_DONE + 2,
  MASK_FULL = XCHG + 2,  // [4]: the key mask of tile j is in slot j & 3
  Q8_READY = MASK_FULL + 4  // FP8: the e4m3 Q tile is written
};
static_assert(Q8_READY + 1 == Smem<false>::kNumBars, "barrier plan and count agree");

// Byte offset of 16-byte chunk c of row r of a 128-row tile stored as
// [2 halves][128 rows][128 B] with the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (BM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

struct ExtendMaps {
  CUtensorMap q;
  CUtensorMap k;
  CUtensorMap v;
};

// ---------------------------------------------------------------- kernel

template <bool FP8>
__global__ void __launch_bounds__(NTHREADS, 1)
extend_tc_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ ExtendMaps maps) {
  using SM = Smem<FP8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw;
  const uint32_t sbase = smem_addr(smem);
  uint32_t *sMask = reinterpret_cast<uint32_t *>(smem + SM::kMask);
  uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + SM::kTmemSlot);
  auto bar = [&](int id) { return sbase + SM::kBar + 8u * id; };

  const int n_qt = gridDim.x;
  const int qt = n_qt - 1 - blockIdx.x;  // longest tiles first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int q_begin = p.cu_seqlens_q[b];
  const int q_len = p.cu_seqlens_q[b + 1] - q_begin;
  const int kv_len = p.cache_seqlens[b];
  const int u0 = qt * BM;
  if (u0 >= q_len || q_begin < 0 || q_begin + u0 >= p.total_q) return;  // uniform
  if ((sbase & 1023u) != 0) {  // layout assumption violated: refuse, flag
    if (tid == 0) atomicOr(p.err, PKV_EFLAG_LAYOUT);
    return;
  }
  const int n_rows = min(BM, min(q_len - u0, p.total_q - (q_begin + u0)));
  const int kvh = h / p.group;

  // key range of the tile and its 128-key tiles
  const int i_min = kv_len - q_len + u0;
  const int i_max = i_min + n_rows - 1;
  int kv_end = kv_len;
  if (p.causal || p.window_left >= 0) kv_end = min(kv_end, i_max + 1);
  int kv_begin = 0;
  if (p.window_left >= 0) kv_begin = max(0, i_min - p.window_left);
  kv_end = max(kv_end, kv_begin);
  const int jt0 = kv_begin / BN;
  const int n_kv = (kv_end + BN - 1) / BN - jt0;

  if (tid == 0) {
    mbar_init(bar(Q_FULL), 1);
    for (int s = 0; s < NKV; ++s) {
      mbar_init(bar(K_FULL + s), 1);
      mbar_init(bar(V_FULL + s), 1);
      mbar_init(bar(K_EMPTY + s), 1);
      mbar_init(bar(V_EMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(S_FULL + s), 1);
      mbar_init(bar(S_FREE + s), 1);  // PV of the tile that used the buffer is done
      mbar_init(bar(P_FULL + s), NSM_WARPS);
      mbar_init(bar(O_DONE + s), 1);
      mbar_init(bar(XCHG + s), NSM_WARPS);
    }
    for (int s = 0; s < 4; ++s) mbar_init(bar(MASK_FULL + s), 1);
    mbar_init(bar(Q8_READY), NSM_WARPS);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    fence_proxy_async();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
                     smem_addr(sTmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS0 = tmem, tO = tmem + 256;  // O_A at tO, O_B at tO + 128

  if (warp == kProducerWarp) {
    // ================================ producer ================================
    const int P = p.page_size;
    const int pbox = P <= BN ? P : BN;
    const int nbox = BN / pbox;
    if (lane == 0 && n_kv > 0) {  // (no keys: nothing may stay in flight)
      mbar_arrive_expect_tx(bar(Q_FULL), kTileBytes);
      tma_load_3d(sbase + SM::kQ, &maps.q, 0, h, q_begin + u0, bar(Q_FULL));
      tma_load_3d(sbase + SM::kQ + BM * 128, &maps.q, 64, h, q_begin + u0, bar(Q_FULL));
    }
    for (int jj = 0; jj < n_kv; ++jj) {
      const int s = jj % NKV;
      const uint32_t prev = ((jj / NKV) & 1) ^ 1;
      // ---- K tile (stage freed when QK of tile jj-NKV completed) ----
      if (jj >= NKV && !mbar_wait_sleep(bar(K_EMPTY + s), prev)) {
        if (lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
        break;
      }
      const int key0 = (jt0 + jj) * BN;
      bool box_ok = false;
      int page = 0, inpage = 0;
      const int bpos0 = key0 + lane * pbox;
      if (lane < nbox && bpos0 < kv_len) {
        const int pidx = bpos0 / P;
        inpage = bpos0 - pidx * P;
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
      // bytes of the tile: a box row is 256 B of bf16 (two 64-column boxes)
      // or 128 B of codes (one box of all 128 columns)
      uint32_t bytes = box_ok ? static_cast<uint32_t>(pbox) * (FP8 ? 128u : 256u) : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
      const uint32_t roff = static_cast<uint32_t>(lane * pbox) * 128u;
      // key-validity mask of the tile (inside the sequence, page loaded),
      // published with K: slot jj & 3 was last read by the softmax of tile
      // jj - 4, which finished before the V stage this loop waited on below
      // for tile jj - 1 was released (the PV of tile jj - 1 - NKV >= jj - 4)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        const int okr = __shfl_sync(0xffffffffu, box_ok ? 1 : 0, r / pbox);
        const uint32_t bits = __ballot_sync(0xffffffffu, okr && key0 + r < kv_len);
        if (lane == 0) sMask[(jj & 3) * 4 + i] = bits;
      }
      if (lane == 0) mbar_arrive(bar(MASK_FULL + (jj & 3)));
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(bar(K_FULL + s), bytes);
      __syncwarp();
      if (box_ok) {
        const uint32_t kdst = sbase + SM::kK + s * SM::kKStage + roff;
        tma_load_4d(kdst, &maps.k, 0, kvh, inpage, page, bar(K_FULL + s));
        if (!FP8) tma_load_4d(kdst + BN * 128, &maps.k, 64, kvh, inpage, page, bar(K_FULL + s));
      }
      // ---- V tile (stage freed when the PV of tile jj-NKV completed) ----
      if (jj >= NKV && !mbar_wait_sleep(bar(V_EMPTY + s), prev)) {
        if (lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(bar(V_FULL + s), bytes);
      __syncwarp();
      if (box_ok) {
        const uint32_t vdst = sbase + SM::kV + s * SM::kKStage + roff;
        tma_load_4d(vdst, &maps.v, 0, kvh, inpage, page, bar(V_FULL + s));
        if (!FP8) tma_load_4d(vdst + BN * 128, &maps.v, 64, kvh, inpage, page, bar(V_FULL + s));
      }
    }
  } else if (warp == kMmaWarp) {
    // ================================== MMA ==================================
    if (lane == 0) {
      // bf16: QK^T and PV kind::f16 on bf16; FP8: QK^T kind::f8f6f4 on e4m3
      // (K 32 a step), PV kind::f16 on f16 (P in f16, V widened to f16)
      constexpr uint32_t kIdescQK = FP8 ? idesc_e4m3(BM, BN) : idesc_bf16(BM, BN, false);
      constexpr uint32_t kIdescPV = FP8 ? idesc_f16(BM, BN, true) : idesc_bf16(BM, BN, true);
      bool ok = n_kv == 0 || mbar_wait_sleep(bar(FP8 ? Q8_READY : Q_FULL), 0);
      const uint64_t qd0 = smem_desc(sbase + (FP8 ? SM::kQ8 : SM::kQ), 0, 1024, 2);
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {  // S_j = Q K_j^T
          const int s = j & 1, sk = j % NKV;
          ok = mbar_wait_sleep(bar(K_FULL + sk), (j / NKV) & 1) &&
               (j < 2 || mbar_wait_sleep(bar(S_FREE + s), ((j >> 1) - 1) & 1));
          if (!ok) break;
          tc_fence_after();
          // descriptors formed once per tile; a K step adds a constant to the
          // start-address field (16-byte units), so the single issuing
          // thread does no 64-bit descriptor arithmetic per MMA
          const uint64_t kd0 = smem_desc(sbase + SM::kK + sk * SM::kKStage, 0, 1024, 2);
          if (FP8) {
            // one 128-byte row holds all 128 dims: four K = 32 steps of 32 B
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_f8(tS0 + s * 128, qd0 + ks * 2, kd0 + ks * 2, kIdescQK, ks > 0);
          } else {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint64_t koff = ((ks >> 2) * (BM * 128) + (ks & 3) * 32) >> 4;
              umma(tS0 + s * 128, qd0 + koff, kd0 + koff, kIdescQK, ks > 0);
            }
          }
          umma_commit(bar(S_FULL + s));
          umma_commit(bar(K_EMPTY + sk));
        }
        if (j >= 1) {  // O += P_{j-1} V_{j-1}
          const int jj = j - 1;
          const int s = jj & 1, sv = jj % NKV;
          // FP8: P_FULL also says the softmax warps widened V_jj to f16
          ok = mbar_wait_sleep(bar(P_FULL + s), (jj >> 1) & 1) &&
               (FP8 || mbar_wait_sleep(bar(V_FULL + sv), (jj / NKV) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint64_t vd0 =
              smem_desc(sbase + (FP8 ? SM::kV16 + (jj & 1) * kTileBytes : SM::kV + sv * kTileBytes),
                        BN * 128, 1024, 2);
          // keys 0-63 of the tile accumulate into O_A, keys 64-127 into O_B
          // (each half of the softmax keeps its own reference max); P_j is
          // read from TMEM: keys 64h + 16k.. at column 128 s + 64 h + 8 k
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            umma_ts(tO + (ks >> 2) * 128, tS0 + s * 128 + (ks >> 2) * 64 + (ks & 3) * 8,
                    vd0 + ((ks * 2048) >> 4), kIdescPV, (jj > 0 || (ks & 3) > 0) ? 1u : 0u);
          umma_commit(bar(O_DONE + s));
          umma_commit(bar(V_EMPTY + sv));
          umma_commit(bar(S_FREE + s));  // S/P buffer s may take S_{jj+2}
        }
      }
      if (!ok) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
    }
  } else {
    // ================================ softmax ================================
    const int quad = warp & 3;               // TMEM lane quadrant
    const int hf = warp >> 2;                // which 64 key columns
    const int row = quad * 32 + lane;        // query row = TMEM lane
    const int u = u0 + row;
    const int i_r = kv_len - q_len + u;
    const bool use_upper = p.causal || p.window_left >= 0;
    const int lo_r = p.window_left >= 0 ? i_r - p.window_left : INT_MIN;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t col0 = hf * HALF;
    // the softmax scale (log2 domain), times k_descale of the (request, KV
    // head) for an fp8 cache; the row maxima below are of raw scores, so a
    // negative product flips the scores' sign instead
    float c = p.scale_log2;
    float vdesc = 1.f;
    if (FP8) {
      const int64_t di = static_cast<int64_t>(b) * p.h_kv + kvh;
      if (p.k_descale != nullptr) c *= p.k_descale[di];
      if (p.v_descale != nullptr) vdesc = p.v_descale[di];
    }
    const bool flip = c < 0.f;
    c = fabsf(c);
    float *xchg = reinterpret_cast<float *>(smem + SM::kXchg);  // [m, l][2 halves][128]
    float m_ref = -INFINITY;  // reference max (log2 domain) of O and l
    float l = 0.f;            // this half's share of the row sum
    bool ok = true;

    if (FP8 && n_kv > 0) {
      // Q rounded to e4m3 (the cache's type) once: bf16 tile [2 halves][128
      // rows][128 B] -> e4m3 tile [128 rows][128 B], both 128-byte swizzled;
      // 16-byte chunk c8 of a row holds dims 16 c8 .. 16 c8 + 15
      ok = mbar_wait_sleep(bar(Q_FULL), 0);
      if (ok) {
        const int t = warp * 32 + lane;  // 0..255
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int pr = t + 256 * k;
          const int r = pr >> 3, c8 = pr & 7;
          const uint4 a = *reinterpret_cast<const uint4 *>(smem + SM::kQ + tile_off(r, 2 * c8));
          const uint4 bq = *reinterpret_cast<const uint4 *>(smem + SM::kQ + tile_off(r, 2 * c8 + 1));
          const uint32_t w[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
          uint32_t o4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t lo = w[2 * i], hi = w[2 * i + 1];  // dims 4i .. 4i + 3
            o4[i] = round_e4m3x2(__uint_as_float(lo << 16), __uint_as_float(lo & 0xffff0000u)) |
                    (round_e4m3x2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u))
                     << 16);
          }
          *reinterpret_cast<uint4 *>(smem + SM::kQ8 + r * 128 + ((c8 ^ (r & 7)) << 4)) =
              make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
        fence_proxy_async();  // generic writes -> the tensor core's reads
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Q8_READY));
    }

    for (int jj = 0; jj < n_kv; ++jj) {
      const int s = jj & 1;
      const uint32_t ph = (jj >> 1) & 1;
      if (!(ok = mbar_wait_sleep(bar(S_FULL + s), ph))) break;
      tc_fence_after();
      float x[HALF];
      tmem_ld64(tS0 + s * 128 + col0 + lane_off, x);
      if (FP8 && flip) {
#pragma unroll
        for (int i = 0; i < HALF; ++i) x[i] = -x[i];
      }

      // the tile's key mask (its slot is rewritten only for tile jj + 4,
      // after this softmax is done, so the phase cannot run ahead)
      const int skv = jj % NKV;
      const uint32_t pkv = (jj / NKV) & 1;
      if (!(ok = mbar_wait_sleep(bar(MASK_FULL + (jj & 3)), (jj >> 2) & 1))) break;
      const int ms = (jj & 3) * 4;
      const int key0 = (jt0 + jj) * BN + col0;  // key of this thread's column 0
      const uint32_t mk0 = sMask[ms + 2 * hf], mk1 = sMask[ms + 2 * hf + 1];
      const uint32_t m_all = sMask[ms] & sMask[ms + 1] & sMask[ms + 2] & sMask[ms + 3];
      const bool all_valid = m_all == 0xffffffffu;
      const int tile_key0 = (jt0 + jj) * BN;
      const bool edge = !all_valid || (use_upper && tile_key0 + BN - 1 > i_min) ||
                        (p.window_left >= 0 && tile_key0 < i_max - p.window_left);
      if (edge) {
#pragma unroll
        for (int i = 0; i < HALF; ++i) {
          const int key = key0 + i;
          const uint32_t w = i < 32 ? mk0 : mk1;
          const bool msk = !((w >> (i & 31)) & 1u) || (use_upper && key > i_r) || key < lo_r;
          x[i] = msk ? -INFINITY : x[i];
        }
      }
      // row max over this half's 64 keys (raw scores): eight chains of
      // three-input maxima
      float pm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = ptx::fmax3(x[k], x[k + 8], x[k + 16]);
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = ptx::fmax3(pm[k], x[k + 24], x[k + 32]);
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = ptx::fmax3(pm[k], x[k + 40], x[k + 48]);
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = fmaxf(pm[k], x[k + 56]);
      float mx = ptx::fmax3(ptx::fmax3(pm[0], pm[1], pm[2]), ptx::fmax3(pm[3], pm[4], pm[5]),
                            fmaxf(pm[6], pm[7]));
      mx *= c;  // this half's max; it owns its own accumulator O_hf

      // lazy rescale: move the reference only when the max grew by > 2^8
      bool need = false;
      float factor = 1.f;
      if (mx > m_ref + 8.f) {
        need = m_ref != -INFINITY;  // O and l hold data only then
        factor = need ? fast_exp2(m_ref - mx) : 1.f;
        m_ref = mx;
      }
      if (__any_sync(0xffffffffu, need)) {
        // O holds P V of tiles 0..jj-1: wait for the last of them, scale
        const int t = jj - 1;
        if (!(ok = mbar_wait_sleep(bar(O_DONE + (t & 1)), (t >> 1) & 1))) break;
        tc_fence_after();
        const uint32_t tOh = tO + hf * 128 + lane_off;  // this half's O
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float v[32];
          tmem_ld32(tOh + ch * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= factor;
          tmem_st32(tOh + ch * 32, v);
        }
        tmem_st_wait();
      }
      l *= factor;

      // P = 2^(x c - m_ref): packed-pair FFMA, one MUFU per element,
      // packed-pair running sums (four pair accumulators)
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < HALF; i += 2) {
        ptx::ffma2(x[i], x[i + 1], c, -mu);
        x[i] = fast_exp2(x[i]);
        x[i + 1] = fast_exp2(x[i + 1]);
        ptx::fadd2(ps[(i >> 1) & 3], ps[4 + ((i >> 1) & 3)], x[i], x[i + 1]);
      }
      l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));

      // P (bf16 pairs) over this half's own first 32 S columns: the PV's A
      // operand in TMEM (the buffer was free for S_jj, so for P_jj too)
      {
        uint32_t pw[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          pw[i] = FP8 ? pack_f16(x[2 * i], x[2 * i + 1]) : pack_bf16(x[2 * i], x[2 * i + 1]);
        tmem_st32u(tS0 + s * 128 + col0 + lane_off, pw);
      }
      // V rows of keys outside the sequence or in skipped pages must be zero
      // (P is 0 there, but 0 * NaN would still poison the product); key row
      // `row` of the tile, this thread's half of its columns
      const uint32_t own = quad == 0 ? sMask[ms] : quad == 1 ? sMask[ms + 1]
                         : quad == 2 ? sMask[ms + 2] : sMask[ms + 3];
      if (FP8) {
        // key row `row` of V_jj, this thread's 64 columns: codes widened to
        // f16 into the tile the PV reads (zeros for keys outside the
        // sequence or in skipped pages).  The f16 tile jj & 1 was last read
        // by the PV of tile jj - 2, done before S_jj (its QK^T waited for
        // that buffer).
        if (!(ok = mbar_wait_sleep(bar(V_FULL + skv), pkv))) break;
        uint8_t *vt = smem + SM::kV16 + (jj & 1) * kTileBytes;
        const uint8_t *vc = smem + SM::kV + skv * SM::kKStage + row * 128;
        const bool live = (own >> lane) & 1u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // 16 codes -> two 16-byte f16 chunks
          uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
          if (live) {
            const uint4 cw = *reinterpret_cast<const uint4 *>(vc + (((hf * 4 + i) ^ (row & 7)) << 4));
            o0 = make_uint4(e4m3x2_to_f16x2(cw.x), e4m3x2_to_f16x2(cw.x >> 16),
                            e4m3x2_to_f16x2(cw.y), e4m3x2_to_f16x2(cw.y >> 16));
            o1 = make_uint4(e4m3x2_to_f16x2(cw.z), e4m3x2_to_f16x2(cw.z >> 16),
                            e4m3x2_to_f16x2(cw.w), e4m3x2_to_f16x2(cw.w >> 16));
          }
          *reinterpret_cast<uint4 *>(vt + tile_off(row, hf * 8 + 2 * i)) = o0;
          *reinterpret_cast<uint4 *>(vt + tile_off(row, hf * 8 + 2 * i + 1)) = o1;
        }
        fence_proxy_async();  // the f16 rows visible to the tensor core
      } else {
        if (!all_valid && !(ok = mbar_wait_sleep(bar(V_FULL + skv), pkv))) break;  // rows to zero
        if (!all_valid && !((own >> lane) & 1u)) {
          uint8_t *vt = smem + SM::kV + skv * kTileBytes;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<uint4 *>(vt + tile_off(row, hf * 8 + cc)) = make_uint4(0, 0, 0, 0);
        }
        if (!all_valid) fence_proxy_async();  // zeroed V rows visible to the tensor core
      }
      tmem_st_wait();     // P in TMEM
      tc_fence_before();  // (and the rescaled O columns)
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P_FULL + s));
    }

    // epilogue: the two halves' states (m, l, O_hf) meet once: this thread
    // writes output columns col0..col0+63 from O_A and O_B
    float oa[HALF], ob[HALF];
#pragma unroll
    for (int i = 0; i < HALF; ++i) oa[i] = ob[i] = 0.f;
    if (ok && n_kv > 0) {
      const int t = n_kv - 1;
      ok = mbar_wait_sleep(bar(O_DONE + (t & 1)), (t >> 1) & 1);
      if (ok) {
        tc_fence_after();
        tmem_ld64(tO + lane_off + col0, oa);
        tmem_ld64(tO + 128 + lane_off + col0, ob);
      }
    }
    float m_oth = -INFINITY, l_oth = 0.f;
    if (ok) {  // the only use of the exchange barrier: its first phase
      xchg[hf * BM + row] = m_ref;
      xchg[(2 + hf) * BM + row] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(XCHG));
      ok = mbar_wait_sleep(bar(XCHG), 0);
      if (ok) {
        m_oth = xchg[(hf ^ 1) * BM + row];
        l_oth = xchg[(2 + (hf ^ 1)) * BM + row];
      }
    }
    if (!ok && lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
    // this thread's (m, l) belong to O_hf; the partner's to the other one
    const float m_a = hf == 0 ? m_ref : m_oth, l_a = hf == 0 ? l : l_oth;
    const float m_b = hf == 0 ? m_oth : m_ref, l_b = hf == 0 ? l_oth : l;
    const float m_tot = fmaxf(m_a, m_b);
    const float f_a = m_a == -INFINITY ? 0.f : fast_exp2(m_a - m_tot);
    const float f_b = m_b == -INFINITY ? 0.f : fast_exp2(m_b - m_tot);
    const float l_tot = l_a * f_a + l_b * f_b;
    float o[HALF];
#pragma unroll
    for (int i = 0; i < HALF; ++i) o[i] = oa[i] * f_a + ob[i] * f_b;
    m_ref = m_tot;
    if (row < n_rows) {
      const float inv = l_tot > 0.f ? vdesc / l_tot : 0.f;  // v_descale: fp8 cache
      const int tok = q_begin + u;
      bf16 *dst = p.out + static_cast<int64_t>(tok) * p.o_st + static_cast<int64_t>(h) * p.o_sh +
                  col0;
#pragma unroll
      for (int cc = 0; cc < HALF; cc += 8) {
        uint4 w;
        w.x = pack_bf16(o[cc] * inv, o[cc + 1] * inv);
        w.y = pack_bf16(o[cc + 2] * inv, o[cc + 3] * inv);
        w.z = pack_bf16(o[cc + 4] * inv, o[cc + 5] * inv);
        w.w = pack_bf16(o[cc + 6] * inv, o[cc + 7] * inv);
        *reinterpret_cast<uint4 *>(dst + cc) = w;
      }
      if (p.lse != nullptr && hf == 0)
        p.lse[static_cast<int64_t>(tok) * p.lse_st + static_cast<int64_t>(h) * p.lse_sh] =
            l_tot > 0.f ? (m_ref + log2f(l_tot)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem)
                 : "memory");
  }
}

// ------------------------------------------------------------------- host

}  // namespace

bool extend_eligible(const AttnParams &p) {
  if (p.topk != nullptr || p.d != D || p.dv != D) return false;
  const int P = p.page_size;
  if (P % 8 != 0) return false;
  if (P <= BN ? (BN % P != 0) : (P % BN != 0)) return false;
  if (p.num_pages > 0xffffffffLL) return false;
  auto nests = [&](int64_t sh, int64_t spos, int64_t sp) {
    return sh >= D && spos >= sh * p.h_kv && sp >= spos * P;
  };
  return nests(p.k_sh, p.k_spos, p.k_sp) && nests(p.v_sh, p.v_spos, p.v_sp) &&
         p.q_sh >= D && p.q_st >= p.q_sh * p.h_q;
}

int launch_extend_tc(const AttnParams &p, cudaStream_t stream) {
  if (p.batch == 0 || p.total_q == 0 || p.max_seqlen_q == 0) return PKV_OK;
  if (!extend_eligible(p)) return PKV_ERR_UNSUPPORTED;
  const int n_qt = (p.max_seqlen_q + BM - 1) / BM;
  if (p.h_q > 65535 || p.batch > 65535) return PKV_ERR_UNSUPPORTED;
  ExtendMaps maps;
  memset(&maps, 0, sizeof(maps));
  const int pbox = p.page_size <= BN ? p.page_size : BN;
  {
    cuuint64_t dims[3] = {D, static_cast<cuuint64_t>(p.h_q), static_cast<cuuint64_t>(p.total_q)};
    cuuint64_t str[2] = {static_cast<cuuint64_t>(p.q_sh) * 2, static_cast<cuuint64_t>(p.q_st) * 2};
    cuuint32_t box[3] = {64, 1, BM};
    if (!encode_tensor_map(&maps.q, p.q, 3, dims, str, box)) return PKV_ERR_UNSUPPORTED;
  }
  const bool fp8 = p.kv_fp8 != 0;
  {
    // bf16: boxes of 64 columns (128 B) per half; fp8 codes: one box of all
    // 128 columns (128 B); strides in bytes
    const cuuint64_t eb = fp8 ? 1 : 2;
    cuuint64_t dims[4] = {D, static_cast<cuuint64_t>(p.h_kv), static_cast<cuuint64_t>(p.page_size),
                          static_cast<cuuint64_t>(p.num_pages)};
    cuuint32_t box[4] = {fp8 ? 128u : 64u, 1, static_cast<cuuint32_t>(pbox), 1};
    cuuint64_t sk[3] = {static_cast<cuuint64_t>(p.k_sh) * eb, static_cast<cuuint64_t>(p.k_spos) * eb,
                        static_cast<cuuint64_t>(p.k_sp) * eb};
    cuuint64_t sv[3] = {static_cast<cuuint64_t>(p.v_sh) * eb, static_cast<cuuint64_t>(p.v_spos) * eb,
                        static_cast<cuuint64_t>(p.v_sp) * eb};
    if (!encode_tensor_map(&maps.k, p.k, 4, dims, sk, box, fp8) ||
        !encode_tensor_map(&maps.v, p.v, 4, dims, sv, box, fp8))
      return PKV_ERR_UNSUPPORTED;
  }
  static std::atomic<bool> configured[64] = {};  // per device; calls may race
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(extend_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Smem<false>::kDynamic)) != cudaSuccess ||
        cudaFuncSetAttribute(extend_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Smem<true>::kDynamic)) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  dim3 grid(n_qt, p.h_q, p.batch);
  if (fp8)
    extend_tc_kernel<true><<<grid, NTHREADS, Smem<true>::kDynamic, stream>>>(p, maps);
  else
    extend_tc_kernel<false><<<grid, NTHREADS, Smem<false>::kDynamic, stream>>>(p, maps);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
