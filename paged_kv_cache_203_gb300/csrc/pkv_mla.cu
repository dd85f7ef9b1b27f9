// pkv_mla.cu -- absorbed-MLA paged attention over top-k sparse key lists on
// the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Computes the absorbed multi-latent attention of flashattention_backend.py
// (`flash_attn_with_kvcache(q=q_rope, k_cache=k_rope, v_cache=c_kv,
// qv=q_nope)`: score = q_nope . c_kv + q_rope . k_rope, output = P c_kv) over
// the keys listed in each query's top-k row (nsa_backend.py `forward_decode`,
// `TopkTransformMethod.PAGED`: logical position -> page-table slot; -1 =
// skip).  Each key is one 576-wide latent row (512 c_kv + 64 k_rope); its
// first 512 entries are the value row, so every gathered row is read once.
//
// One CTA = (query token, 256-wide half of the value dims, chunk of its key
// list).  The output accumulator for 128 heads x 256 value dims fills half
// of TMEM; both halves recompute the scores (the full 128 x 512 accumulator
// would leave no TMEM columns for them).  The first 448 columns of Q live in
// TMEM as the A operand of Q K^T and the other 128 in shared memory, which
// leaves shared memory for five 32-key tiles: the gather is the limit, and
// a deeper ring measured faster than wider tiles (2 x 64 keys: 866 GB/s,
// 3 x 48: 1303, 5 x 32: 1357).
//   warps 5-12 producers: per 32-key tile, gather the 576-wide rows with
//            16-byte cp.async into a [9 chunks][32 rows][128 B] 128-byte-
//            swizzled tile (zero rows for skipped keys), four rows per warp,
//            completion on mbarriers, up to five tiles in flight.  The list
//            entries and page ids of a tile are loaded one and two tiles
//            ahead, so the two dependent lookups stay off the copy path
//            (with them on it, each tile waited two global round trips);
//   warp 4   MMA issuer: S = Q K^T (M 128 heads, N 32 keys, K 576: 36
//            MMAs, K-major), then O += P V (M 128, N 256 value dims, K 32
//            keys: V is an MN-major view of the same key tile).  Descriptors
//            are formed once per tile and the K steps fully unrolled (a lone
//            issuing thread that rebuilt them per step took longer than the
//            MMAs);
//   warps 0-3 softmax (thread = head = TMEM lane): scores from TMEM, masks,
//            online softmax in the log2 domain with a lazy reference max
//            (O rescaled in TMEM only when the row max grows by > 2^8), P
//            (bf16) to shared memory in the unswizzled core-matrix layout.
// Split lists are merged by the last CTA of each (token, half).  Every wait
// is bounded (PKV_EFLAG_TIMEOUT on expiry).
#include <limits.h>
#include <string.h>

#include <atomic>

#include "pkv_ptx.cuh"

namespace pkv {
namespace {

using namespace ptx;

constexpr int H = 128;        // query heads (the M dimension)
constexpr int DQK = 576;      // latent + rope
constexpr int DV = 512;       // latent (value) dims
constexpr int DVH = 256;      // value dims per CTA
constexpr int BKEYS = 32;     // keys per tile
constexpr int NSTG = 5;       // key-tile stages
constexpr int NCH_TM = 7;     // 64-column Q chunks held in TMEM (A operand)
constexpr int NCH = DQK / 64; // 64-column chunks of a row (9)
constexpr int NSOFT = 4, NPROD = 8;
constexpr int kMmaWarp = NSOFT;
constexpr int kProdWarp0 = NSOFT + 1;
constexpr int NTHREADS = (NSOFT + 1 + NPROD) * 32;
constexpr int kRowsPerWarp = BKEYS / NPROD;         // 4
constexpr uint32_t kQBytes = (NCH - NCH_TM) * H * 128;  // the shared-memory part: 49152
// TMEM columns: S (32) | Q chunks 0-6 (224) | O (256)
constexpr uint32_t kTmS = 0, kTmQ = 32, kTmO = 256;
static_assert(BKEYS <= kTmQ, "S fits its TMEM columns");
static_assert(kTmQ + NCH_TM * 32 <= kTmO, "TMEM plan overflows");
constexpr uint32_t kKTile = NCH * BKEYS * 128;      // 36864
constexpr int kLook = 2;                          // look-ahead of each lookup level (tiles)
constexpr int kRingA = 2 * kLook + 1, kRingB = kLook + 1;
constexpr uint32_t kPTile = H * BKEYS * 2;          // 8192

struct Smem {
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kQBytes;          // NSTG stages
  static constexpr uint32_t kP = kK + NSTG * kKTile;
  static constexpr uint32_t kPos = kP + kPTile;         // int [NSTG][BKEYS]
  // producers' look-ahead rings, per warp: list entries [RA][8], page ids [RB][8]
  static constexpr uint32_t kRing = kPos + NSTG * BKEYS * 4;
  static constexpr uint32_t kBar = kRing + NPROD * (kRingA + kRingB) * kRowsPerWarp * 4;
  // q_full, full[NSTG], empty[NSTG], s_full, s_free, p_full, o_done, q_tmem
  static constexpr int kNumBars = 2 * NSTG + 6;
  static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
  static constexpr uint32_t kFlag = kTmemSlot + 16;     // softmax: split ticket
  static constexpr uint32_t kEnd = kFlag + 16;
  static constexpr size_t kDynamic = kEnd;  // base must be 1024-aligned (checked)
};
static_assert(Smem::kDynamic <= 232448, "shared memory plan exceeds 227 KB");
enum BarId {
  Q_FULL = 0,
  FULL = 1,
  EMPTY = FULL + NSTG,
  S_FULL = EMPTY + NSTG,
  S_FREE = S_FULL + 1,
  P_FULL = S_FREE + 1,
  O_DONE = P_FULL + 1,
  Q_TMEM = O_DONE + 1
};

// byte offset of 16-byte chunk c (0..71) of row r in a 128-byte-swizzled
// [9][nrows][128 B] tile
template <int NROWS>
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (NROWS * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}
// P [128 heads][BKEYS keys] bf16, unswizzled core matrices: 8 rows x 16 B,
// 128 B apart along the keys, BKEYS * 16 B apart along the heads
__device__ __forceinline__ uint32_t p_off(int m, int c) {
  return static_cast<uint32_t>((m >> 3) * (BKEYS * 16) + c * 128 + (m & 7) * 16);
}

struct MlaMaps {
  CUtensorMap q;
};

__global__ void __launch_bounds__(NTHREADS, 1)
mla_topk_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ MlaMaps maps) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  int *sPos = reinterpret_cast<int *>(smem + Smem::kPos);
  uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + Smem::kTmemSlot);
  int *sFlag = reinterpret_cast<int *>(smem + Smem::kFlag);
  auto bar = [&](int id) { return sbase + Smem::kBar + 8u * id; };

  const int split = blockIdx.x;
  const int hv = blockIdx.y;        // value half
  const int t = blockIdx.z;         // query token
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  if ((sbase & 1023u) != 0) {
    if (tid == 0) atomicOr(p.err, PKV_EFLAG_LAYOUT);
    return;
  }
  // request of token t: largest b with cu[b] <= t
  int b = 0;
  {
    int lo = 0, hi = p.batch;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.cu_seqlens_q[mid] <= t) lo = mid; else hi = mid;
    }
    b = lo;
  }
  const int q_begin = p.cu_seqlens_q[b];
  const int q_len = p.cu_seqlens_q[b + 1] - q_begin;
  const bool covered = p.batch > 0 && q_begin <= t && t < q_begin + q_len;
  const int kv_len = covered ? p.cache_seqlens[b] : 0;
  const int i_pos = kv_len - q_len + (t - q_begin);  // absolute position of the token

  // this split's 32-key tiles of the token's list
  const int n_tiles_all = covered ? (p.topk_len + BKEYS - 1) / BKEYS : 0;
  const int per = (n_tiles_all + p.num_splits - 1) / p.num_splits;
  const int tile0 = min(n_tiles_all, split * per);
  const int n_kv = min(n_tiles_all, tile0 + per) - tile0;

  if (tid == 0) {
    mbar_init(bar(Q_FULL), 1);
    for (int s = 0; s < NSTG; ++s) {
      mbar_init(bar(FULL + s), NPROD * 32);
      mbar_init(bar(EMPTY + s), 1);
    }
    mbar_init(bar(S_FULL), 1);
    mbar_init(bar(S_FREE), NSOFT);
    mbar_init(bar(P_FULL), NSOFT);
    mbar_init(bar(O_DONE), 1);
    mbar_init(bar(Q_TMEM), NSOFT);
    mbar_init_fence();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(sTmem), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS0 = tmem + kTmS, tQ = tmem + kTmQ, tO = tmem + kTmO;

  if (warp >= kProdWarp0) {
    // ================================ producers ================================
    const int ptid = tid - kProdWarp0 * 32;  // 0..127
    if (ptid == 0 && n_kv > 0) {
      mbar_arrive_expect_tx(bar(Q_FULL), kQBytes);
#pragma unroll 1
      for (int c = NCH_TM; c < NCH; ++c)
        tma_load_3d(sbase + Smem::kQ + (c - NCH_TM) * (H * 128), &maps.q, c * 64, 0, t,
                    bar(Q_FULL));
    }
    const int32_t *list = p.topk + static_cast<int64_t>(t) * p.topk_stride;
    const int pw = warp - kProdWarp0;  // producer warp: rows pw + 8 i of each tile
    const int end_j = (tile0 + n_kv) * BKEYS;
    // Lane i < 8 of producer warp pw owns row pw + 8 i of every tile.  Its
    // list entry is fetched 2 * kLook tiles ahead and its page id kLook tiles
    // ahead, both with 4-byte cp.async into this warp's rings (one commit
    // group per tile), so no global load is waited on in the copy loop.
    const int myrow = pw + NPROD * lane;
    const bool keyl = lane < kRowsPerWarp;
    int *ringA = reinterpret_cast<int *>(smem + Smem::kRing) +
                 pw * (kRingA + kRingB) * kRowsPerWarp;
    int *ringB = ringA + kRingA * kRowsPerWarp;
    const uint32_t ringA_s = sbase + Smem::kRing + pw * (kRingA + kRingB) * kRowsPerWarp * 4;
    const uint32_t ringB_s = ringA_s + kRingA * kRowsPerWarp * 4;
    auto fetchA = [&](int tile) {  // list entry of this lane's row (or -1)
      if (!keyl) return;
      const int slot = (tile % kRingA) * kRowsPerWarp + lane;
      const int j = (tile0 + tile) * BKEYS + myrow;
      if (tile < n_kv && j < end_j && j < p.topk_len) cp_async4(ringA_s + slot * 4, list + j);
      else ringA[slot] = -1;
    };
    auto fetchB = [&](int tile) {  // page id of that entry (-1: no key, -2: row too short)
      if (!keyl) return;
      const int idx = ringA[(tile % kRingA) * kRowsPerWarp + lane];
      const int slot = (tile % kRingB) * kRowsPerWarp + lane;
      if (idx >= 0 && idx < kv_len) {
        const int pidx = idx / p.page_size;
        if (pidx < p.pt_cols)
          cp_async4(ringB_s + slot * 4,
                    p.page_table + static_cast<int64_t>(b) * p.pt_stride + pidx);
        else
          ringB[slot] = -2;
      } else {
        ringB[slot] = -1;
      }
    };
    for (int x = 0; x < 2 * kLook; ++x) fetchA(x);
    cp_async_commit();
    cp_async_wait_all();
    for (int x = 0; x < kLook; ++x) fetchB(x);
    cp_async_commit();
    cp_async_wait_all();
    for (int jj = 0; jj < n_kv; ++jj) {
      const int s = jj % NSTG;
      // entries of tile jj + kLook and page ids of tile jj have landed
      cp_async_wait_group<kLook - 1>();
      fetchB(jj + kLook);
      fetchA(jj + 2 * kLook);
      cp_async_commit();
      // this lane's row of tile jj: position (or -1) and row offset
      int pos = -1;
      int64_t off = -1;
      if (keyl) {
        const int ic = ringA[(jj % kRingA) * kRowsPerWarp + lane];
        const int64_t pc = ringB[(jj % kRingB) * kRowsPerWarp + lane];
        if (ic < -1 || ic >= kv_len) {
          if (ic != -1) atomicOr(p.err, PKV_EFLAG_TOPK_OOB);
        } else if (ic >= 0) {
          if (pc == -2) {
            atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
          } else if (pc < 0 || pc >= p.num_pages) {
            atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
          } else {
            pos = ic;
            off = pc * p.k_sp +
                  static_cast<int64_t>(ic - (ic / p.page_size) * p.page_size) * p.k_spos;
          }
        }
      }
      int ok = 1;
      if (lane == 0 && jj >= NSTG)
        ok = mbar_wait(bar(EMPTY + s), ((jj / NSTG) & 1) ^ 1) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
        break;
      }
      if (keyl) sPos[s * BKEYS + myrow] = pos;
      // gather this warp's rows: 72 chunks of 16 B each, lanes along the row
      const uint32_t kdst = sbase + Smem::kK + s * kKTile;
#pragma unroll 2
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const int r = pw + NPROD * i;
        const int64_t ro = __shfl_sync(0xffffffffu, off, i);
        const bf16 *src = ro >= 0 ? p.k + ro : p.k;
        const int nbytes = ro >= 0 ? 16 : 0;
#pragma unroll
        for (int c = lane; c < DQK / 8; c += 32)
          cp_async16(kdst + sw_off<BKEYS>(r, c), ro >= 0 ? src + c * 8 : src, nbytes);
      }
      cp_async_arrive(bar(FULL + s));
      mbar_arrive(bar(FULL + s));
    }
  } else if (warp == kMmaWarp) {
    // ================================== MMA ==================================
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_bf16(H, BKEYS, false);
      constexpr uint32_t kIdescPV = idesc_bf16(H, DVH, true);
      bool ok = n_kv == 0 || (mbar_wait(bar(Q_FULL), 0) && mbar_wait(bar(Q_TMEM), 0));
      const uint64_t qd0 = smem_desc(sbase + Smem::kQ, 0, 1024, 2);
      const uint64_t pd0 = smem_desc(sbase + Smem::kP, 128, BKEYS * 16, 0);
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {  // S_j = Q K_j^T (S is free once the softmax loaded S_{j-1})
          const int s = j % NSTG;
          ok = mbar_wait(bar(FULL + s), (j / NSTG) & 1) &&
               (j < 1 || mbar_wait(bar(S_FREE), (j - 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd0 = smem_desc(sbase + Smem::kK + s * kKTile, 0, 1024, 2);
          // K step ks: 16 columns = 32 bytes within chunk ks / 4 (descriptor
          // addresses are in 16-byte units)
#pragma unroll
          for (int ks = 0; ks < NCH_TM * 4; ++ks)  // A = Q columns from TMEM
            umma_ts(tS0, tQ + ks * 8,
                    kd0 + static_cast<uint64_t>(((ks >> 2) * (BKEYS * 128) + (ks & 3) * 32) >> 4),
                    kIdescQK, ks > 0 ? 1u : 0u);
#pragma unroll
          for (int ks = NCH_TM * 4; ks < DQK / 16; ++ks)  // A = Q columns from smem
            umma(tS0,
                 qd0 + static_cast<uint64_t>((((ks >> 2) - NCH_TM) * (H * 128) + (ks & 3) * 32) >> 4),
                 kd0 + static_cast<uint64_t>(((ks >> 2) * (BKEYS * 128) + (ks & 3) * 32) >> 4),
                 kIdescQK, 1u);
          umma_commit(bar(S_FULL));
        }
        if (j >= 1) {  // O += P_{j-1} V_{j-1}
          const int jj = j - 1;
          const int s = jj % NSTG;
          ok = mbar_wait(bar(P_FULL), jj & 1);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vd0 =
              smem_desc(sbase + Smem::kK + s * kKTile + hv * 4 * (BKEYS * 128), BKEYS * 128, 1024, 2);
#pragma unroll
          for (int ks = 0; ks < BKEYS / 16; ++ks)  // 16 keys = 2 P chunks = 2 V row groups
            umma(tO, pd0 + static_cast<uint64_t>((ks * 256) >> 4),
                 vd0 + static_cast<uint64_t>((ks * 2048) >> 4), kIdescPV,
                 (jj > 0 || ks > 0) ? 1u : 0u);
          umma_commit(bar(O_DONE));
          umma_commit(bar(EMPTY + s));
        }
      }
      if (!ok) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
    }
  } else {
    // ================================ softmax ================================
    const int row = tid;  // head = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float c = p.scale_log2;
    const bool use_upper = p.causal || p.window_left >= 0;
    const int lo_r = p.window_left >= 0 ? i_pos - p.window_left : INT_MIN;
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    if (n_kv > 0) {
      // Q row `row`, columns 0..447, as packed bf16 pairs into TMEM columns
      // tQ .. tQ + 223 of this thread's lane (the A operand of Q K^T)
      const uint4 *qsrc = reinterpret_cast<const uint4 *>(
          p.q + static_cast<int64_t>(t) * p.q_st + static_cast<int64_t>(row) * p.q_sh);
#pragma unroll 1
      for (int cb = 0; cb < NCH_TM; ++cb) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 w = qsrc[cb * 8 + i];
          r[4 * i] = w.x;
          r[4 * i + 1] = w.y;
          r[4 * i + 2] = w.z;
          r[4 * i + 3] = w.w;
        }
        tmem_st32u(tQ + lane_off + cb * 32, r);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Q_TMEM));
    }
    for (int jj = 0; jj < n_kv; ++jj) {
      const int s = jj % NSTG;
      if (!(ok = mbar_wait(bar(S_FULL), jj & 1) && mbar_wait(bar(FULL + s), (jj / NSTG) & 1)))
        break;
      tc_fence_after();
      float x[BKEYS];
      {
        static_assert(BKEYS == 32, "S row load below is written for 32 keys");
        tmem_ld32(tS0 + lane_off, x);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(S_FREE));
      float mx = -INFINITY;
      const int4 *pos4 = reinterpret_cast<const int4 *>(sPos + s * BKEYS);
#pragma unroll
      for (int i4 = 0; i4 < BKEYS / 4; ++i4) {
        const int4 pp = pos4[i4];
        const int pv[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = 4 * i4 + u;
          const int pos = pv[u];
          const bool msk = pos < 0 || (use_upper && pos > i_pos) || pos < lo_r;
          x[i] = msk ? -INFINITY : x[i] * c;
          mx = fmaxf(mx, x[i]);
        }
      }
      bool need = false;
      float factor = 1.f;
      if (mx > m_ref + 8.f) {
        need = m_ref != -INFINITY;
        factor = need ? fast_exp2(m_ref - mx) : 1.f;
        m_ref = mx;
      }
      // P buffer (and O) are free once the PV of tile jj-1 completed
      if (jj >= 1 && !(ok = mbar_wait(bar(O_DONE), (jj - 1) & 1))) break;
      if (__any_sync(0xffffffffu, need)) {
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < DVH / 32; ++ch) {
          float v[32];
          tmem_ld32(tO + lane_off + ch * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= factor;
          tmem_st32(tO + lane_off + ch * 32, v);
        }
        tmem_st_wait();
      }
      l *= factor;
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < BKEYS; ++i) {
        x[i] = fast_exp2(x[i] - mu);
        sum += x[i];
      }
      l += sum;
#pragma unroll
      for (int cc = 0; cc < BKEYS / 8; ++cc) {
        uint4 w;
        w.x = pack_bf16(x[8 * cc], x[8 * cc + 1]);
        w.y = pack_bf16(x[8 * cc + 2], x[8 * cc + 3]);
        w.z = pack_bf16(x[8 * cc + 4], x[8 * cc + 5]);
        w.w = pack_bf16(x[8 * cc + 6], x[8 * cc + 7]);
        *reinterpret_cast<uint4 *>(smem + Smem::kP + p_off(row, cc)) = w;
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P_FULL));
    }

    // ---- epilogue: this CTA's normalised state for its 256 value dims ----
    bool have_o = false;
    if (ok && n_kv > 0) {
      ok = mbar_wait(bar(O_DONE), (n_kv - 1) & 1);
      have_o = ok;
      if (ok) tc_fence_after();
    }
    if (!ok && lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_nat = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
    const int64_t rows_total = static_cast<int64_t>(p.total_q) * p.h_q;
    const int64_t grow = static_cast<int64_t>(t) * p.h_q + row;
    const bool split_mode = p.num_splits > 1;
#pragma unroll 1
    for (int ch = 0; ch < DVH / 32; ++ch) {
      float v[32];
      if (have_o) {
        tmem_ld32(tO + lane_off + ch * 32, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      const int col = hv * DVH + ch * 32;
      if (!split_mode) {
        if (covered) {
          bf16 *dst = p.out + static_cast<int64_t>(t) * p.o_st + static_cast<int64_t>(row) * p.o_sh + col;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16(v[i] * inv, v[i + 1] * inv);
            w.y = pack_bf16(v[i + 2] * inv, v[i + 3] * inv);
            w.z = pack_bf16(v[i + 4] * inv, v[i + 5] * inv);
            w.w = pack_bf16(v[i + 6] * inv, v[i + 7] * inv);
            *reinterpret_cast<uint4 *>(dst + i) = w;
          }
        }
      } else {
        float *dst = p.ws_o + (static_cast<int64_t>(split) * rows_total + grow) * p.dv + col;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          __stcg(reinterpret_cast<float4 *>(dst + i),
                 make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv));
      }
    }
    if (!split_mode) {
      if (covered && hv == 0 && p.lse != nullptr)
        p.lse[static_cast<int64_t>(t) * p.lse_st + static_cast<int64_t>(row) * p.lse_sh] = lse_nat;
    } else {
      // both value halves see the same scores, so each keeps its own copy of
      // every split's lse ([half][split][token][head]) and merges from it
      const int ns = p.num_splits;
      float *lse_half = p.ws_lse + static_cast<int64_t>(hv) * ns * rows_total;
      __stcg(lse_half + split * rows_total + grow, lse_nat);
      __threadfence();
      asm volatile("bar.sync 1, %0;\n" ::"n"(NSOFT * 32) : "memory");
      if (tid == 0) {
        int32_t *ctr = p.ws_counter + static_cast<int64_t>(t) * 2 + hv;
        *sFlag = (atomicAdd(ctr, 1) == ns - 1);
      }
      asm volatile("bar.sync 1, %0;\n" ::"n"(NSOFT * 32) : "memory");
      if (*sFlag && covered) {
        __threadfence();  // every split's state is visible from here on
        float Ms = -INFINITY;
        for (int sp = 0; sp < ns; ++sp) Ms = fmaxf(Ms, __ldcg(lse_half + sp * rows_total + grow));
        float wsum = 0.f;
        for (int sp = 0; sp < ns; ++sp)
          wsum += Ms == -INFINITY ? 0.f
                                  : exp2f((__ldcg(lse_half + sp * rows_total + grow) - Ms) * kLog2e);
        const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
        bf16 *dst = p.out + static_cast<int64_t>(t) * p.o_st + static_cast<int64_t>(row) * p.o_sh +
                    hv * DVH;
#pragma unroll 1
        for (int cc = 0; cc < DVH; cc += 8) {
          float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int sp = 0; sp < ns; ++sp) {
            const float ls = __ldcg(lse_half + sp * rows_total + grow);
            const float w = Ms == -INFINITY ? 0.f : exp2f((ls - Ms) * kLog2e);
            const float *src = p.ws_o + (static_cast<int64_t>(sp) * rows_total + grow) * p.dv +
                               hv * DVH + cc;
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(src));
            const float4 bq = __ldcg(reinterpret_cast<const float4 *>(src + 4));
            acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
            acc[4] += w * bq.x; acc[5] += w * bq.y; acc[6] += w * bq.z; acc[7] += w * bq.w;
          }
          uint4 wv;
          wv.x = pack_bf16(acc[0] * winv, acc[1] * winv);
          wv.y = pack_bf16(acc[2] * winv, acc[3] * winv);
          wv.z = pack_bf16(acc[4] * winv, acc[5] * winv);
          wv.w = pack_bf16(acc[6] * winv, acc[7] * winv);
          *reinterpret_cast<uint4 *>(dst + cc) = wv;
        }
        if (hv == 0 && p.lse != nullptr)
          p.lse[static_cast<int64_t>(t) * p.lse_st + static_cast<int64_t>(row) * p.lse_sh] =
              wsum > 0.f ? Ms + logf(wsum) : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_mla_topk(const AttnParams &p, cudaStream_t stream) {
  if (p.total_q == 0) return PKV_OK;
  if (p.topk == nullptr || p.h_q != H || p.h_kv != 1 || p.d != DQK || p.dv != DV)
    return PKV_ERR_UNSUPPORTED;
  if (p.v != p.k || p.v_sp != p.k_sp || p.v_spos != p.k_spos) return PKV_ERR_UNSUPPORTED;
  if (p.q_sh < DQK || p.q_st < p.q_sh * H || p.num_splits > 64) return PKV_ERR_UNSUPPORTED;
  if (p.total_q > 65535) return PKV_ERR_UNSUPPORTED;
  MlaMaps maps;
  memset(&maps, 0, sizeof(maps));
  cuuint64_t dims[3] = {DQK, H, static_cast<cuuint64_t>(p.total_q)};
  cuuint64_t str[2] = {static_cast<cuuint64_t>(p.q_sh) * 2, static_cast<cuuint64_t>(p.q_st) * 2};
  cuuint32_t box[3] = {64, H, 1};
  if (!encode_tensor_map(&maps.q, p.q, 3, dims, str, box)) return PKV_ERR_UNSUPPORTED;
  static std::atomic<bool> configured[64] = {};  // per device; calls may race
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(mla_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Smem::kDynamic)) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  dim3 grid(p.num_splits, 2, p.total_q);
  mla_topk_kernel<<<grid, NTHREADS, Smem::kDynamic, stream>>>(p, maps);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
