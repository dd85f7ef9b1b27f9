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
// would leave no TMEM columns for them).
//   warps 5-12 producers: per 16-key tile, gather the 576-wide rows with
//            16-byte cp.async into a [9 chunks][16 rows][128 B] 128-byte-
//            swizzled tile (zero rows for skipped keys), two rows per warp,
//            completion on mbarriers, four tiles in flight.  The list
//            entries and page ids of a tile are loaded one and two tiles
//            ahead, so the two dependent lookups stay off the copy path
//            (with them on it, each tile waited two global round trips);
//   warp 4   MMA issuer: S = Q K^T (M 128 heads, N 16 keys, K 576: 36
//            MMAs, both operands K-major), then O += P V (M 128, N 256 value
//            dims, K 16 keys: V is an MN-major view of the same key tile);
//   warps 0-3 softmax (thread = head = TMEM lane): scores from TMEM, masks,
//            online softmax in the log2 domain with a lazy reference max
//            (O rescaled in TMEM only when the row max grows by > 2^8), P
//            (bf16) to shared memory in the unswizzled core-matrix layout.
// Split lists are merged by the last CTA of each (token, half).  Every wait
// is bounded (PKV_EFLAG_TIMEOUT on expiry).
#include <limits.h>
#include <string.h>

#include "pkv_ptx.cuh"

namespace pkv {
namespace {

using namespace ptx;

constexpr int H = 128;        // query heads (the M dimension)
constexpr int DQK = 576;      // latent + rope
constexpr int DV = 512;       // latent (value) dims
constexpr int DVH = 256;      // value dims per CTA
constexpr int BKEYS = 16;     // keys per tile
constexpr int NSTG = 4;       // key-tile stages
constexpr int NCH = DQK / 64; // 64-column chunks of a row (9)
constexpr int NSOFT = 4, NPROD = 8;
constexpr int kMmaWarp = NSOFT;
constexpr int kProdWarp0 = NSOFT + 1;
constexpr int NTHREADS = (NSOFT + 1 + NPROD) * 32;
constexpr int kRowsPerWarp = BKEYS / NPROD;         // 2
constexpr uint32_t kQBytes = NCH * H * 128;         // 147456
constexpr uint32_t kKTile = NCH * BKEYS * 128;      // 18432
constexpr uint32_t kPTile = H * BKEYS * 2;          // 4096

struct Smem {
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kQBytes;          // NSTG stages
  static constexpr uint32_t kP = kK + NSTG * kKTile;
  static constexpr uint32_t kPos = kP + kPTile;         // int [NSTG][BKEYS]
  static constexpr uint32_t kBar = kPos + NSTG * BKEYS * 4;
  // q_full, full[NSTG], empty[NSTG], s_full[2], s_free[2], p_full, o_done
  static constexpr int kNumBars = 3 + 2 * NSTG + 4;
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
  S_FREE = S_FULL + 2,
  P_FULL = S_FREE + 2,
  O_DONE = P_FULL + 1
};

// byte offset of 16-byte chunk c (0..71) of row r in a 128-byte-swizzled
// [9][nrows][128 B] tile
template <int NROWS>
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (NROWS * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}
// P [128 heads][16 keys] bf16, unswizzled core matrices: 8 rows x 16 B,
// 128 B apart along the keys, 256 B apart along the heads
__device__ __forceinline__ uint32_t p_off(int m, int c) {
  return static_cast<uint32_t>((m >> 3) * 256 + c * 128 + (m & 7) * 16);
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(S_FULL + s), 1);
      mbar_init(bar(S_FREE + s), NSOFT);
    }
    mbar_init(bar(P_FULL), NSOFT);
    mbar_init(bar(O_DONE), 1);
    mbar_init_fence();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(sTmem), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS0 = tmem, tO = tmem + 256;

  if (warp >= kProdWarp0) {
    // ================================ producers ================================
    const int ptid = tid - kProdWarp0 * 32;  // 0..127
    if (ptid == 0 && n_kv > 0) {
      mbar_arrive_expect_tx(bar(Q_FULL), kQBytes);
#pragma unroll 1
      for (int c = 0; c < NCH; ++c)
        tma_load_3d(sbase + Smem::kQ + c * (H * 128), &maps.q, c * 64, 0, t, bar(Q_FULL));
    }
    const int32_t *list = p.topk + static_cast<int64_t>(t) * p.topk_stride;
    const int pw = warp - kProdWarp0;  // producer warp: rows pw + 8 i of each tile
    const int end_j = (tile0 + n_kv) * BKEYS;
    // lanes 0-15 follow key lane of the tile two ahead (list entry), one
    // ahead (page id) and current (row offset)
    auto load_idx = [&](int tile) -> int {
      const int j = (tile0 + tile) * BKEYS + lane;
      return (lane < BKEYS && tile < n_kv && j < end_j && j < p.topk_len) ? list[j] : -1;
    };
    auto page_of = [&](int idx) -> int64_t {
      if (idx < 0 || idx >= kv_len) return -1;
      const int pidx = idx / p.page_size;
      if (pidx >= p.pt_cols) return -2;
      return p.page_table[static_cast<int64_t>(b) * p.pt_stride + pidx];
    };
    int idx_cur = load_idx(0);
    int64_t pg_cur = page_of(idx_cur);
    int idx_nxt = load_idx(1);
    for (int jj = 0; jj < n_kv; ++jj) {
      const int s = jj % NSTG;
      // lookups for the next tiles go out first; their latency overlaps this
      // tile's wait and copies
      const int64_t pg_nxt = page_of(idx_nxt);
      const int idx_nn = load_idx(jj + 2);
      // this tile's key lane: position (or -1) and row offset
      int pos = -1;
      int64_t off = -1;
      if (lane < BKEYS) {
        if (idx_cur < -1 || idx_cur >= kv_len) {
          if (pw == 0 && idx_cur != -1 && (tile0 + jj) * BKEYS + lane < p.topk_len)
            atomicOr(p.err, PKV_EFLAG_TOPK_OOB);
        } else if (idx_cur >= 0) {
          if (pg_cur == -2) {
            if (pw == 0) atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
          } else if (pg_cur < 0 || pg_cur >= p.num_pages) {
            if (pw == 0) atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
          } else {
            pos = idx_cur;
            off = pg_cur * p.k_sp +
                  static_cast<int64_t>(idx_cur - (idx_cur / p.page_size) * p.page_size) * p.k_spos;
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
      if (pw == 0 && lane < BKEYS) sPos[s * BKEYS + lane] = pos;
      // gather this warp's rows: 72 chunks of 16 B each, lanes along the row
      const uint32_t kdst = sbase + Smem::kK + s * kKTile;
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const int r = pw + NPROD * i;
        const int64_t ro = __shfl_sync(0xffffffffu, off, r);
        const bf16 *src = ro >= 0 ? p.k + ro : p.k;
        const int nbytes = ro >= 0 ? 16 : 0;
#pragma unroll
        for (int c = lane; c < DQK / 8; c += 32)
          cp_async16(kdst + sw_off<BKEYS>(r, c), ro >= 0 ? src + c * 8 : src, nbytes);
      }
      cp_async_arrive(bar(FULL + s));
      mbar_arrive(bar(FULL + s));
      idx_cur = idx_nxt;
      pg_cur = pg_nxt;
      idx_nxt = idx_nn;
    }
  } else if (warp == kMmaWarp) {
    // ================================== MMA ==================================
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_bf16(H, BKEYS, false);
      constexpr uint32_t kIdescPV = idesc_bf16(H, DVH, true);
      bool ok = n_kv == 0 || mbar_wait(bar(Q_FULL), 0);
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {  // S_j = Q K_j^T
          const int s = j % NSTG, sb = j & 1;
          ok = mbar_wait(bar(FULL + s), (j / NSTG) & 1) &&
               (j < 2 || mbar_wait(bar(S_FREE + sb), ((j >> 1) - 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint32_t kb = sbase + Smem::kK + s * kKTile;
#pragma unroll 4
          for (int ks = 0; ks < DQK / 16; ++ks) {
            const uint32_t qoff = (ks >> 2) * (H * 128) + (ks & 3) * 32;
            const uint32_t koff = (ks >> 2) * (BKEYS * 128) + (ks & 3) * 32;
            umma(tS0 + sb * BKEYS, smem_desc(sbase + Smem::kQ + qoff, 0, 1024, 2),
                 smem_desc(kb + koff, 0, 1024, 2), kIdescQK, ks > 0);
          }
          umma_commit(bar(S_FULL + sb));
        }
        if (j >= 1) {  // O += P_{j-1} V_{j-1}
          const int jj = j - 1;
          const int s = jj % NSTG;
          ok = mbar_wait(bar(P_FULL), jj & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vb = sbase + Smem::kK + s * kKTile + hv * 4 * (BKEYS * 128);
          static_assert(BKEYS == 16, "one K=16 step of P V per tile");
          umma(tO, smem_desc(sbase + Smem::kP, 128, 256, 0),
               smem_desc(vb, BKEYS * 128, 1024, 2), kIdescPV, jj > 0 ? 1u : 0u);
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
    for (int jj = 0; jj < n_kv; ++jj) {
      const int s = jj % NSTG, sb = jj & 1;
      if (!(ok = mbar_wait(bar(S_FULL + sb), (jj >> 1) & 1) &&
                 mbar_wait(bar(FULL + s), (jj / NSTG) & 1)))
        break;
      tc_fence_after();
      float x[BKEYS];
      tmem_ld16(tS0 + sb * BKEYS + lane_off, x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(S_FREE + sb));
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < BKEYS; ++i) {
        const int pos = sPos[s * BKEYS + i];
        const bool msk = pos < 0 || (use_upper && pos > i_pos) || pos < lo_r;
        x[i] = msk ? -INFINITY : x[i] * c;
        mx = fmaxf(mx, x[i]);
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
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 64 && !configured[dev]) {
    if (cudaFuncSetAttribute(mla_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Smem::kDynamic)) != cudaSuccess)
      return PKV_ERR_CUDA;
    configured[dev] = true;
  }
  dim3 grid(p.num_splits, 2, p.total_q);
  mla_topk_kernel<<<grid, NTHREADS, Smem::kDynamic, stream>>>(p, maps);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
