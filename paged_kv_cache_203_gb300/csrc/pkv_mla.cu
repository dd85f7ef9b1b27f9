// pkv_mla.cu -- absorbed-MLA paged attention over top-k sparse key lists on
// the 5th-generation tensor cores (tcgen05 + TMEM), one 2-CTA cluster per
// (query token, chunk of its key list).
//
// Computes the absorbed multi-latent attention of flashattention_backend.py
// (`flash_attn_with_kvcache(q=q_rope, k_cache=k_rope, v_cache=c_kv,
// qv=q_nope)`: score = q_nope . c_kv + q_rope . k_rope, output = P c_kv) over
// the keys listed in each query's top-k row (nsa_backend.py `forward_decode`,
// `TopkTransformMethod.PAGED`: logical position -> page-table slot; -1 =
// skip).  Each key is one 576-wide latent row (512 c_kv + 64 k_rope); its
// first 512 entries are the value row.
//
// TMEM holds 512 fp32 columns per SM: the 128 x 512 output accumulator fills
// all of it, leaving nothing for the scores.  So the work of one (token,
// chunk) is split by kind, not by value columns, over the two CTAs of a
// cluster, and every score is computed once:
//   rank 0 ("score CTA"): Q (all 576 columns, bf16) in TMEM as the A operand;
//     per 64-key tile S = Q K^T (M 128 heads, N 64 keys, K 576: 36 MMAs) into
//     one of two TMEM score buffers; four softmax warps (thread = head) add
//     the key mask, run the online softmax in the log2 domain with a lazy
//     reference max, and store P (bf16) and the per-head rescale factors
//     straight into the value CTA's shared memory (distributed shared-memory
//     stores, an async-proxy fence, a remote barrier arrive).  At the end it
//     sends 1/l and the lse of each head.
//   rank 1 ("value CTA"): O (128 x 512 fp32) in all of TMEM; per tile
//     O += P V (M 128, N 2 x 256 value columns, K 64 keys: 8 MMAs); when the
//     score CTA raised a head's reference max, its four epilogue warps
//     rescale those O rows in TMEM first.  Epilogue: O * (1/l) -> bf16 output
//     (or a split partial, merged by the last CTA of the token).
// Each CTA gathers the columns it needs of every listed row (score CTA: 576,
// value CTA: the first 512) with 16-byte cp.async into 128-byte-swizzled
// [chunks][64 keys][128 B] tiles, three stages each, so neither pipeline
// waits on the other's stage recycling; the second read of a row is an L2
// hit.  (Gathering each row once and exchanging halves between the CTAs was
// measured slower: the exchange ties the score CTA's stages to the value
// CTA's, which are freed only after the softmax and PV.)  The gather loop is
// bound by its issue rate through the shared-memory/MIO pipe, which it shares
// with shuffles and barrier polls, so row offsets are broadcast once per tile
// and every wait sleeps in hardware between polls.
// Warps: 0-3 softmax (score) / epilogue + rescale (value); 4 MMA issuer;
// 5 forwarder of "P consumed" to the score CTA (value CTA; idle in the score
// CTA); 6-13 producers.  Every wait is bounded (PKV_EFLAG_TIMEOUT on expiry).
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
constexpr int BK = 64;        // keys per tile
constexpr int NCH = DQK / 64; // 64-column (128-byte) chunks of a key row (9)
constexpr int NSTG = 3;       // stages on each side
constexpr int NSOFT = 4, NPROD = 8;
constexpr int kMmaWarp = NSOFT;
constexpr int kFwdWarp = NSOFT + 1;
constexpr int kProdWarp0 = NSOFT + 2;
constexpr int NTHREADS = (NSOFT + 2 + NPROD) * 32;  // 448
constexpr int kRowsPerWarp = BK / NPROD;            // 8
constexpr uint32_t kChunk = BK * 128;               // 8192: one chunk of a tile
constexpr uint32_t kKTile = NCH * kChunk;           // 73728 (score CTA: all 9 chunks)
constexpr uint32_t kVTile = 8 * kChunk;             // 65536 (value CTA: chunks 0-7)
constexpr uint32_t kPTile = H * BK * 2;             // 16384: P [128 heads][64 keys] bf16
constexpr uint32_t kFacWarp = 144;                  // 32 factors, a flag word, padding
constexpr uint32_t kPXfer = kPTile + NSOFT * kFacWarp;  // 16960 bytes per P buffer
constexpr uint32_t kFinBytes = H * 8;               // (1/l, lse) per head
// fp8 cache: two MMA stages of f16 tiles plus two staging tiles of the
// gathered codes (rows of 576 B on the score side, 512 B on the value side)
// take the bytes of the three bf16 stages
constexpr int NSTG_F8 = 2;
constexpr uint32_t kStgScore = BK * DQK;            // 36864
constexpr uint32_t kStgValue = BK * DV;             // 32768
static_assert(NSTG_F8 * kKTile + 2 * kStgScore <= NSTG * kKTile &&
                  NSTG_F8 * kVTile + 2 * kStgValue <= NSTG * kVTile,
              "fp8 staging fits the bf16 stage budget");
// TMEM columns.  Score CTA: Q [0, 288) as packed bf16 pairs, S0 at 384, S1 at
// 448.  Value CTA: O [0, 512).
constexpr uint32_t kTmQ = 0, kTmS = 384;
static_assert(kTmQ + DQK / 2 <= kTmS && kTmS + 2 * BK <= 512, "TMEM plan");

constexpr uint32_t kQRow = DQK * 2 + 16;  // a staged Q row (padded: 4-way banked reads)
struct Smem {
  // score CTA
  static constexpr uint32_t kK = 0;                          // NSTG key tiles
  // bf16: Q rows staged by bulk copies in the bytes of stages 1-2 (and a
  // little past them) until the softmax warps have moved them to TMEM
  static constexpr uint32_t kQStage = kK + kKTile;
  static constexpr uint32_t kBias = kQStage + H * kQRow;     // float [NSTG][BK]: 0 or -inf
  // value CTA
  static constexpr uint32_t kV = 0;                          // NSTG value tiles
  static constexpr uint32_t kP = kV + NSTG * kVTile;         // P as received [2][kPXfer]
  static constexpr uint32_t kFin = kP + 2 * kPXfer;          // float2 [H]
  // both (same offsets in both CTAs: each CTA addresses the peer's barriers
  // by their local offsets)
  static constexpr uint32_t kCtl = kFin + kFinBytes;
  static constexpr int kNumBars = 16;
  static constexpr uint32_t kTmemSlot = kCtl + kNumBars * 8;
  static constexpr uint32_t kWord = kTmemSlot + 16;          // int[4]: ticket, rescale tile
  static constexpr uint32_t kEnd = kWord + 16;
  static constexpr size_t kDynamic = kEnd;  // base must be 1024-aligned (checked)
};
static_assert(Smem::kBias + NSTG * BK * 4 <= Smem::kCtl, "score-CTA plan overlaps the control block");
static_assert(Smem::kBias >= Smem::kK + NSTG * kKTile && Smem::kBias >= NSTG_F8 * kKTile + 2 * BK * DQK,
              "key masks past every score-CTA stage");
static_assert(Smem::kDynamic <= 232448, "shared memory plan exceeds 227 KB");
static_assert(kPXfer % 16 == 0 && kFacWarp % 16 == 0, "16-byte aligned P buffers");

enum BarId {
  FULL = 0,          // [3] the stage's rows landed (producers' cp.async)
  EMPTY = 3,         // [3] the stage was consumed
  P_FREE = 6,        // [2] score CTA: the value CTA finished the PV of P buffer b (remote)
  S_FULL = 8,        // [2] score CTA: QK^T done      | value CTA: P_FULL (4 remote arrivals)
  P_FULL = 8,
  S_FREE = 10,       // [2] score CTA: S read         | value CTA: PV_DONE
  PV_DONE = 10,
  Q_TMEM = 12,       //     score CTA: Q is in TMEM   | value CTA: O_DONE (each PV done)
  O_DONE = 12,
  CORR_REQ = 13,     // value CTA: rescale request (or stop) to the epilogue warps
  Q_LANDED = 13,     // score CTA: the staged Q rows landed (bytes)
  CORR_DONE = 14,    // value CTA: rescale done
  Q_STAGED = 14,     // score CTA: the staged rows are in TMEM (stages 1-2 reusable)
  FIN = 15           // value CTA: (1/l, lse) landed (4 remote arrivals)
};

// byte offset of 16-byte unit c (0..71) of row r in a 128-byte-swizzled
// [chunks][BK rows][128 B] tile
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * kChunk + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}
// P [128 heads][64 keys] bf16 in unswizzled core matrices (8 heads x 16 B):
// 128 B apart along the keys, 1024 B apart along the heads.
__device__ __forceinline__ uint32_t p_off(int m, int c) {
  return static_cast<uint32_t>((m >> 3) * (BK * 16) + c * 128 + (m & 7) * 16);
}

// One producer lane's view of a key: list position -> slot row offset.
struct RowRef {
  int pos;      // logical key position, or -1 (no key)
  int64_t off;  // element offset of its row in the cache, or -1
};

__device__ __forceinline__ int list_entry(const AttnParams &p, const int32_t *list, int j,
                                          int end_j) {
  return (j < end_j && j < p.topk_len) ? __ldg(list + j) : -1;
}
// Page id of a list entry: the page-table load (or -1: no key / bad entry,
// -2: the row is too short).
__device__ __forceinline__ int page_of(const AttnParams &p, int b, int e, int kv_len) {
  if (e < 0 || e >= kv_len) return -1;
  const int pidx = e / p.page_size;
  if (pidx >= p.pt_cols) return -2;
  return __ldg(p.page_table + static_cast<int64_t>(b) * p.pt_stride + pidx);
}
__device__ __forceinline__ RowRef resolve(const AttnParams &p, int e, int pc, int kv_len,
                                          bool report) {
  RowRef r{-1, -1};
  if (e < -1 || e >= kv_len) {
    if (report && e != -1) atomicOr(p.err, PKV_EFLAG_TOPK_OOB);
  } else if (e >= 0) {
    if (pc == -2) {
      if (report) atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
    } else if (pc < 0 || pc >= p.num_pages) {
      if (report) atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
    } else {
      r.pos = e;
      r.off = static_cast<int64_t>(pc) * p.k_sp +
              static_cast<int64_t>(e - (e / p.page_size) * p.page_size) * p.k_spos;
    }
  }
  return r;
}

template <bool FP8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
mla_topk_kernel(const __grid_constant__ AttnParams p) {
  constexpr int NS = FP8 ? NSTG_F8 : NSTG;  // MMA stages
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + Smem::kTmemSlot);
  volatile int *sWord = reinterpret_cast<volatile int *>(smem + Smem::kWord);
  auto bar = [&](int id) { return sbase + Smem::kCtl + 8u * id; };

  const uint32_t rank = cluster_ctarank();  // 0: scores + softmax, 1: values
  const uint32_t peer = rank ^ 1u;
  const bool score = rank == 0;
  const int split = blockIdx.x >> 1;
  const int t = blockIdx.z;                 // query token
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  if ((sbase & 1023u) != 0) {  // the same in both CTAs of a launch
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

  // this split's 64-key tiles of the token's list
  const int n_tiles_all = covered ? (p.topk_len + BK - 1) / BK : 0;
  const int per = (n_tiles_all + p.num_splits - 1) / p.num_splits;
  const int tile0 = min(n_tiles_all, split * per);
  const int n_kv = min(n_tiles_all, tile0 + per) - tile0;

  // bf16 Q rows go through shared memory by bulk copies when their rows are
  // 16-byte aligned (else each softmax thread loads its row from global)
  const bool qstage = !FP8 && (reinterpret_cast<uintptr_t>(p.q) & 15) == 0 && p.q_st % 8 == 0 &&
                      p.q_sh % 8 == 0;
  if (score && warp < NSOFT && covered && !qstage) {  // warm L2 with this head's Q row
    const bf16 *qrow = p.q + static_cast<int64_t>(t) * p.q_st + static_cast<int64_t>(tid) * p.q_sh;
#pragma unroll
    for (int i = 0; i < NCH; ++i) prefetch_line_l2(qrow + i * 64);
  }
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(FULL + s), NPROD * 32);
      mbar_init(bar(EMPTY + s), score ? 1 + NSOFT : 1);
    }
    if (score) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(bar(S_FULL + i), 1);
        mbar_init(bar(S_FREE + i), NSOFT);
        mbar_init(bar(P_FREE + i), 1);
      }
      mbar_init(bar(Q_TMEM), NSOFT);
      mbar_init(bar(Q_LANDED), 1);
      mbar_init(bar(Q_STAGED), NSOFT);
    } else {
      for (int i = 0; i < 2; ++i) {
        mbar_init(bar(P_FULL + i), NSOFT);
        mbar_init(bar(PV_DONE + i), 1);
      }
      mbar_init(bar(O_DONE), 1);
      mbar_init(bar(CORR_REQ), 1);
      mbar_init(bar(CORR_DONE), NSOFT);
      mbar_init(bar(FIN), NSOFT);
    }
    mbar_init_fence();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(sTmem), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers are initialised before any remote use
  const uint32_t tmem = *sTmem;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const int end_j = (tile0 + n_kv) * BK;
  const int32_t *list = p.topk + static_cast<int64_t>(t) * p.topk_stride;
  const uint32_t ring = sbase + (score ? Smem::kK : Smem::kV);
  const uint32_t tile_bytes = score ? kKTile : kVTile;

  if (warp >= kProdWarp0) {
    // ================================ producers ================================
    // Lane l < 8 of producer warp pw owns row pw * 8 + l of every tile.  Its
    // list entry is loaded kAhead + kLagP + kLagE tiles ahead, its page id
    // kAhead + kLagP tiles ahead and the row resolved kAhead tiles ahead, all
    // in registers: each load has kLagE (kLagP) iterations to land before its
    // value is used, since loads issued behind the SM's in-flight gathers
    // take as long as the gathers.  Per tile: wait for the stage, gather this
    // CTA's columns of the 64 rows (zeros for skipped keys), and (score CTA)
    // publish each key's additive mask: 0, or -inf for no key / outside the
    // causal or window bound.
    constexpr int kAhead = 2, kLagP = 3, kLagE = 3;
    const int pw = warp - kProdWarp0;
    const bool own = lane < kRowsPerWarp;
    const int myrow = pw * kRowsPerWarp + lane;
    const bool use_upper = p.causal || p.window_left >= 0;
    const int lo_r = p.window_left >= 0 ? i_pos - p.window_left : INT_MIN;
    auto entry = [&](int tile) {
      return (own && tile < n_kv) ? list_entry(p, list, (tile0 + tile) * BK + myrow, end_j) : -1;
    };
    auto page = [&](int e) { return own ? page_of(p, b, e, kv_len) : -1; };
    auto res = [&](int e, int pg) {
      return own ? resolve(p, e, pg, kv_len, score) : RowRef{-1, -1};
    };
    RowRef rr[kAhead + 1];        // rows of tiles jj .. jj + kAhead
    int E[kLagP + kLagE + 1];     // entries of tiles jj + kAhead .. + kLagP + kLagE
    int G[kLagP + 1];             // page ids of tiles jj + kAhead .. + kLagP
#pragma unroll
    for (int k = 0; k < kAhead; ++k) {
      const int e = entry(k);
      rr[k] = res(e, page(e));
    }
#pragma unroll
    for (int k = 0; k < kLagP + kLagE; ++k) E[k] = entry(kAhead + k);
#pragma unroll
    for (int k = 0; k < kLagP; ++k) G[k] = page(E[k]);
    float *sBias = reinterpret_cast<float *>(smem + Smem::kBias);
    auto key_bias = [&](int pos) {
      const bool vis = pos >= 0 && !(use_upper && pos > i_pos) && pos >= lo_r;
      return vis ? 0.f : -INFINITY;
    };
    // fp8 cache: the codes of tile jj land in staging slot jj & 1 (rows of
    // 576 / 512 B); one tile later this warp widens its own 8 rows to f16
    // into MMA stage jj % NS (exact: an e4m3 value is an f16 value), writes
    // the key mask, and arrives on the stage's barrier
    const uint8_t *k8 = reinterpret_cast<const uint8_t *>(p.k);
    const uint32_t stg_row = score ? DQK : DV;
    const uint32_t stg0 = ring + NS * tile_bytes;
    auto widen = [&](int jt, int pos, bool last) -> bool {
      const int s = jt % NS;
      if (last) cp_async_wait_group<0>();
      else cp_async_wait_group<1>();
      __syncwarp();  // the warp's other lanes' copies are visible
      int ok = 1;
      if (lane == 0 && jt >= NS) ok = mbar_wait_sleep(bar(EMPTY + s), ((jt / NS) & 1) ^ 1) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      if (score && own) sBias[s * BK + myrow] = key_bias(pos);
      const uint32_t dst0 = ring + s * tile_bytes;
      const uint32_t src0 = stg0 + (jt & 1) * (BK * stg_row);
#pragma unroll
      for (int rl = 0; rl < kRowsPerWarp; ++rl) {  // value columns: 16 codes a lane
        const int row = pw * kRowsPerWarp + rl;
        uint4 cw;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(cw.x), "=r"(cw.y), "=r"(cw.z), "=r"(cw.w)
                     : "r"(src0 + row * stg_row + lane * 16));
        const uint4 o0 = make_uint4(e4m3x2_to_f16x2(cw.x), e4m3x2_to_f16x2(cw.x >> 16),
                                    e4m3x2_to_f16x2(cw.y), e4m3x2_to_f16x2(cw.y >> 16));
        const uint4 o1 = make_uint4(e4m3x2_to_f16x2(cw.z), e4m3x2_to_f16x2(cw.z >> 16),
                                    e4m3x2_to_f16x2(cw.w), e4m3x2_to_f16x2(cw.w >> 16));
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(dst0 + sw_off(row, 2 * lane)),
                     "r"(o0.x), "r"(o0.y), "r"(o0.z), "r"(o0.w) : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(dst0 + sw_off(row, 2 * lane + 1)),
                     "r"(o1.x), "r"(o1.y), "r"(o1.z), "r"(o1.w) : "memory");
      }
      if (score) {  // rope columns: 4 lanes a row
        const int row = pw * kRowsPerWarp + (lane >> 2), c = lane & 3;
        uint4 cw;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(cw.x), "=r"(cw.y), "=r"(cw.z), "=r"(cw.w)
                     : "r"(src0 + row * stg_row + DV + c * 16));
        const uint4 o0 = make_uint4(e4m3x2_to_f16x2(cw.x), e4m3x2_to_f16x2(cw.x >> 16),
                                    e4m3x2_to_f16x2(cw.y), e4m3x2_to_f16x2(cw.y >> 16));
        const uint4 o1 = make_uint4(e4m3x2_to_f16x2(cw.z), e4m3x2_to_f16x2(cw.z >> 16),
                                    e4m3x2_to_f16x2(cw.w), e4m3x2_to_f16x2(cw.w >> 16));
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"r"(dst0 + sw_off(row, 64 + 2 * c)),
                     "r"(o0.x), "r"(o0.y), "r"(o0.z), "r"(o0.w) : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};\n"
                     ::"r"(dst0 + sw_off(row, 64 + 2 * c + 1)),
                     "r"(o1.x), "r"(o1.y), "r"(o1.z), "r"(o1.w) : "memory");
      }
      fence_proxy_async();  // generic writes -> the tensor core's reads
      mbar_arrive(bar(FULL + s));
      return true;
    };
    int prev_pos = -1;  // fp8: the key of this lane's row in the tile being widened
    bool ok_all = true;
    for (int jj = 0; jj < n_kv; ++jj) {
      const int s = jj % NS;
      E[kLagP + kLagE] = entry(jj + kAhead + kLagP + kLagE);
      G[kLagP] = page(E[kLagP]);
      rr[kAhead] = res(E[0], G[0]);
      // the warp's 8 row offsets, broadcast once (shuffles share the pipe
      // with the copies and barrier polls); skipped keys read zeros
      int64_t ro[kRowsPerWarp];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) ro[r] = __shfl_sync(0xffffffffu, rr[0].off, r);
      if (FP8) {
        const uint32_t stg = stg0 + (jj & 1) * (BK * stg_row);
#pragma unroll
        for (int rl = 0; rl < kRowsPerWarp; ++rl)  // 512 codes of a row per instruction
          cp_async16(stg + (pw * kRowsPerWarp + rl) * stg_row + lane * 16,
                     ro[rl] >= 0 ? k8 + ro[rl] + lane * 16 : k8, ro[rl] >= 0 ? 16 : 0);
        if (score) {  // the 64 rope codes: 8 rows per instruction
          const int rl = lane >> 2, c = lane & 3;
          const int64_t r8 = __shfl_sync(0xffffffffu, rr[0].off, rl);
          cp_async16(stg + (pw * kRowsPerWarp + rl) * stg_row + DV + c * 16,
                     r8 >= 0 ? k8 + r8 + DV + c * 16 : k8, r8 >= 0 ? 16 : 0);
        }
        cp_async_commit();
        if (jj >= 1 && !widen(jj - 1, prev_pos, false)) {
          ok_all = false;
          break;
        }
        prev_pos = rr[0].pos;
      } else {
        int ok = 1;
        if (lane == 0 && jj >= NS)
          ok = mbar_wait_sleep(bar(EMPTY + s), ((jj / NS) & 1) ^ 1) ? 1 : 0;
        // stages 1-2 hold the staged Q rows until they are in TMEM
        if (lane == 0 && ok && score && qstage && jj == 1)
          ok = mbar_wait_sleep(bar(Q_STAGED), 0) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          ok_all = false;
          break;
        }
        const uint32_t dst0 = ring + s * tile_bytes;
        if (score && own) sBias[s * BK + myrow] = key_bias(rr[0].pos);
        // value chunks 0-7: half a row (512 B) per instruction, row known at
        // compile time
#pragma unroll
        for (int i = 0; i < 2 * kRowsPerWarp; ++i) {
          const int rl = i >> 1;
          const int c = lane + 32 * (i & 1);
          const bf16 *src = ro[rl] >= 0 ? p.k + ro[rl] + c * 8 : p.k;
          cp_async16(dst0 + sw_off(pw * kRowsPerWarp + rl, c), src, ro[rl] >= 0 ? 16 : 0);
        }
        if (score) {
          // the rope chunk (8): 4 rows per instruction
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int rl = (lane >> 3) + 4 * i;
            const int c = (NCH - 1) * 8 + (lane & 7);
            const int64_t r8 = __shfl_sync(0xffffffffu, rr[0].off, rl);
            const bf16 *src = r8 >= 0 ? p.k + r8 + c * 8 : p.k;
            cp_async16(dst0 + sw_off(pw * kRowsPerWarp + rl, c), src, r8 >= 0 ? 16 : 0);
          }
        }
        cp_async_arrive(bar(FULL + s));
        mbar_arrive(bar(FULL + s));
      }
#pragma unroll
      for (int k = 0; k < kAhead; ++k) rr[k] = rr[k + 1];
#pragma unroll
      for (int k = 0; k < kLagP + kLagE; ++k) E[k] = E[k + 1];
#pragma unroll
      for (int k = 0; k < kLagP; ++k) G[k] = G[k + 1];
    }
    if (FP8 && ok_all && n_kv >= 1 && !widen(n_kv - 1, prev_pos, true)) ok_all = false;
    if (!ok_all && lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
    cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ================================== MMA ==================================
    if (lane == 0 && score) {
      // fp8 cache: f16 operands (codes widened exactly, q rounded to e4m3)
      constexpr uint32_t kIdescQK = FP8 ? idesc_f16(H, BK, false) : idesc_bf16(H, BK, false);
      bool ok = n_kv == 0 || mbar_wait_sleep(bar(Q_TMEM), 0);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % NS, bb = j & 1;
        ok = mbar_wait_sleep(bar(FULL + s), (j / NS) & 1) &&
             (j < 2 || mbar_wait_sleep(bar(S_FREE + bb), ((j >> 1) - 1) & 1));
        if (!ok) break;
        fence_proxy_async();
        tc_fence_after();
        const uint64_t kd0 = smem_desc(ring + s * kKTile, 0, 1024, 2);
        const uint32_t dS = tmem + kTmS + bb * BK;
        // K step ks: 16 columns = 32 bytes within chunk ks / 4 (descriptor
        // addresses are in 16-byte units); A = Q columns from TMEM
#pragma unroll
        for (int ks = 0; ks < DQK / 16; ++ks)
          umma_ts(dS, tmem + kTmQ + ks * 8,
                  kd0 + static_cast<uint64_t>(((ks >> 2) * kChunk + (ks & 3) * 32) >> 4),
                  kIdescQK, ks > 0 ? 1u : 0u);
        umma_commit(bar(S_FULL + bb));
        umma_commit(bar(EMPTY + s));
      }
      if (!ok) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
    } else if (lane == 0) {
      constexpr uint32_t kIdescPV = FP8 ? idesc_f16(H, 256, true) : idesc_bf16(H, 256, true);
      bool ok = true;
      int n_corr = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % NS, bb = j & 1;
        ok = mbar_wait_sleep(bar(FULL + s), (j / NS) & 1) &&
             mbar_wait_cluster_sleep(bar(P_FULL + bb), (j >> 1) & 1);
        if (!ok) break;
        // did the score CTA raise any head's reference max for this tile?
        const uint8_t *fac = smem + Smem::kP + bb * kPXfer + kPTile;
        int any = 0;
#pragma unroll
        for (int w = 0; w < NSOFT; ++w)
          any |= *reinterpret_cast<const volatile int *>(fac + w * kFacWarp + 128);
        if (any) {
          sWord[1] = j;
          mbar_arrive(bar(CORR_REQ));
          ok = mbar_wait_sleep(bar(CORR_DONE), n_corr & 1);
          ++n_corr;
          if (!ok) break;
        }
        fence_proxy_async();
        tc_fence_after();
        const uint64_t pd0 = smem_desc(sbase + Smem::kP + bb * kPXfer, 128, BK * 16, 0);
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint64_t vd = smem_desc(ring + s * kVTile + h * 4 * kChunk, kChunk, 1024, 2);
            umma(tmem + h * 256, pd0 + static_cast<uint64_t>((ks * 256) >> 4),
                 vd + static_cast<uint64_t>((ks * 2048) >> 4), kIdescPV,
                 (j > 0 || ks > 0) ? 1u : 0u);
          }
        }
        umma_commit(bar(EMPTY + s));
        umma_commit(bar(PV_DONE + bb));
        umma_commit(bar(O_DONE));
      }
      if (!ok) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
      sWord[1] = -1;  // stop the epilogue warps' rescale loop
      mbar_arrive(bar(CORR_REQ));
    }
  } else if (warp == kFwdWarp) {
    // ======================= forwarder (value CTA only) =======================
    // The PV of P buffer b is done: tell the score CTA it may refill it.
    if (!score && lane == 0) {
      const uint32_t remote0 = map_to_cta(bar(P_FREE), peer);
      for (int j = 0; j < n_kv; ++j) {
        const int bb = j & 1;
        if (!mbar_wait_sleep(bar(PV_DONE + bb), (j >> 1) & 1)) {
          atomicOr(p.err, PKV_EFLAG_TIMEOUT);
          break;
        }
        mbar_arrive_remote(remote0 + 8u * bb);
      }
    }
  } else if (score) {
    // ============================ softmax (score CTA) ============================
    const int row = tid;  // head = TMEM lane
    // softmax scale (log2 domain), times the request's k_descale (fp8)
    const float c = p.scale_log2 * ((FP8 && p.k_descale != nullptr) ? p.k_descale[b] : 1.f);
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    const uint32_t peer_P = map_to_cta(sbase + Smem::kP, peer);
    const uint32_t peer_pfull = map_to_cta(bar(P_FULL), peer);
    if (n_kv > 0) {
      // Q row `row` (576 bf16) as packed pairs into TMEM columns 0..287 of
      // this thread's lane: the A operand of Q K^T.  bf16 (aligned rows):
      // one bulk copy per row into shared memory, read back 384 bytes at a
      // time; else three 192-column loads from global in flight at a time
      // (the row's lines were warmed at kernel start)
      const uint4 *qsrc = reinterpret_cast<const uint4 *>(
          p.q + static_cast<int64_t>(t) * p.q_st + static_cast<int64_t>(row) * p.q_sh);
      const uint32_t qs = sbase + Smem::kQStage + static_cast<uint32_t>(row) * kQRow;
      if (qstage) {
        if (row == 0) mbar_arrive_expect_tx(bar(Q_LANDED), H * DQK * 2);
        asm volatile("bar.sync 2, %0;\n" ::"n"(NSOFT * 32) : "memory");  // expectation first
        bulk_g2s(qs, qsrc, DQK * 2, bar(Q_LANDED));
        if (!mbar_wait_sleep(bar(Q_LANDED), 0)) {
          ok = false;
          if (lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
        }
      }
#pragma unroll 1
      for (int cb0 = 0; cb0 < NCH; cb0 += 3) {
        uint4 w[24];
        if (qstage) {
#pragma unroll
          for (int i = 0; i < 24; ++i)
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                         : "=r"(w[i].x), "=r"(w[i].y), "=r"(w[i].z), "=r"(w[i].w)
                         : "r"(qs + (cb0 * 8 + i) * 16));
        } else {
#pragma unroll
          for (int i = 0; i < 24; ++i) w[i] = qsrc[cb0 * 8 + i];
        }
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          uint32_t r[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            r[4 * i] = w[8 * k + i].x;
            r[4 * i + 1] = w[8 * k + i].y;
            r[4 * i + 2] = w[8 * k + i].z;
            r[4 * i + 3] = w[8 * k + i].w;
          }
          if (FP8) {  // q rounded to e4m3 (the cache's type), held as f16 pairs
#pragma unroll
            for (int i = 0; i < 32; ++i)
              r[i] = e4m3x2_to_f16x2(round_e4m3x2(__uint_as_float(r[i] << 16),
                                                  __uint_as_float(r[i] & 0xffff0000u)));
          }
          tmem_st32u(tmem + kTmQ + lane_off + (cb0 + k) * 32, r);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(Q_TMEM));
        if (qstage) mbar_arrive(bar(Q_STAGED));  // the staged rows were read
      }
    }
    const float *sBias = reinterpret_cast<const float *>(smem + Smem::kBias);
    for (int jj = 0; jj < n_kv; ++jj) {
      const int s = jj % NS, bb = jj & 1;
      if (!(ok = mbar_wait_sleep(bar(S_FULL + bb), (jj >> 1) & 1) &&
                 mbar_wait_sleep(bar(FULL + s), (jj / NS) & 1)))
        break;
      tc_fence_after();
      float x[BK];
      {
        float (&x0)[32] = *reinterpret_cast<float (*)[32]>(&x[0]);
        float (&x1)[32] = *reinterpret_cast<float (*)[32]>(&x[32]);
        tmem_ld32(tmem + kTmS + bb * BK + lane_off, x0);
        tmem_ld32(tmem + kTmS + bb * BK + 32 + lane_off, x1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(S_FREE + bb));
      // scale to the log2 domain and add the key mask (0 / -inf)
      const float4 *b4 = reinterpret_cast<const float4 *>(sBias + s * BK);
#pragma unroll
      for (int i4 = 0; i4 < BK / 4; ++i4) {
        const float4 bq = b4[i4];
        ffma2v(x[4 * i4], x[4 * i4 + 1], c, bq.x, bq.y);
        ffma2v(x[4 * i4 + 2], x[4 * i4 + 3], c, bq.z, bq.w);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(EMPTY + s));  // mask read: the stage may refill
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < BK; i += 2) mx = fmax3(mx, x[i], x[i + 1]);
      bool need = false;
      float factor = 1.f;
      if (mx > m_ref + 8.f) {
        need = m_ref != -INFINITY;
        factor = need ? fast_exp2(m_ref - mx) : 1.f;
        m_ref = mx;
      }
      l *= factor;
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int i = 0; i < BK; i += 2) {
        fadd2(x[i], x[i + 1], -mu, -mu);
        x[i] = fast_exp2(x[i]);
        x[i + 1] = fast_exp2(x[i + 1]);
        fadd2(s0, s1, x[i], x[i + 1]);
      }
      l += s0 + s1;
      // the value CTA's P buffer bb is free once its PV of tile jj-2 is done
      int okw = 1;
      if (lane == 0 && jj >= 2) okw = mbar_wait_cluster_sleep(bar(P_FREE + bb), ((jj >> 1) - 1) & 1);
      if (!(ok = __shfl_sync(0xffffffffu, okw, 0) != 0)) break;
      const uint32_t dst = peer_P + bb * kPXfer;
#pragma unroll
      for (int cc = 0; cc < BK / 8; ++cc) {
        uint4 w;
        if (FP8) {  // the value CTA's PV runs on f16
          w.x = pack_f16(x[8 * cc], x[8 * cc + 1]);
          w.y = pack_f16(x[8 * cc + 2], x[8 * cc + 3]);
          w.z = pack_f16(x[8 * cc + 4], x[8 * cc + 5]);
          w.w = pack_f16(x[8 * cc + 6], x[8 * cc + 7]);
        } else {
          w.x = pack_bf16(x[8 * cc], x[8 * cc + 1]);
          w.y = pack_bf16(x[8 * cc + 2], x[8 * cc + 3]);
          w.z = pack_bf16(x[8 * cc + 4], x[8 * cc + 5]);
          w.w = pack_bf16(x[8 * cc + 6], x[8 * cc + 7]);
        }
        st_cluster_v4(dst + p_off(row, cc), w);
      }
      const uint32_t fac = dst + kPTile + warp * kFacWarp;
      st_cluster_b32(fac + lane * 4, __float_as_uint(factor));
      const int any = __any_sync(0xffffffffu, need) ? 1 : 0;
      if (lane == 0) st_cluster_b32(fac + 128, static_cast<uint32_t>(any));
      fence_proxy_async_cluster();  // P is read by the value CTA's MMAs
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(peer_pfull + 8u * bb);
    }
    if (!ok && lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
    // final (1/l, lse) of each head to the value CTA
    st_cluster_v2f(map_to_cta(sbase + Smem::kFin, peer) + row * 8, l > 0.f ? 1.f / l : 0.f,
                   l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY);
    __syncwarp();
    if (lane == 0) {
      mbar_arrive_remote(map_to_cta(bar(FIN), peer));
      // every arrival the value CTA sends here has landed before this CTA ends
      if (warp == 0 && ok) {
        for (int bb = 0; bb < 2; ++bb) {
          const int uses = (n_kv - bb + 1) / 2;  // tiles jj < n_kv with jj & 1 == bb
          if (uses > 0 && !mbar_wait_cluster_sleep(bar(P_FREE + bb), (uses - 1) & 1))
            atomicOr(p.err, PKV_EFLAG_TIMEOUT);
        }
      }
    }
  } else {
    // ==================== epilogue + rescale (value CTA) ====================
    const int row = tid;  // head = TMEM lane
    bool ok = true;
    for (int ev = 0;; ++ev) {
      if (!mbar_wait_sleep(bar(CORR_REQ), ev & 1)) {
        ok = false;
        break;
      }
      const int j = sWord[1];
      if (j < 0) break;
      const float f =
          reinterpret_cast<const float *>(smem + Smem::kP + (j & 1) * kPXfer + kPTile +
                                          warp * kFacWarp)[lane];
      if (__any_sync(0xffffffffu, f != 1.f)) {
        // O holds tiles 0..j-1: wait for the last of them, then scale rows
        if (j >= 1 && !(ok = mbar_wait_sleep(bar(O_DONE), (j - 1) & 1))) break;
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < DV / 32; ++ch) {
          float v[32];
          tmem_ld32(tmem + lane_off + ch * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= f;
          tmem_st32(tmem + lane_off + ch * 32, v);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(CORR_DONE));
    }
    if (ok) ok = mbar_wait_cluster_sleep(bar(FIN), 0);
    bool have_o = false;
    if (ok && n_kv > 0) {
      ok = mbar_wait_sleep(bar(O_DONE), (n_kv - 1) & 1);
      have_o = ok;
      if (ok) tc_fence_after();
    }
    if (!ok && lane == 0) atomicOr(p.err, PKV_EFLAG_TIMEOUT);
    const float2 fl = ok ? reinterpret_cast<const float2 *>(smem + Smem::kFin)[row]
                         : make_float2(0.f, -INFINITY);
    // v_descale of the request multiplies the output (and every partial:
    // the merge is linear)
    const float inv = fl.x * ((FP8 && p.v_descale != nullptr) ? p.v_descale[b] : 1.f);
    const float lse_nat = fl.y;
    const int64_t rows_total = static_cast<int64_t>(p.total_q) * p.h_q;
    const int64_t grow = static_cast<int64_t>(t) * p.h_q + row;
    const bool split_mode = p.num_splits > 1;
#pragma unroll 1
    for (int ch = 0; ch < DV / 32; ++ch) {
      float v[32];
      if (have_o) {
        tmem_ld32(tmem + lane_off + ch * 32, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      const int col = ch * 32;
      if (!split_mode) {
        if (covered) {
          bf16 *dst = p.out + static_cast<int64_t>(t) * p.o_st +
                      static_cast<int64_t>(row) * p.o_sh + col;
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
        float *dst = p.ws_o + (static_cast<int64_t>(split) * rows_total + grow) * DV + col;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          __stcg(reinterpret_cast<float4 *>(dst + i),
                 make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv));
      }
    }
    if (!split_mode) {
      if (covered && p.lse != nullptr)
        p.lse[static_cast<int64_t>(t) * p.lse_st + static_cast<int64_t>(row) * p.lse_sh] = lse_nat;
    } else {
      const int ns = p.num_splits;
      __stcg(p.ws_lse + split * rows_total + grow, lse_nat);
      __threadfence();
      asm volatile("bar.sync 1, %0;\n" ::"n"(NSOFT * 32) : "memory");
      if (tid == 0) sWord[0] = (atomicAdd(p.ws_counter + t, 1) == ns - 1);
      asm volatile("bar.sync 1, %0;\n" ::"n"(NSOFT * 32) : "memory");
      if (sWord[0] && covered) {
        __threadfence();  // every split's state is visible from here on
        float Ms = -INFINITY;
        for (int sp = 0; sp < ns; ++sp) Ms = fmaxf(Ms, __ldcg(p.ws_lse + sp * rows_total + grow));
        float wsum = 0.f;
        for (int sp = 0; sp < ns; ++sp)
          wsum += Ms == -INFINITY
                      ? 0.f
                      : exp2f((__ldcg(p.ws_lse + sp * rows_total + grow) - Ms) * kLog2e);
        const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
        bf16 *dst = p.out + static_cast<int64_t>(t) * p.o_st + static_cast<int64_t>(row) * p.o_sh;
#pragma unroll 1
        for (int cc = 0; cc < DV; cc += 8) {
          float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int sp = 0; sp < ns; ++sp) {
            const float ls = __ldcg(p.ws_lse + sp * rows_total + grow);
            const float w = Ms == -INFINITY ? 0.f : exp2f((ls - Ms) * kLog2e);
            const float *src = p.ws_o + (static_cast<int64_t>(sp) * rows_total + grow) * DV + cc;
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
        if (p.lse != nullptr)
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
  cluster_sync();  // no CTA leaves while the other may still address it
}

}  // namespace

int launch_mla_topk(const AttnParams &p, cudaStream_t stream) {
  if (p.total_q == 0) return PKV_OK;
  if (p.topk == nullptr || p.h_q != H || p.h_kv != 1 || p.d != DQK || p.dv != DV)
    return PKV_ERR_UNSUPPORTED;
  if (p.v != p.k || p.v_sp != p.k_sp || p.v_spos != p.k_spos) return PKV_ERR_UNSUPPORTED;
  if (p.q_sh < DQK || p.q_st < p.q_sh * H || p.num_splits > kMlaMaxSplits)
    return PKV_ERR_UNSUPPORTED;
  if (p.total_q > 65535) return PKV_ERR_UNSUPPORTED;
  static std::atomic<bool> configured[64] = {};  // per device; calls may race
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(mla_topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Smem::kDynamic)) != cudaSuccess ||
        cudaFuncSetAttribute(mla_topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Smem::kDynamic)) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  dim3 grid(2 * p.num_splits, 1, p.total_q);
  if (p.kv_fp8)
    mla_topk_kernel<true><<<grid, NTHREADS, Smem::kDynamic, stream>>>(p);
  else
    mla_topk_kernel<false><<<grid, NTHREADS, Smem::kDynamic, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
