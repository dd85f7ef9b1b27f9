// pkv_decode.cu -- paged attention for decode and short query runs (GQA).
//
// Computes, for the query rows of one (request, KV head, row tile) and one
// contiguous chunk of that request's keys, the state (O, lse) of
// flashattention_backend.py's `flash_attn_with_kvcache` call, and combines
// the chunks of a split request with the log-sum-exp state merge
// (dual_chunk_flashattention_backend.py, `_merge_attn_outputs`).
//
// Design (HBM-bound: every K/V byte is read once per KV head):
//  * One CTA = 4 warps = one tile of 16 query rows.  The rows are the
//    (new token, q head) pairs that share one KV head, so all GQA heads of a
//    KV head are served by a single read of its K/V rows.
//  * Keys stream through a NSTAGE-deep cp.async pipeline of 64-key stages.
//    Each key row (D * 2 bytes, contiguous) is gathered through the page
//    table with 16-byte cp.async into XOR-swizzled shared memory (16-byte
//    chunk index ^= row & 7), so ldmatrix reads are bank-conflict free.
//  * Warp w owns keys [16w, 16w + 16) of every stage: S = Q K^T and O += P V
//    on bf16 mma.sync m16n8k16 tensor-core tiles with fp32 accumulation and a
//    per-warp online softmax in the log2 domain.  The four warps' states are
//    merged through shared memory at the end.
//  * Split-KV: the CTA for chunk s writes its normalised partial (O_s, lse_s)
//    to the workspace; the last CTA of the (request, KV head, tile) to finish
//    (atomic ticket, no waiting) merges all partials and writes the output.
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int BK = 64;       // keys per pipeline stage
constexpr int NWARP = 4;
constexpr int NTHREAD = NWARP * 32;
constexpr int ROWS = kDecodeRowTile;  // 16

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src,
                                           int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
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

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// byte offset of 16-byte chunk c of row r in a swizzled [rows][D] bf16 tile
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((r * D + ((c ^ (r & 7)) << 3)) * 2);
}

struct RowInfo {
  int tok;    // query token index, -1 if the row is padding
  int head;   // q head
  int pos;    // absolute position i of the token
};

// Row r (0..15) of tile `tile` of request b / KV head kvh.
__device__ __forceinline__ RowInfo row_info(const AttnParams &p, int b,
                                            int kvh, int tile, int r,
                                            int q_len, int kv_len,
                                            int q_begin) {
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

template <int D, int NSTAGE>
__global__ void __launch_bounds__(NTHREAD, 2)
decode_gqa_kernel(const AttnParams p) {
  constexpr int CPR = D / 8;             // 16-byte chunks per row
  constexpr int RPP = NTHREAD / CPR;     // rows per producer pass
  constexpr int PASSES = BK / RPP;
  constexpr int KT = D / 16;             // k-steps of QK^T
  constexpr int NT = D / 8;              // n-tiles of PV
  constexpr uint32_t STAGE_BYTES = BK * D * 2;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *sQ = smem;                                   // [16][D] bf16
  uint8_t *sK = sQ + ROWS * D * 2;                      // [NSTAGE][BK][D]
  uint8_t *sV = sK + NSTAGE * STAGE_BYTES;              // [NSTAGE][BK][D]
  int *sPos = reinterpret_cast<int *>(sV + NSTAGE * STAGE_BYTES);  // [NSTAGE][BK]
  float *sM = reinterpret_cast<float *>(sPos + NSTAGE * BK);       // [NWARP][16]
  float *sL = sM + NWARP * ROWS;                                   // [NWARP][16]
  int *sFlag = reinterpret_cast<int *>(sL + NWARP * ROWS);

  const int split = blockIdx.x;
  const int kvh = blockIdx.y / p.n_row_tiles;
  const int tile = blockIdx.y % p.n_row_tiles;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int q_begin = p.cu_seqlens_q[b];
  const int q_len = p.cu_seqlens_q[b + 1] - q_begin;
  const int kv_len = p.cache_seqlens[b];

  // ---- rows of this tile; CTAs past the request's rows have no work ----
  int n_valid_rows = 0, u_min = 0x7fffffff, u_max = -1;
  {
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
  }
  if (n_valid_rows == 0) return;  // uniform over the CTA

  // ---- key range of this tile, then this split's chunk of it ----
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
  int k0, k1;
  {
    const int len = hi - lo;
    int chunk = (len + p.num_splits - 1) / p.num_splits;
    chunk = (chunk + BK - 1) / BK * BK;
    k0 = min(hi, lo + split * chunk);
    k1 = min(hi, k0 + chunk);
  }
  const int n_kt = (k1 - k0 + BK - 1) / BK;

  // ---- stage Q rows into shared memory (zero rows for padding) ----
  for (int e = tid; e < ROWS * CPR; e += NTHREAD) {
    const int r = e / CPR, c = e % CPR;
    const RowInfo ri = row_info(p, b, kvh, tile, r, q_len, kv_len, q_begin);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (ri.tok >= 0)
      val = *reinterpret_cast<const uint4 *>(
          p.q + static_cast<int64_t>(ri.tok) * p.q_st +
          static_cast<int64_t>(ri.head) * p.q_sh + c * 8);
    *reinterpret_cast<uint4 *>(sQ + swz<D>(r, c)) = val;
  }

  // ---- producer: gather one 64-key stage of K and V rows ----
  const int prow = tid / CPR;   // row within a pass
  const int pchunk = tid % CPR;
  const int topk_tok = q_begin + u_min;  // top-k mode: one token per tile
  auto issue_stage = [&](int kt) {
    const int st = kt % NSTAGE;
    const int base = k0 + kt * BK;
    const uint32_t kdst0 = smem_addr(sK + st * STAGE_BYTES);
    const uint32_t vdst0 = smem_addr(sV + st * STAGE_BYTES);
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int r = ps * RPP + prow;
      const int j = base + r;
      int pos = -1;
      const bf16 *ksrc = p.k;
      const bf16 *vsrc = p.v;
      if (j < k1) {
        pos = j;
        bool ok = true;
        if (p.topk != nullptr) {
          pos = p.topk[static_cast<int64_t>(topk_tok) * p.topk_stride + j];
          if (pos < 0 || pos >= kv_len) {
            if (pos != -1 && pchunk == 0) atomicOr(p.err, PKV_EFLAG_TOPK_OOB);
            ok = false;
          }
        }
        if (ok) {
          const int pidx = pos / p.page_size;
          if (pidx >= p.pt_cols) {
            if (pchunk == 0) atomicOr(p.err, PKV_EFLAG_ROW_TOO_SHORT);
            ok = false;
          } else {
            const int64_t page = p.page_table[static_cast<int64_t>(b) * p.pt_stride + pidx];
            if (page < 0 || page >= p.num_pages) {
              if (pchunk == 0) atomicOr(p.err, PKV_EFLAG_PAGE_OOB);
              ok = false;
            } else {
              const int inpage = pos - pidx * p.page_size;
              ksrc = p.k + page * p.k_sp + inpage * p.k_spos + kvh * p.k_sh + pchunk * 8;
              vsrc = p.v + page * p.v_sp + inpage * p.v_spos + kvh * p.v_sh + pchunk * 8;
            }
          }
        }
        if (!ok) pos = -1;
      }
      const int bytes = pos >= 0 ? 16 : 0;
      cp_async16(kdst0 + swz<D>(r, pchunk), ksrc, bytes);
      cp_async16(vdst0 + swz<D>(r, pchunk), vsrc, bytes);
      if (pchunk == 0) sPos[st * BK + r] = pos;
    }
  };

#pragma unroll
  for (int s = 0; s < NSTAGE - 1; ++s) {
    if (s < n_kt) issue_stage(s);
    cp_async_commit();
  }
  __syncthreads();  // Q tile visible

  // ---- Q fragments (A operand, 16 x D) ----
  uint32_t qf[KT][4];
  {
    const uint32_t qbase = smem_addr(sQ);
    const int m = lane >> 3;
    const int r = (m & 1) * 8 + (lane & 7);
#pragma unroll
    for (int kk = 0; kk < KT; ++kk)
      ldsm_x4(qbase + swz<D>(r, 2 * kk + (m >> 1)), qf[kk][0], qf[kk][1],
              qf[kk][2], qf[kk][3]);
  }

  // positions of this thread's two rows (g and g + 8)
  const int g = lane >> 2;
  const int tq = lane & 3;
  int rpos[2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    rpos[h] = row_info(p, b, kvh, tile, g + 8 * h, q_len, kv_len, q_begin).pos;
  const bool use_upper = p.causal || p.window_left >= 0;

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  // ---- main loop ----
  for (int kt = 0; kt < n_kt; ++kt) {
    cp_async_wait<NSTAGE - 2>();
    __syncthreads();
    if (kt + NSTAGE - 1 < n_kt) issue_stage(kt + NSTAGE - 1);
    cp_async_commit();

    const int st = kt % NSTAGE;
    const uint32_t kbase = smem_addr(sK + st * STAGE_BYTES);
    const uint32_t vbase = smem_addr(sV + st * STAGE_BYTES);
    const int key0 = warp * 16;

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
        ldsm_x4(kbase + swz<D>(kr, 2 * kk + kc), b0, b1, b2, b3);
        mma_bf16(s[0], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
        mma_bf16(s[1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
      }
    }

    // masks, scale to log2 domain
    int kpos[2][2];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      kpos[n][0] = sPos[st * BK + key0 + n * 8 + 2 * tq];
      kpos[n][1] = sPos[st * BK + key0 + n * 8 + 2 * tq + 1];
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
      float mx = fmaxf(fmaxf(s[0][2 * h], s[0][2 * h + 1]),
                       fmaxf(s[1][2 * h], s[1][2 * h + 1]));
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
        ldsm_x4_t(vbase + swz<D>(vr, 2 * cc + vc), b0, b1, b2, b3);
        mma_bf16(o[2 * cc], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[2 * cc + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // pipeline buffers free for the epilogue

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
  __syncthreads();
  constexpr int OSTRIDE = D + 4;  // padded fp32 row
  float *sO = reinterpret_cast<float *>(sK);  // [NWARP][16][D + 4]
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = g + 8 * h;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) M = fmaxf(M, sM[w * ROWS + r]);
    const float f = M == -INFINITY ? 0.f : exp2f(m_run[h] - M);
    float *dst = sO + (warp * ROWS + r) * OSTRIDE;
#pragma unroll
    for (int n = 0; n < NT; ++n)
      *reinterpret_cast<float2 *>(dst + n * 8 + 2 * tq) =
          make_float2(o[n][2 * h] * f, o[n][2 * h + 1] * f);
  }
  __syncthreads();

  // each thread: one row, D/8 consecutive columns
  constexpr int CPT = D / 8;  // columns per thread
  const int fr = tid >> 3;
  const int fc = (tid & 7) * CPT;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) M = fmaxf(M, sM[w * ROWS + fr]);
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    const float mw = sM[w * ROWS + fr];
    L += (M == -INFINITY) ? 0.f : sL[w * ROWS + fr] * exp2f(mw - M);
  }
  float acc[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) acc[c] = 0.f;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    const float *src = sO + (w * ROWS + fr) * OSTRIDE + fc;
#pragma unroll
    for (int c = 0; c < CPT; c += 4) {
      const float4 v4 = *reinterpret_cast<const float4 *>(src + c);
      acc[c] += v4.x; acc[c + 1] += v4.y; acc[c + 2] += v4.z; acc[c + 3] += v4.w;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const float lse_nat = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  const RowInfo fri = row_info(p, b, kvh, tile, fr, q_len, kv_len, q_begin);

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
  __syncthreads();
  if (tid == 0) {
    int32_t *ctr = p.ws_counter +
                   (static_cast<int64_t>(b) * p.h_kv + kvh) * p.n_row_tiles + tile;
    const int ticket = atomicAdd(ctr, 1);
    *sFlag = (ticket == p.num_splits - 1);
  }
  __syncthreads();
  if (!*sFlag) return;
  __threadfence();  // every other chunk's state is visible from here on

  // ---- last CTA: merge all chunks (the state merge of merge_state) ----
  if (fri.tok < 0) return;
  const int64_t row = static_cast<int64_t>(fri.tok) * p.h_q + fri.head;
  float Ms = -INFINITY;
  for (int sp = 0; sp < p.num_splits; ++sp)
    Ms = fmaxf(Ms, __ldcg(p.ws_lse + sp * rows_total + row));
  float out[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) out[c] = 0.f;
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
        out[c] += w * v4.x; out[c + 1] += w * v4.y;
        out[c + 2] += w * v4.z; out[c + 3] += w * v4.w;
      }
    }
  }
  const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
  bf16 *dst = p.out + static_cast<int64_t>(fri.tok) * p.o_st +
              static_cast<int64_t>(fri.head) * p.o_sh + fc;
#pragma unroll
  for (int c = 0; c < CPT; c += 8) {
    uint4 u;
    u.x = pack_bf16(out[c] * winv, out[c + 1] * winv);
    u.y = pack_bf16(out[c + 2] * winv, out[c + 3] * winv);
    u.z = pack_bf16(out[c + 4] * winv, out[c + 5] * winv);
    u.w = pack_bf16(out[c + 6] * winv, out[c + 7] * winv);
    *reinterpret_cast<uint4 *>(dst + c) = u;
  }
  if (p.lse != nullptr && (tid & 7) == 0)
    p.lse[static_cast<int64_t>(fri.tok) * p.lse_st + fri.head * p.lse_sh] =
        wsum > 0.f ? Ms + logf(wsum) : -INFINITY;
}

template <int D, int NSTAGE>
constexpr size_t decode_smem_bytes() {
  return ROWS * D * 2 + 2 * NSTAGE * BK * D * 2 + NSTAGE * BK * 4 +
         2 * NWARP * ROWS * 4 + 16;
}

template <int D, int NSTAGE>
int launch_typed(const AttnParams &p, cudaStream_t stream) {
  constexpr size_t smem = decode_smem_bytes<D, NSTAGE>();
  static_assert(NWARP * ROWS * (D + 4) * 4 <= 2 * NSTAGE * BK * D * 2,
                "epilogue buffer must fit in the pipeline buffers");
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 64 && !configured[dev]) {
    if (cudaFuncSetAttribute(decode_gqa_kernel<D, NSTAGE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return PKV_ERR_CUDA;
    configured[dev] = true;
  }
  dim3 grid(p.num_splits, p.h_kv * p.n_row_tiles, p.batch);
  decode_gqa_kernel<D, NSTAGE><<<grid, NTHREAD, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

int launch_decode_gqa(const AttnParams &p, cudaStream_t stream) {
  if (p.batch == 0 || p.n_row_tiles == 0) return PKV_OK;
  if (p.h_kv * p.n_row_tiles > 65535 || p.batch > 65535 || p.num_splits > 65535)
    return PKV_ERR_UNSUPPORTED;
  if (p.d == 128 && p.dv == 128) return launch_typed<128, 3>(p, stream);
  if (p.d == 64 && p.dv == 64) return launch_typed<64, 4>(p, stream);
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
