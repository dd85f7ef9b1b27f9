// pkv_merge.cu -- log-sum-exp merge of two attention states
// (dual_chunk_flashattention_backend.py `_merge_attn_outputs`; the
// merge_state_v2 call of flashattention_backend.py's cascade decode).
//
// HBM-bound elementwise work: each thread owns 8 consecutive elements of one
// (n, h) row, reads both states with 16-byte (bf16) or 2x16-byte (fp32)
// vector loads and writes the merged row once.  The row's two lse values are
// read by every thread of the row (L1 broadcast).
#include "pkv_internal.h"

namespace pkv {
namespace {

template <typename T>
struct Vec8;
template <>
struct Vec8<bf16> {
  __device__ static void load(const bf16 *p, float (&x)[8]) {
    uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
  __device__ static void store(bf16 *p, const float (&x)[8]) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    *reinterpret_cast<uint4 *>(p) = u;
  }
};
template <>
struct Vec8<float> {
  __device__ static void load(const float *p, float (&x)[8]) {
    float4 a = *reinterpret_cast<const float4 *>(p);
    float4 b = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  __device__ static void store(float *p, const float (&x)[8]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
  }
};

template <typename TI, typename TO>
__global__ void __launch_bounds__(256)
merge_state_kernel(const TI *__restrict__ va, const TI *__restrict__ vb,
                   TO *vo, int64_t n, int h, int d, int64_t va_sn,
                   int64_t va_sh, int64_t vb_sn, int64_t vb_sh, int64_t vo_sn,
                   int64_t vo_sh, const float *__restrict__ la, int64_t la_sn,
                   int64_t la_sh, const float *__restrict__ lb, int64_t lb_sn,
                   int64_t lb_sh, float *lo, int64_t lo_sn, int64_t lo_sh) {
  const int chunks = d >> 3;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rows = n * h;
  if (gid >= rows * chunks) return;
  const int64_t row = gid / chunks;
  const int c = static_cast<int>(gid - row * chunks);
  const int64_t i = row / h;
  const int hh = static_cast<int>(row - i * h);
  const float lse_a = la[i * la_sn + hh * la_sh];
  const float lse_b = lb[i * lb_sn + hh * lb_sh];
  const float m = fmaxf(lse_a, lse_b);
  float wa, wb, lse;
  if (m == -INFINITY) {  // both states empty
    wa = 0.f; wb = 0.f; lse = -INFINITY;
  } else {
    const float ea = exp2f((lse_a - m) * kLog2e);
    const float eb = exp2f((lse_b - m) * kLog2e);
    const float s = ea + eb;
    wa = ea / s;
    wb = eb / s;
    lse = m + log2f(s) * kLn2;
  }
  float xa[8], xb[8], y[8];
  Vec8<TI>::load(va + i * va_sn + hh * va_sh + c * 8, xa);
  Vec8<TI>::load(vb + i * vb_sn + hh * vb_sh + c * 8, xb);
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = wa * xa[e] + wb * xb[e];
  Vec8<TO>::store(vo + i * vo_sn + hh * vo_sh + c * 8, y);
  if (lo != nullptr && c == 0) lo[i * lo_sn + hh * lo_sh] = lse;
}

template <typename TI, typename TO>
int launch_typed(const void *va, const void *vb, void *vo, int64_t n, int h,
                 int d, int64_t va_sn, int64_t va_sh, int64_t vb_sn,
                 int64_t vb_sh, int64_t vo_sn, int64_t vo_sh, const float *la,
                 int64_t la_sn, int64_t la_sh, const float *lb, int64_t lb_sn,
                 int64_t lb_sh, float *lo, int64_t lo_sn, int64_t lo_sh,
                 cudaStream_t stream) {
  const int64_t total = n * h * (d / 8);
  if (total == 0) return PKV_OK;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  merge_state_kernel<TI, TO><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const TI *>(va), static_cast<const TI *>(vb),
      static_cast<TO *>(vo), n, h, d, va_sn, va_sh, vb_sn, vb_sh, vo_sn, vo_sh,
      la, la_sn, la_sh, lb, lb_sn, lb_sh, lo, lo_sn, lo_sh);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

int launch_merge_state(const void *va, const void *vb, void *vo, int v_dtype,
                       int o_dtype, int64_t n, int h, int d, int64_t va_sn,
                       int64_t va_sh, int64_t vb_sn, int64_t vb_sh,
                       int64_t vo_sn, int64_t vo_sh, const float *la,
                       int64_t la_sn, int64_t la_sh, const float *lb,
                       int64_t lb_sn, int64_t lb_sh, float *lo, int64_t lo_sn,
                       int64_t lo_sh, cudaStream_t stream) {
#define PKV_MERGE_ARGS                                                      \
  va, vb, vo, n, h, d, va_sn, va_sh, vb_sn, vb_sh, vo_sn, vo_sh, la, la_sn, \
      la_sh, lb, lb_sn, lb_sh, lo, lo_sn, lo_sh, stream
  if (v_dtype == PKV_BF16 && o_dtype == PKV_BF16) return launch_typed<bf16, bf16>(PKV_MERGE_ARGS);
  if (v_dtype == PKV_BF16 && o_dtype == PKV_F32) return launch_typed<bf16, float>(PKV_MERGE_ARGS);
  if (v_dtype == PKV_F32 && o_dtype == PKV_BF16) return launch_typed<float, bf16>(PKV_MERGE_ARGS);
  if (v_dtype == PKV_F32 && o_dtype == PKV_F32) return launch_typed<float, float>(PKV_MERGE_ARGS);
#undef PKV_MERGE_ARGS
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
