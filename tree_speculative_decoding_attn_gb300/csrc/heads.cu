// Medusa residual heads.
//
// "Medusa, explained", procedure step 1: head k computes
// W2_k (SiLU(W1_k h) + h); "Medusa and EAGLE ... explained", section
// "Implementation sketch": the first linear layer may carry a bias.
//
// At the heads' batch (one hidden state per sequence) both projections are
// matrix-vector products that stream their weights once: 2 flops per 2-byte
// weight, far below any tensor-core ridge, so they run on CUDA cores with
// one warp per weight row, 16-byte streaming loads kept eight deep per lane,
// and a warp-shuffle reduction.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kGemvWarps = 8;
constexpr int kDepth = 8;  // 16-byte weight loads in flight per lane
constexpr int kSms = 152;

enum Epilogue { kPlain = 0, kSiluResidual = 1 };

template <typename TX>
__device__ __forceinline__ void load_x8(const TX *x, float *f);
template <>
__device__ __forceinline__ void load_x8<__nv_bfloat16>(const __nv_bfloat16 *x, float *f) {
  sv::bf16x8_to_f32(*reinterpret_cast<const uint4 *>(x), f);
}
template <>
__device__ __forceinline__ void load_x8<float>(const float *x, float *f) {
  const float4 a = *reinterpret_cast<const float4 *>(x), b = *reinterpret_cast<const float4 *>(x + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// y[b, head k, o] for all weight rows.  W is [n_heads * rows_per_head, d]
// (bf16); x for head k and batch b is x + k * x_head_stride + b *
// x_batch_stride; y index b * y_batch_stride + k * rows_per_head + o.
template <typename TX, int B, int EPI>
__global__ void __launch_bounds__(kGemvWarps * 32)
    gemv_rows_kernel(const __nv_bfloat16 *__restrict__ W, const TX *__restrict__ x,
                     int64_t x_head_stride, int64_t x_batch_stride, int total_rows,
                     int rows_per_head, int d, float *__restrict__ y, int64_t y_batch_stride,
                     const __nv_bfloat16 *__restrict__ bias, const __nv_bfloat16 *__restrict__ resid,
                     int64_t resid_batch_stride) {
  const int lane = threadIdx.x & 31;
  const int warp_global = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
  const int n_warps = gridDim.x * kGemvWarps;
  const int n_vec = d / 8;
  for (int row = warp_global; row < total_rows; row += n_warps) {
    const int k = row / rows_per_head, o = row % rows_per_head;
    const __nv_bfloat16 *w = W + (int64_t)row * d;
    const TX *xk = x + (int64_t)k * x_head_stride;
    float acc[B];
#pragma unroll
    for (int bb = 0; bb < B; ++bb) acc[bb] = 0.f;
    for (int v0 = lane; v0 < n_vec; v0 += 32 * kDepth) {
      uint4 wv[kDepth];
#pragma unroll
      for (int u = 0; u < kDepth; ++u) {
        const int vi = v0 + u * 32;
        wv[u] = vi < n_vec ? sv::ldg_stream(w + (int64_t)vi * 8) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kDepth; ++u) {
        const int vi = v0 + u * 32;
        if (vi >= n_vec) break;
        float wf[8];
        sv::bf16x8_to_f32(wv[u], wf);
#pragma unroll
        for (int bb = 0; bb < B; ++bb) {
          float xf[8];
          load_x8<TX>(xk + bb * x_batch_stride + (int64_t)vi * 8, xf);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[bb] = fmaf(wf[j], xf[j], acc[bb]);
        }
      }
    }
#pragma unroll
    for (int bb = 0; bb < B; ++bb) acc[bb] = sv::warp_sum(acc[bb]);
    if (lane < B) {
      float a = 0.f;
#pragma unroll
      for (int bb = 0; bb < B; ++bb)
        if (bb == lane) a = acc[bb];
      if (EPI == kSiluResidual) {
        if (bias) a += __bfloat162float(bias[row]);
        const float s = a / (1.f + expf(-a));
        a = __bfloat162float(resid[lane * resid_batch_stride + o]) + s;
      }
      y[lane * y_batch_stride + (int64_t)k * rows_per_head + o] = a;
    }
  }
}

template <typename TX, int EPI>
int launch_gemv(int batch, const __nv_bfloat16 *W, const TX *x, int64_t xhs, int64_t xbs,
                int total_rows, int rows_per_head, int d, float *y, int64_t ybs,
                const __nv_bfloat16 *bias, const __nv_bfloat16 *resid, int64_t rbs,
                cudaStream_t stream) {
  int blocks = (total_rows + kGemvWarps - 1) / kGemvWarps;
  if (blocks > kSms * 16) blocks = kSms * 16;
#define SV_GEMV_CASE(BB)                                                                     \
  case BB:                                                                                   \
    gemv_rows_kernel<TX, BB, EPI><<<blocks, kGemvWarps * 32, 0, stream>>>(                   \
        W, x, xhs, xbs, total_rows, rows_per_head, d, y, ybs, bias, resid, rbs);             \
    break;
  switch (batch) {
    SV_GEMV_CASE(1)
    SV_GEMV_CASE(2)
    SV_GEMV_CASE(3)
    SV_GEMV_CASE(4)
    SV_GEMV_CASE(5)
    SV_GEMV_CASE(6)
    SV_GEMV_CASE(7)
    SV_GEMV_CASE(8)
    default:
      return SPEC_ERR_UNSUPPORTED;
  }
#undef SV_GEMV_CASE
  return sv_launch_status();
}

}  // namespace

int sv_medusa_heads(const void *h, const void *w1, const void *b1, const void *w2, int batch,
                    int n_heads, int hidden, int vocab, float *z, float *logits,
                    cudaStream_t stream) {
  // z[b, k, :] = h[b] + SiLU(W1_k h[b] + b1_k)
  int rc = launch_gemv<__nv_bfloat16, kSiluResidual>(
      batch, (const __nv_bfloat16 *)w1, (const __nv_bfloat16 *)h, 0, hidden, n_heads * hidden,
      hidden, hidden, z, (int64_t)n_heads * hidden, (const __nv_bfloat16 *)b1,
      (const __nv_bfloat16 *)h, hidden, stream);
  if (rc != SPEC_OK) return rc;
  // logits[b, k, :] = W2_k z[b, k]
  return launch_gemv<float, kPlain>(batch, (const __nv_bfloat16 *)w2, z, hidden,
                                    (int64_t)n_heads * hidden, n_heads * vocab, vocab, hidden,
                                    logits, (int64_t)n_heads * vocab, nullptr, nullptr, 0, stream);
}
