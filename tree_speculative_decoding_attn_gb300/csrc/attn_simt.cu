// Tree attention on CUDA cores (float32 math): the general path for f32
// inputs, head_dim 64 and shapes the tensor-core kernel does not take, and
// the split-KV combine shared by both kernels.
//
// "5.3 Medusa、EAGLE 与 MTP" (infra-guide), sections 3.1 and 8: node i attends
// to the shared prefix and to its ancestors-or-self; "Medusa, explained",
// step 6: every node is scored in one pass.
//
// Work split: one CTA per (16 query rows, KV split, sequence x KV head).
// Query row r of a (sequence, KV head) is node r / G, query head
// kvh * G + r % G, so every K/V tile staged in shared memory serves all G
// heads of the group and all tree nodes of the CTA.  The prefix keys of the
// sequence are cut into `splits` chunks; the last split also takes the
// tree keys, whose visibility comes from the node's ancestor bitmask.
// Online softmax in base 2 (scores pre-multiplied by log2 e).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;
constexpr int kKeyTile = 32;
constexpr int kSms = 152;

// Stage `nrows` rows of [.., D] starting at `src` (row stride D) into
// shared memory as float32; rows past nrows are zero.
template <typename T, int D, int LD>
__device__ __forceinline__ void stage_rows(float *dst, const T *src, int nrows) {
  constexpr int kVec = 16 / sizeof(T);
  constexpr int kVecPerRow = D / kVec;
  for (int e = threadIdx.x; e < kKeyTile * kVecPerRow; e += kWarps * 32) {
    const int r = e / kVecPerRow, c = (e % kVecPerRow) * kVec;
    float f[kVec];
    if (r < nrows) {
      const uint4 u = *reinterpret_cast<const uint4 *>(src + (int64_t)r * D + c);
      if constexpr (sizeof(T) == 2) {
        sv::bf16x8_to_f32(u, f);
      } else {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kVec; ++j) f[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < kVec; ++j) dst[r * LD + c + j] = f[j];
  }
}

template <typename T, int D, int MW>
__global__ void __launch_bounds__(kWarps * 32)
    attn_simt_kernel(const T *__restrict__ q, const T *__restrict__ kc, const T *__restrict__ vc,
                     const T *__restrict__ kt, const T *__restrict__ vt,
                     const int32_t *__restrict__ prefix_len, const uint64_t *__restrict__ anc,
                     T *__restrict__ out, int N, int Hq, int Hkv, int s_max, int max_prefix,
                     int splits, int chunk, float scale_log2, float *ws, int32_t *status, const sv::KvPages pg) {
  constexpr int DL = D / 32;  // output dims per lane
  __shared__ float sK[kKeyTile * (D + 1)];
  __shared__ float sV[kKeyTile * D];
  __shared__ float sQ[kRowsPerCta * D];

  const int G = Hq / Hkv;
  const int R = N * G;
  const int rg = blockIdx.x, split = blockIdx.y, bh = blockIdx.z;
  const int b = bh / Hkv, kvh = bh % Hkv;
  const int P = prefix_len[b];
  if (P < 0 || P > max_prefix || P > s_max) {
    if (threadIdx.x == 0) sv::report(status, SPEC_DEV_CAPACITY);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int e = threadIdx.x; e < kRowsPerCta * D; e += kWarps * 32) {
    const int rr = e / D, d = e % D, r = rg * kRowsPerCta + rr;
    float v = 0.f;
    if (r < R) v = sv::to_f32(q[(((int64_t)b * N + r / G) * Hq + kvh * G + r % G) * D + d]);
    sQ[e] = v;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DL];
  // the row's ancestor mask: MW words of 64 nodes (ceil(N / 64) stored per node)
  const int nw = (N + 63) >> 6;
  uint64_t am[kRowsPerWarp][MW];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int r = rg * kRowsPerCta + warp * kRowsPerWarp + k;
#pragma unroll
    for (int w = 0; w < MW; ++w) am[k][w] = r < R && w < nw ? anc[((int64_t)b * N + r / G) * nw + w] : 0ull;
    m[k] = -INFINITY;
    l[k] = 0.f;
#pragma unroll
    for (int dd = 0; dd < DL; ++dd) acc[k][dd] = 0.f;
  }

  const int k0 = split * chunk;
  const int k1 = min(P, k0 + chunk);
  const bool with_tree = split == splits - 1;
  const int n_prefix_tiles = k1 > k0 ? (k1 - k0 + kKeyTile - 1) / kKeyTile : 0;
  const int n_tree_tiles = with_tree ? (N + kKeyTile - 1) / kKeyTile : 0;
  const int64_t kv_base = ((int64_t)b * Hkv + kvh) * s_max * D;
  const int64_t kt_base = ((int64_t)b * Hkv + kvh) * N * D;

  for (int tile = 0; tile < n_prefix_tiles + n_tree_tiles; ++tile) {
    const bool tree = tile >= n_prefix_tiles;
    const int t0 = tree ? (tile - n_prefix_tiles) * kKeyTile : k0 + tile * kKeyTile;
    const int nvalid = tree ? min(kKeyTile, N - t0) : min(kKeyTile, k1 - t0);
    __syncthreads();  // previous tile fully consumed (and sQ written on entry)
    if (tree) {
      stage_rows<T, D, D + 1>(sK, kt + kt_base + (int64_t)t0 * D, nvalid);
      stage_rows<T, D, D>(sV, vt + kt_base + (int64_t)t0 * D, nvalid);
    } else {
      // a 32-key tile lies inside one cache block (block sizes are multiples of 32)
      const int row = pg.table ? sv::kv_row(pg, b, Hkv, kvh, s_max, t0, status) : 0;
      const T *ks = pg.table ? kc + (int64_t)(row < 0 ? 0 : row) * D : kc + kv_base + (int64_t)t0 * D;
      const T *vs = pg.table ? vc + (int64_t)(row < 0 ? 0 : row) * D : vc + kv_base + (int64_t)t0 * D;
      stage_rows<T, D, D + 1>(sK, ks, row < 0 ? 0 : nvalid);
      stage_rows<T, D, D>(sV, vs, row < 0 ? 0 : nvalid);
    }
    __syncthreads();
    // The warp's rows go through each step together, so their dot products,
    // reductions and P.V updates are independent chains, and every staged
    // K/V value is read once for all of them.
    constexpr int RW = kRowsPerWarp;
    const float *kr = sK + lane * (D + 1);
    const float *qw = sQ + warp * RW * D;
    float sc[RW];
#pragma unroll
    for (int k = 0; k < RW; ++k) sc[k] = 0.f;
#pragma unroll 8
    for (int d = 0; d < D; ++d) {
      const float kd = kr[d];
#pragma unroll
      for (int k = 0; k < RW; ++k) sc[k] = fmaf(qw[k * D + d], kd, sc[k]);
    }
    float mx[RW], p[RW];
    // a 32-key tree tile lies inside one mask word (t0 is a multiple of 32)
#pragma unroll
    for (int k = 0; k < RW; ++k) {
      uint64_t word = am[k][0];
#pragma unroll
      for (int w = 1; w < MW; ++w)
        if ((t0 >> 6) == w) word = am[k][w];
      const bool vis = lane < nvalid && (!tree || ((word >> ((t0 & 63) + lane)) & 1ull));
      sc[k] = vis ? sc[k] * scale_log2 : -INFINITY;
      mx[k] = sc[k];
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
#pragma unroll
      for (int k = 0; k < RW; ++k) mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], o));
#pragma unroll
    for (int k = 0; k < RW; ++k) {
      const float mn = fmaxf(m[k], mx[k]);
      const bool live = mn != -INFINITY;  // something visible so far
      p[k] = live && sc[k] != -INFINITY ? exp2f(sc[k] - mn) : 0.f;
      const float corr = live ? exp2f(m[k] - mn) : 1.f;  // 0 when m was -inf
      mx[k] = p[k];                                      // reused for the row sum
      l[k] *= corr;
#pragma unroll
      for (int dd = 0; dd < DL; ++dd) acc[k][dd] *= corr;
      m[k] = mn;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
#pragma unroll
      for (int k = 0; k < RW; ++k) mx[k] += __shfl_xor_sync(0xffffffffu, mx[k], o);
#pragma unroll
    for (int k = 0; k < RW; ++k) l[k] += mx[k];
    for (int j = 0; j < nvalid; ++j) {
      float v[DL];
#pragma unroll
      for (int dd = 0; dd < DL; ++dd) v[dd] = sV[j * D + lane + 32 * dd];
#pragma unroll
      for (int k = 0; k < RW; ++k) {
        const float pj = __shfl_sync(0xffffffffu, p[k], j);
#pragma unroll
        for (int dd = 0; dd < DL; ++dd) acc[k][dd] = fmaf(pj, v[dd], acc[k][dd]);
      }
    }
  }

#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int r = rg * kRowsPerCta + warp * kRowsPerWarp + k;
    if (r >= R) continue;
    if (splits == 1) {
      const float inv = l[k] > 0.f ? 1.f / l[k] : 0.f;
      T *o = out + (((int64_t)b * N + r / G) * Hq + kvh * G + r % G) * D;
#pragma unroll
      for (int dd = 0; dd < DL; ++dd) o[lane + 32 * dd] = sv::from_f32<T>(acc[k][dd] * inv);
    } else {
      const int64_t slot = (((int64_t)b * Hkv + kvh) * splits + split) * R + r;
      float *wa = ws + slot * sv_partial_stride(D);
#pragma unroll
      for (int dd = 0; dd < DL; ++dd) wa[lane + 32 * dd] = acc[k][dd];
      if (lane == 0) {
        wa[D] = m[k];
        wa[D + 1] = l[k];
      }
    }
  }
}

// Merge split partials (m_s, l_s, acc_s) of one query row:
// out = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s.
template <typename T, int D>
__global__ void __launch_bounds__(128)
    attn_combine_kernel(const float *__restrict__ ws, T *__restrict__ out,
                        const int32_t *__restrict__ prefix_len, int N, int Hq, int Hkv, int splits,
                        int s_max, int max_prefix) {
  constexpr int DL = D / 32;
  const int G = Hq / Hkv, R = N * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 4 + warp, bh = blockIdx.y;
  if (r >= R) return;
  const int b = bh / Hkv, kvh = bh % Hkv;
  const int P = prefix_len[b];
  if (P < 0 || P > max_prefix || P > s_max) return;  // reported by the main kernel
  const float *w0 = ws + ((int64_t)bh * splits * R + r) * sv_partial_stride(D);
  const int64_t sstride = (int64_t)R * sv_partial_stride(D);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, w0[s * sstride + D]);
  float L = 0.f, acc[DL];
#pragma unroll
  for (int dd = 0; dd < DL; ++dd) acc[dd] = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float *w = w0 + s * sstride;
    const float ms = w[D];
    if (ms == -INFINITY) continue;
    const float f = exp2f(ms - M);
    L = fmaf(f, w[D + 1], L);
#pragma unroll
    for (int dd = 0; dd < DL; ++dd) acc[dd] = fmaf(f, w[lane + 32 * dd], acc[dd]);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  T *o = out + (((int64_t)b * N + r / G) * Hq + kvh * G + r % G) * D;
#pragma unroll
  for (int dd = 0; dd < DL; ++dd) o[lane + 32 * dd] = sv::from_f32<T>(acc[dd] * inv);
}

template <typename T, int D>
int launch_simt(const SvAttnShape &s, const SvAttnPlan &p, const void *q, const void *kc,
                const void *vc, const void *kt, const void *vt, const int32_t *prefix_len,
                const uint64_t *anc, void *out, float scale, void *ws, int32_t *status,
                cudaStream_t stream) {
  const int R = s.n_nodes * (s.hq / s.hkv);
  dim3 grid((R + kRowsPerCta - 1) / kRowsPerCta, p.splits, s.batch * s.hkv);
  auto kern = s.n_nodes <= 64 ? attn_simt_kernel<T, D, 1> : attn_simt_kernel<T, D, 4>;
  kern<<<grid, kWarps * 32, 0, stream>>>((const T *)q, (const T *)kc, (const T *)vc, (const T *)kt, (const T *)vt,
                                         prefix_len, anc, (T *)out, s.n_nodes, s.hq, s.hkv, s.s_max, s.max_prefix,
                                         p.splits, p.chunk, scale * 1.4426950408889634f, (float *)ws, status,
                                         sv::KvPages{s.block_table, s.block_size, s.max_blocks, s.num_blocks});
  return sv_launch_status();
}

template <typename T, int D>
int launch_combine(const SvAttnShape &s, const SvAttnPlan &p, const void *ws, void *out,
                   const int32_t *prefix_len, cudaStream_t stream) {
  const int R = s.n_nodes * (s.hq / s.hkv);
  dim3 grid((R + 3) / 4, s.batch * s.hkv);
  attn_combine_kernel<T, D><<<grid, 128, 0, stream>>>((const float *)ws, (T *)out, prefix_len,
                                                      s.n_nodes, s.hq, s.hkv, p.splits, s.s_max,
                                                      s.max_prefix);
  return sv_launch_status();
}

}  // namespace

SvAttnPlan sv_attn_simt_plan(const SvAttnShape &s, int num_splits) {
  SvAttnPlan p{};
  p.use_tc = 0;
  const int R = s.n_nodes * (s.hq / s.hkv);
  const int base = ((R + kRowsPerCta - 1) / kRowsPerCta) * s.batch * s.hkv;
  const int max_useful = s.max_prefix > 0 ? (s.max_prefix + kKeyTile - 1) / kKeyTile : 1;
  int splits = num_splits > 0 ? num_splits : (2 * kSms + base - 1) / base;
  splits = splits < 1 ? 1 : (splits > max_useful ? max_useful : splits);
  if (splits > 64) splits = 64;
  int chunk = s.max_prefix > 0 ? (s.max_prefix + splits - 1) / splits : 0;
  chunk = (chunk + kKeyTile - 1) / kKeyTile * kKeyTile;
  p.splits = splits;
  p.chunk = chunk;
  p.ws_bytes = splits > 1 ? (size_t)s.batch * s.hkv * splits * R * sv_partial_stride(s.head_dim) * sizeof(float) : 0;
  return p;
}

int sv_attn_simt(const SvAttnShape &s, const SvAttnPlan &p, const void *q, const void *kc,
                 const void *vc, const void *kt, const void *vt, const int32_t *prefix_len,
                 const uint64_t *anc, void *out, float scale, void *ws, int32_t *status,
                 cudaStream_t stream) {
  if (s.dtype == SPEC_BF16) {
    return s.head_dim == 128 ? launch_simt<__nv_bfloat16, 128>(s, p, q, kc, vc, kt, vt, prefix_len, anc, out, scale, ws, status, stream)
                             : launch_simt<__nv_bfloat16, 64>(s, p, q, kc, vc, kt, vt, prefix_len, anc, out, scale, ws, status, stream);
  }
  return s.head_dim == 128 ? launch_simt<float, 128>(s, p, q, kc, vc, kt, vt, prefix_len, anc, out, scale, ws, status, stream)
                           : launch_simt<float, 64>(s, p, q, kc, vc, kt, vt, prefix_len, anc, out, scale, ws, status, stream);
}

int sv_attn_combine(const SvAttnShape &s, const SvAttnPlan &p, const void *ws, void *out,
                    const int32_t *prefix_len, cudaStream_t stream) {
  if (s.dtype == SPEC_BF16) {
    return s.head_dim == 128 ? launch_combine<__nv_bfloat16, 128>(s, p, ws, out, prefix_len, stream)
                             : launch_combine<__nv_bfloat16, 64>(s, p, ws, out, prefix_len, stream);
  }
  return s.head_dim == 128 ? launch_combine<float, 128>(s, p, ws, out, prefix_len, stream)
                           : launch_combine<float, 64>(s, p, ws, out, prefix_len, stream);
}
