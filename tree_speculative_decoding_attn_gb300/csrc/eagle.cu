// One EAGLE drafting round on the GPU: the draft layer applied to the
// frontier nodes of a drafted tree, then the confidence-product expansion.
//
// "Medusa and EAGLE: self-speculative decoding heads, explained", section
// "EAGLE: autoregression over features": the draft reads the feature of a
// position together with the embedding of the token after it, reduces the
// 2d-vector to d with a fully connected layer, runs one decoder layer to
// predict the next feature, and reuses the target's LM head to turn features
// into tokens.  "5.3 Medusa、EAGLE 与 MTP", sections 4.1 (FC + one decoder
// layer) and 5.2 (grow the nodes of highest path value).
//
// The decoder layer is a pre-norm block with rotary attention and a SwiGLU
// MLP (the target's architecture).  Per round, for the F frontier nodes of
// each sequence (R = batch * F rows):
//   inputs_kernel     x = [feature(parent) ; embedding(token)]      bf16 [R, 2d]
//   GEMM              h0 = x W_fc^T                                 f32  [R, d]
//   rmsnorm_kernel    n1 = RMSNorm(h0) w_ln1                        bf16
//   GEMM              qkv = n1 W_qkv^T                              f32
//   compact_kernel    the round's draft tree: frontier + ancestors (pool
//                     order, frontier last), parents, pool index map
//   rope_kernel       rotary Q (compact rows) and K, V into the node cache
//   gather_kv_kernel  node K/V rows of the compact tree
//   tree build + tree attention over the draft prefix cache and the tree
//   gather_out_kernel attention rows of the frontier                bf16 [R, Hq D]
//   GEMM + rmsnorm    h1 = h0 + a W_o^T; n2 = RMSNorm(h1) w_ln2
//   GEMM + swiglu     act = SiLU(n2 W_gate^T) * (n2 W_up^T)         bf16 [R, f]
//   GEMM + rmsnorm    f = h1 + act W_down^T (stored as the node's feature);
//                     n3 = RMSNorm(f) w_lnf
//   GEMM              draft logits = n3 W_lm^T                      f32  [R, V]
//   tree expansion    top-k children, path values, next frontier
// Every GEMM is the weight-streaming tensor-core GEMM; the small kernels are
// row-parallel CUDA-core kernels.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxCompact = 64;  // nodes of a round's draft tree (one mask word)
constexpr float kRmsEps = 1e-6f;
constexpr double kRopeBase = 10000.0;

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__device__ __forceinline__ float block_sum(float v, float *red) {
  v = sv::warp_sum(v);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  return t;
}

// The row kernels that feed a GEMM let it launch at once (programmatic
// dependent launch): the GEMM streams its first weights while the row
// kernel runs and reads the row kernel's output only after
// griddepcontrol.wait, which returns once this grid has completed.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// x[r] = [feat[b, parent(v)] ; emb[tok(v)]] for frontier node v = frontier[b, f];
// the root's parent feature is slot pool_cap.
__global__ void __launch_bounds__(kThreads)
    inputs_kernel(const __nv_bfloat16 *__restrict__ feat, const __nv_bfloat16 *__restrict__ emb,
                  const int32_t *__restrict__ pool_parent, const int32_t *__restrict__ pool_tok,
                  const int32_t *__restrict__ frontier, int F, int pool_cap, int d, int V,
                  __nv_bfloat16 *__restrict__ x, int32_t *status) {
  pdl_trigger();
  const int r = blockIdx.x, b = r / F;
  const int v = frontier[r];
  const bool ok = v >= 0 && v < pool_cap;
  const int p = ok ? pool_parent[(int64_t)b * pool_cap + v] : 0;
  const int t = ok ? pool_tok[(int64_t)b * pool_cap + v] : 0;
  if (threadIdx.x == 0 && (!ok || t < 0 || t >= V || p >= pool_cap)) sv::report(status, SPEC_DEV_BAD_POOL);
  const int slot = p < 0 || p >= pool_cap ? pool_cap : p;
  const uint4 *src0 = reinterpret_cast<const uint4 *>(feat + ((int64_t)b * (pool_cap + 1) + slot) * d);
  const uint4 *src1 = reinterpret_cast<const uint4 *>(emb + (int64_t)(t < 0 || t >= V ? 0 : t) * d);
  uint4 *dst = reinterpret_cast<uint4 *>(x + (int64_t)r * 2 * d);
  for (int i = threadIdx.x; i < d / 8; i += kThreads) {
    dst[i] = src0[i];
    dst[d / 8 + i] = src1[i];
  }
}

// y = RMSNorm(x (+ add)) w, bf16; with `add` the sum is also written back to
// x_out (float32, the residual stream) and, optionally, as bf16 to feat_out
// at the frontier node's slot.  d is a multiple of 8 (16-byte rows); the
// row stays in registers between the two passes.
constexpr int kRmsVec = 8;  // float4 per thread: d <= 4 * kRmsVec * kThreads = 8192
__global__ void __launch_bounds__(kThreads)
    rmsnorm_kernel(const float *__restrict__ x, const float *__restrict__ add, float *__restrict__ x_out,
                   const __nv_bfloat16 *__restrict__ w, int d, __nv_bfloat16 *__restrict__ y,
                   __nv_bfloat16 *__restrict__ feat_out, const int32_t *__restrict__ frontier, int F, int pool_cap) {
  __shared__ float red[kThreads / 32];
  pdl_trigger();
  const int r = blockIdx.x;
  const float4 *xr = reinterpret_cast<const float4 *>(x + (int64_t)r * d);
  const float4 *ar = add ? reinterpret_cast<const float4 *>(add + (int64_t)r * d) : nullptr;
  const int n4 = d / 4;
  float4 v[kRmsVec];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < kRmsVec; ++q) {
    const int i = (int)threadIdx.x + q * kThreads;
    v[q] = i < n4 ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (ar && i < n4) {
      const float4 a = ar[i];
      v[q].x += a.x;
      v[q].y += a.y;
      v[q].z += a.z;
      v[q].w += a.w;
    }
    ss = fmaf(v[q].x, v[q].x, fmaf(v[q].y, v[q].y, fmaf(v[q].z, v[q].z, fmaf(v[q].w, v[q].w, ss))));
  }
  const float inv = rsqrtf(block_sum(ss, red) / (float)d + kRmsEps);
  __nv_bfloat16 *fo = nullptr;
  if (feat_out) {
    const int b = r / F, fv = frontier[r];
    if (fv >= 0 && fv < pool_cap) fo = feat_out + ((int64_t)b * (pool_cap + 1) + fv) * d;
  }
#pragma unroll
  for (int q = 0; q < kRmsVec; ++q) {
    const int i = (int)threadIdx.x + q * kThreads;
    if (i >= n4) break;
    if (x_out) reinterpret_cast<float4 *>(x_out + (int64_t)r * d)[i] = v[q];
    if (fo) {
      reinterpret_cast<__nv_bfloat162 *>(fo)[2 * i] = __floats2bfloat162_rn(v[q].x, v[q].y);
      reinterpret_cast<__nv_bfloat162 *>(fo)[2 * i + 1] = __floats2bfloat162_rn(v[q].z, v[q].w);
    }
    const __nv_bfloat162 w01 = reinterpret_cast<const __nv_bfloat162 *>(w)[2 * i];
    const __nv_bfloat162 w23 = reinterpret_cast<const __nv_bfloat162 *>(w)[2 * i + 1];
    __nv_bfloat162 *yr = reinterpret_cast<__nv_bfloat162 *>(y + (int64_t)r * d);
    yr[2 * i] = __floats2bfloat162_rn(v[q].x * inv * __low2float(w01), v[q].y * inv * __high2float(w01));
    yr[2 * i + 1] = __floats2bfloat162_rn(v[q].z * inv * __low2float(w23), v[q].w * inv * __high2float(w23));
  }
}

// The round's draft tree per sequence: the frontier nodes and all their
// ancestors, ancestors in pool order (a parent precedes its child), the
// frontier last in frontier order.  Outputs: cpar [B, C] (compact parents,
// -1 past the valid count), n_valid [B], cpool [B, C] (pool index, -1
// past), cidx [B, F] (compact index of each frontier node).
__global__ void __launch_bounds__(kThreads)
    compact_kernel(const int32_t *__restrict__ pool_parent, const int32_t *__restrict__ frontier, int F, int pool_cap,
                   int C, int32_t *cpar, int32_t *n_valid, int32_t *cpool, int32_t *cidx, int32_t *status) {
  extern __shared__ int sm[];
  int *mark = sm;                 // [pool_cap]: 0 absent, 1 ancestor, 2 frontier
  int *newi = sm + pool_cap;      // [pool_cap]: compact index
  int *pp = sm + 2 * pool_cap;    // [pool_cap]: the pool's parents (walked from shared memory)
  __shared__ int s_n, s_bad, s_run, s_wc[kThreads / 32];
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < pool_cap; i += kThreads) {
    mark[i] = 0;
    pp[i] = pool_parent[(int64_t)b * pool_cap + i];
  }
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  for (int f = threadIdx.x; f < F; f += kThreads) {
    const int v = frontier[(int64_t)b * F + f];
    if (v < 0 || v >= pool_cap) {
      atomicOr(&s_bad, 1);
      continue;
    }
    mark[v] = 2;
  }
  __syncthreads();
  // ancestors (bounded walks; a parent must precede its child)
  for (int f = threadIdx.x; f < F; f += kThreads) {
    const int v = frontier[(int64_t)b * F + f];
    if (v < 0 || v >= pool_cap) continue;
    int u = pp[v];
    for (int guard = 0; u >= 0 && guard < kMaxCompact; ++guard) {
      if (u >= pool_cap || mark[u] == 2) {  // a frontier node is never another's ancestor
        atomicOr(&s_bad, 1);
        break;
      }
      mark[u] = 1;
      u = pp[u];
    }
  }
  // ancestors numbered in pool order: a block-wide count of the marked
  // entries before each one
  if (threadIdx.x == 0) s_run = 0;
  __syncthreads();
  for (int c0 = 0; c0 < pool_cap; c0 += kThreads) {
    const int i = c0 + (int)threadIdx.x;
    const bool is_anc = i < pool_cap && mark[i] == 1;
    const unsigned bal = __ballot_sync(0xffffffffu, is_anc);
    if (lane == 0) s_wc[warp] = __popc(bal);
    __syncthreads();
    int off = s_run;
    for (int w = 0; w < warp; ++w) off += s_wc[w];
    if (is_anc) newi[i] = off + __popc(bal & ((1u << lane) - 1u));
    __syncthreads();
    if (threadIdx.x == 0)
      for (int w = 0; w < kThreads / 32; ++w) s_run += s_wc[w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int n = s_run;
    for (int f = 0; f < F; ++f) {
      const int v = frontier[(int64_t)b * F + f];
      if (v >= 0 && v < pool_cap && mark[v] == 2) {
        mark[v] = 3;  // once, even if listed twice
        newi[v] = n++;
      }
    }
    if (n > C) s_bad = 1;
    s_n = n;
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) {
      sv::report(status, SPEC_DEV_BAD_POOL);
      n_valid[b] = 1;
    }
    for (int i = threadIdx.x; i < C; i += kThreads) {
      cpar[(int64_t)b * C + i] = -1;
      cpool[(int64_t)b * C + i] = -1;
    }
    for (int f = threadIdx.x; f < F; f += kThreads) cidx[(int64_t)b * F + f] = 0;
    return;
  }
  for (int i = threadIdx.x; i < C; i += kThreads) {
    cpar[(int64_t)b * C + i] = -1;
    cpool[(int64_t)b * C + i] = -1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < pool_cap; i += kThreads) {
    if (mark[i] == 0) continue;
    const int ci = newi[i], p = pp[i];
    cpool[(int64_t)b * C + ci] = i;
    cpar[(int64_t)b * C + ci] = p >= 0 && p < pool_cap && mark[p] ? newi[p] : -1;
  }
  for (int f = threadIdx.x; f < F; f += kThreads) {
    const int v = frontier[(int64_t)b * F + f];
    cidx[(int64_t)b * F + f] = newi[v];
  }
  if (threadIdx.x == 0) n_valid[b] = s_n;
}

// Rotary embedding (rotate-half: dims i and i + D/2 by pos * base^(-2i/D))
// of the frontier rows' Q and K at position prefix_len + depth; Q goes to
// its compact row, K and V to the node cache slot of the frontier node.  The
// D/2 angles of the row's position are taken once per row, in double, then
// rounded to float cosines and sines.
constexpr int kMaxHalf = 128;
__global__ void __launch_bounds__(kThreads)
    rope_kernel(const float *__restrict__ qkv, int F, int hq, int hkv, int D, const int32_t *__restrict__ frontier,
                const int32_t *__restrict__ cidx, int C, const int32_t *__restrict__ prefix_len, int depth,
                int pool_cap, __nv_bfloat16 *__restrict__ qc, __nv_bfloat16 *__restrict__ k_nodes,
                __nv_bfloat16 *__restrict__ v_nodes) {
  __shared__ float2 cs[kMaxHalf];
  const int r = blockIdx.x, b = r / F, f = r % F;
  const int v = frontier[r];
  if (v < 0 || v >= pool_cap) return;
  const int ci = cidx[(int64_t)b * F + f];
  const int half = D / 2;
  for (int i = threadIdx.x; i < half; i += kThreads) {
    double sn, c;
    sincos((double)(prefix_len[b] + depth) * pow(kRopeBase, -2.0 * i / D), &sn, &c);
    cs[i] = make_float2((float)c, (float)sn);
  }
  __syncthreads();
  const float *row = qkv + (int64_t)r * (hq + 2 * hkv) * D;
#pragma unroll 4
  for (int e = threadIdx.x; e < (hq + 2 * hkv) * half; e += kThreads) {
    const int h = e / half, i = e % half;
    const float x1 = row[h * D + i], x2 = row[h * D + i + half];
    if (h < hq + hkv) {
      const float c = cs[i].x, s = cs[i].y;
      const float y1 = x1 * c - x2 * s, y2 = x2 * c + x1 * s;
      __nv_bfloat16 *dst = h < hq ? qc + (((int64_t)b * C + ci) * hq + h) * D
                                  : k_nodes + (((int64_t)b * hkv + (h - hq)) * pool_cap + v) * D;
      dst[i] = __float2bfloat16_rn(y1);
      dst[i + half] = __float2bfloat16_rn(y2);
    } else {
      __nv_bfloat16 *dst = v_nodes + (((int64_t)b * hkv + (h - hq - hkv)) * pool_cap + v) * D;
      dst[i] = __float2bfloat16_rn(x1);
      dst[i + half] = __float2bfloat16_rn(x2);
    }
  }
}

// Node K/V rows of the compact tree ([B, hkv, C, D]); rows past the valid
// count are zero.
__global__ void __launch_bounds__(kThreads)
    gather_kv_kernel(const __nv_bfloat16 *__restrict__ k_nodes, const __nv_bfloat16 *__restrict__ v_nodes,
                     const int32_t *__restrict__ cpool, int C, int hkv, int D, int pool_cap,
                     __nv_bfloat16 *__restrict__ kt, __nv_bfloat16 *__restrict__ vt) {
  const int b = blockIdx.y, h = blockIdx.x;
  const int vec = D / 8;
  for (int e = threadIdx.x; e < C * vec; e += kThreads) {
    const int i = e / vec, c = e % vec;
    const int u = cpool[(int64_t)b * C + i];
    uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (u >= 0 && u < pool_cap) {
      const int64_t src = (((int64_t)b * hkv + h) * pool_cap + u) * D;
      kv = reinterpret_cast<const uint4 *>(k_nodes + src)[c];
      vv = reinterpret_cast<const uint4 *>(v_nodes + src)[c];
    }
    const int64_t dst = (((int64_t)b * hkv + h) * C + i) * D;
    reinterpret_cast<uint4 *>(kt + dst)[c] = kv;
    reinterpret_cast<uint4 *>(vt + dst)[c] = vv;
  }
}

// Attention rows of the frontier nodes, [R, hq * D] bf16.
__global__ void __launch_bounds__(kThreads)
    gather_out_kernel(const __nv_bfloat16 *__restrict__ out, const int32_t *__restrict__ cidx, int F, int C, int hqd,
                      __nv_bfloat16 *__restrict__ a) {
  pdl_trigger();
  const int r = blockIdx.x, b = r / F;
  const int ci = cidx[r];
  const uint4 *src = reinterpret_cast<const uint4 *>(out + ((int64_t)b * C + ci) * hqd);
  uint4 *dst = reinterpret_cast<uint4 *>(a + (int64_t)r * hqd);
  for (int i = threadIdx.x; i < hqd / 8; i += kThreads) dst[i] = src[i];
}

// act = SiLU(gate) * up from the [R, 2, f] float32 product, bf16; grid
// (chunks of 4 * kThreads, R), f a multiple of 4.
__global__ void __launch_bounds__(kThreads)
    swiglu_kernel(const float *__restrict__ gu, int f, __nv_bfloat16 *__restrict__ act) {
  pdl_trigger();
  const int r = blockIdx.y, i = (int)(blockIdx.x * kThreads + threadIdx.x);
  if (4 * i >= f) return;
  const float4 g = reinterpret_cast<const float4 *>(gu + (int64_t)r * 2 * f)[i];
  const float4 u = reinterpret_cast<const float4 *>(gu + (int64_t)r * 2 * f + f)[i];
  auto silu = [](float x) { return x / (1.f + __expf(-x)); };
  __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(act + (int64_t)r * f);
  dst[2 * i] = __floats2bfloat162_rn(silu(g.x) * u.x, silu(g.y) * u.y);
  dst[2 * i + 1] = __floats2bfloat162_rn(silu(g.z) * u.z, silu(g.w) * u.w);
}

struct Layout {
  size_t x, h0, n1, qkv, qc, kt, vt, cpar, nval, cpool, cidx, depth, pos, anc, fc, ns, attn_out, attn_ws, a, o, h1,
      n2, gu, act, dn, n3, logits, gemm, total;
  SvAttnShape as;
  SvAttnPlan ap;
  size_t gemm_bytes;
};

Layout layout(int B, int F, int d, int hq, int hkv, int D, int ffn, int V, int s_max, int max_prefix) {
  Layout l{};
  const int R = B * F, C = kMaxCompact;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  l.x = take((size_t)R * 2 * d * 2);
  l.h0 = take((size_t)R * d * 4);
  l.n1 = take((size_t)R * d * 2);
  l.qkv = take((size_t)R * (hq + 2 * hkv) * D * 4);
  l.qc = take((size_t)B * C * hq * D * 2);
  l.kt = take((size_t)B * hkv * C * D * 2);
  l.vt = take((size_t)B * hkv * C * D * 2);
  l.cpar = take((size_t)B * C * 4);
  l.nval = take((size_t)B * 4);
  l.cpool = take((size_t)B * C * 4);
  l.cidx = take((size_t)R * 4);
  l.depth = take((size_t)B * C * 4);
  l.pos = take((size_t)B * C * 4);
  l.anc = take((size_t)B * C * 8);
  l.fc = take((size_t)B * C * 4);
  l.ns = take((size_t)B * C * 4);
  l.attn_out = take((size_t)B * C * hq * D * 2);
  l.as = SvAttnShape{SPEC_BF16, B, C, hq, hkv, D, s_max, max_prefix};
  l.ap = sv_attn_plan(l.as, 0);
  l.attn_ws = take(l.ap.ws_bytes > 0 ? l.ap.ws_bytes : 16);
  l.a = take((size_t)R * hq * D * 2);
  l.o = take((size_t)R * d * 4);
  l.h1 = take((size_t)R * d * 4);
  l.n2 = take((size_t)R * d * 2);
  l.gu = take((size_t)R * 2 * ffn * 4);
  l.act = take((size_t)R * ffn * 2);
  l.dn = take((size_t)R * d * 4);
  l.n3 = take((size_t)R * d * 2);
  l.logits = take((size_t)R * V * 4);
  // one GEMM workspace share, sized for the largest of the round's GEMMs
  size_t g = 0;
  const int shapes[6][3] = {{d, 2 * d, 1}, {(hq + 2 * hkv) * D, d, 1}, {d, hq * D, 1}, {ffn, d, 2}, {d, ffn, 1},
                            {V, d, 1}};
  for (auto &sh : shapes) {
    const SvGemmPlan p = sv_wgemm_plan(sh[0], sh[1], sh[2], R);
    const size_t need = p.partial_bytes;
    g = need > g ? need : g;
  }
  l.gemm_bytes = g;
  l.gemm = take(g);
  l.total = off;
  return l;
}

}  // namespace

size_t sv_eagle_round_ws_bytes(int batch, int n_front, int hidden, int hq, int hkv, int head_dim, int ffn,
                               int vocab, int s_max, int max_prefix) {
  return layout(batch, n_front, hidden, hq, hkv, head_dim, ffn, vocab, s_max, max_prefix).total;
}

int sv_eagle_round(const SvEagleWeights &w, int batch, int hidden, int hq, int hkv, int head_dim, int ffn, int vocab,
                   const void *k_prefix, const void *v_prefix, int s_max, const int32_t *prefix_len, int max_prefix,
                   void *k_nodes, void *v_nodes, void *feat, const int32_t *frontier, int n_front, int depth, int k,
                   float temperature, int32_t *pool_parent, int32_t *pool_tok, float *pool_conf, float *pool_val,
                   int32_t *pool_count, int pool_cap, int32_t *next_frontier, int n_next, float *logits_out,
                   void *ws, int32_t *status, cudaStream_t stream) {
  const int B = batch, F = n_front, d = hidden, D = head_dim, R = B * F, C = kMaxCompact;
  const Layout l = layout(B, F, d, hq, hkv, D, ffn, vocab, s_max, max_prefix);
  uint8_t *base = reinterpret_cast<uint8_t *>(ws);
  auto at = [&](size_t off) { return base + off; };
  auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16 *>(base + off); };
  auto f32 = [&](size_t off) { return reinterpret_cast<float *>(base + off); };
  auto i32 = [&](size_t off) { return reinterpret_cast<int32_t *>(base + off); };
  // a GEMM whose output is float32 rows [R, G, M], the workspace share reused;
  // launched as a programmatic dependent of the row kernel that feeds it
  auto gemm = [&](const void *W, const void *X, int M, int K, int G, float *out) {
    const SvGemmPlan p = sv_wgemm_plan(M, K, G, R);
    return sv_wgemm(p, W, X, 0, M, K, G, R, 0, out, nullptr, nullptr, nullptr, reinterpret_cast<float *>(at(l.gemm)),
                    true, status, stream);
  };
  int rc;
  inputs_kernel<<<R, kThreads, 0, stream>>>(reinterpret_cast<const __nv_bfloat16 *>(feat),
                                            reinterpret_cast<const __nv_bfloat16 *>(w.emb), pool_parent, pool_tok,
                                            frontier, F, pool_cap, d, vocab, bf(l.x), status);
  if ((rc = gemm(w.fc, bf(l.x), d, 2 * d, 1, f32(l.h0))) != SPEC_OK) return rc;
  rmsnorm_kernel<<<R, kThreads, 0, stream>>>(f32(l.h0), nullptr, nullptr,
                                             reinterpret_cast<const __nv_bfloat16 *>(w.ln1), d, bf(l.n1), nullptr,
                                             nullptr, F, pool_cap);
  if ((rc = gemm(w.qkv, bf(l.n1), (hq + 2 * hkv) * D, d, 1, f32(l.qkv))) != SPEC_OK) return rc;
  // the round's draft tree, its Q / K / V and masks
  compact_kernel<<<B, kThreads, (size_t)3 * pool_cap * sizeof(int), stream>>>(
      pool_parent, frontier, F, pool_cap, C, i32(l.cpar), i32(l.nval), i32(l.cpool), i32(l.cidx), status);
  if (cudaMemsetAsync(at(l.qc), 0, (size_t)B * C * hq * D * 2, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  rope_kernel<<<R, kThreads, 0, stream>>>(f32(l.qkv), F, hq, hkv, D, frontier, i32(l.cidx), C, prefix_len, depth,
                                          pool_cap, bf(l.qc), reinterpret_cast<__nv_bfloat16 *>(k_nodes),
                                          reinterpret_cast<__nv_bfloat16 *>(v_nodes));
  gather_kv_kernel<<<dim3(hkv, B), kThreads, 0, stream>>>(reinterpret_cast<const __nv_bfloat16 *>(k_nodes),
                                                          reinterpret_cast<const __nv_bfloat16 *>(v_nodes),
                                                          i32(l.cpool), C, hkv, D, pool_cap, bf(l.kt), bf(l.vt));
  if ((rc = sv_build_batch(i32(l.cpar), C, i32(l.nval), nullptr, nullptr, nullptr, 0, 1, nullptr, prefix_len, B, C,
                           nullptr, i32(l.depth), i32(l.pos), reinterpret_cast<uint64_t *>(at(l.anc)), i32(l.fc),
                           i32(l.ns), status, stream)) != SPEC_OK)
    return rc;
  if ((rc = sv_attn_run(l.as, l.ap, bf(l.qc), k_prefix, v_prefix, bf(l.kt), bf(l.vt), prefix_len,
                        reinterpret_cast<const uint64_t *>(at(l.anc)), bf(l.attn_out), 1.0f / sqrtf((float)D),
                        at(l.attn_ws), l.ap.ws_bytes, status, stream)) != SPEC_OK)
    return rc;
  gather_out_kernel<<<R, kThreads, 0, stream>>>(bf(l.attn_out), i32(l.cidx), F, C, hq * D, bf(l.a));
  // O projection, residual, MLP, residual
  if ((rc = gemm(w.o, bf(l.a), d, hq * D, 1, f32(l.o))) != SPEC_OK) return rc;
  rmsnorm_kernel<<<R, kThreads, 0, stream>>>(f32(l.o), f32(l.h0), f32(l.h1),
                                             reinterpret_cast<const __nv_bfloat16 *>(w.ln2), d, bf(l.n2), nullptr,
                                             nullptr, F, pool_cap);
  if ((rc = gemm(w.gate_up, bf(l.n2), ffn, d, 2, f32(l.gu))) != SPEC_OK) return rc;
  swiglu_kernel<<<dim3((ffn / 4 + kThreads - 1) / kThreads, R), kThreads, 0, stream>>>(f32(l.gu), ffn, bf(l.act));
  if ((rc = gemm(w.down, bf(l.act), d, ffn, 1, f32(l.dn))) != SPEC_OK) return rc;
  // the node's feature (f = h1 + down) and the final norm before the LM head
  rmsnorm_kernel<<<R, kThreads, 0, stream>>>(f32(l.dn), f32(l.h1), nullptr,
                                             reinterpret_cast<const __nv_bfloat16 *>(w.lnf), d, bf(l.n3),
                                             reinterpret_cast<__nv_bfloat16 *>(feat), frontier, F, pool_cap);
  float *logits = logits_out ? logits_out : f32(l.logits);
  if ((rc = gemm(w.lm, bf(l.n3), vocab, d, 1, logits)) != SPEC_OK) return rc;
  if ((rc = sv_launch_status()) != SPEC_OK) return rc;
  return sv_tree_expand(logits, SPEC_F32, B, F, vocab, frontier, k, temperature, pool_parent, pool_tok, pool_conf,
                        pool_val, pool_count, pool_cap, next_frontier, n_next, status, stream);
}
