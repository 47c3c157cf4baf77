// Fused LM head + acceptance: the target logits of every tree node are
// reduced to softmax statistics inside the LM-head GEMM's epilogue, so the
// [rows, vocabulary] logits never reach HBM.
//
// "Medusa, explained", step 6 (one pass of the base model scores every
// node) and step 7 / section "Typical acceptance" (greedy: a node is valid
// when its token is the target's argmax at its parent; typical: p(x) >
// min(eps, delta exp(-H)); the step's first token is the greedy one);
// "Drafters: ...", section "Why the answer does not change".
//
// 1. The GEMM (statistics epilogue) writes, per tree node, vocabulary tile and
//    epilogue warp (the 32 * MT vocabulary rows that warp holds), (max logit,
//    sum exp(z - zmax), sum exp(z - zmax)(z - zmax), argmax) with z = logit / T.
// 2. fold_kernel, one CTA per (node, sequence): merges the node's records in
//    a fixed order into (max, S, Q, argmax) and, for typical acceptance,
//    computes each child's logit as the dot product of the node's hidden
//    state with the child token's LM-head row (float32) and its probability
//    exp(z - max) / S.  Then it takes a ticket on the sequence's counter;
//    the CTA that completes the sequence walks the tree: greedy from the
//    root, or typical over all nodes at once (every node's threshold is
//    known, so no node is visited twice).  No CTA waits for another.
// Rejection sampling needs the whole residual row and keeps the logits
// (spec_lm_head + spec_accept).
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxNodes = SPEC_MAX_NODES;

struct __align__(16) RowStat {
  float m, S, Q;  // max z, sum exp(z - m), sum exp(z - m)(z - m)
  int amax;
};

// Union of two disjoint sets' statistics (both moved to the larger max).
__device__ __forceinline__ void merge(float &m, float &S, float &Q, float m2, float S2, float Q2) {
  if (!(S2 > 0.f)) return;
  if (!(S > 0.f)) {
    m = m2; S = S2; Q = Q2;
    return;
  }
  const float mn = fmaxf(m, m2), da = m - mn, db = m2 - mn;
  const float ea = __expf(da), eb = __expf(db);
  const float nS = fmaf(ea, S, eb * S2);
  Q = fmaf(ea, fmaf(da, S, Q), eb * fmaf(db, S2, Q2));
  S = nS;
  m = mn;
}

__global__ void __launch_bounds__(kThreads)
    fold_kernel(int mode, const float4 *__restrict__ stats, int rec_stride, const __nv_bfloat16 *__restrict__ hid,
                const __nv_bfloat16 *__restrict__ w, int N, int hidden, int V, const int32_t *__restrict__ tok,
                const int32_t *__restrict__ parents, const int32_t *__restrict__ first_child,
                const int32_t *__restrict__ next_sibling, float inv_t, float eps, float delta, int path_cap,
                RowStat *rowstat, float *childp, int *counters, int32_t *acc_len, int32_t *acc_path,
                int32_t *bonus, int32_t *status) {
  __shared__ float s_m[kWarps], s_S[kWarps], s_Q[kWarps];
  __shared__ unsigned long long s_k[kWarps];
  __shared__ RowStat s_row;
  __shared__ int s_last;
  const int v = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)b * N + v;
  // the records were written by the previous kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // 1. merge this node's records: strided per thread, then a fixed butterfly
  float m = -FLT_MAX, S = 0.f, Q = 0.f;
  unsigned long long key = 0ull;
  const float4 *rec = stats + row * rec_stride;
  for (int i = threadIdx.x; i < rec_stride; i += kThreads) {
    const float4 r = rec[i];
    if (!(r.y > 0.f)) continue;
    const int am = __float_as_int(r.w);
    merge(m, S, Q, r.x * inv_t, r.y, r.z);
    const unsigned long long k = sv::rank_key(r.x, (uint32_t)am);
    key = k > key ? k : key;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), S2 = __shfl_xor_sync(0xffffffffu, S, o);
    const float Q2 = __shfl_xor_sync(0xffffffffu, Q, o);
    merge(m, S, Q, m2, S2, Q2);
    const unsigned long long k = __shfl_xor_sync(0xffffffffu, key, o);
    key = k > key ? k : key;
  }
  if (lane == 0) {
    s_m[warp] = m; s_S[warp] = S; s_Q[warp] = Q; s_k[warp] = key;
  }
  __syncthreads();
  if (warp == 0) {
    m = lane < kWarps ? s_m[lane] : -FLT_MAX;
    S = lane < kWarps ? s_S[lane] : 0.f;
    Q = lane < kWarps ? s_Q[lane] : 0.f;
    key = lane < kWarps ? s_k[lane] : 0ull;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), S2 = __shfl_xor_sync(0xffffffffu, S, o);
      const float Q2 = __shfl_xor_sync(0xffffffffu, Q, o);
      merge(m, S, Q, m2, S2, Q2);
      const unsigned long long k = __shfl_xor_sync(0xffffffffu, key, o);
      key = k > key ? k : key;
    }
    if (lane == 0) {
      s_row = RowStat{m, S, Q, (int)sv::key_index(key)};
      rowstat[row] = s_row;
    }
  }
  __syncthreads();

  // 2. typical: each child's probability from its own logit (one warp per
  // child, 16-byte loads of the hidden state and the LM-head row)
  if (mode == SPEC_ACCEPT_TYPICAL) {
    int c = first_child[row];
    for (int k = 0; k < warp && c >= 0 && c < N; ++k) c = next_sibling[(int64_t)b * N + c];
    for (int guard = 0; c >= 0 && c < N && guard < kMaxNodes; ++guard) {
      const int x = tok[(int64_t)b * N + c];
      float p = -1.f;
      if (x >= 0 && x < V) {
        const uint4 *hv = reinterpret_cast<const uint4 *>(hid + row * hidden);
        const uint4 *wv = reinterpret_cast<const uint4 *>(w + (int64_t)x * hidden);
        float acc = 0.f;
        for (int i = lane; i < hidden / 8; i += 32) {
          float a8[8], b8[8];
          sv::bf16x8_to_f32(hv[i], a8);
          sv::bf16x8_to_f32(wv[i], b8);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc = fmaf(a8[j], b8[j], acc);
        }
        acc = sv::warp_sum(acc);
        p = __expf(acc * inv_t - s_row.m) / s_row.S;
      } else if (lane == 0) {
        sv::report(status, SPEC_DEV_BAD_TOKEN);
      }
      if (lane == 0) childp[(int64_t)b * N + c] = p;
      // next child of this warp: kWarps siblings further on
      for (int k = 0; k < kWarps && c >= 0 && c < N; ++k) c = next_sibling[(int64_t)b * N + c];
    }
  }

  // 3. the CTA completing the sequence takes the decisions
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&counters[b], 1) == N - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  __shared__ int s_par[kMaxNodes], s_ok[kMaxNodes], s_depth[kMaxNodes], s_path[kMaxNodes + 1];
  __shared__ float s_thr[kMaxNodes];
  const int64_t base = (int64_t)b * N;
  for (int i = threadIdx.x; i < N; i += kThreads) {
    s_par[i] = parents[base + i];
    if (mode == SPEC_ACCEPT_TYPICAL) {
      // written by other CTAs: read past L1
      const float4 rs = __ldcg(reinterpret_cast<const float4 *>(rowstat) + base + i);
      const float H = logf(rs.y) - rs.z / rs.y;
      s_thr[i] = fminf(eps, delta * expf(-H));
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int len = 1, bon = -1;
    s_path[0] = 0;
    if (mode == SPEC_ACCEPT_GREEDY) {
      int u = 0;
      for (int guard = 0; guard < kMaxNodes; ++guard) {
        const int a = __ldcg(&rowstat[base + u].amax);
        int nxt = -1;
        for (int c = first_child[base + u], n = 0; c >= 0 && c < N && n < kMaxNodes;
             c = next_sibling[base + c], ++n)
          if (tok[base + c] == a) {
            nxt = c;
            break;
          }
        if (nxt < 0) {
          bon = a;
          break;
        }
        s_path[len++] = nxt;
        u = nxt;
      }
    } else {
      // a node is reachable when its parent is and its probability passes
      // the parent's threshold; the deepest reachable node (lowest index on
      // ties) ends the accepted path
      s_ok[0] = 1;
      s_depth[0] = 0;
      int best = 0;
      for (int i = 1; i < N; ++i) {
        const int p = s_par[i];
        const bool pv = p >= 0 && p < i;
        if (!pv) sv::report(status, SPEC_DEV_BAD_PARENTS);
        s_depth[i] = pv ? s_depth[p] + 1 : 0;
        s_ok[i] = pv && s_ok[p] && __ldcg(&childp[base + i]) > s_thr[p];
        if (s_ok[i] && s_depth[i] > s_depth[best]) best = i;
      }
      int d = s_depth[best];
      len = d + 1;
      for (int u = best; d >= 0; --d) {
        s_path[d] = u;
        u = s_par[u];
      }
      bon = __ldcg(&rowstat[base + best].amax);
    }
    if (len > path_cap) {
      sv::report(status, SPEC_DEV_CAPACITY);
      len = path_cap;
    }
    acc_len[b] = len - 1;
    for (int j = 0; j < path_cap; ++j) acc_path[(int64_t)b * path_cap + j] = j < len ? s_path[j] : -1;
    bonus[b] = bon;
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  SvGemmPlan p;
  size_t fold_counters, partial, stats, rowstat, childp, total;
};

Layout layout(int batch, int n_nodes, int hidden, int vocab) {
  Layout l{};
  const int rows = batch * n_nodes;
  l.p = sv_wgemm_plan(vocab, hidden, 1, rows);
  const int rec = l.p.tiles_pg * 4;  // one record per (row, tile, epilogue warp)
  l.fold_counters = 0;
  l.partial = l.fold_counters + align256((size_t)batch * 4);
  l.stats = l.partial + l.p.partial_bytes;
  l.rowstat = l.stats + align256((size_t)rows * rec * 16);
  l.childp = l.rowstat + align256((size_t)rows * sizeof(RowStat));
  l.total = l.childp + align256((size_t)rows * 4);
  return l;
}

}  // namespace

size_t sv_lm_head_accept_ws_bytes(int batch, int n_nodes, int hidden, int vocab) {
  return layout(batch, n_nodes, hidden, vocab).total;
}

int sv_lm_head_accept(int mode, const void *hid, const void *w, int batch, int n_nodes, int hidden, int vocab,
                      const int32_t *tok, const int32_t *parents, const int32_t *first_child,
                      const int32_t *next_sibling, float temperature, float eps, float delta, int path_cap,
                      int32_t *acc_len, int32_t *acc_path, int32_t *bonus, void *ws, int32_t *status,
                      cudaStream_t stream) {
  const Layout l = layout(batch, n_nodes, hidden, vocab);
  uint8_t *base = reinterpret_cast<uint8_t *>(ws);
  const int rows = batch * n_nodes;
  // the per-sequence tickets start at zero
  if (cudaMemsetAsync(base, 0, l.partial, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  const float inv_t = 1.f / temperature;
  int rc = sv_wgemm(l.p, w, hid, 0, vocab, hidden, 1, rows, 2, nullptr, nullptr, nullptr, nullptr,
                    reinterpret_cast<float *>(base + l.partial), false, status, stream, inv_t, base + l.stats);
  if (rc != SPEC_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_nodes, batch);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fold_kernel, mode, reinterpret_cast<const float4 *>(base + l.stats),
                         l.p.tiles_pg * 4, reinterpret_cast<const __nv_bfloat16 *>(hid),
                         reinterpret_cast<const __nv_bfloat16 *>(w), n_nodes, hidden, vocab, tok, parents,
                         first_child, next_sibling, inv_t, eps, delta, path_cap,
                         reinterpret_cast<RowStat *>(base + l.rowstat), reinterpret_cast<float *>(base + l.childp),
                         reinterpret_cast<int *>(base + l.fold_counters), acc_len, acc_path, bonus,
                         status) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}
