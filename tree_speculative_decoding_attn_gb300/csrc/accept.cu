// Acceptance of the longest target-agreeing path and the bonus token.
//
// Greedy: "Drafters: draft models, Medusa, EAGLE, MTP, DFlash, DSpark",
// section "Why the answer does not change" (keep a draft only if it is the
// target's own pick; at the first disagreement use the target's token);
// "Medusa, explained", step 7.  Typical: "Medusa, explained", section
// "Typical acceptance" (p(x) > min(eps, delta exp(-H)); the step's first
// token is the greedy one).  Rejection: "Drafters: ...", same section
// (min(1, p/q); on rejection sample the target minus the drafter), with
// the point-mass proposal of a deterministic tree sibling.
//
// One cluster of nc CTAs per sequence (8; 4 at batch >= 32).
// The cluster walks the tree from the root: each visited node's vocabulary
// row is reduced in slices (CTA c reduces the c-th slice with 16-byte loads),
// the nc partial results are exchanged through distributed shared memory and
// combined in CTA order, so every CTA of the cluster holds the same totals
// and takes the same decisions without a broadcast.  Only the rows on the
// walk are read (plus, for typical acceptance, the rows of every node
// reachable through valid children).  Logits are scaled by 1/T as a product;
// the softmax exponentials use the fast exp.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxNodes = SPEC_MAX_NODES;
constexpr int kMaxCluster = 8;  // CTAs per sequence (4 at batch >= 32)

struct Red {
  float f[kWarps];
  unsigned long long u[kWarps];
  float bf;
  unsigned long long bu;
  // cluster exchange slots, double-buffered by reduction parity: a slot is
  // rewritten two reductions later, after every CTA has passed the barrier
  // that follows its last read of it
  float xf[2][2];
  unsigned long long xu[2];
  float cf[2];
  unsigned long long cu;
};

__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t remote(const void *local, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(sv::ptx_smem(local)), "r"(cta));
  return r;
}
__device__ __forceinline__ float ld_remote_f32(const void *local, uint32_t cta) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote(local, cta)) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_remote_u64(const void *local, uint32_t cta) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(remote(local, cta)) : "memory");
  return v;
}

template <typename Op>
__device__ float block_reduce(float v, float ident, Red &r, Op op) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) r.f[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = threadIdx.x < kWarps ? r.f[threadIdx.x] : ident;
#pragma unroll
    for (int o = 16; o; o >>= 1) w = op(w, __shfl_xor_sync(0xffffffffu, w, o));
    if (threadIdx.x == 0) r.bf = w;
  }
  __syncthreads();
  const float out = r.bf;
  __syncthreads();
  return out;
}

__device__ unsigned long long block_max_u64(unsigned long long v, Red &r) {
  v = sv::warp_max_u64(v);
  if ((threadIdx.x & 31) == 0) r.u[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned long long w = threadIdx.x < kWarps ? r.u[threadIdx.x] : 0ull;
    w = sv::warp_max_u64(w);
    if (threadIdx.x == 0) r.bu = w;
  }
  __syncthreads();
  const unsigned long long out = r.bu;
  __syncthreads();
  return out;
}

// Cluster-wide reductions: every CTA gets the identical result (partials
// combined in CTA order).  All threads of all CTAs must call them together.
struct ClusterOps {
  Red &r;
  int parity;
  uint32_t nc;  // CTAs in the cluster

  __device__ float max(float v) {
    v = block_reduce(v, -INFINITY, r, [](float a, float b) { return fmaxf(a, b); });
    if (threadIdx.x == 0) r.xf[parity][0] = v;
    cluster_barrier();
    if (threadIdx.x == 0) {
      float m = -INFINITY;
      for (uint32_t c = 0; c < nc; ++c) m = fmaxf(m, ld_remote_f32(&r.xf[parity][0], c));
      r.cf[0] = m;
    }
    __syncthreads();
    const float out = r.cf[0];
    __syncthreads();
    parity ^= 1;
    return out;
  }
  // two sums at once
  __device__ void sum2(float &a, float &b) {
    a = block_reduce(a, 0.f, r, [](float x, float y) { return x + y; });
    b = block_reduce(b, 0.f, r, [](float x, float y) { return x + y; });
    if (threadIdx.x == 0) {
      r.xf[parity][0] = a;
      r.xf[parity][1] = b;
    }
    cluster_barrier();
    if (threadIdx.x == 0) {
      float sa = 0.f, sb = 0.f;
      for (uint32_t c = 0; c < nc; ++c) {
        sa += ld_remote_f32(&r.xf[parity][0], c);
        sb += ld_remote_f32(&r.xf[parity][1], c);
      }
      r.cf[0] = sa;
      r.cf[1] = sb;
    }
    __syncthreads();
    a = r.cf[0];
    b = r.cf[1];
    __syncthreads();
    parity ^= 1;
  }
  __device__ unsigned long long max_u64(unsigned long long v) {
    v = block_max_u64(v, r);
    if (threadIdx.x == 0) r.xu[parity] = v;
    cluster_barrier();
    if (threadIdx.x == 0) {
      unsigned long long m = 0ull;
      for (uint32_t c = 0; c < nc; ++c) {
        const unsigned long long w = ld_remote_u64(&r.xu[parity], c);
        m = w > m ? w : m;
      }
      r.cu = m;
    }
    __syncthreads();
    const unsigned long long out = r.cu;
    __syncthreads();
    parity ^= 1;
    return out;
  }
};

// Visit every element of this CTA's slice [lo, hi) of a logits row:
// f(x, value) with x the column.  16-byte loads when the slice start is
// aligned and its length a multiple of the vector width, issued kBatch at a
// time per thread before any is used, so a CTA keeps kThreads * kBatch * 16
// bytes in flight.
constexpr int kBatch = 8;
template <typename T, typename F>
__device__ __forceinline__ void for_slice(const T *row, int lo, int hi, F &&f) {
  constexpr int kVec = 16 / sizeof(T);
  if (((hi - lo) % kVec) == 0 && (reinterpret_cast<uintptr_t>(row + lo) & 15) == 0) {
    const int nv = (hi - lo) / kVec;
    const uint4 *src = reinterpret_cast<const uint4 *>(row + lo);
    for (int v0 = threadIdx.x; v0 < nv; v0 += kBatch * kThreads) {
      uint4 u[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int vi = v0 + i * kThreads;
        u[i] = vi < nv ? src[vi] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int vi = v0 + i * kThreads;
        if (vi >= nv) break;
        float v[kVec];
        if constexpr (sizeof(T) == 2) {
          sv::bf16x8_to_f32(u[i], v);
        } else {
          v[0] = __uint_as_float(u[i].x);
          v[1] = __uint_as_float(u[i].y);
          v[2] = __uint_as_float(u[i].z);
          v[3] = __uint_as_float(u[i].w);
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j) f(lo + vi * kVec + j, v[j]);
      }
    }
  } else {
    for (int x = lo + threadIdx.x; x < hi; x += kThreads) f(x, sv::to_f32(row[x]));
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    accept_kernel(int mode, const T *__restrict__ logits, int N, int V,
                  const int32_t *__restrict__ tok, const int32_t *__restrict__ parents,
                  const int32_t *__restrict__ first_child, const int32_t *__restrict__ next_sibling,
                  float temp, float eps, float delta, uint64_t seed, uint64_t step, int path_cap,
                  int32_t *acc_len, int32_t *acc_path, int32_t *bonus_out, int32_t *status) {
  __shared__ Red red;
  __shared__ int s_path[kMaxNodes + 1];
  __shared__ int s_len, s_next, s_bonus;
  __shared__ int s_fc[kMaxNodes], s_ns[kMaxNodes], s_tok[kMaxNodes], s_par[kMaxNodes];
  __shared__ int s_ok[kMaxNodes], s_depth[kMaxNodes];
  __shared__ int s_exc[kMaxNodes];
  __shared__ int s_nexc;

  const uint32_t cta = blockIdx.x;  // rank in the cluster (cluster spans x)
  const int b = blockIdx.y;
  const int nc = (int)gridDim.x;  // the cluster spans x
  const int slice = ((V + nc - 1) / nc + 7) / 8 * 8;
  const int lo = min(V, (int)cta * slice), hi = min(V, lo + slice);
  ClusterOps cl{red, 0, (uint32_t)nc};

  const int64_t row0 = (int64_t)b * N;
  // 1/T once: logits are scaled by a product, not a division per element
  const float inv_t = 1.f / temp;
  for (int i = threadIdx.x; i < N; i += kThreads) {
    s_fc[i] = first_child[row0 + i];
    s_ns[i] = next_sibling[row0 + i];
    s_tok[i] = tok[row0 + i];
    s_par[i] = parents[row0 + i];
  }
  if (threadIdx.x == 0) {
    s_len = 1;
    s_path[0] = 0;
  }
  __syncthreads();
  const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  const uint32_t st = (uint32_t)step;
  const T *base = logits + row0 * V;

  auto row_argmax = [&](const T *row) -> int {
    unsigned long long best = 0ull;
    for_slice(row, lo, hi, [&](int x, float v) {
      const unsigned long long k = sv::rank_key(v, (uint32_t)x);
      best = k > best ? k : best;
    });
    return (int)sv::key_index(cl.max_u64(best));
  };
  auto row_max_z = [&](const T *row) -> float {
    float m = -INFINITY;
    for_slice(row, lo, hi, [&](int, float v) { m = fmaxf(m, v * inv_t); });
    return cl.max(m);
  };

  if (mode == SPEC_ACCEPT_GREEDY) {
    int v = 0;
    for (int guard = 0; guard < kMaxNodes; ++guard) {
      const int a = row_argmax(base + (int64_t)v * V);
      if (threadIdx.x == 0) {
        int nxt = -1;
        for (int c = s_fc[v]; c >= 0 && c < N; c = s_ns[c])
          if (s_tok[c] == a) {
            nxt = c;
            break;
          }
        s_next = nxt;
        if (nxt >= 0) s_path[s_len++] = nxt;
        else s_bonus = a;
      }
      __syncthreads();
      if (s_next < 0) break;
      v = s_next;
      __syncthreads();
    }
  } else if (mode == SPEC_ACCEPT_TYPICAL) {
    if (threadIdx.x == 0) {
      s_ok[0] = 1;
      s_depth[0] = 0;
      for (int i = 1; i < N; ++i) {
        s_ok[i] = 0;
        s_depth[i] = s_depth[s_par[i] >= 0 && s_par[i] < i ? s_par[i] : 0] + 1;
      }
    }
    __syncthreads();
    for (int v = 0; v < N; ++v) {
      if (!s_ok[v] || s_fc[v] < 0) continue;  // uniform: shared flags, identical in every CTA
      const T *row = base + (int64_t)v * V;
      const float m = row_max_z(row);
      float S = 0.f, Q = 0.f;
      for_slice(row, lo, hi, [&](int, float x) {
        const float z = x * inv_t - m;
        const float e = __expf(z);
        S += e;
        Q = fmaf(e, z, Q);
      });
      cl.sum2(S, Q);
      if (threadIdx.x == 0) {
        const float H = logf(S) - Q / S;
        const float thr = fminf(eps, delta * expf(-H));
        for (int c = s_fc[v]; c >= 0 && c < N; c = s_ns[c]) {
          const int x = s_tok[c];
          if (x < 0 || x >= V) {
            sv::report(status, SPEC_DEV_BAD_TOKEN);
            continue;
          }
          const float p = __expf(sv::to_f32(row[x]) * inv_t - m) / S;
          s_ok[c] = p > thr;
        }
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      int best = 0;
      for (int i = 1; i < N; ++i)
        if (s_ok[i] && s_depth[i] > s_depth[best]) best = i;
      int d = s_depth[best];  // root-first path of `best`
      s_len = d + 1;
      for (int u = best; d >= 0; --d) {
        s_path[d] = u;
        u = s_par[u];
      }
      s_next = best;
    }
    __syncthreads();
    const int a = row_argmax(base + (int64_t)s_next * V);
    if (threadIdx.x == 0) s_bonus = a;
  } else {  // SPEC_ACCEPT_REJECT
    int v = 0;
    for (int guard = 0; guard < kMaxNodes; ++guard) {
      const T *row = base + (int64_t)v * V;
      const float m = row_max_z(row);
      float S = 0.f, unused = 0.f;
      for_slice(row, lo, hi, [&](int, float x) { S += __expf(x * inv_t - m); });
      cl.sum2(S, unused);
      if (threadIdx.x == 0) {
        int nxt = -1;
        float removed = 0.f;
        s_nexc = 0;
        for (int c = s_fc[v]; c >= 0 && c < N; c = s_ns[c]) {
          const int x = s_tok[c];
          bool seen = false;
          for (int e = 0; e < s_nexc; ++e) seen |= s_exc[e] == x;
          float r = 0.f, ex = 0.f;
          if (x < 0 || x >= V) {
            sv::report(status, SPEC_DEV_BAD_TOKEN);
            seen = true;
          } else if (!seen) {
            ex = __expf(sv::to_f32(row[x]) * inv_t - m);
            r = ex / (S - removed);
          }
          const sv::u32x4 w = sv::philox4x32_10(sv::u32x4{(uint32_t)c, 0u, (uint32_t)b, st}, k0, k1);
          const float u = (float)(w.x >> 8) * 5.9604644775390625e-8f;  // 2^-24
          if (u < r) {
            nxt = c;
            break;
          }
          if (!seen) {
            s_exc[s_nexc++] = x;
            removed = removed + ex;
          }
        }
        s_next = nxt;
        if (nxt >= 0) s_path[s_len++] = nxt;
      }
      __syncthreads();
      if (s_next >= 0) {
        v = s_next;
        __syncthreads();
        continue;
      }
      // residual sample: exponential race in log form over non-removed tokens
      const int nexc = s_nexc;
      unsigned long long best = 0ull;
      for_slice(row, lo, hi, [&](int x, float val) {
        for (int e = 0; e < nexc; ++e)
          if (s_exc[e] == x) return;
        const sv::u32x4 w =
            sv::philox4x32_10(sv::u32x4{(uint32_t)x, 256u + (uint32_t)v, (uint32_t)b, st}, k0, k1);
        const float up = ((float)(w.x >> 9) + 0.5f) * 1.1920928955078125e-7f;  // 2^-23
        const float g = -logf(-logf(up));
        const float key = val * inv_t + g;
        const unsigned long long k = sv::rank_key(key, (uint32_t)x);
        best = k > best ? k : best;
      });
      best = cl.max_u64(best);
      if (threadIdx.x == 0) s_bonus = (int)sv::key_index(best);
      __syncthreads();
      break;
    }
  }
  __syncthreads();
  if (cta == 0 && threadIdx.x == 0) {
    int len = s_len;
    if (len > path_cap) {
      sv::report(status, SPEC_DEV_CAPACITY);
      len = path_cap;
    }
    acc_len[b] = len - 1;
    for (int j = 0; j < path_cap; ++j) acc_path[(int64_t)b * path_cap + j] = j < len ? s_path[j] : -1;
    bonus_out[b] = s_bonus;
  }
  cluster_barrier();  // partners' reads of this CTA's exchange slots are done
}

template <typename T>
int launch_accept(int mode, const void *logits, int batch, int n_nodes, int vocab, const int32_t *tok,
                  const int32_t *parents, const int32_t *first_child, const int32_t *next_sibling,
                  float temperature, float eps, float delta, uint64_t seed, uint64_t step, int path_cap,
                  int32_t *acc_len, int32_t *acc_path, int32_t *bonus, int32_t *status, cudaStream_t stream) {
  // CTAs per sequence (the kernel reads it from gridDim.x): at batch >= 32
  // four, so every sequence's cluster is resident in one wave
  const int nc = batch >= 32 ? 4 : kMaxCluster;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nc, batch);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, accept_kernel<T>, mode, (const T *)logits, n_nodes, vocab, tok, parents,
                            first_child, next_sibling, temperature, eps, delta, seed, step, path_cap, acc_len,
                            acc_path, bonus, status) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

}  // namespace

int sv_accept(int mode, const void *logits, int dtype, int batch, int n_nodes, int vocab,
              const int32_t *tok, const int32_t *parents, const int32_t *first_child,
              const int32_t *next_sibling, float temperature, float eps, float delta,
              uint64_t seed, uint64_t step, int path_cap, int32_t *acc_len, int32_t *acc_path,
              int32_t *bonus, int32_t *status, cudaStream_t stream) {
  if (dtype == SPEC_BF16)
    return launch_accept<__nv_bfloat16>(mode, logits, batch, n_nodes, vocab, tok, parents, first_child,
                                        next_sibling, temperature, eps, delta, seed, step, path_cap, acc_len,
                                        acc_path, bonus, status, stream);
  return launch_accept<float>(mode, logits, batch, n_nodes, vocab, tok, parents, first_child, next_sibling,
                              temperature, eps, delta, seed, step, path_cap, acc_len, acc_path, bonus, status,
                              stream);
}
