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
// One CTA per sequence walks the tree from the root; each visited node's
// vocabulary row is reduced by the whole CTA with 16-byte loads, so only
// the rows on the walk are read (plus, for typical acceptance, the rows of
// every node reachable through valid children).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxNodes = SPEC_MAX_NODES;

struct Red {
  float f[kWarps];
  unsigned long long u[kWarps];
  float bf;
  unsigned long long bu;
};

__device__ float block_max(float v, Red &r) {
  v = sv::warp_max(v);
  if ((threadIdx.x & 31) == 0) r.f[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = threadIdx.x < kWarps ? r.f[threadIdx.x] : -INFINITY;
    w = sv::warp_max(w);
    if (threadIdx.x == 0) r.bf = w;
  }
  __syncthreads();
  const float out = r.bf;
  __syncthreads();
  return out;
}

__device__ float block_sum(float v, Red &r) {
  v = sv::warp_sum(v);
  if ((threadIdx.x & 31) == 0) r.f[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = threadIdx.x < kWarps ? r.f[threadIdx.x] : 0.f;
    w = sv::warp_sum(w);
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

// Visit every element of a logits row: f(x, value).  16-byte loads when the
// row is aligned and its length a multiple of the vector width.
template <typename T, typename F>
__device__ __forceinline__ void for_row(const T *row, int V, F &&f) {
  constexpr int kVec = 16 / sizeof(T);
  if ((V % kVec) == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
    for (int vi = threadIdx.x; vi < V / kVec; vi += kThreads) {
      const uint4 u = *reinterpret_cast<const uint4 *>(row + (int64_t)vi * kVec);
      float v[kVec];
      if constexpr (sizeof(T) == 2) {
        sv::bf16x8_to_f32(u, v);
      } else {
        v[0] = __uint_as_float(u.x);
        v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z);
        v[3] = __uint_as_float(u.w);
      }
#pragma unroll
      for (int j = 0; j < kVec; ++j) f(vi * kVec + j, v[j]);
    }
  } else {
    for (int x = threadIdx.x; x < V; x += kThreads) f(x, sv::to_f32(row[x]));
  }
}

template <typename T>
__device__ int row_argmax(const T *row, int V, Red &r) {
  unsigned long long best = 0ull;
  for_row(row, V, [&](int x, float v) {
    const unsigned long long k = sv::rank_key(v, (uint32_t)x);
    best = k > best ? k : best;
  });
  return (int)sv::key_index(block_max_u64(best, r));
}

// max of z = logits / T over the row
template <typename T>
__device__ float row_max_z(const T *row, int V, float T_, Red &r) {
  float m = -INFINITY;
  for_row(row, V, [&](int, float v) { m = fmaxf(m, v / T_); });
  return block_max(m, r);
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

  const int b = blockIdx.x;
  const int64_t row0 = (int64_t)b * N;
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

  if (mode == SPEC_ACCEPT_GREEDY) {
    int v = 0;
    for (int guard = 0; guard < kMaxNodes; ++guard) {
      const int a = row_argmax(base + (int64_t)v * V, V, red);
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
      if (!s_ok[v] || s_fc[v] < 0) continue;  // uniform: shared flags
      const T *row = base + (int64_t)v * V;
      const float m = row_max_z(row, V, temp, red);
      float S = 0.f, Q = 0.f;
      for_row(row, V, [&](int, float x) {
        const float z = x / temp - m;
        const float e = expf(z);
        S += e;
        Q = fmaf(e, z, Q);
      });
      S = block_sum(S, red);
      Q = block_sum(Q, red);
      if (threadIdx.x == 0) {
        const float H = logf(S) - Q / S;
        const float thr = fminf(eps, delta * expf(-H));
        for (int c = s_fc[v]; c >= 0 && c < N; c = s_ns[c]) {
          const int x = s_tok[c];
          if (x < 0 || x >= V) {
            sv::report(status, SPEC_DEV_BAD_TOKEN);
            continue;
          }
          const float p = expf(sv::to_f32(row[x]) / temp - m) / S;
          s_ok[c] = p > thr;
        }
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      int best = 0;
      for (int i = 1; i < N; ++i)
        if (s_ok[i] && s_depth[i] > s_depth[best]) best = i;
      // root-first path of `best`
      int d = s_depth[best];
      s_len = d + 1;
      for (int u = best; d >= 0; --d) {
        s_path[d] = u;
        u = s_par[u];
      }
      s_next = best;
    }
    __syncthreads();
    const int a = row_argmax(base + (int64_t)s_next * V, V, red);
    if (threadIdx.x == 0) s_bonus = a;
  } else {  // SPEC_ACCEPT_REJECT
    int v = 0;
    for (int guard = 0; guard < kMaxNodes; ++guard) {
      const T *row = base + (int64_t)v * V;
      const float m = row_max_z(row, V, temp, red);
      float S = 0.f;
      for_row(row, V, [&](int, float x) { S += expf(x / temp - m); });
      S = block_sum(S, red);
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
            ex = expf(sv::to_f32(row[x]) / temp - m);
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
      for_row(row, V, [&](int x, float val) {
        for (int e = 0; e < nexc; ++e)
          if (s_exc[e] == x) return;
        const sv::u32x4 w =
            sv::philox4x32_10(sv::u32x4{(uint32_t)x, 256u + (uint32_t)v, (uint32_t)b, st}, k0, k1);
        const float up = ((float)(w.x >> 9) + 0.5f) * 1.1920928955078125e-7f;  // 2^-23
        const float g = -logf(-logf(up));
        const float key = val / temp + g;
        const unsigned long long k = sv::rank_key(key, (uint32_t)x);
        best = k > best ? k : best;
      });
      best = block_max_u64(best, red);
      if (threadIdx.x == 0) s_bonus = (int)sv::key_index(best);
      __syncthreads();
      break;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int len = s_len;
    if (len > path_cap) {
      sv::report(status, SPEC_DEV_CAPACITY);
      len = path_cap;
    }
    acc_len[b] = len - 1;
    for (int j = 0; j < path_cap; ++j) acc_path[(int64_t)b * path_cap + j] = j < len ? s_path[j] : -1;
    bonus_out[b] = s_bonus;
  }
}

}  // namespace

int sv_accept(int mode, const void *logits, int dtype, int batch, int n_nodes, int vocab,
              const int32_t *tok, const int32_t *parents, const int32_t *first_child,
              const int32_t *next_sibling, float temperature, float eps, float delta,
              uint64_t seed, uint64_t step, int path_cap, int32_t *acc_len, int32_t *acc_path,
              int32_t *bonus, int32_t *status, cudaStream_t stream) {
  if (dtype == SPEC_BF16)
    accept_kernel<__nv_bfloat16><<<batch, kThreads, 0, stream>>>(
        mode, (const __nv_bfloat16 *)logits, n_nodes, vocab, tok, parents, first_child,
        next_sibling, temperature, eps, delta, seed, step, path_cap, acc_len, acc_path, bonus,
        status);
  else
    accept_kernel<float><<<batch, kThreads, 0, stream>>>(
        mode, (const float *)logits, n_nodes, vocab, tok, parents, first_child, next_sibling,
        temperature, eps, delta, seed, step, path_cap, acc_len, acc_path, bonus, status);
  return sv_launch_status();
}
