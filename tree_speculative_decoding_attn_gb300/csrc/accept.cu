// Acceptance of the longest target-agreeing path and the bonus token.
//
// Greedy: "Drafters: draft models, Medusa, EAGLE, MTP, DFlash, DSpark",
// section "Why the answer does not change" (keep a draft only if it is the
// target's own pick; at the first disagreement use the target's token);
// "Medusa, explained", step 7.  Typical: "Medusa, explained", section
// "Typical acceptance" (p(x) > min(eps, delta exp(-H)); the step's first
// token is the greedy one).  Rejection: "Drafters: ...", same section
// (min(1, p/q); on rejection sample the target minus the drafter), with
// the point-mass proposal of a deterministic tree sibling, or with siblings
// drawn from the drafter's distribution q at their parent (SpecInfer-style
// multi-draft verification, "Medusa and EAGLE ... explained", section
// "Medusa: heads, losses and trees").
//
// One cluster of nc CTAs per sequence (16 at batch < 16, 8 below 32, else
// 4).  The cluster walks the tree from the root: each visited node's
// vocabulary row is reduced in slices (CTA c reduces the c-th slice with
// 16-byte loads), the nc partial results are exchanged through distributed
// shared memory and combined in the same fixed order in every CTA, so all
// CTAs hold the same totals and take the same decisions without a
// broadcast.  Only the rows on the walk are read (plus, for typical
// acceptance, the rows of every node reachable through valid children).
// The softmax statistics of a row (max, sum of exponentials and, for the
// entropy, their first moment) come from one online pass.  A node's
// children are examined by one warp in parallel; only the rejection rule's
// residual bookkeeping runs serially, on values already in shared memory.
#include <float.h>
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxNodes = SPEC_MAX_NODES;

// Softmax statistics of a set of scaled logits z: m = max z, S = sum
// exp(z - m), Q = sum exp(z - m) (z - m).  S == 0 marks the empty set.
struct Stats {
  float m, S, Q;
};
__device__ __forceinline__ Stats stats_empty() { return Stats{-FLT_MAX, 0.f, 0.f}; }
// The union of two disjoint sets: both are brought to the larger max
// (exp(z - m') = exp(m - m') exp(z - m), and z - m' = (z - m) + (m - m')).
__device__ __forceinline__ Stats stats_merge(Stats a, Stats b) {
  if (!(b.S > 0.f)) return a;
  if (!(a.S > 0.f)) return b;
  const float mn = fmaxf(a.m, b.m), da = a.m - mn, db = b.m - mn;
  const float ea = __expf(da), eb = __expf(db);
  return Stats{mn, fmaf(ea, a.S, eb * b.S), fmaf(ea, fmaf(da, a.S, a.Q), eb * fmaf(db, b.S, b.Q))};
}
// One more element z (kQ: keep the first moment as well).
template <bool kQ>
__device__ __forceinline__ void stats_add(Stats &s, float z) {
  if (z > s.m) {  // new max: rescale what is there
    if (s.S > 0.f) {
      const float d = s.m - z, e = __expf(d);
      if (kQ) s.Q = e * fmaf(d, s.S, s.Q);
      s.S *= e;
    }
    s.m = z;
  }
  const float d = z - s.m, e = __expf(d);
  s.S += e;
  if (kQ) s.Q = fmaf(e, d, s.Q);
}
__device__ __forceinline__ Stats shfl_stats(Stats s, int o) {
  return Stats{__shfl_xor_sync(0xffffffffu, s.m, o), __shfl_xor_sync(0xffffffffu, s.S, o),
               __shfl_xor_sync(0xffffffffu, s.Q, o)};
}
// Butterfly over a warp.  Lane 0 ends with the union of all lanes' sets,
// combined in a fixed order: warps holding the same inputs get the same
// lane-0 value bit for bit (other lanes may differ in rounding).
__device__ __forceinline__ Stats warp_stats(Stats s) {
#pragma unroll
  for (int o = 16; o; o >>= 1) s = stats_merge(s, shfl_stats(s, o));
  return s;
}

struct Red {
  Stats ws[kWarps];              // per-warp partials
  unsigned long long wu[kWarps];
  // cluster exchange slots, double-buffered by reduction parity: a slot is
  // rewritten two reductions later, after every CTA has passed the barrier
  // that follows its last read of it
  Stats xs[2];
  unsigned long long xu[2];
  Stats cs;                      // the cluster's result
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

// Cluster-wide reductions: every CTA gets the identical result.  Warp
// partials go through shared memory to warp 0, which combines them, posts
// the CTA's partial, and after the cluster barrier reads all nc partials
// at once (lane c reads CTA c) and combines them by the same butterfly in
// every CTA.  All threads of all CTAs must call them together.
struct ClusterOps {
  Red &r;
  int parity;
  uint32_t nc;  // CTAs in the cluster (<= 32)

  __device__ Stats stats(Stats s) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    s = warp_stats(s);
    if (lane == 0) r.ws[w] = s;
    __syncthreads();
    if (w == 0) {
      Stats c = lane < kWarps ? r.ws[lane] : stats_empty();
      c = warp_stats(c);
      if (lane == 0) r.xs[parity] = c;
    }
    cluster_barrier();
    if (w == 0) {
      Stats c = stats_empty();
      if (lane < (int)nc)
        c = Stats{ld_remote_f32(&r.xs[parity].m, lane), ld_remote_f32(&r.xs[parity].S, lane),
                  ld_remote_f32(&r.xs[parity].Q, lane)};
      c = warp_stats(c);
      if (lane == 0) r.cs = c;
    }
    __syncthreads();
    const Stats out = r.cs;
    parity ^= 1;
    return out;
  }
  __device__ unsigned long long max_u64(unsigned long long v) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = sv::warp_max_u64_redux(v);
    if (lane == 0) r.wu[w] = v;
    __syncthreads();
    if (w == 0) {
      unsigned long long c = lane < kWarps ? r.wu[lane] : 0ull;
      c = sv::warp_max_u64_redux(c);
      if (lane == 0) r.xu[parity] = c;
    }
    cluster_barrier();
    if (w == 0) {
      unsigned long long c = lane < (int)nc ? ld_remote_u64(&r.xu[parity], lane) : 0ull;
      c = sv::warp_max_u64_redux(c);
      if (lane == 0) r.cu = c;
    }
    __syncthreads();
    const unsigned long long out = r.cu;
    parity ^= 1;
    return out;
  }
};

// Visit this CTA's slice [lo, hi) of a logits row.  Where the slice start
// is 16-byte aligned and its length a multiple of the vector width, fv(x0,
// v) gets kVec consecutive values from column x0 (x0 a multiple of kVec,
// since lo is a multiple of 8); loads are issued kBatch at a time per
// thread before any is used, so a CTA keeps kThreads * kBatch * 16 bytes in
// flight (kB loads, for a caller that needs registers for its own work).
// Otherwise f1(x, value) gets one column at a time.
constexpr int kBatch = 8;
template <int kB = kBatch, typename T, typename FV, typename F1>
__device__ __forceinline__ void for_slice_v(const T *row, int lo, int hi, FV &&fv, F1 &&f1) {
  constexpr int kVec = 16 / sizeof(T);
  if (((hi - lo) % kVec) == 0 && (reinterpret_cast<uintptr_t>(row + lo) & 15) == 0) {
    const int nv = (hi - lo) / kVec;
    const uint4 *src = reinterpret_cast<const uint4 *>(row + lo);
    for (int v0 = threadIdx.x; v0 < nv; v0 += kB * kThreads) {
      uint4 u[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        const int vi = v0 + i * kThreads;
        u[i] = vi < nv ? src[vi] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < kB; ++i) {
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
        fv(lo + vi * kVec, v);
      }
    }
  } else {
    for (int x = lo + threadIdx.x; x < hi; x += kThreads) f1(x, sv::to_f32(row[x]));
  }
}
template <typename T, typename F>
__device__ __forceinline__ void for_slice(const T *row, int lo, int hi, F &&f) {
  constexpr int kVec = 16 / sizeof(T);
  for_slice_v(
      row, lo, hi,
      [&](int x0, const float *v) {
#pragma unroll
        for (int j = 0; j < kVec; ++j) f(x0 + j, v[j]);
      },
      f);
}
// The first column this thread visits in for_slice_v (hi if none).
template <typename T>
__device__ __forceinline__ int first_column(const T *row, int lo, int hi) {
  constexpr int kVec = 16 / sizeof(T);
  const bool vec = ((hi - lo) % kVec) == 0 && (reinterpret_cast<uintptr_t>(row + lo) & 15) == 0;
  return min(hi, lo + (int)threadIdx.x * (vec ? kVec : 1));
}

// Visit this CTA's slice of two rows at the same columns (two rows of one
// [.., V] layout: equal alignment): f(x, a[x], b[x]).
template <typename T, typename F>
__device__ __forceinline__ void for_slice2(const T *ra, const T *rb, int lo, int hi, F &&f) {
  constexpr int kVec = 16 / sizeof(T);
  if (((hi - lo) % kVec) == 0 && (reinterpret_cast<uintptr_t>(ra + lo) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(rb + lo) & 15) == 0) {
    const int nv = (hi - lo) / kVec;
    const uint4 *sa = reinterpret_cast<const uint4 *>(ra + lo);
    const uint4 *sb = reinterpret_cast<const uint4 *>(rb + lo);
    for (int vi = threadIdx.x; vi < nv; vi += kThreads) {
      const uint4 ua = sa[vi], ub = sb[vi];
      float a[kVec], c[kVec];
      if constexpr (sizeof(T) == 2) {
        sv::bf16x8_to_f32(ua, a);
        sv::bf16x8_to_f32(ub, c);
      } else {
        a[0] = __uint_as_float(ua.x); a[1] = __uint_as_float(ua.y);
        a[2] = __uint_as_float(ua.z); a[3] = __uint_as_float(ua.w);
        c[0] = __uint_as_float(ub.x); c[1] = __uint_as_float(ub.y);
        c[2] = __uint_as_float(ub.z); c[3] = __uint_as_float(ub.w);
      }
#pragma unroll
      for (int j = 0; j < kVec; ++j) f(lo + vi * kVec + j, a[j], c[j]);
    }
  } else {
    for (int x = lo + threadIdx.x; x < hi; x += kThreads) f(x, sv::to_f32(ra[x]), sv::to_f32(rb[x]));
  }
}

// Uniform in (0, 1) for the sampling race from a 32-bit Philox word:
// ((w >> 9) + 1/2) 2^-23, exact in float32.
__device__ __forceinline__ float race_uniform(uint32_t w) {
  return ((float)(w >> 9) + 0.5f) * 1.1920928955078125e-7f;
}
// Race key z + G, G = -log(-log u) a Gumbel variate.  The inner log keeps
// full precision (u near 1 gives the largest G); the outer one takes the
// fast log, whose absolute error is far below the keys' spacing.
__device__ __forceinline__ float race_key(float z, uint32_t w) {
  return z - __logf(-logf(race_uniform(w)));
}

// Two CTAs per SM (<= 64 registers), so that 4-CTA clusters of a batch
// of 64 are all resident in one wave.
template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
    accept_kernel(int mode, const T *__restrict__ logits, const T *__restrict__ draft, int N, int V,
                  const int32_t *__restrict__ tok, const int32_t *__restrict__ parents,
                  const int32_t *__restrict__ first_child, const int32_t *__restrict__ next_sibling,
                  float temp, float eps, float delta, uint64_t seed, uint64_t step, int path_cap,
                  int32_t *acc_len, int32_t *acc_path, int32_t *bonus_out, int32_t *status, const SvCommit cm) {
  __shared__ Red red;
  __shared__ int s_path[kMaxNodes + 1];
  __shared__ int s_len, s_next, s_bonus;
  __shared__ int s_fc[kMaxNodes], s_ns[kMaxNodes], s_tok[kMaxNodes], s_par[kMaxNodes];
  __shared__ int s_ok[kMaxNodes], s_depth[kMaxNodes];
  __shared__ int s_kid[kMaxNodes], s_nkid;   // children of the node being examined, in node order
  __shared__ float s_kex[kMaxNodes];         // exp(z - m) of each child's token
  __shared__ float s_ku[kMaxNodes];          // each child's accept draw
  __shared__ float s_kq[kMaxNodes];          // stochastic siblings: q(tok) of each child
  __shared__ int s_exc[kMaxNodes];           // tokens removed from the residual
  __shared__ int s_nexc;

  const uint32_t cta = blockIdx.x;  // rank in the cluster (cluster spans x)
  const int b = blockIdx.y;
  const int nc = (int)gridDim.x;  // the cluster spans x
  const int slice = ((V + nc - 1) / nc + 7) / 8 * 8;
  const int lo = min(V, (int)cta * slice), hi = min(V, lo + slice);
  const int lane = threadIdx.x & 31;
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

  // argmax with ties to the lowest column: each thread keeps its first
  // largest value (it visits columns in increasing order), the cluster
  // takes the largest (value, lowest column) key
  auto row_argmax = [&](const T *row) -> int {
    float best = -INFINITY;
    int bx = first_column(row, lo, hi);
    for_slice(row, lo, hi, [&](int x, float v) {
      if (v > best) {
        best = v;
        bx = x;
      }
    });
    return (int)sv::key_index(cl.max_u64(bx < hi ? sv::rank_key(best, (uint32_t)bx) : 0ull));
  };
  // softmax statistics of z = logits / T over the row, one pass
  auto row_stats = [&](const T *row, auto with_q) -> Stats {
    Stats s = stats_empty();
    for_slice(row, lo, hi, [&](int, float v) { stats_add<decltype(with_q)::value>(s, v * inv_t); });
    return cl.stats(s);
  };
  // node v's children in node order into s_kid (thread 0; bounded walk)
  auto list_children = [&](int v) {
    if (threadIdx.x == 0) {
      int n = 0;
      for (int c = s_fc[v]; c >= 0 && c < N && n < kMaxNodes; c = s_ns[c]) s_kid[n++] = c;
      s_nkid = n;
    }
    __syncthreads();
  };

  if (mode == SPEC_ACCEPT_GREEDY) {
    int v = 0;
    for (int guard = 0; guard < kMaxNodes; ++guard) {
      const int a = row_argmax(base + (int64_t)v * V);
      if (threadIdx.x == 0) {
        int nxt = -1;
        for (int c = s_fc[v], n = 0; c >= 0 && c < N && n < kMaxNodes; c = s_ns[c], ++n)
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
      const Stats s = row_stats(row, std::true_type{});
      list_children(v);
      if (threadIdx.x < 32) {
        const float H = logf(s.S) - s.Q / s.S;
        const float thr = fminf(eps, delta * expf(-H));
        for (int j = lane; j < s_nkid; j += 32) {
          const int c = s_kid[j], x = s_tok[c];
          if (x < 0 || x >= V) {
            sv::report(status, SPEC_DEV_BAD_TOKEN);
            continue;
          }
          const float p = __expf(sv::to_f32(row[x]) * inv_t - s.m) / s.S;
          s_ok[c] = p > thr;
        }
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      int best = 0;
      for (int i = 1; i < N; ++i)
        if (s_ok[i] && s_depth[i] > s_depth[best]) best = i;
      // root-first path of `best` along parents[]: every step must go to an
      // earlier node and end at the root, else parents[] disagrees with the
      // child links (reported; the root alone is accepted)
      const int d = s_depth[best];
      bool good = true;
      for (int u = best, k = d; k >= 0; --k) {
        if (u < 0 || u >= N || (k == 0) != (u == 0)) {
          good = false;
          break;
        }
        s_path[k] = u;
        if (k > 0) {
          const int p = s_par[u];
          if (p < 0 || p >= u) {
            good = false;
            break;
          }
          u = p;
        }
      }
      if (!good) {
        sv::report(status, SPEC_DEV_BAD_PARENTS);
        best = 0;
        s_path[0] = 0;
      }
      s_len = good ? d + 1 : 1;
      s_next = best;
    }
    __syncthreads();
    const int a = row_argmax(base + (int64_t)s_next * V);
    if (threadIdx.x == 0) s_bonus = a;
  } else if (mode == SPEC_ACCEPT_REJECT_STOCHASTIC) {
    const T *qbase = draft + row0 * V;
    int v = 0;
    for (int guard = 0; guard < kMaxNodes; ++guard) {
      const T *row = base + (int64_t)v * V, *qrow = qbase + (int64_t)v * V;
      const Stats sp = row_stats(row, std::false_type{});
      const Stats sq = row_stats(qrow, std::false_type{});
      list_children(v);
      if (threadIdx.x < 32) {
        for (int j = lane; j < s_nkid; j += 32) {
          const int c = s_kid[j], x = s_tok[c];
          const bool ok = x >= 0 && x < V;
          if (!ok) sv::report(status, SPEC_DEV_BAD_TOKEN);
          s_kex[j] = ok ? __expf(sv::to_f32(row[x]) * inv_t - sp.m) / sp.S : 0.f;
          s_kq[j] = ok ? __expf(sv::to_f32(qrow[x]) * inv_t - sq.m) / sq.S : -1.f;  // -1: never accepted
          const sv::u32x4 w = sv::philox4x32_10(sv::u32x4{(uint32_t)c, 0u, (uint32_t)b, st}, k0, k1);
          s_ku[j] = (float)(w.x >> 8) * 5.9604644775390625e-8f;  // 2^-24
        }
      }
      __syncthreads();
      // children in node order; every CTA holds the same shared values and
      // the same cluster sums, so all take the same branch
      float cq = 0.f, D = 1.f;
      int nxt = -1;
      const int nk = s_nkid;
      for (int j = 0; j < nk; ++j) {
        const float pj = s_kex[j], qj = s_kq[j];
        if (qj < 0.f) continue;  // bad token: reported, never accepted, residual unchanged
        // accept iff u < r(x) / q(x); q(x) = 0 (a token the drafter cannot
        // propose) is always kept
        if (!(qj > 0.f) || s_ku[j] * (D * qj) < fmaxf(pj - cq * qj, 0.f)) {
          nxt = s_kid[j];
          break;
        }
        const float c2 = cq + D;
        float part = 0.f;
        for_slice2(row, qrow, lo, hi, [&](int, float zp, float zq) {
          part += fmaxf(__expf(zp * inv_t - sp.m) / sp.S - c2 * (__expf(zq * inv_t - sq.m) / sq.S), 0.f);
        });
        const float D2 = cl.stats(Stats{0.f, part, 0.f}).S;
        if (!(D2 > 0.f)) {  // nothing left (rounding): sample from the target itself
          cq = 0.f;
          D = 1.f;
          break;
        }
        cq = c2;
        D = D2;
      }
      if (threadIdx.x == 0 && nxt >= 0) s_path[s_len++] = nxt;
      if (nxt >= 0) {
        v = nxt;
        __syncthreads();
        continue;
      }
      // residual sample: exponential race argmax_x log r(x) + G over the
      // tokens with r(x) > 0 (same draws as the point-mass rule)
      float bk = -INFINITY;
      int bx = hi;
      for_slice2(row, qrow, lo, hi, [&](int x, float zp, float zq) {
        const float r = __expf(zp * inv_t - sp.m) / sp.S - cq * (__expf(zq * inv_t - sq.m) / sq.S);
        if (!(r > 0.f)) return;
        const sv::u32x4 w =
            sv::philox4x32_10(sv::u32x4{(uint32_t)x >> 2, 256u + (uint32_t)v, (uint32_t)b, st}, k0, k1);
        const uint32_t wx = (x & 2) ? ((x & 1) ? w.w : w.z) : ((x & 1) ? w.y : w.x);
        const float key = race_key(__logf(r), wx);
        if (key > bk) {
          bk = key;
          bx = x;
        }
      });
      const unsigned long long best = cl.max_u64(bx < hi ? sv::rank_key(bk, (uint32_t)bx) : 0ull);
      const int a = best ? (int)sv::key_index(best) : row_argmax(row);  // empty residual: the argmax
      if (threadIdx.x == 0) s_bonus = a;
      __syncthreads();
      break;
    }
  } else {  // SPEC_ACCEPT_REJECT
    int v = 0;
    for (int guard = 0; guard < kMaxNodes; ++guard) {
      const T *row = base + (int64_t)v * V;
      const Stats s = row_stats(row, std::false_type{});
      list_children(v);
      if (threadIdx.x < 32) {
        // every child's exp(z - m) and accept draw, in parallel
        for (int j = lane; j < s_nkid; j += 32) {
          const int c = s_kid[j], x = s_tok[c];
          s_kex[j] = x >= 0 && x < V ? __expf(sv::to_f32(row[x]) * inv_t - s.m) : 0.f;
          const sv::u32x4 w = sv::philox4x32_10(sv::u32x4{(uint32_t)c, 0u, (uint32_t)b, st}, k0, k1);
          s_ku[j] = (float)(w.x >> 8) * 5.9604644775390625e-8f;  // 2^-24
        }
        __syncwarp();
        // the residual's bookkeeping, child after child: accept c iff
        // u < r(tok c); otherwise tok c leaves the residual
        if (lane == 0) {
          int nxt = -1, nexc = 0;
          float removed = 0.f;
          for (int j = 0; j < s_nkid; ++j) {
            const int c = s_kid[j], x = s_tok[c];
            bool seen = false;
            for (int e = 0; e < nexc; ++e) seen |= s_exc[e] == x;
            float r = 0.f;
            if (x < 0 || x >= V) {
              sv::report(status, SPEC_DEV_BAD_TOKEN);
              seen = true;
            } else if (!seen) {
              // the residual's mass is at least this token's own; the last
              // token left in the vocabulary holds all of it
              r = nexc + 1 >= V ? 1.f : s_kex[j] / fmaxf(s.S - removed, s_kex[j]);
            }
            if (s_ku[j] < r) {
              nxt = c;
              break;
            }
            if (!seen) {
              s_exc[nexc++] = x;
              removed = removed + s_kex[j];
            }
          }
          s_nexc = nexc;
          s_next = nxt;
          if (nxt >= 0) s_path[s_len++] = nxt;
        }
      }
      __syncthreads();
      if (s_next >= 0) {
        v = s_next;
        __syncthreads();
        continue;
      }
      // residual sample: exponential race in log form over the tokens not
      // removed.  One Philox call gives the draws of four consecutive
      // tokens: token x uses word x % 4 of counter (x / 4, 256 + v, b, step).
      const int nexc = s_nexc;
      float bk = -INFINITY;
      int bx = hi;
      auto race4 = [&](int x0, const float *z4, unsigned skip) {
        const sv::u32x4 w =
            sv::philox4x32_10(sv::u32x4{(uint32_t)x0 >> 2, 256u + (uint32_t)v, (uint32_t)b, st}, k0, k1);
        const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int l = 0; l < 4; ++l) {
          if ((skip >> l) & 1u) continue;
          const float key = race_key(z4[l] * inv_t, wd[l]);
          if (key > bk) {
            bk = key;
            bx = x0 + l;
          }
        }
      };
      // (four loads in flight: the race's arithmetic hides the latency)
      for_slice_v<4>(
          row, lo, hi,
          [&](int x0, const float *vals) {
            constexpr int kVec = 16 / sizeof(T);
            unsigned skip = 0;  // removed tokens among x0 .. x0 + kVec - 1
            for (int e = 0; e < nexc; ++e) {
              const unsigned d = (unsigned)(s_exc[e] - x0);
              if (d < (unsigned)kVec) skip |= 1u << d;
            }
#pragma unroll
            for (int q = 0; q < kVec / 4; ++q) race4(x0 + 4 * q, vals + 4 * q, skip >> (4 * q));
          },
          [&](int x, float val) {
            for (int e = 0; e < nexc; ++e)
              if (s_exc[e] == x) return;
            const sv::u32x4 w =
                sv::philox4x32_10(sv::u32x4{(uint32_t)x >> 2, 256u + (uint32_t)v, (uint32_t)b, st}, k0, k1);
            const uint32_t wx = (x & 2) ? ((x & 1) ? w.w : w.z) : ((x & 1) ? w.y : w.x);
            const float key = race_key(val * inv_t, wx);
            if (key > bk) {
              bk = key;
              bx = x;
            }
          });
      const unsigned long long best = cl.max_u64(bx < hi ? sv::rank_key(bk, (uint32_t)bx) : 0ull);
      // an empty residual (not reached in exact arithmetic): the row's argmax
      const int a = best ? (int)sv::key_index(best) : row_argmax(row);
      if (threadIdx.x == 0) s_bonus = a;
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
  // the fused commit (kv_commit's copies): the cluster's CTAs share the
  // accepted rows of every (K or V, layer, KV head), 16-byte vectors
  int P = 0, len = 0;
  bool fits = false;
  if (cm.kc) {
    P = cm.prefix_len[b];
    len = min(s_len, path_cap);
    fits = P >= 0 && P + len <= cm.s_max;
    if (cta == 0 && threadIdx.x == 0 && !fits) sv::report(status, SPEC_DEV_CAPACITY);
    if (fits) {
      const int n = len * cm.vec_per_row;  // vectors of one (layer, head) for K or V
      const int total = 2 * cm.n_layers * cm.hkv * n;
      const int nb = (int)gridDim.y;
#pragma unroll 4
      for (int idx = (int)(cta * kThreads + threadIdx.x); idx < total; idx += nc * kThreads) {
        const int it = idx / n, e = idx - it * n;
        const int j = e / cm.vec_per_row, c = e - j * cm.vec_per_row;
        const int lh = it >> 1;  // layer * hkv + head
        const int layer = lh / cm.hkv, h = lh % cm.hkv;
        const int64_t lb = ((int64_t)layer * nb + b) * cm.hkv + h;
        const uint4 v = ((it & 1) ? cm.vt : cm.kt)[(lb * N + s_path[j]) * cm.vec_per_row + c];
        ((it & 1) ? cm.vc : cm.kc)[(lb * cm.s_max + P + j) * cm.vec_per_row + c] = v;
      }
    }
  }
  cluster_barrier();  // partners' reads of this CTA's exchange slots (and of prefix_len) are done
  if (cm.kc && cm.prefix_len_out && cta == 0 && threadIdx.x == 0) cm.prefix_len_out[b] = fits ? P + len : P;
}

// CTAs per sequence (the kernel reads it from gridDim.x): enough to fill
// the GPU at small batch, few enough that every cluster is resident in one
// wave at large batch.  Sixteen is a non-portable cluster size; it is used
// only where the device accepts it for this kernel.
template <typename T>
int cluster_size(int batch) {
  if (batch >= 32) return 4;
  if (batch >= 16) return 8;
  if (cudaFuncSetAttribute(accept_kernel<T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    (void)cudaGetLastError();
    return 8;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16, batch);
  cfg.blockDim = dim3(kThreads);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 16;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxPotentialClusterSize(&n, accept_kernel<T>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 8;
  }
  return n >= 16 ? 16 : 8;
}

template <typename T>
int launch_accept(int mode, const void *logits, const void *draft, int batch, int n_nodes, int vocab,
                  const int32_t *tok,
                  const int32_t *parents, const int32_t *first_child, const int32_t *next_sibling,
                  float temperature, float eps, float delta, uint64_t seed, uint64_t step, int path_cap,
                  int32_t *acc_len, int32_t *acc_path, int32_t *bonus, int32_t *status, cudaStream_t stream,
                  const SvCommit &cm) {
  const int nc = cluster_size<T>(batch);
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
  return cudaLaunchKernelEx(&cfg, accept_kernel<T>, mode, (const T *)logits, (const T *)draft, n_nodes, vocab,
                            tok, parents,
                            first_child, next_sibling, temperature, eps, delta, seed, step, path_cap, acc_len,
                            acc_path, bonus, status, cm) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

}  // namespace

int sv_accept(int mode, const void *logits, const void *draft, int dtype, int batch, int n_nodes, int vocab,
              const int32_t *tok, const int32_t *parents, const int32_t *first_child,
              const int32_t *next_sibling, float temperature, float eps, float delta,
              uint64_t seed, uint64_t step, int path_cap, int32_t *acc_len, int32_t *acc_path,
              int32_t *bonus, int32_t *status, cudaStream_t stream, SvCommit commit) {
  if (dtype == SPEC_BF16)
    return launch_accept<__nv_bfloat16>(mode, logits, draft, batch, n_nodes, vocab, tok, parents, first_child,
                                        next_sibling, temperature, eps, delta, seed, step, path_cap, acc_len,
                                        acc_path, bonus, status, stream, commit);
  return launch_accept<float>(mode, logits, draft, batch, n_nodes, vocab, tok, parents, first_child, next_sibling,
                              temperature, eps, delta, seed, step, path_cap, acc_len, acc_path, bonus, status,
                              stream, commit);
}
