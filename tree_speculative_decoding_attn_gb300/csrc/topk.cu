// Top-s candidate selection and one confidence-product expansion round.
//
// "Medusa and EAGLE ... explained", section "Medusa: heads, losses and
// trees": head k contributes its top s_k tokens to the tree.
// "5.3 Medusa、EAGLE 与 MTP", section 5.2: a node's value is the product of
// draft confidences on its path; expansion grows the highest-value nodes.
//
// Selection order everywhere: larger value first, equal values by lower
// index -- one 64-bit key per element (value bits made order-preserving in
// the high word, the complemented index in the low word), so every
// comparison is a single integer max.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxS = 16;  // largest s / k (per-thread sorted list length)

// Bitonic sorting network on S keys (S a power of two), descending: every
// stage is S/2 independent compare-exchanges.
template <int S>
__device__ __forceinline__ void bitonic_sort_desc(unsigned long long (&a)[S]) {
#pragma unroll
  for (int k = 2; k <= S; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
      for (int i = 0; i < S; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const unsigned long long x = a[i], y = a[l];
          const bool sw = (i & k) == 0 ? x < y : x > y;
          a[i] = sw ? y : x;
          a[l] = sw ? x : y;
        }
      }
}
// Sorts a bitonic sequence of S keys descending.
template <int S>
__device__ __forceinline__ void bitonic_merge_desc(unsigned long long (&a)[S]) {
#pragma unroll
  for (int j = S >> 1; j > 0; j >>= 1)
#pragma unroll
    for (int i = 0; i < S; ++i) {
      const int l = i ^ j;
      if (l > i) {
        const unsigned long long x = a[i], y = a[l];
        a[i] = x > y ? x : y;
        a[l] = x > y ? y : x;
      }
    }
}
// Folds a batch of S keys (any order; consumed) into the sorted top-S list:
// the batch is sorted, the pairwise maxima of the list and the reversed
// batch form a bitonic sequence holding the top S of both, which is sorted.
template <int S>
__device__ __forceinline__ void fold_batch(unsigned long long (&best)[S], unsigned long long (&c)[S], bool first) {
  bitonic_sort_desc<S>(c);
  if (first) {
#pragma unroll
    for (int i = 0; i < S; ++i) best[i] = c[i];
    return;
  }
#pragma unroll
  for (int i = 0; i < S; ++i) best[i] = best[i] > c[S - 1 - i] ? best[i] : c[S - 1 - i];
  bitonic_merge_desc<S>(best);
}

// Top-s of the CTA from the per-thread sorted lists (keys are unique; 0 =
// empty).  Each warp takes its own top-s by s warp-wide maxima of the list
// heads, the winning lane popping its head (no block barrier per round);
// then the kWarps * s warp winners are ranked by counting the larger ones.
// out[0..s) in shared memory, descending; contains __syncthreads.
template <int S>
__device__ void merge_top(unsigned long long (&best)[S], int s, unsigned long long *out) {
  __shared__ unsigned long long cand[kWarps][S];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int r = 0; r < s; ++r) {
    const unsigned long long w = sv::warp_max_u64_redux(best[0]);
    if (lane == 0) cand[warp][r] = w;
    if (w != 0ull && best[0] == w) {
#pragma unroll
      for (int j = 0; j < S - 1; ++j) best[j] = best[j + 1];
      best[S - 1] = 0ull;
    }
  }
  if (threadIdx.x < s) out[threadIdx.x] = 0ull;
  __syncthreads();
  if (threadIdx.x < kWarps * s) {
    const unsigned long long k = cand[threadIdx.x / s][threadIdx.x % s];
    int rank = 0;
    for (int w = 0; w < kWarps; ++w)
      for (int r = 0; r < s; ++r) rank += cand[w][r] > k;
    if (k != 0ull && rank < s) out[rank] = k;
  }
  __syncthreads();
}

// Top-s of one row by a cluster of kCluster CTAs: CTA c ranks the c-th slice
// of the row, then CTA 0 gathers the kCluster candidate lists through
// distributed shared memory and keeps the s best (keys are unique, so a
// key's rank is the number of larger keys).
constexpr int kCluster = 8;

__device__ __forceinline__ uint64_t ld_cluster_u64(const void *local, uint32_t cta) {
  uint32_t remote;
  uint64_t v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(sv::ptx_smem(local)), "r"(cta));
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(remote) : "memory");
  return v;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <typename T, int S>
__global__ void __launch_bounds__(kThreads)
    topk_cluster_kernel(const T *__restrict__ rows, int row_len, int64_t row_stride, int s,
                        int32_t *__restrict__ idx, float *__restrict__ val) {
  __shared__ unsigned long long top[32];
  __shared__ unsigned long long all[kCluster * S];
  const uint32_t cta = blockIdx.x;  // rank within the cluster (cluster spans x)
  const int slice = ((row_len + kCluster - 1) / kCluster + 7) / 8 * 8;
  const int lo = min(row_len, (int)cta * slice), hi = min(row_len, lo + slice);
  unsigned long long best[S];
#pragma unroll
  for (int j = 0; j < S; ++j) best[j] = 0ull;
  const T *row = rows + (int64_t)blockIdx.y * row_stride;
  // batches of S keys per thread (coalesced: element lo + threadIdx.x + j kThreads)
  for (int base = lo + threadIdx.x; base < hi; base += S * kThreads) {
    unsigned long long c[S];
#pragma unroll
    for (int j = 0; j < S; ++j) {
      const int x = base + j * kThreads;
      c[j] = x < hi ? sv::rank_key(sv::to_f32(row[x]), (uint32_t)x) : 0ull;
    }
    fold_batch<S>(best, c, base == lo + (int)threadIdx.x);
  }
  merge_top<S>(best, s, top);  // top[0..s) of this slice (0 = empty)
  cluster_barrier();
  if (cta == 0) {
    for (int e = threadIdx.x; e < kCluster * s; e += kThreads) all[e] = ld_cluster_u64(&top[e % s], e / s);
    __syncthreads();
    for (int e = threadIdx.x; e < kCluster * s; e += kThreads) {
      const unsigned long long k = all[e];
      int rank = 0;
      for (int f = 0; f < kCluster * s; ++f) rank += all[f] > k;
      if (k != 0ull && rank < s) {
        idx[(int64_t)blockIdx.y * s + rank] = (int32_t)sv::key_index(k);
        if (val) val[(int64_t)blockIdx.y * s + rank] = sv::key_value(k);
      }
    }
  }
  cluster_barrier();  // remote reads done before any CTA of the cluster exits
}

// ---------------------------------------------------------------------------
// Expansion round, part 1: one cluster of kExpandCluster CTAs per (sequence,
// frontier node) row.  CTA c reads the c-th slice of the draft row once,
// keeping its top-k keys and the online softmax statistics (running max of
// z = logit / T and the sum of exp(z - max)); CTA 0 merges the slices'
// lists and statistics through distributed shared memory and appends the k
// children (token, probability, path value) to the pool.
// ---------------------------------------------------------------------------
constexpr int kExpandCluster = 4;  // 4, 2 and 8 CTAs per row measured within 10 %; 4 fastest

struct Soft {
  float m, s;  // max of z, sum of exp(z - m)
};
__device__ __forceinline__ Soft soft_merge(Soft a, Soft b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return Soft{m, 0.f};
  return Soft{m, (a.m == -INFINITY ? 0.f : a.s * expf(a.m - m)) + (b.m == -INFINITY ? 0.f : b.s * expf(b.m - m))};
}

// A warp's top list: lanes 0..15 hold the 16 largest keys offered so far
// (descending; 0 = empty), lanes 16..31 hold 0; the k-th entry (k <= 16) is
// the admission threshold.  warp_offer offers one key per lane.  No lane
// beating the threshold -- the common case -- costs one compare and one
// ballot.  A few lanes are inserted one at a time (a ballot finds the
// position, a shuffle shifts the tail).  Many lanes (the first offers, while
// the list fills) are sorted across the warp by a bitonic network and merged
// with the list: the larger of entry i and batch entry 15 - i form a bitonic
// sequence holding the top 16 of both, which a bitonic merge sorts.
struct WarpTop {
  unsigned long long l = 0ull;   // this lane's entry
  unsigned long long thr = 0ull; // the k-th entry (warp-uniform)
  float thr_v = -INFINITY;       // its value (-inf while the list is not full)
};
__device__ __forceinline__ unsigned long long u64max(unsigned long long a, unsigned long long b) { return a > b ? a : b; }
__device__ __forceinline__ unsigned long long u64min(unsigned long long a, unsigned long long b) { return a > b ? b : a; }
__device__ __forceinline__ void warp_offer(WarpTop &w, unsigned long long key, int k) {
  const int lane = threadIdx.x & 31;
  unsigned bal = __ballot_sync(0xffffffffu, key > w.thr);
  if (__popc(bal) > 6) {
    unsigned long long x = key > w.thr ? key : 0ull;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, x, stride);
        const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0 || size == 32);
        x = keep_max ? u64max(x, o) : u64min(x, o);
      }
    const unsigned long long b = __shfl_sync(0xffffffffu, x, (15 - lane) & 31);
    unsigned long long c = lane < 16 ? u64max(w.l, b) : 0ull;
#pragma unroll
    for (int stride = 8; stride > 0; stride >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, c, stride);
      c = (lane & stride) == 0 ? u64max(c, o) : u64min(c, o);
    }
    w.l = c;
    w.thr = __shfl_sync(0xffffffffu, w.l, k - 1);
    w.thr_v = w.thr ? sv::key_value(w.thr) : -INFINITY;
    return;
  }
  while (bal) {
    const int src = __ffs(bal) - 1;
    bal &= bal - 1u;
    const unsigned long long kk = __shfl_sync(0xffffffffu, key, src);
    if (kk <= w.thr) continue;  // (uniform) beaten since the ballot
    const int pos = __popc(__ballot_sync(0xffffffffu, lane < 16 && w.l > kk));
    const unsigned long long up = __shfl_up_sync(0xffffffffu, w.l, 1);
    if (lane > pos && lane < 16) w.l = up;
    if (lane == pos) w.l = kk;
    w.thr = __shfl_sync(0xffffffffu, w.l, k - 1);
    w.thr_v = w.thr ? sv::key_value(w.thr) : -INFINITY;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    expand_rows_kernel(const T *__restrict__ logits, int n_front, int V, const int32_t *frontier,
                       int k, float temp, int32_t *pool_parent, int32_t *pool_tok, float *pool_conf,
                       float *pool_val, const int32_t *pool_count, int pool_cap, int32_t *status) {
  __shared__ unsigned long long cand[kWarps * kMaxS];
  __shared__ unsigned long long top[kMaxS];
  __shared__ unsigned long long all[kExpandCluster * kMaxS];
  __shared__ Soft red[kWarps];
  __shared__ unsigned long long s_soft;  // this CTA's (m, s), read by CTA 0
  __shared__ Soft s_tot;
  const uint32_t cta = blockIdx.x;       // rank in the cluster (cluster spans x)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.y, b = r / n_front, f = r % n_front;
  const int base = pool_count[b];
  // (every CTA of the cluster takes the same branch: same inputs)
  if (base + n_front * k > pool_cap) {
    if (cta == 0 && threadIdx.x == 0) sv::report(status, SPEC_DEV_CAPACITY);
    return;
  }
  const int src = frontier[(int64_t)b * n_front + f];
  if (src < 0 || src >= base) {
    if (cta == 0 && threadIdx.x == 0) sv::report(status, SPEC_DEV_BAD_POOL);
    return;
  }
  const T *row = logits + (int64_t)r * V;
  const int slice = ((V + kExpandCluster - 1) / kExpandCluster + 7) / 8 * 8;
  const int lo = min(V, (int)cta * slice), hi = min(V, lo + slice);
  const float inv_t = 1.f / temp;
  WarpTop wt;
  Soft st{-INFINITY, 0.f};
  // every lane of a warp calls visit together (key 0 and z = -inf: no element)
  // The list's k-th value as a float prefilter (-inf while the list is not
  // full): a lane's elements are offered only when one of them reaches it.
  // n values of one lane (warp-uniform call): the top-k offers, then the
  // online statistics moved once to the group's max (fast exponentials: the
  // normaliser is a sum of many positive terms)
  auto visit_group = [&](bool in, int x, const float *v, auto n_c) {
    constexpr int n = decltype(n_c)::value;
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < n; ++e) mx = fmaxf(mx, v[e]);
    if (__any_sync(0xffffffffu, in && mx >= wt.thr_v)) {
#pragma unroll
      for (int e = 0; e < n; ++e) {
        const bool c = in && v[e] >= wt.thr_v;
        warp_offer(wt, c ? sv::rank_key(v[e], (uint32_t)(x + e)) : 0ull, k);
      }
    }
    if (!in) return;
    const float zmax = mx * inv_t;
    if (zmax > st.m) {
      st.s = st.m == -INFINITY ? 0.f : st.s * __expf(st.m - zmax);
      st.m = zmax;
    }
    if (st.m == -INFINITY) return;  // every value so far is -inf
    float add = 0.f;
#pragma unroll
    for (int e = 0; e < n; ++e) add += __expf(fmaf(v[e], inv_t, -st.m));
    st.s += add;
  };
  constexpr int kVec = 16 / sizeof(T);
  constexpr int kUnroll = sizeof(T) == 2 ? 2 : 4;
  int vec_end = lo;
  if ((reinterpret_cast<uintptr_t>(row + lo) & 15) == 0) {
    vec_end = lo + (hi - lo) / kVec * kVec;
    // several 16-byte loads in flight per thread; warp-uniform trip count
    for (int x0 = lo + (int)threadIdx.x * kVec; __any_sync(0xffffffffu, x0 < vec_end);
         x0 += kUnroll * kThreads * kVec) {
      uint4 u[kUnroll];
#pragma unroll
      for (int q = 0; q < kUnroll; ++q) {
        const int x = x0 + q * kThreads * kVec;
        u[q] = x < vec_end ? sv::ldg_stream(row + x) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < kUnroll; ++q) {
        const int x = x0 + q * kThreads * kVec;
        float v[kVec];
        if constexpr (sizeof(T) == 2) {
          sv::bf16x8_to_f32(u[q], v);
        } else {
          v[0] = __uint_as_float(u[q].x);
          v[1] = __uint_as_float(u[q].y);
          v[2] = __uint_as_float(u[q].z);
          v[3] = __uint_as_float(u[q].w);
        }
        visit_group(x < vec_end, x, v, std::integral_constant<int, kVec>{});
      }
    }
  }
  for (int x = vec_end + (int)threadIdx.x; __any_sync(0xffffffffu, x < hi); x += kThreads) {
    const float v = x < hi ? sv::to_f32(row[x]) : 0.f;
    visit_group(x < hi, x, &v, std::integral_constant<int, 1>{});
  }
  // the CTA's statistics (warps in order) and its top-k (rank by counting)
#pragma unroll
  for (int o = 16; o; o >>= 1) st = soft_merge(st, Soft{__shfl_xor_sync(0xffffffffu, st.m, o),
                                                         __shfl_xor_sync(0xffffffffu, st.s, o)});
  if (lane == 0) red[warp] = st;
  if (lane < k) cand[warp * k + lane] = wt.l;
  if (threadIdx.x < k) top[threadIdx.x] = 0ull;
  __syncthreads();
  if (threadIdx.x < kWarps * k) {
    const unsigned long long key = cand[threadIdx.x];
    int rank = 0;
    for (int e = 0; e < kWarps * k; ++e) rank += cand[e] > key;
    if (key != 0ull && rank < k) top[rank] = key;
  }
  if (threadIdx.x == 0) {
    Soft t = red[0];
    for (int w = 1; w < kWarps; ++w) t = soft_merge(t, red[w]);
    s_soft = ((unsigned long long)__float_as_uint(t.s) << 32) | __float_as_uint(t.m);
  }
  cluster_barrier();
  if (cta == 0) {
    for (int e = threadIdx.x; e < kExpandCluster * k; e += kThreads) all[e] = ld_cluster_u64(&top[e % k], e / k);
    if (threadIdx.x == 0) {
      Soft t{-INFINITY, 0.f};
      for (int c = 0; c < kExpandCluster; ++c) {
        const unsigned long long w = ld_cluster_u64(&s_soft, c);
        t = soft_merge(t, Soft{__uint_as_float((uint32_t)w), __uint_as_float((uint32_t)(w >> 32))});
      }
      s_tot = t;
    }
    __syncthreads();
    const Soft t = s_tot;
    for (int e = threadIdx.x; e < kExpandCluster * k; e += kThreads) {
      const unsigned long long key = all[e];
      int rank = 0;
      for (int g = 0; g < kExpandCluster * k; ++g) rank += all[g] > key;
      if (key == 0ull || rank >= k) continue;
      const int x = (int)sv::key_index(key);
      const float p = expf(sv::key_value(key) * inv_t - t.m) / t.s;
      const int64_t slot = (int64_t)b * pool_cap + base + f * k + rank;
      pool_parent[slot] = src;
      pool_tok[slot] = x;
      pool_conf[slot] = p;
      pool_val[slot] = __fmul_rn(pool_val[(int64_t)b * pool_cap + src], p);
    }
  }
  cluster_barrier();  // remote reads done before any CTA of the cluster exits
}

// Part 2: one CTA per sequence ranks the n_front * k new children by
// (value desc, pool index asc), writes the next frontier, bumps the count.
__global__ void __launch_bounds__(1024)
    expand_select_kernel(int n_new, const float *__restrict__ pool_val, int32_t *pool_count,
                         int pool_cap, int32_t *next_frontier, int n_next) {
  __shared__ unsigned long long keys[1024];
  const int b = blockIdx.x;
  const int base = pool_count[b];
  if (base + n_new > pool_cap) return;  // reported by part 1
  const int t = threadIdx.x;
  if (t < n_new) {
    const float v = pool_val[(int64_t)b * pool_cap + base + t];
    keys[t] = ((unsigned long long)(0xFFFFFFFFu - (__float_as_uint(v) & 0x7FFFFFFFu)) << 32) |  // v >= 0
              (unsigned)(base + t);
  }
  __syncthreads();
  if (t < n_new) {
    int r = 0;
    for (int j = 0; j < n_new; ++j) r += keys[j] < keys[t];
    if (r < n_next) next_frontier[(int64_t)b * n_next + r] = base + t;
  }
  for (int r = n_new + t; r < n_next; r += blockDim.x) next_frontier[(int64_t)b * n_next + r] = -1;
  __syncthreads();
  if (t == 0) pool_count[b] = base + n_new;
}

template <typename T, int S>
int launch_topk(const void *rows, int n_rows, int row_len, int row_stride, int s, int32_t *idx, float *val,
                cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCluster, n_rows);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel<T, S>, (const T *)rows, row_len, (int64_t)row_stride, s,
                            idx, val) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

}  // namespace

int sv_topk(const void *rows, int dtype, int n_rows, int row_len, int row_stride, int s,
            int32_t *idx, float *val, cudaStream_t stream) {
  if (s > kMaxS) return SPEC_ERR_UNSUPPORTED;
  // per-thread lists no longer than needed: s rounded up to 4, 8 or 16
  if (dtype == SPEC_BF16) {
    if (s <= 4) return launch_topk<__nv_bfloat16, 4>(rows, n_rows, row_len, row_stride, s, idx, val, stream);
    if (s <= 8) return launch_topk<__nv_bfloat16, 8>(rows, n_rows, row_len, row_stride, s, idx, val, stream);
    return launch_topk<__nv_bfloat16, kMaxS>(rows, n_rows, row_len, row_stride, s, idx, val, stream);
  }
  if (s <= 4) return launch_topk<float, 4>(rows, n_rows, row_len, row_stride, s, idx, val, stream);
  if (s <= 8) return launch_topk<float, 8>(rows, n_rows, row_len, row_stride, s, idx, val, stream);
  return launch_topk<float, kMaxS>(rows, n_rows, row_len, row_stride, s, idx, val, stream);
}

int sv_tree_expand(const void *logits, int dtype, int batch, int n_front, int vocab,
                   const int32_t *frontier, int k, float temperature, int32_t *pool_parent,
                   int32_t *pool_tok, float *pool_conf, float *pool_val, int32_t *pool_count,
                   int pool_cap, int32_t *next_frontier, int n_next, int32_t *status,
                   cudaStream_t stream) {
  if (k > kMaxS) return SPEC_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kExpandCluster, batch * n_front);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kExpandCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      dtype == SPEC_BF16
          ? cudaLaunchKernelEx(&cfg, expand_rows_kernel<__nv_bfloat16>, (const __nv_bfloat16 *)logits, n_front,
                               vocab, frontier, k, temperature, pool_parent, pool_tok, pool_conf, pool_val, pool_count,
                               pool_cap, status)
          : cudaLaunchKernelEx(&cfg, expand_rows_kernel<float>, (const float *)logits, n_front, vocab, frontier,
                               k, temperature, pool_parent, pool_tok, pool_conf, pool_val, pool_count, pool_cap,
                               status);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  expand_select_kernel<<<batch, 1024, 0, stream>>>(n_front * k, pool_val, pool_count, pool_cap,
                                                   next_frontier, n_next);
  return sv_launch_status();
}
