// Tree bookkeeping of the verify pass: depth, ancestor bitmask, depth
// position ids, child links; static (Medusa) token placement and the
// confidence-product rerank (EAGLE-2).
//
// "5.3 Medusa、EAGLE 与 MTP" (infra-guide): section 3.1 (a node sees the
// prefix and its ancestors only), 3.2 (position id = depth; siblings share
// one), 5.2 (path value = product of draft confidences; the best nodes go to
// verification), 8 (parents array with parent < node, ancestor walk).
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kMaxNodes = SPEC_MAX_NODES;

// Emits depth/pos/mask/child links for one sequence's parents array held in
// shared memory, with kids[v * MW + w] = word w of the set of v's children
// (MW words of 64 bits; trees of up to 64 * MW nodes).  The ancestor mask of
// node i is written as `nw` = ceil(N / 64) words.  One thread per node; the
// walk is bounded because the caller validated parent < node.
template <int MW>
__device__ void emit_tree_arrays(const int *par, const unsigned long long *kids, int i, int nw, int prefix,
                                 int64_t row, int32_t *depth, int32_t *pos, uint64_t *anc,
                                 int32_t *first_child, int32_t *next_sibling, int *depth_out) {
  uint64_t m[MW];
#pragma unroll
  for (int w = 0; w < MW; ++w) m[w] = 0;
  int d = -1;
  for (int c = i; c != -1; c = par[c]) {
#pragma unroll
    for (int w = 0; w < MW; ++w)
      if ((c >> 6) == w) m[w] |= 1ull << (c & 63);
    ++d;
  }
  // first child: the lowest child; next sibling: the parent's lowest child above i
  int fc = -1;
#pragma unroll
  for (int w = MW - 1; w >= 0; --w)
    if (kids[i * MW + w]) fc = w * 64 + __ffsll((long long)kids[i * MW + w]) - 1;
  int ns = -1;
  if (i > 0 && par[i] >= 0) {
    const int p = par[i];
#pragma unroll
    for (int w = MW - 1; w >= 0; --w) {
      const int lo = i + 1 - w * 64;  // first bit of word w above i
      const unsigned long long k = kids[p * MW + w];
      const unsigned long long later = lo <= 0 ? k : lo >= 64 ? 0ull : k & (~0ull << lo);
      if (later) ns = w * 64 + __ffsll((long long)later) - 1;
    }
  }
  depth[row + i] = d;
  pos[row + i] = prefix + d;
  for (int w = 0; w < nw; ++w) anc[(row + i) * nw + w] = w < MW ? m[w] : 0ull;
  first_child[row + i] = fc;
  next_sibling[row + i] = ns;
  *depth_out = d;
}

// One CTA per sequence.  parents: shared [N] (par_stride 0) or per sequence
// [batch, N] (par_stride N).  n_valid (optional, [batch]): nodes at and past
// it are absent (a smaller tree padded to N): they are nobody's child and
// get depth 0, position prefix_len, a mask of themselves and no links.
// Tokens: tok_in [batch, N] copied when given, else the static candidate
// table (cand_tok), else not written.
template <int MW>
__global__ void __launch_bounds__(64 * MW)
    build_static_kernel(const int32_t *__restrict__ parents, int par_stride, const int32_t *__restrict__ n_valid,
                        const int32_t *__restrict__ tok_in, const int32_t *__restrict__ rank,
                        const int32_t *__restrict__ cand_tok, int cand_levels, int cand_s,
                        const int32_t *__restrict__ root_tok, const int32_t *__restrict__ prefix_len,
                        int N, int32_t *tok, int32_t *depth, int32_t *pos, uint64_t *anc,
                        int32_t *first_child, int32_t *next_sibling, int32_t *status) {
  __shared__ int par[64 * MW];
  __shared__ unsigned long long kids[64 * MW * MW];
  __shared__ int bad;
  const int b = blockIdx.x, i = threadIdx.x;
  // every load that does not depend on the tree walk is issued up front
  const int nv = n_valid ? n_valid[b] : N;
  const int p = i < N ? parents[(int64_t)b * par_stride + i] : 0;
  const int P = prefix_len[b];
  const int r = tok && !tok_in && i > 0 && i < N ? rank[i] : 0;
  const int t0 = tok && !tok_in && i == 0 ? root_tok[b] : -1;
  const int tin = tok && tok_in && i < N ? tok_in[(int64_t)b * N + i] : -1;
  if (i == 0) bad = nv < 1 || nv > N;
#pragma unroll
  for (int w = 0; w < MW; ++w) kids[i * MW + w] = 0ull;
  __syncthreads();
  if (i < N) {
    par[i] = i < nv ? p : -1;
    if (i >= nv) {
      // absent node
    } else if (i == 0 ? p != -1 : (p < 0 || p >= i)) {
      atomicOr(&bad, 1);
    } else if (i > 0) {
      atomicOr(&kids[p * MW + (i >> 6)], 1ull << (i & 63));
    }
  }
  __syncthreads();
  if (bad) {
    if (i == 0) sv::report(status, SPEC_DEV_BAD_PARENTS);
    return;
  }
  if (i >= N) return;
  const int64_t row = (int64_t)b * N;
  int d;
  emit_tree_arrays<MW>(par, kids, i, (N + 63) >> 6, P, row, depth, pos, anc, first_child, next_sibling, &d);
  if (tok && tok_in) {
    tok[row + i] = tin;
  } else if (tok) {
    int t = -1;
    if (i == 0) {
      t = t0;
    } else if (i >= nv) {
      t = -1;
    } else {
      if (d - 1 < cand_levels && r >= 0 && r < cand_s)
        t = cand_tok[((int64_t)b * cand_levels + (d - 1)) * cand_s + r];
      else
        sv::report(status, SPEC_DEV_BAD_PARENTS);
    }
    tok[row + i] = t;
  }
}

// ---------------------------------------------------------------------------
// Confidence-product rerank.  One CTA per sequence.
//   1. val[i] = val[parent] * conf[i] in root-to-node order (float32).
//   2. the pool sorted by (val desc, depth asc, index asc); the n first
//      nodes are kept (the root comes first).
//   3. breadth-first renumbering, level by level: (new parent, val desc,
//      index asc).
// ---------------------------------------------------------------------------
constexpr int kDynThreads = 512;
constexpr int kMaxPool = 4096;
constexpr int kMaxPoolDepth = 64;

// Bitonic compare-exchange steps with partner distance j0, j0/2, .., 1 of
// the merge of width k, for element i held in a register; the partner
// i ^ j lies in the same warp because j < 32.  Ascending where i & k == 0.
__device__ __forceinline__ unsigned long long bitonic_steps_reg(unsigned long long a, int i, int k, int j0) {
  for (int j = j0; j > 0; j >>= 1) {
    const unsigned long long c = __shfl_xor_sync(0xffffffffu, a, j);
    const bool keep_min = ((i & j) == 0) == ((i & k) == 0);
    a = keep_min ? (c < a ? c : a) : (c < a ? a : c);
  }
  return a;
}

template <int MW>
__global__ void __launch_bounds__(kDynThreads)
    build_dynamic_kernel(const int32_t *__restrict__ pool_parent, const int32_t *__restrict__ pool_tok,
                         const float *__restrict__ pool_conf, int M, const int32_t *__restrict__ prefix_len,
                         int N, int32_t *tok, int32_t *parents_out, int32_t *depth, int32_t *pos,
                         uint64_t *anc, int32_t *first_child, int32_t *next_sibling, int32_t *pool_index,
                         float *val_out, int32_t *status) {
  extern __shared__ __align__(16) unsigned char smem[];
  int M2 = 1;  // M rounded up to a power of two: the sort width
  while (M2 < M) M2 <<= 1;
  unsigned long long *key = reinterpret_cast<unsigned long long *>(smem);  // [M2]
  int *ppar = reinterpret_cast<int *>(key + M2);                         // [M]
  float *val = reinterpret_cast<float *>(ppar + M);                      // [M]
  float *conf = val + M;                                                 // [M]
  int *pdep = reinterpret_cast<int *>(conf + M);                         // [M]
  int *ptok = pdep + M;                                                  // [M]
  __shared__ int kept_new[kMaxNodes];   // new (breadth-first) index of kept slot r
  __shared__ int new_par[kMaxNodes];    // parents by new index
  __shared__ int bad, s_dmax;

  const int b = blockIdx.x, t = threadIdx.x;
  const int64_t prow = (int64_t)b * M;
  // every global load is issued here, so their latencies overlap
  const int P = t < N ? prefix_len[b] : 0;
  if (t == 0) {
    bad = 0;
    s_dmax = 0;
  }
  __syncthreads();
  for (int i = t; i < M; i += kDynThreads) {
    const int p = pool_parent[prow + i];
    const float c = pool_conf[prow + i];
    ptok[i] = pool_tok[prow + i];
    ppar[i] = p;
    conf[i] = c;
    if (i == 0 ? p != -1 : (p < 0 || p >= i || !(c >= 0.f && c <= 1.f))) atomicOr(&bad, 1);
  }
  __syncthreads();
  if (bad) {
    if (t == 0) sv::report(status, SPEC_DEV_BAD_POOL);
    return;
  }
  // 1. depths (parent walk in shared memory), then path values level by
  // level: v[i] = v[parent] * conf[i] multiplies in root-to-node order, the
  // parent's value being complete one level earlier
  int dmax_t = 0;
  for (int i = t; i < M; i += kDynThreads) {
    int d = 0, c = i;
    while (c > 0 && d < kMaxPoolDepth) {
      c = ppar[c];
      ++d;
    }
    if (c != 0) {
      atomicOr(&bad, 1);
      d = 0;
    }
    pdep[i] = d;
    dmax_t = max(dmax_t, d);
  }
  if (dmax_t > 0) atomicMax(&s_dmax, dmax_t);
  __syncthreads();
  if (bad) {
    if (t == 0) sv::report(status, SPEC_DEV_BAD_POOL);
    return;
  }
  if (t == 0) val[0] = 1.0f;
  for (int d = 1; d <= s_dmax; ++d) {
    __syncthreads();  // level d - 1 complete
    for (int i = t; i < M; i += kDynThreads)
      if (pdep[i] == d) val[i] = __fmul_rn(val[ppar[i]], conf[i]);
  }
  __shared__ int lvl_count[kMaxPoolDepth + 2];  // kept nodes per depth
  __shared__ __align__(16) unsigned lkey[kMaxNodes];  // sort keys of one level
  for (int i = t; i < kMaxPoolDepth + 2; i += kDynThreads) lvl_count[i] = 0;
  __syncthreads();
  // conf is dead once the values are formed: it becomes the map from pool
  // index to kept slot (-1: not kept)
  int *slot_of = reinterpret_cast<int *>(conf);
  for (int i = t; i < M2; i += kDynThreads) {
    // v >= 0, so clearing the sign bit only maps -0 to +0; padding sorts last
    key[i] = i < M ? ((unsigned long long)(0xFFFFFFFFu - (__float_as_uint(val[i]) & 0x7FFFFFFFu)) << 32) |
                         ((unsigned long long)pdep[i] << 16) | (unsigned long long)i
                   : ~0ull;
    if (i < M) slot_of[i] = -1;
  }
  __syncthreads();
  // 2. keep the N smallest keys: bitonic sort of the (unique) keys,
  // ascending.  Steps with partner distance >= 32 exchange through shared
  // memory; the shorter ones run on registers.  Merges up to width 32 run
  // entirely on registers (over a whole warp: past M2 the lanes hold
  // padding that only ever meets padding).
  const int M2w = M2 < 32 ? 32 : M2;
  for (int i = t; i < M2w; i += kDynThreads) {
    unsigned long long a = i < M2 ? key[i] : ~0ull;
    for (int k = 2; k <= 32 && k <= M2; k <<= 1) a = bitonic_steps_reg(a, i, k, k >> 1);
    if (i < M2) key[i] = a;
  }
  __syncthreads();
  for (int k = 64; k <= M2; k <<= 1) {
    for (int j = k >> 1; j >= 32; j >>= 1) {
      for (int i = t; i < M2; i += kDynThreads) {
        const int l = i ^ j;
        if (l > i) {
          const unsigned long long a = key[i], c = key[l];
          if ((a > c) == ((i & k) == 0)) {
            key[i] = c;
            key[l] = a;
          }
        }
      }
      __syncthreads();
    }
    for (int i = t; i < M2; i += kDynThreads) key[i] = bitonic_steps_reg(key[i], i, k, 16);
    __syncthreads();
  }
  // kept slot t = the t-th smallest key; its parent's slot through the map
  int my_pool = -1, my_depth = 0, my_pslot = -1;
  if (t < N) {
    my_pool = (int)(key[t] & 0xFFFFull);
    my_depth = pdep[my_pool];
    slot_of[my_pool] = t;
    atomicAdd(&lvl_count[min(my_depth, kMaxPoolDepth + 1)], 1);
  }
  __syncthreads();
  if (t > 0 && t < N) {
    my_pslot = slot_of[ppar[my_pool]];
    if (my_pslot < 0) atomicOr(&bad, 1);  // the kept set is not closed under parents
  }
  __syncthreads();
  if (bad) {
    if (t == 0) sv::report(status, SPEC_DEV_BAD_POOL);
    return;
  }
  // breadth-first renumbering, one level per round: a node's place on its
  // level is the number of level nodes with a smaller (new parent, slot);
  // slots are in key order, so this orders siblings by value
  int base = 0;
  for (int d = 0; d <= kMaxPoolDepth; ++d) {
    const int here = lvl_count[d];
    if (here == 0) break;
    int mp = -1;
    unsigned mine = 0xFFFFFFFFu;
    if (t < N && my_depth == d) {
      mp = t == 0 ? -1 : kept_new[my_pslot];  // the parent was numbered one level up
      mine = ((unsigned)(mp + 1) << 8) | (unsigned)t;
    }
    if (t < 64 * MW) lkey[t] = mine;
    __syncthreads();
    if (t < N && my_depth == d) {
      int before = 0;
#pragma unroll
      for (int r = 0; r < 64 * MW; r += 4) {
        const uint4 q = *reinterpret_cast<const uint4 *>(&lkey[r]);
        before += (q.x < mine) + (q.y < mine) + (q.z < mine) + (q.w < mine);
      }
      kept_new[t] = base + before;
      new_par[base + before] = mp;
    }
    base += here;
    __syncthreads();
  }
  // 3. outputs by new index
  if (t < N) {
    const int ni = kept_new[t];
    const int64_t row = (int64_t)b * N;
    tok[row + ni] = ptok[my_pool];
    parents_out[row + ni] = new_par[ni];
    if (pool_index) pool_index[row + ni] = my_pool;
    if (val_out) val_out[row + ni] = val[my_pool];
  }
  __shared__ unsigned long long kids[kMaxNodes * MW];
  if (t < N)
    for (int w = 0; w < MW; ++w) kids[t * MW + w] = 0ull;
  __syncthreads();
  if (t > 0 && t < N) atomicOr(&kids[new_par[t] * MW + (t >> 6)], 1ull << (t & 63));
  __syncthreads();
  if (t < N) {
    int d;
    emit_tree_arrays<MW>(new_par, kids, t, (N + 63) >> 6, P, (int64_t)b * N, depth, pos, anc, first_child,
                         next_sibling, &d);
  }
}

}  // namespace

int sv_build_static(const int32_t *parents, const int32_t *rank, const int32_t *cand_tok,
                    int cand_levels, int cand_s, const int32_t *root_tok, const int32_t *prefix_len,
                    int batch, int n, int32_t *tok, int32_t *depth, int32_t *pos, uint64_t *anc,
                    int32_t *first_child, int32_t *next_sibling, int32_t *status,
                    cudaStream_t stream) {
  return sv_build_batch(parents, 0, nullptr, nullptr, rank, cand_tok, cand_levels, cand_s, root_tok, prefix_len,
                        batch, n, tok, depth, pos, anc, first_child, next_sibling, status, stream);
}

int sv_build_batch(const int32_t *parents, int par_stride, const int32_t *n_valid, const int32_t *tok_in,
                   const int32_t *rank, const int32_t *cand_tok, int cand_levels, int cand_s,
                   const int32_t *root_tok, const int32_t *prefix_len, int batch, int n, int32_t *tok,
                   int32_t *depth, int32_t *pos, uint64_t *anc, int32_t *first_child, int32_t *next_sibling,
                   int32_t *status, cudaStream_t stream) {
  if (n <= 64)
    build_static_kernel<1><<<batch, 64, 0, stream>>>(parents, par_stride, n_valid, tok_in, rank, cand_tok,
                                                     cand_levels, cand_s, root_tok, prefix_len, n, tok, depth, pos,
                                                     anc, first_child, next_sibling, status);
  else
    build_static_kernel<4><<<batch, 256, 0, stream>>>(parents, par_stride, n_valid, tok_in, rank, cand_tok,
                                                      cand_levels, cand_s, root_tok, prefix_len, n, tok, depth, pos,
                                                      anc, first_child, next_sibling, status);
  return sv_launch_status();
}

int sv_build_dynamic(const int32_t *pool_parent, const int32_t *pool_tok, const float *pool_conf,
                     int M, const int32_t *prefix_len, int batch, int n, int32_t *tok,
                     int32_t *parents_out, int32_t *depth, int32_t *pos, uint64_t *anc,
                     int32_t *first_child, int32_t *next_sibling, int32_t *pool_index, float *val,
                     int32_t *status, cudaStream_t stream) {
  if (M > kMaxPool) return SPEC_ERR_UNSUPPORTED;
  size_t M2 = 1;
  while (M2 < (size_t)M) M2 <<= 1;
  const size_t smem = M2 * 8 + (size_t)M * (4 + 4 + 4 + 4 + 4);  // key (sort width), parent, value, conf, depth, token
  auto kern = n <= 64 ? build_dynamic_kernel<1> : build_dynamic_kernel<4>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  kern<<<batch, kDynThreads, smem, stream>>>(pool_parent, pool_tok, pool_conf, M, prefix_len, n, tok, parents_out,
                                             depth, pos, anc, first_child, next_sibling, pool_index, val, status);
  return sv_launch_status();
}
