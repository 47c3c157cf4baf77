// Tree attention for GQA groups with more than 128 query rows per KV head,
// or trees of more than 64 nodes (up to 256), bf16 in, float32 softmax and
// accumulation, head_dim 128, on pairs of SMs: tcgen05.mma.cta_group::2 with
// M = 256, a persistent grid, and a stream-K split of the work.
//
// "5.3 Medusa、EAGLE 与 MTP" (infra-guide), sections 3.1 and 8: every node
// attends to the shared prefix and to its ancestors-or-self; "Medusa,
// explained", step 6: all nodes are scored in one pass.
//
// Rows.  Query row r of a (sequence, KV head) is node r / G, query head
// kvh*G + r % G, so the G heads of a GQA group and all tree nodes share
// every K/V tile.  A row group is (sequence, KV head, pair of 128-row query
// tiles): CTA k of a cluster owns rows [256 p + 128 k, +128) of pair p.
//
// Work.  The units of a row group are its tree tiles of 128 keys (units
// 0 .. nt-1, nt = ceil(N / 128)) and its prefix tiles of 128 keys (units
// nt ..).  All units of all row groups, in order (sequence, KV head, pair,
// unit), form one sequence of U units, split into C contiguous ranges of
// equal weight: a prefix tile weighs 1 and the tree tiles together
// nt + kSegW, the row group's fixed cost (pipeline drain, epilogue, mask)
// included, so ranges with more row-group starts hold fewer tiles.  No range
// starts between two tree tiles, so the first tile of every part of a row
// group (its first tree tile, holding the root, or a prefix tile) shows
// every row at least one key.  A row group that lies wholly inside one
// cluster's range is normalised and written out; the parts of a row group cut by range ends leave partials
// (unnormalised O in bf16, running max in log2 units and row sum in
// float32) in workspace slots (2c + 1 for the part cut at cluster c's range
// end, 2c for the one cut at its start), merged by attn_tc2_combine_kernel.
//
// Pair MMA.  The even CTA issues every MMA for both.  M = 256: each CTA
// holds its own 128 query rows (Q in shared memory; S, P and O in its own
// TMEM) and half of every K/V tile: CTA k stages keys [64k, 64k+64) of K and
// head dims [64k, 64k+64) of V, 16 KB each, so five-deep K and V rings and
// two Q buffers fit in one SM's shared memory.
//
//   warp 0   Q and K loads; warp 10: V loads (TMA, 128-byte swizzle; one
//            warp each, so neither ring waits on the other's releases).
//            The even CTA's Q/K loads signal its full barriers directly; the
//            odd CTA's signal local barriers
//   warp 1   pair TMEM allocation; in the even CTA it issues
//              S(g) = Q K(g)^T   into TMEM columns [128 (g%3), +128)
//            once PV(g-3), which read that buffer's P, has completed; in the
//            odd CTA it forwards the arrival of its Q/K halves to the even CTA
//   warp 11  in the even CTA, issues
//              O   += P(g) V(g)  (P over S(g)'s first 64 columns, bf16 pairs)
//            Two issuing threads: one thread's tcgen05.mma / commit stream
//            (about 60 cycles per instruction) would otherwise bound the tile
//            rate
//   warps 2-9  softmax and epilogue: each owns 16 TMEM lanes (rows) and
//            reads all 128 keys of a tile with the 16-lane load shape, so a
//            row lives in 4 threads of one warp and its exact tile max is two
//            shuffles away; the running max moves only when a tile exceeds
//            it by 2^16 (then the sum and O are rescaled).  P = 2^(s - m) is
//            written as bf16 pairs over the tile's first 64 S columns.
//            V: before PV(g) the even CTA's PV issuer waits for its own V
//            half to land and zeroes the V rows past the last key of a
//            partial tile (stale cache rows need not be finite); the odd
//            CTA's warp 11 does the same for its half and then arrives on the
//            even CTA's P barrier of the tile.
//
// Every mbarrier wait is bounded; on a timeout the CTA reports
// SPEC_DEV_TIMEOUT, lets its own copies and the pair's MMAs finish, frees
// TMEM and returns.
#include <math.h>

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace {

using namespace sv::ptx;

constexpr int kBN = 128;                     // keys per tile
constexpr int kD = 128;                      // head_dim
constexpr int kKS = 5;                       // K ring stages
constexpr int kVS = 5;                       // V ring stages
constexpr int kQB = 2;                       // Q buffers
constexpr int kPrefetch = 0;                 // L2 prefetch distance in tiles (0: none)
constexpr int kThreads = 384;
constexpr int kPairRows = 256;
constexpr uint32_t kQBytes = 128 * kD * 2;   // 128 rows x 128 dims
constexpr uint32_t kQHalf = kQBytes / 2;     // one 64-dim swizzle column
constexpr uint32_t kKBytes = 64 * kD * 2;    // 64 keys x 128 dims
constexpr uint32_t kKHalf = kKBytes / 2;
constexpr uint32_t kVBytes = kBN * 64 * 2;   // 128 keys x 64 dims
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kSB = 3;                       // S/P buffers in TMEM (128 columns each)
constexpr uint32_t kColO = kSB * 128;        // O after them (128 columns; 512 in all)
// The running max moves only when a tile exceeds it by more than kTau (log2
// units): P = 2^(s - m) then stays below 2^16, far inside bf16's and float32's
// exponent range, and its relative precision does not depend on its size.  A
// small bound made the first prefix tile after a tree tile (whose rows see
// only a few keys) move the max and rescale O in most row groups.
constexpr float kTau = 16.f;
constexpr float kSumBound = 65536.f;  // 2^kTau
constexpr uint16_t kBoth = 3;                // CTA mask of the pair
constexpr int kStoreThread = 64;             // softmax thread that issues the output stores (warp 2, lane 0)
// A partial row: 128 bf16 of unnormalised O (256 B), then the running max
// (log2 units) and the sum as float32, padded to 272 B.
constexpr int kPartialBytes = kD * 2 + 16;

struct Bars {
  uint64_t kland[kKS], kempty[kKS], kfull[kKS];
  uint64_t vland[kVS], vempty[kVS];
  uint64_t qland[kQB], qempty[kQB], qfull[kQB];
  uint64_t sfull[kSB], pfull[kSB], ofull[kSB], drain;
  uint32_t tmem;
  volatile int abort;
  int start_b, start_gi, start_t, n_tiles;     // this cluster's first unit and unit count
  int start_raw, start_raw_next;               // prefix_len[start_b], prefix_len[start_b + 1] (0 past the batch)
};
constexpr uint32_t kTileBytes = kQB * kQBytes + kKS * kKBytes + kVS * kVBytes;
constexpr uint32_t kSmemBytes = kTileBytes + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KB");

constexpr uint32_t kIdescS = idesc_bf16_f32(256, 128, 0, 0);   // Q, K both K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(256, 128, 0, 1);  // V MN-major (dims contiguous)

// ---------------------------------------------------------------------------
// Work schedule
// ---------------------------------------------------------------------------
struct Sched {
  const int32_t *prefix_len;
  int batch, hkv, pairs, n_nodes, s_max, max_prefix, n_clusters;
  int nt, mw;                                              // tree tiles; ancestor-mask words per node
  sv::KvPages pg;                                          // prefix cache addressing
  __device__ int gpb() const { return hkv * pairs; }  // row groups per sequence
};

// A row group's fixed cost (the pipeline drain and epilogue at its end, the
// tree mask) in tile equivalents, carried by its tree tiles in the balanced
// split: a row group of n tiles weighs n + kSegW, and its unit t starts at
// weight unit_start_w(t) within it (all tree tiles at 0: no range starts
// between them).
constexpr int kSegW = 3;
__device__ __forceinline__ int unit_start_w(int t, int nt) { return t < nt ? 0 : kSegW + t; }

// A prefix length out of bounds counts as 0 (the sequence is reported and
// its output left unwritten).
__device__ __forceinline__ bool prefix_ok(const Sched &s, int raw) {
  return raw >= 0 && raw <= s.max_prefix && raw <= s.s_max;
}
__device__ __forceinline__ int seq_tiles(const Sched &s, int P) { return s.nt + (P + kBN - 1) / kBN; }
__device__ __forceinline__ int tiles_of(const Sched &s, int raw) { return seq_tiles(s, prefix_ok(s, raw) ? raw : 0); }

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ long long warp_incl_ll(long long v) {  // inclusive prefix sum over lanes
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Prefix lengths of sequences 32 i + lane (i < 4) in a warp's registers,
// loaded in one round; chunks of 32 sequences past the first 128 are loaded
// where they are walked.
constexpr int kTabSeqs = 128;
struct SeqTab {
  int raw[4];
};
__device__ __forceinline__ void tab_load(const Sched &s, SeqTab &tb) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) tb.raw[i] = 32 * i + lane < s.batch ? s.prefix_len[32 * i + lane] : 0;
}
// f(i, raw) for the chunks i of 32 sequences in order (raw: the lane's
// sequence 32 i + lane, 0 past the batch) until f returns true (uniform).
template <typename F>
__device__ __forceinline__ void for_chunks(const Sched &s, const SeqTab &tb, F f) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (32 * i >= s.batch || f(i, tb.raw[i])) return;
  }
  for (int i = 4; 32 * i < s.batch; ++i)
    if (f(i, 32 * i + lane < s.batch ? s.prefix_len[32 * i + lane] : 0)) return;
}
// prefix_len[b] for a warp-uniform b (0 past the batch).
__device__ __forceinline__ int warp_raw(const Sched &s, const SeqTab &tb, int b) {
  if (b >= s.batch) return 0;
  if (b >= kTabSeqs) return s.prefix_len[b];
  int v = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int x = __shfl_sync(0xffffffffu, tb.raw[i], b & 31);
    if ((b >> 5) == i) v = x;
  }
  return v;
}
// Total weight W and units U of all row groups.
__device__ __forceinline__ void warp_totals(const Sched &s, const SeqTab &tb, long long *W, long long *U) {
  const int lane = threadIdx.x & 31;
  long long n = 0;
  for_chunks(s, tb, [&](int i, int raw) {
    n += 32 * i + lane < s.batch ? tiles_of(s, raw) : 0;
    return false;
  });
  const long long nt = warp_sum_ll(n);
  *U = nt * s.gpb();
  *W = (nt + (long long)kSegW * s.batch) * s.gpb();
}

// A unit: sequence, row group, tile; its index among all units; the start
// weight of its row group.
struct Pos {
  int b, gi, t;
  long long u, wrg;
};
// The first units whose start weights are >= x0 and >= x1 (past the last
// unit: b = batch, u = U, wrg = W), in one walk over the sequences.
__device__ void warp_seek2(const Sched &s, const SeqTab &tb, long long x0, long long x1, Pos *p0, Pos *p1) {
  const int lane = threadIdx.x & 31;
  const int gpb = s.gpb();
  long long W0 = 0, U0 = 0;
  *p0 = *p1 = Pos{s.batch, 0, 0, 0, 0};
  bool found0 = false, found1 = false;
  for_chunks(s, tb, [&](int i, int raw) -> bool {
    const bool in = 32 * i + lane < s.batch;
    const int n = in ? tiles_of(s, raw) : 0;
    const long long w = in ? (long long)gpb * (n + kSegW) : 0, uu = (long long)gpb * n;
    const long long wi = warp_incl_ll(w), ui = warp_incl_ll(uu);
    auto place = [&](long long x, Pos *p, bool *found) {
      const unsigned hit = __ballot_sync(0xffffffffu, in && W0 + wi > x);
      if (!hit) return;
      const int l = __ffs(hit) - 1;
      const long long wb = W0 + __shfl_sync(0xffffffffu, wi - w, l);
      const long long ub = U0 + __shfl_sync(0xffffffffu, ui - uu, l);
      const int nl = __shfl_sync(0xffffffffu, n, l);
      int gi = (int)((x - wb) / (nl + kSegW));
      const int r = (int)(x - wb - (long long)gi * (nl + kSegW));
      int t = r == 0 ? 0 : max(s.nt, r - kSegW);
      int b = 32 * i + l;
      p->u = ub + (long long)gi * nl + t;
      p->wrg = wb + (long long)gi * (nl + kSegW);
      if (t >= nl) {  // past the row group's last tile: the next row group's tree tile
        t = 0;
        p->wrg += nl + kSegW;
        if (++gi == gpb) {
          gi = 0;
          ++b;
        }
      }
      p->b = b;
      p->gi = gi;
      p->t = t;
      *found = true;
    };
    if (!found0) place(x0, p0, &found0);
    if (!found1) place(x1, p1, &found1);
    W0 += __shfl_sync(0xffffffffu, wi, 31);
    U0 += __shfl_sync(0xffffffffu, ui, 31);
    return found0 && found1;
  });
  if (!found0) {
    p0->u = U0;
    p0->wrg = W0;
  }
  if (!found1) {
    p1->u = U0;
    p1->wrg = W0;
  }
}

// Clusters in use: each range is at least as wide as the heaviest run of
// units with one start weight (a row group's tree tiles), so every range
// holds a unit's start.
__device__ __forceinline__ long long clusters_used(const Sched &s, long long W) {
  return max(1ll, min((long long)s.n_clusters, W / (s.nt + kSegW)));
}
__device__ __forceinline__ long long range_start(long long c, long long W, long long C) { return c * W / C; }
// Cluster whose range holds weight x (the largest c with range_start(c) <= x).
__device__ __forceinline__ int cluster_of(long long x, long long W, long long C) {
  return (int)(((x + 1) * C - 1) / W);
}

// Range boundary k (the start of cluster k's range, k >= 1): whether it is
// the first range start inside a row group cut by range ends, that row
// group, and the last cluster holding a part of it (the first is k - 1).
// Written by cluster k for every k of the grid, read by the merge kernel.
struct CutDesc {
  int usable, b, gi, c_hi;
};
__device__ __forceinline__ CutDesc *cut_descs(void *ws, int n_clusters) {
  return reinterpret_cast<CutDesc *>(reinterpret_cast<uint8_t *>(ws) +
                                     (size_t)n_clusters * 2 * kPairRows * kPartialBytes);
}

// Walks the tiles of a cluster's range in order.  The next sequence's
// prefix length is loaded one sequence ahead: a global load waited for at a
// sequence boundary would stall the walk for a full memory latency.
struct Cur {
  int b, gi, t;   // sequence, row group within it, tile within the row group
  int n, P;       // tiles of the row group, effective prefix
  bool ok;        // prefix within bounds
  int raw_next;   // prefix_len[b + 1] (0 past the batch)
};
__device__ __forceinline__ int load_prefix(const Sched &s, int b) { return b < s.batch ? s.prefix_len[b] : 0; }
__device__ __forceinline__ void cur_apply(Cur &c, const Sched &s, int raw) {
  c.ok = prefix_ok(s, raw);
  c.P = c.ok ? raw : 0;
  c.n = seq_tiles(s, c.P);
}
__device__ __forceinline__ Cur cur_begin(const Bars *bars, const Sched &s) {
  Cur c;
  c.b = bars->start_b;
  c.gi = bars->start_gi;
  c.t = bars->start_t;
  cur_apply(c, s, bars->start_raw);
  c.raw_next = bars->start_raw_next;
  return c;
}
__device__ __forceinline__ void cur_next(Cur &c, const Sched &s) {
  if (++c.t == c.n) {
    c.t = 0;
    if (++c.gi == s.gpb()) {
      c.gi = 0;
      ++c.b;
      cur_apply(c, s, c.raw_next);
      c.raw_next = load_prefix(s, c.b + 1);
    }
  }
}
// Valid keys of tile t: a tree tile (t < nt) or a prefix tile.
__device__ __forceinline__ int tile_keys(const Cur &c, const Sched &s) {
  return c.t < s.nt ? min(kBN, s.n_nodes - c.t * kBN) : min(kBN, c.P - (c.t - s.nt) * kBN);
}

__device__ __forceinline__ void give_up(Bars *bars, int32_t *status) {
  bars->abort = 1;
  sv::report(status, SPEC_DEV_TIMEOUT);
}
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, kWaitLimit));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Waits for this CTA's V half of tile g to land and zeroes its rows past the
// last key of a partial tile, up to the next multiple of 16 (the last PV
// k-step reads them with zero probabilities; stale cache rows need not be
// finite).  Full warp; false on timeout.
__device__ __forceinline__ bool v_ready(Bars *bars, uint8_t *sV, int g, int nkeys) {
  const int st = g % kVS;
  if (!warp_wait(&bars->vland[st], (g / kVS) & 1)) return false;
  if (nkeys < kBN) {
    uint4 *v = reinterpret_cast<uint4 *>(sV + st * kVBytes);
    const int end = min(kBN, (nkeys + 15) & ~15) * 8;
    for (int e = nkeys * 8 + (int)(threadIdx.x & 31); e < end; e += 32) v[e] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  __syncwarp();
  return true;
}

// MAXW: ancestor-mask words per node, rounded up to 1, 2 or 4 (trees of up
// to 64, 128 or 256 nodes; one, one or two tree tiles).
template <int MAXW>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_tc2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                    const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kt,
                    const __grid_constant__ CUtensorMap tm_vt, const __grid_constant__ CUtensorMap tm_o,
                    const Sched s_in, const uint64_t *__restrict__ anc, void *__restrict__ ws, int Hq,
                    float scale_log2, int32_t *status) {
  // the tree-tile count as a compile-time constant in every schedule step
  const Sched s = [&] {
    Sched t = s_in;
    t.nt = (MAXW + 1) / 2;
    return t;
  }();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + kQB * kQBytes;
  uint8_t *sV = sK + kKS * kKBytes;
  Bars *bars = reinterpret_cast<Bars *>(sV + kVS * kVBytes);

  const int N = s.n_nodes, G = Hq / s.hkv, R = N * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cluster = blockIdx.x >> 1;

  // The 128-byte swizzle needs 1024-byte aligned tiles; both CTAs of a
  // cluster see the same layout, so they leave together.
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) sv::report(status, SPEC_DEV_INTERNAL);
    return;
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kc);
    tma_prefetch_desc(&tm_vc);
    tma_prefetch_desc(&tm_kt);
    tma_prefetch_desc(&tm_vt);
    tma_prefetch_desc(&tm_o);
  }
  // The range lookup (warp 0) overlaps the barrier and TMEM set-up (warp 1).
  if (warp == 0) {
    SeqTab tb;
    tab_load(s, tb);
    long long W, U;
    warp_totals(s, tb, &W, &U);
    const long long C = clusters_used(s, W);
    Pos p0{s.batch, 0, 0, 0, 0}, p1;
    int T = 0;
    if (cluster < C) {
      warp_seek2(s, tb, range_start(cluster, W, C), range_start(cluster + 1, W, C), &p0, &p1);
      T = (int)(p1.u - p0.u);  // (range_start(C) = W: no unit starts there, p1.u = U)
    }
    const int raw0 = warp_raw(s, tb, p0.b), raw1 = warp_raw(s, tb, p0.b + 1);
    if (lane == 0) {
      bars->start_b = p0.b;
      bars->start_gi = p0.gi;
      bars->start_t = p0.t;
      bars->n_tiles = T;
      bars->start_raw = raw0;
      bars->start_raw_next = raw1;
      if (rank == 0 && cluster >= 1) {
        CutDesc d{0, 0, 0, 0};
        if (cluster < C && p0.t != 0) {  // this range starts inside row group (b, gi)
          d.usable = cluster_of(p0.wrg, W, C) == cluster - 1;
          d.b = p0.b;
          d.gi = p0.gi;
          d.c_hi = cluster_of(p0.wrg + unit_start_w(tiles_of(s, raw0) - 1, s.nt), W, C);
        }
        cut_descs(ws, s.n_clusters)[cluster] = d;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < kKS; ++i) {
        mbar_init(&bars->kland[i], 1);
        mbar_init(&bars->kempty[i], 1);
        mbar_init(&bars->kfull[i], 2);
      }
      for (int i = 0; i < kVS; ++i) {
        mbar_init(&bars->vland[i], 1);
        mbar_init(&bars->vempty[i], 1);
      }
      for (int i = 0; i < kQB; ++i) {
        mbar_init(&bars->qland[i], 1);
        mbar_init(&bars->qempty[i], 2);  // the segment's last S MMA, and its output store
        mbar_init(&bars->qfull[i], 2);
      }
      for (int i = 0; i < kSB; ++i) {
        mbar_init(&bars->sfull[i], 1);
        mbar_init(&bars->ofull[i], 1);
        // one arrival per softmax warp of both CTAs and one for the odd CTA's
        // V half; the softmax may finish tiles g .. g+kSB-1 before the PV
        // issuer observes tile g, never g+kSB (it needs S(g+kSB), issued
        // after PV(g) completed)
        mbar_init(&bars->pfull[i], 17);
      }
      mbar_init(&bars->drain, 2);  // one commit from each MMA-issuing warp
      bars->abort = 0;
      mbar_fence_init();
    }
    __syncwarp();
    tmem_alloc_pair(&bars->tmem, 512);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the partner's barriers exist before any remote arrival or commit
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const int T = bars->n_tiles;
  if (T == 0) {  // same (empty) range for both CTAs of the cluster
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
    return;
  }
  // the merge grid may be scheduled (from a softmax thread: the producers'
  // first copies come first)
  if (threadIdx.x == 96) grid_dep_launch();
  const int pairs = s.pairs;

  if (warp == 0 || warp == 10) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      const bool is_v = warp == 10;
      Cur c = cur_begin(bars, s);
      int seg = 0, issued = 0, q_issued = 0;
      Cur cpf = c;  // kPrefetch tiles ahead of c
      for (int i = 0; i < kPrefetch && i < T; ++i) cur_next(cpf, s);
      for (int g = 0; g < T; ++g) {
        const bool first = g == 0 || c.t == 0;
        if (first && g > 0) ++seg;
        const int kvh = c.gi / pairs, pair = c.gi % pairs;
        const int bh = c.b * s.hkv + kvh;
        if (kPrefetch > 0 && g + kPrefetch < T) {
          // warm L2 with this CTA's half of tile g + kPrefetch
          const int pbh = cpf.b * s.hkv + cpf.gi / pairs;
          const bool ptree = cpf.t < s.nt;
          const int prow = ptree ? pbh * N + cpf.t * kBN
                                 : sv::kv_row(s.pg, cpf.b, s.hkv, cpf.gi / pairs, s.s_max, (cpf.t - s.nt) * kBN, nullptr);
          if (is_v) {
            tma_prefetch_2d(ptree ? &tm_vt : &tm_vc, 64 * (int)rank, prow);
          } else {
            tma_prefetch_2d(ptree ? &tm_kt : &tm_kc, 0, prow + 64 * (int)rank);
            tma_prefetch_2d(ptree ? &tm_kt : &tm_kc, 64, prow + 64 * (int)rank);
          }
          cur_next(cpf, s);
        }
        if (!is_v && first) {
          const int qb = seg % kQB;
          // (a buffer's first use needs no wait: a completed-phase poll still costs a few hundred cycles)
          if ((seg >= kQB && !mbar_wait_cluster(&bars->qempty[qb], ((seg / kQB) & 1) ^ 1, kWaitLimit)) || bars->abort) {
            give_up(bars, status);
            break;
          }
          uint64_t *qbar = rank == 0 ? &bars->qfull[qb] : &bars->qland[qb];
          mbar_expect_tx(qbar, kQBytes);
          const int node0 = c.b * N + (pair * kPairRows + (int)rank * 128) / G;
          tma_load_4d(sQ + qb * kQBytes, &tm_q, 0, 0, kvh, node0, qbar);
          tma_load_4d(sQ + qb * kQBytes + kQHalf, &tm_q, 64, 0, kvh, node0, qbar);
          ++q_issued;
        }
        const int st = g % (is_v ? kVS : kKS);
        const int use = g / (is_v ? kVS : kKS);
        uint64_t *empty = is_v ? &bars->vempty[st] : &bars->kempty[st];
        uint64_t *land = is_v ? &bars->vland[st] : (rank == 0 ? &bars->kfull[st] : &bars->kland[st]);
        if ((use > 0 && !mbar_wait_cluster(empty, (use & 1) ^ 1, kWaitLimit)) || bars->abort) {
          give_up(bars, status);
          break;
        }
        const bool tree = c.t < s.nt;
        // (a 128-key tile lies inside one cache block: block sizes are
        // multiples of 128; a bad block id gives row -1, read as zeros)
        const int row0 =
            tree ? bh * N + c.t * kBN : sv::kv_row(s.pg, c.b, s.hkv, kvh, s.s_max, (c.t - s.nt) * kBN, status);
        if (is_v) {
          mbar_expect_tx(land, kVBytes);
          tma_load_2d(sV + st * kVBytes, tree ? &tm_vt : &tm_vc, 64 * (int)rank, row0, land);
        } else {
          mbar_expect_tx(land, kKBytes);
          const CUtensorMap *m = tree ? &tm_kt : &tm_kc;
          tma_load_2d(sK + st * kKBytes, m, 0, row0 + 64 * (int)rank, land);
          tma_load_2d(sK + st * kKBytes + kKHalf, m, 64, row0 + 64 * (int)rank, land);
        }
        ++issued;
        cur_next(c, s);
      }
      if (bars->abort) {  // let the copies into this CTA land before it exits (bounded)
        // (a full barrier of the even CTA completes only with the odd CTA's
        // half as well; its own copies are then done too)
        const int ns = is_v ? kVS : kKS;
        for (int j = issued > ns ? issued - ns : 0; j < issued; ++j)
          mbar_wait_cluster(is_v ? &bars->vland[j % ns] : (rank == 0 ? &bars->kfull[j % ns] : &bars->kland[j % ns]),
                            (j / ns) & 1, kWaitLimit);
        if (!is_v)
          for (int j = q_issued > kQB ? q_issued - kQB : 0; j < q_issued; ++j)
            mbar_wait_cluster(rank == 0 ? &bars->qfull[j % kQB] : &bars->qland[j % kQB], (j / kQB) & 1, kWaitLimit);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (rank == 0) {
      const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK);
      Cur cs = cur_begin(bars, s);
      int seg_s = 0;
      // S(g) = Q K(g)^T into S buffer g % kSB; called for g = 0, 1, 2, ...
      // in order.  Descriptors are a base plus constant offsets (the start
      // address field is the low 14 bits, in 16-byte units).
      auto issue_s = [&](int g) -> bool {
        const bool first = g == 0 || cs.t == 0;
        if (first && g > 0) ++seg_s;
        const int qb = seg_s % kQB, st = g % kKS;
        if (first && !warp_wait(&bars->qfull[qb], (seg_s / kQB) & 1)) return false;
        if (!warp_wait(&bars->kfull[st], (g / kKS) & 1)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t qd = smem_desc_sw128(qa + (uint32_t)qb * kQBytes, 16, 1024);
          const uint64_t kd = smem_desc_sw128(ka + (uint32_t)st * kKBytes, 16, 1024);
          const uint32_t d = tmem + (uint32_t)(g % kSB) * 128u;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_ss_pair(d, qd + (uint64_t)(((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4),
                        kd + (uint64_t)(((kk >> 2) * kKHalf + (kk & 3) * 32) >> 4), kIdescS, kk > 0);
          mma_commit_pair_mc(&bars->sfull[g % kSB], kBoth);
          mma_commit_pair_mc(&bars->kempty[st], kBoth);
          if (g == T - 1 || cs.t == cs.n - 1) mma_commit_pair_mc(&bars->qempty[qb], kBoth);
        }
        __syncwarp();
        cur_next(cs, s);
        return true;
      };
      bool ok = true;
      for (int g = 0; ok && g < T; ++g) {
        // S(g) overwrites the buffer whose P PV(g - kSB) read
        if (g >= kSB && !(ok = warp_wait(&bars->ofull[g % kSB], ((g - kSB) / kSB) & 1))) break;
        ok = issue_s(g);
      }
      if (!ok) give_up(bars, status);
      if (lane == 0) mma_commit_pair_mc(&bars->drain, kBoth);  // after every MMA issued above
      __syncwarp();
    } else {
      // odd CTA: its Q and K halves have landed -> arrive on the even CTA's
      // full barriers
      Cur c = cur_begin(bars, s);
      int seg = 0;
      for (int g = 0; g < T; ++g) {
        const bool first = g == 0 || c.t == 0;
        if (first && g > 0) ++seg;
        if (first) {
          const int qb = seg % kQB;
          if (!warp_wait(&bars->qland[qb], (seg / kQB) & 1) || bars->abort) {
            give_up(bars, status);
            break;
          }
          if (lane == 0) mbar_arrive_cluster(mapa_cluster(&bars->qfull[qb], 0));
        }
        const int st = g % kKS;
        if (!warp_wait(&bars->kland[st], (g / kKS) & 1) || bars->abort) {
          give_up(bars, status);
          break;
        }
        if (lane == 0) mbar_arrive_cluster(mapa_cluster(&bars->kfull[st], 0));
        cur_next(c, s);
      }
      __syncwarp();
    }
    // both CTAs: every pair MMA (and its commits into this CTA) done
    mbar_wait_cluster(&bars->drain, 0, kWaitLimit);
    __syncwarp();
  } else if (warp == 11) {
    // ------------------------------------------------------------ PV issuer
    if (rank == 0) {
      const uint32_t va = smem_u32(sV);
      Cur cp = cur_begin(bars, s);
      bool ok = true;
      for (int g = 0; ok && g < T; ++g) {
        // O += P(g) V(g) once P of both CTAs is ready (which also covers both
        // V halves of tile g)
        const int nkeys = tile_keys(cp, s);
        if (!(ok = warp_wait(&bars->pfull[g % kSB], (g / kSB) & 1) && v_ready(bars, sV, g, nkeys))) break;
        tc_fence_after();
        const bool first = g == 0 || cp.t == 0;
        const int st = g % kVS;
        const int ksteps = (nkeys + 15) >> 4;
        if (lane == 0) {
          const uint64_t vd = smem_desc_sw128(va + (uint32_t)st * kVBytes, kVBytes, 1024);
          const uint32_t pbase = tmem + (uint32_t)(g % kSB) * 128u;  // P of keys [16kk, +16) at + 8kk
          const uint32_t acc0 = first ? 0u : 1u;
          if (ksteps == kBN / 16) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              mma_ts_pair(tmem + kColO, pbase + (uint32_t)kk * 8u, vd + (uint64_t)((kk * 2048) >> 4), kIdescPV,
                          kk > 0 ? 1u : acc0);
          } else {
            for (int kk = 0; kk < ksteps; ++kk)
              mma_ts_pair(tmem + kColO, pbase + (uint32_t)kk * 8u, vd + (uint64_t)((kk * 2048) >> 4), kIdescPV,
                          kk > 0 ? 1u : acc0);
          }
          mma_commit_pair_mc(&bars->vempty[st], kBoth);
          mma_commit_pair_mc(&bars->ofull[g % kSB], kBoth);
        }
        __syncwarp();
        cur_next(cp, s);
      }
      if (!ok) give_up(bars, status);
      if (lane == 0) mma_commit_pair_mc(&bars->drain, kBoth);  // after every MMA issued above
      __syncwarp();
    } else {
      // odd CTA: its V half of each tile is ready -> arrive on the even
      // CTA's P barrier of that tile.  V runs ahead of the softmax, so this
      // arrival first waits for S(g) to complete: S(g) was issued after
      // PV(g-kSB) completed, i.e. after the barrier's phase for tile g-kSB,
      // so the arrival cannot fall into that earlier phase.
      const uint32_t pfull_even0 = mapa_cluster(&bars->pfull[0], 0);  // pfull[i] at + 8 i
      Cur c = cur_begin(bars, s);
      for (int g = 0; g < T; ++g) {
        if (!warp_wait(&bars->sfull[g % kSB], (g / kSB) & 1) || !v_ready(bars, sV, g, tile_keys(c, s)) ||
            bars->abort) {
          give_up(bars, status);
          break;
        }
        if (lane == 0) mbar_arrive_cluster(pfull_even0 + (uint32_t)(g % kSB) * (uint32_t)sizeof(uint64_t));
        cur_next(c, s);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w owns TMEM lanes [32 (w%4) + 16 u, +16), u = (w - 2) / 4: thread
    // t holds rows lb + t/4 and lb + t/4 + 8 (lb = that lane base), 32 key
    // columns of each row (pairs 2 (t%4), +1 of every 8-key group), so a
    // row's max and sum are reduced over the 4 threads t%4 with shuffles.
    const int quarter = warp & 3;
    const int u = (warp - 2) >> 2;
    const int lb = quarter * 32 + u * 16;  // lane base of this warp
    const int tq = lane & 3;
    const int ra = lb + (lane >> 2), rb = ra + 8;  // this thread's rows (TMEM lanes)
    const uint32_t lane_off = (uint32_t)lb << 16;
    // the 8 softmax warps of this CTA (named barrier 1)
    auto softmax_sync = [&]() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
    const uint32_t pfull_even0 = mapa_cluster(&bars->pfull[0], 0);  // pfull[i] at + 8 i
    const float NEG_INF = -INFINITY;
    Cur c = cur_begin(bars, s);
    int seg = 0;        // segment (row group part) of this range: Q buffer seg % kQB
    int q_pending = 0;  // 1 + the Q buffer the last output store reads (store thread)
    bool from_start = c.t == 0;
    float ma = NEG_INF, mb = NEG_INF;  // running max of rows ra, rb (log2 units)
    float la = 0.f, lb_sum = 0.f;      // this thread's part of their sums
    // Ancestor bits of a row for tree tile tt (words 2 tt and 2 tt + 1 of its
    // node; padding rows: all tree keys): the first tree tile's loaded one
    // row group ahead, a later tree tile's one tile ahead, so no tree tile
    // waits for them.
    constexpr int NT = (MAXW + 1) / 2;        // tree tiles
    constexpr int MP = MAXW == 1 ? 1 : 2;     // mask words of one tree tile
    const int MW = MAXW == 1 ? 1 : s.mw;
    struct Mask {
      uint64_t w[MP];
    };
    auto grow = [&](int gi, int lane_row) { return (gi % pairs) * kPairRows + (int)rank * 128 + lane_row; };
    auto load_mask = [&](int b, int gi, int lane_row, int tt) -> Mask {
      Mask m;
      const int rr = grow(gi, lane_row);
      const uint64_t *p = anc + ((int64_t)b * N + rr / G) * MW + 2 * tt;
#pragma unroll
      for (int i = 0; i < MP; ++i) m.w[i] = rr >= R ? ~0ull : (MP == 1 || 2 * tt + i < MW) ? p[i] : 0ull;
      return m;
    };
    Mask amask_a{}, amask_b{}, next_a{}, next_b{};
    if (c.t < NT) {
      amask_a = load_mask(c.b, c.gi, ra, c.t);
      amask_b = load_mask(c.b, c.gi, rb, c.t);
    }
    bool ok = true;
    bool s_ready = false;  // S(g) seen complete during tile g - 1
    // A failed wait (timeout) or an abort turns the rest into a no-op that
    // still passes every pair barrier, so the two warps of a pair always
    // execute the same barriers.
    // Outer loop: the segments of the range (a row group, or the part of one
    // the range holds); inner loop: their tiles.  The epilogue and the
    // segment set-up stay out of the per-tile loop.
    for (int g = 0; g < T;) {
      if (g > 0) {  // a later segment starts at a row group's tree tile
        ++seg;
        from_start = true;
        amask_a = next_a;
        amask_b = next_b;
      }
      ma = mb = NEG_INF;
      la = lb_sum = 0.f;
      if (g + (c.n - 1 - c.t) + 1 < T) {  // the next segment's ancestor bits, a segment ahead
        const bool same_b = c.gi + 1 < s.gpb();
        next_a = load_mask(same_b ? c.b : c.b + 1, same_b ? c.gi + 1 : 0, ra, 0);
        next_b = load_mask(same_b ? c.b : c.b + 1, same_b ? c.gi + 1 : 0, rb, 0);
      }
      bool first = true;
      for (;;) {
        if (ok && !s_ready && !warp_wait(&bars->sfull[g % kSB], (g / kSB) & 1)) ok = false;
        const uint32_t s_addr = tmem + lane_off + (uint32_t)(g % kSB) * 128u;
        // sv[4j + e]: row ra, key 8j + 2 tq + e;  sv[4j + 2 + e]: row rb
        uint32_t sv[64];
        if (ok) {
          tc_fence_after();
          tmem_ld_16x256b_x16(s_addr, sv);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) sv[i] = __float_as_uint(0.f);
        }
        const bool tree = c.t < s.nt;
        const int nvalid = tile_keys(c, s);
        // The tile body comes in two instances so that full prefix tiles, the
        // steady state, carry no masking code: the masked one serves the tree
        // tiles and the last, partial prefix tile.
        auto tile = [&](auto masked) {
          if constexpr (decltype(masked)::value) {
            // Visibility of this thread's keys 8j + 2 tq + e as bits 2j + e: the
            // keys below nvalid are a prefix of these bits (they increase with
            // the bit index); on a tree tile also the ancestor bits (keys 0-63
            // of the tile from its first mask word, 64-127 from its second).
            const int m8 = nvalid - 2 * tq;
            const int nb = m8 <= 0 ? 0 : min(32, 2 * (m8 >> 3) + min(2, m8 & 7));
            const uint32_t in = nb >= 32 ? 0xFFFFFFFFu : ((1u << nb) - 1u);
            uint32_t va = in, vb = in;
            if (tree) {
              auto mine = [&](uint64_t m) -> uint32_t {
                uint64_t x = (m >> (2 * tq)) & 0x0303030303030303ull;
                x = (x | (x >> 6)) & 0x000F000F000F000Full;
                x = (x | (x >> 12)) & 0x000000FF000000FFull;
                return (uint32_t)((x | (x >> 24)) & 0xFFFFull);
              };
              if constexpr (MP == 1) {
                va &= mine(amask_a.w[0]);
                vb &= mine(amask_b.w[0]);
              } else {
                va &= mine(amask_a.w[0]) | (mine(amask_a.w[1]) << 16);
                vb &= mine(amask_b.w[0]) | (mine(amask_b.w[1]) << 16);
              }
              if constexpr (NT > 1) {
                if (c.t + 1 < NT) {  // the next tree tile's bits, a tile ahead
                  amask_a = load_mask(c.b, c.gi, ra, c.t + 1);
                  amask_b = load_mask(c.b, c.gi, rb, c.t + 1);
                }
              }
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {  // i = 2j + e: register 4j + e of row ra, 4j + 2 + e of row rb
              if (!((va >> i) & 1u)) sv[4 * (i >> 1) + (i & 1)] = __float_as_uint(NEG_INF);
              if (!((vb >> i) & 1u)) sv[4 * (i >> 1) + 2 + (i & 1)] = __float_as_uint(NEG_INF);
            }
          }
          // S(g + 1) has nearly always completed by now; testing it here lets
          // the barrier's latency overlap this tile's work
          const bool next_done = ok && g + 1 < T && mbar_test(&bars->sfull[(g + 1) % kSB], ((g + 1) / kSB) & 1);
          // P = 2^(s * scale - m) as bf16 pairs: key pair 8j + 2 tq, +1 is P
          // column 4j + tq, written over the tile's first 64 S columns of this
          // warp's lanes (all of them were read above); and the row sums.
          uint32_t pk[32];
          float2 sa2, sb2;
          auto exps = [&]() {
            const float2 sc2 = make_float2(scale_log2, scale_log2);
            const float2 na2 = make_float2(-ma, -ma), nb2 = make_float2(-mb, -mb);
            sa2 = sb2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 xa2 = fma2(make_float2(__uint_as_float(sv[4 * j]), __uint_as_float(sv[4 * j + 1])), sc2, na2);
              const float2 xb2 =
                  fma2(make_float2(__uint_as_float(sv[4 * j + 2]), __uint_as_float(sv[4 * j + 3])), sc2, nb2);
              const float2 pa = make_float2(ex2(xa2.x), ex2(xa2.y));
              const float2 pb = make_float2(ex2(xb2.x), ex2(xb2.y));
              sa2 = add2(sa2, pa);
              sb2 = add2(sb2, pb);
              pk[2 * j] = pack_bf16(pa.x, pa.y);
              pk[2 * j + 1] = pack_bf16(pb.x, pb.y);
            }
          };
          // Past a row group's first tile, P is computed in one pass with the
          // running max as it stands: the exact tile max matters only when some
          // score exceeds the running max by more than kTau, which shows in the
          // row sums (one P above 2^kTau puts its row's sum above it), and then
          // the tile is read again and redone on the exact path (the tree and
          // ragged tiles and a segment's first tile take the exact path at once).
          bool exact = decltype(masked)::value || first;
          for (;;) {
            if (exact) {
              // exact row max of the tile: finite on a part's first tile (the
              // root, or prefix keys, are visible to every row); a later tree
              // tile may hide all its keys from a row (max -inf: the running
              // max stays, and its P is 0)
              float xa[2] = {NEG_INF, NEG_INF}, xb[2] = {NEG_INF, NEG_INF};
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                xa[j & 1] = fmax3(xa[j & 1], __uint_as_float(sv[4 * j]), __uint_as_float(sv[4 * j + 1]));
                xb[j & 1] = fmax3(xb[j & 1], __uint_as_float(sv[4 * j + 2]), __uint_as_float(sv[4 * j + 3]));
              }
              float ta = fmaxf(xa[0], xa[1]), tb = fmaxf(xb[0], xb[1]);
              ta = fmaxf(ta, __shfl_xor_sync(0xffffffffu, ta, 1));
              tb = fmaxf(tb, __shfl_xor_sync(0xffffffffu, tb, 1));
              ta = fmaxf(ta, __shfl_xor_sync(0xffffffffu, ta, 2)) * scale_log2;
              tb = fmaxf(tb, __shfl_xor_sync(0xffffffffu, tb, 2)) * scale_log2;
              // The running max moves only when a tile exceeds it by more than
              // kTau: P = 2^(s - m) stays below 2^kTau, and the sum and O are
              // rescaled (O once PV(g-1) has completed) only then.
              const bool need_a = ta > ma + kTau, need_b = tb > mb + kTau;
              if (ok && __any_sync(0xffffffffu, need_a || need_b)) {
                const float alpha_a = need_a ? ex2(ma - ta) : 1.f;  // 0 when m was -inf
                const float alpha_b = need_b ? ex2(mb - tb) : 1.f;
                if (need_a) {
                  ma = ta;
                  la *= alpha_a;
                }
                if (need_b) {
                  mb = tb;
                  lb_sum *= alpha_b;
                }
                if (!first && __any_sync(0xffffffffu, alpha_a != 1.f || alpha_b != 1.f) &&
                    (ok = warp_wait(&bars->ofull[(g - 1) % kSB], ((g - 1) / kSB) & 1))) {
                  tc_fence_after();
#pragma unroll 1
                  for (int cc = 0; cc < 4; ++cc) {  // O columns [32 cc, +32) of this warp's 16 rows
                    uint32_t o[16];
                    const uint32_t oa = tmem + lane_off + kColO + (uint32_t)cc * 32u;
                    tmem_ld_16x256b_x4(oa, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                      o[4 * j] = __float_as_uint(__uint_as_float(o[4 * j]) * alpha_a);
                      o[4 * j + 1] = __float_as_uint(__uint_as_float(o[4 * j + 1]) * alpha_a);
                      o[4 * j + 2] = __float_as_uint(__uint_as_float(o[4 * j + 2]) * alpha_b);
                      o[4 * j + 3] = __float_as_uint(__uint_as_float(o[4 * j + 3]) * alpha_b);
                    }
                    tmem_st_16x256b_x4(oa, o);
                  }
                }
              }
            }
            if (!ok) break;
            exps();
            // some P above 2^kTau makes its row's partial sum exceed it too (a
            // NaN or infinite sum fails the test as well)
            if (exact || !__any_sync(0xffffffffu, !(fmaxf(sa2.x + sa2.y, sb2.x + sb2.y) <= kSumBound))) break;
            exact = true;
            tmem_ld_16x256b_x16(s_addr, sv);
            tmem_wait_ld();
          }
          if (ok) {
            tmem_st_16x128b_x16(s_addr, pk);
            la += sa2.x + sa2.y;
            lb_sum += sb2.x + sb2.y;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(pfull_even0 + (uint32_t)(g % kSB) * (uint32_t)sizeof(uint64_t));
          }
          s_ready = __all_sync(0xffffffffu, next_done);
        };
        if (__builtin_expect(tree || nvalid < kBN, 0))
          tile(std::true_type{});
        else
          tile(std::false_type{});
        if (q_pending && threadIdx.x == kStoreThread) {  // the previous output store has long read its buffer
          bulk_wait_read();
          mbar_arrive(&bars->qempty[q_pending - 1]);
          q_pending = 0;
        }
        if (g == T - 1 || c.t == c.n - 1) break;
        cur_next(c, s);
        ++g;
        first = false;
      }
      {
        // ---------------------------------------------------- epilogue
        // O of this warp's 16 rows is read in the softmax layout (thread:
        // rows ra, rb, key-column pairs 8j + 2 tq), where each row's running
        // max and sum already sit in its 4 threads.  Complete rows are
        // normalised and staged as bf16 in this segment's Q buffer (its last
        // S MMA has completed) in the output box's 128-byte-swizzled layout,
        // then written by one TMA store per 64-dim half; the producer reloads
        // that buffer only once the store has read it.  The rows of a row
        // group cut by a range end are written as partials.
        if (ok && !warp_wait(&bars->ofull[g % kSB], (g / kSB) & 1)) ok = false;
        float sa = la + __shfl_xor_sync(0xffffffffu, la, 1);
        float sb = lb_sum + __shfl_xor_sync(0xffffffffu, lb_sum, 1);
        sa += __shfl_xor_sync(0xffffffffu, sa, 2);
        sb += __shfl_xor_sync(0xffffffffu, sb, 2);
        const bool complete = from_start && c.t == c.n - 1;
        // a prefix out of bounds: the sequence is reported, its rows left unwritten
        if (!c.ok && warp == 2 && lane == 0 && c.gi == 0) sv::report(status, SPEC_DEV_CAPACITY);
        const int qb = seg % kQB;
        uint8_t *stage = sQ + qb * kQBytes;
        const bool live = ok && !__any_sync(0xffffffffu, bars->abort != 0);
        uint32_t ov[64];  // ov[4j + e]: row ra, column 8j + 2 tq + e;  ov[4j + 2 + e]: row rb
        if (live) {
          tc_fence_after();
          tmem_ld_16x256b_x16(tmem + lane_off + kColO, ov);
          tmem_wait_ld();
        }
        if (live && complete) {
          const float ia = sa > 0.f ? 1.f / sa : 0.f, ib = sb > 0.f ? 1.f / sb : 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) {  // 16-byte chunk j & 7 of 64-dim half j >> 3 of rows ra, rb
            uint8_t *half = stage + (j >> 3) * kQHalf + 4 * tq;
            *reinterpret_cast<uint32_t *>(half + ra * 128 + (((j & 7) ^ (ra & 7)) << 4)) =
                pack_bf16(__uint_as_float(ov[4 * j]) * ia, __uint_as_float(ov[4 * j + 1]) * ia);
            *reinterpret_cast<uint32_t *>(half + rb * 128 + (((j & 7) ^ (rb & 7)) << 4)) =
                pack_bf16(__uint_as_float(ov[4 * j + 2]) * ib, __uint_as_float(ov[4 * j + 3]) * ib);
          }
          fence_proxy_async_smem();  // visible to the TMA store
        } else if (live) {
          // a part cut at the range end: slot 2c + 1; the one cut at its start: 2c
          const int slot = cluster * 2 + (g == T - 1 && c.t != c.n - 1 ? 1 : 0);
          uint8_t *w = reinterpret_cast<uint8_t *>(ws) + ((int64_t)slot * kPairRows + (int)rank * 128) * kPartialBytes;
          const bool oka = grow(c.gi, ra) < R, okb = grow(c.gi, rb) < R;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (oka)
              *reinterpret_cast<uint32_t *>(w + ra * kPartialBytes + 16 * j + 4 * tq) =
                  pack_bf16(__uint_as_float(ov[4 * j]), __uint_as_float(ov[4 * j + 1]));
            if (okb)
              *reinterpret_cast<uint32_t *>(w + rb * kPartialBytes + 16 * j + 4 * tq) =
                  pack_bf16(__uint_as_float(ov[4 * j + 2]), __uint_as_float(ov[4 * j + 3]));
          }
          if (tq == 0) {
            if (oka) *reinterpret_cast<float2 *>(w + ra * kPartialBytes + kD * 2) = make_float2(ma, sa);
            if (okb) *reinterpret_cast<float2 *>(w + rb * kPartialBytes + kD * 2) = make_float2(mb, sb);
          }
        }
        softmax_sync();  // every row of this CTA staged
        if (threadIdx.x == kStoreThread) {
          const int node0 = ((c.gi % pairs) * kPairRows + (int)rank * 128) / G;
          if (live && complete && c.ok && node0 < N) {  // (a CTA past the last node has no rows to write)
            const int kvh = c.gi / pairs;
            tma_store_5d(&tm_o, stage, 0, 0, kvh, node0, c.b);
            tma_store_5d(&tm_o, stage + kQHalf, 64, 0, kvh, node0, c.b);
            bulk_commit();
            q_pending = qb + 1;  // Q buffer released once the store has read it
          } else {
            mbar_arrive(&bars->qempty[qb]);
          }
        }
        if (!ok) give_up(bars, status);
      }
      cur_next(c, s);
      ++g;
    }
    if (threadIdx.x == kStoreThread) {
      if (q_pending) {
        bulk_wait_read();
        mbar_arrive(&bars->qempty[q_pending - 1]);
      }
      bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  // remote arrivals and multicast commits into either CTA are complete once
  // both have passed their own __syncthreads
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Merges the partials of the row groups cut by cluster range ends: block
// (k - 1, y) merges rows [32 y, +32) of the row group whose first range
// start inside it is boundary k, if any (its descriptor, written by cluster
// k).  Thread = (row, 16 head dims), 8 threads per row; each reads every
// contributor's max and sum itself, so a row needs no exchange, and the
// loads of up to kCombBatch contributors are in flight together.  Launched
// as a programmatic dependent of the main kernel: its blocks become
// resident as the main kernel's CTAs leave and wait for it to complete.
constexpr int kCombRows = 32;
constexpr int kCombBatch = 3;
__global__ void __launch_bounds__(256, 4) attn_tc2_combine_kernel(void *__restrict__ ws, __nv_bfloat16 *__restrict__ out,
                                                                  const Sched s, int Hq) {
  const int k = blockIdx.x + 1;                 // boundary between clusters k-1 and k
  const int rr = blockIdx.y * kCombRows + (threadIdx.x >> 3);  // row of the pair
  const int d0 = (threadIdx.x & 7) * 16;        // first head dim
  grid_dep_wait();  // the main kernel's partials and descriptors are written and visible
  const CutDesc d = cut_descs(ws, s.n_clusters)[k];
  if (!d.usable) return;
  const int G = Hq / s.hkv, R = s.n_nodes * G;
  const int kvh = d.gi / s.pairs, pair = d.gi % s.pairs;
  const int rg = pair * kPairRows + rr;
  if (rg >= R) return;
  const int c_lo = k - 1, nc = d.c_hi - c_lo + 1;
  // cluster c's part: slot 2c + 1 when cut at its range end (all but the last)
  auto row_of = [&](int c) -> const uint8_t * {
    const int slot = 2 * c + (c < d.c_hi ? 1 : 0);
    return reinterpret_cast<const uint8_t *>(ws) + ((int64_t)slot * kPairRows + rr) * kPartialBytes;
  };
  float M = -INFINITY, L = 0.f;
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  for (int c0 = 0; c0 < nc; c0 += kCombBatch) {
    float2 ml[kCombBatch];
    uint4 o[kCombBatch][2];
#pragma unroll
    for (int i = 0; i < kCombBatch; ++i) {
      if (c0 + i < nc) {
        const uint8_t *row = row_of(c_lo + c0 + i);
        ml[i] = *reinterpret_cast<const float2 *>(row + kD * 2);
        o[i][0] = *reinterpret_cast<const uint4 *>(row + d0 * 2);
        o[i][1] = *reinterpret_cast<const uint4 *>(row + d0 * 2 + 16);
      } else {
        ml[i] = make_float2(-INFINITY, 0.f);
        o[i][0] = o[i][1] = make_uint4(0, 0, 0, 0);
      }
    }
    float Mb = M;
#pragma unroll
    for (int i = 0; i < kCombBatch; ++i) Mb = fmaxf(Mb, ml[i].x);
    // every part has a finite max (its first tile holds a key visible to every row)
    const float r = exp2f(M - Mb);  // 0 on the first batch
    L *= r;
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] *= r;
#pragma unroll
    for (int i = 0; i < kCombBatch; ++i) {
      const float f = c0 + i < nc ? exp2f(ml[i].x - Mb) : 0.f;
      L = fmaf(f, ml[i].y, L);
      const uint32_t w[8] = {o[i][0].x, o[i][0].y, o[i][0].z, o[i][0].w, o[i][1].x, o[i][1].y, o[i][1].z, o[i][1].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[2 * j] = fmaf(f, __uint_as_float(w[j] << 16), acc[2 * j]);
        acc[2 * j + 1] = fmaf(f, __uint_as_float(w[j] & 0xFFFF0000u), acc[2 * j + 1]);
      }
    }
    M = Mb;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint4 v0, v1;
  v0.x = pack_bf16(acc[0] * inv, acc[1] * inv);
  v0.y = pack_bf16(acc[2] * inv, acc[3] * inv);
  v0.z = pack_bf16(acc[4] * inv, acc[5] * inv);
  v0.w = pack_bf16(acc[6] * inv, acc[7] * inv);
  v1.x = pack_bf16(acc[8] * inv, acc[9] * inv);
  v1.y = pack_bf16(acc[10] * inv, acc[11] * inv);
  v1.z = pack_bf16(acc[12] * inv, acc[13] * inv);
  v1.w = pack_bf16(acc[14] * inv, acc[15] * inv);
  uint4 *dst = reinterpret_cast<uint4 *>(out + (((int64_t)d.b * s.n_nodes + rg / G) * Hq + kvh * G + rg % G) * kD + d0);
  dst[0] = v0;
  dst[1] = v1;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load();
  if (!f) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<EncodeTiledFn>(p);
      fn.store(f);
    }
  }
  return f;
}

int make_map(CUtensorMap *m, const void *base, cuuint32_t rank, const cuuint64_t *dims, const cuuint64_t *strides,
             const cuuint32_t *box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return SPEC_ERR_CUDA;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SPEC_OK : SPEC_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_clusters[kMaxDevices];

// Clusters of the persistent grid: as many as fit on the current device at
// once (one CTA per SM); looked up once per device.
int tc2_clusters() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = g_clusters[dev].load();
  if (n > 0) return n;
  if (cudaFuncSetAttribute(attn_tc2_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, attn_tc2_kernel<1>, &cfg) != cudaSuccess || clusters < 1) return 0;
  g_clusters[dev].store(clusters);
  return clusters;
}

}  // namespace

bool sv_attn_tc2_supported(const SvAttnShape &s) {
  if (s.dtype != SPEC_BF16 || s.head_dim != kD || s.hkv < 1) return false;
  const int G = s.hq / s.hkv;
  return s.n_nodes <= SPEC_MAX_NODES && G <= 128 && (128 % G) == 0 && (s.n_nodes * G > 128 || s.n_nodes > 64);
}

size_t sv_attn_tc2_ws_bytes() {
  const int c = tc2_clusters();
  return c > 0 ? (size_t)c * (2 * kPairRows * kPartialBytes + sizeof(CutDesc)) : 0;
}

int sv_attn_tc2(const SvAttnShape &s, const void *q, const void *kc, const void *vc, const void *kt, const void *vt,
                const int32_t *prefix_len, const uint64_t *anc, void *out, float scale, void *ws, size_t ws_bytes,
                int32_t *status, cudaStream_t stream) {
  const int C = tc2_clusters();
  if (C < 1) return SPEC_ERR_CUDA;
  if (!ws || ws_bytes < sv_attn_tc2_ws_bytes()) return SPEC_ERR_CAPACITY;
  const int G = s.hq / s.hkv, R = s.n_nodes * G;
  CUtensorMap mq, mkc, mvc, mkt, mvt, mo;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)G, (cuuint64_t)s.hkv, (cuuint64_t)s.batch * s.n_nodes};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)G * kD * 2, (cuuint64_t)s.hq * kD * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)(128 / G)};
    if (make_map(&mq, q, 4, dims, strides, box) != SPEC_OK) return SPEC_ERR_CUDA;
  }
  {
    // output rows of a CTA: 128 / G nodes x the G heads of a KV head; nodes
    // past the sequence's last are outside the map and not written
    const cuuint64_t dims[5] = {(cuuint64_t)kD, (cuuint64_t)G, (cuuint64_t)s.hkv, (cuuint64_t)s.n_nodes,
                                (cuuint64_t)s.batch};
    const cuuint64_t strides[4] = {(cuuint64_t)kD * 2, (cuuint64_t)G * kD * 2, (cuuint64_t)s.hq * kD * 2,
                                   (cuuint64_t)s.n_nodes * s.hq * kD * 2};
    const cuuint32_t box[5] = {64, (cuuint32_t)G, 1, (cuuint32_t)(128 / G), 1};
    if (make_map(&mo, out, 5, dims, strides, box) != SPEC_OK) return SPEC_ERR_CUDA;
  }
  {
    // (at least one row so the map is valid when no prefix tile is ever
    // loaded; a paged cache is one pool of blocks)
    const cuuint64_t rows = s.block_table ? (cuuint64_t)s.num_blocks * s.hkv * s.block_size
                                          : (cuuint64_t)s.batch * s.hkv * s.s_max;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, rows > 0 ? rows : 1};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t kbox[2] = {64, 64}, vbox[2] = {64, (cuuint32_t)kBN};
    if (make_map(&mkc, kc, 2, dims, strides, kbox) != SPEC_OK) return SPEC_ERR_CUDA;
    if (make_map(&mvc, vc, 2, dims, strides, vbox) != SPEC_OK) return SPEC_ERR_CUDA;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)s.batch * s.hkv * s.n_nodes};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t kbox[2] = {64, 64}, vbox[2] = {64, (cuuint32_t)kBN};
    if (make_map(&mkt, kt, 2, dims, strides, kbox) != SPEC_OK) return SPEC_ERR_CUDA;
    if (make_map(&mvt, vt, 2, dims, strides, vbox) != SPEC_OK) return SPEC_ERR_CUDA;
  }
  Sched sc;
  sc.prefix_len = prefix_len;
  sc.batch = s.batch;
  sc.hkv = s.hkv;
  sc.pairs = (R + kPairRows - 1) / kPairRows;
  sc.n_nodes = s.n_nodes;
  sc.s_max = s.s_max;
  sc.max_prefix = s.max_prefix;
  sc.n_clusters = C;
  sc.nt = (s.n_nodes + kBN - 1) / kBN;
  sc.mw = (s.n_nodes + 63) / 64;
  sc.pg = sv::KvPages{s.block_table, s.block_size, s.max_blocks, s.num_blocks};
  // (every instance has the same shared memory and one CTA per SM, so the
  // cluster count looked up for one holds for all)
  auto kern = sc.mw == 1 ? attn_tc2_kernel<1> : sc.mw == 2 ? attn_tc2_kernel<2> : attn_tc2_kernel<4>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
    return SPEC_ERR_CUDA;
  kern<<<2 * C, kThreads, kSmemBytes, stream>>>(mq, mkc, mvc, mkt, mvt, mo, sc, anc, ws, s.hq,
                                               scale * 1.4426950408889634f, status);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (C > 1) {
    // programmatic dependent launch: the merge blocks locate their row groups
    // while the main kernel runs (it triggers its dependents after setup)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C - 1, kPairRows / kCombRows);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, attn_tc2_combine_kernel, ws, (__nv_bfloat16 *)out, sc, s.hq) !=
        cudaSuccess)
      return SPEC_ERR_CUDA;
  }
  return sv_launch_status();
}
