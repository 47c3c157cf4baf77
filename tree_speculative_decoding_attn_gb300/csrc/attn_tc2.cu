// Tree attention for GQA groups with more than 128 query rows per KV head
// (bf16 in, float32 softmax and accumulation, head_dim 128), on pairs of
// SMs: tcgen05.mma.cta_group::2 with M = 256, a persistent grid, and a
// stream-K split of the work.
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
// Work.  The units of a row group are its tree tile (unit 0) and its prefix
// tiles of 128 keys (units 1..).  All units of all row groups, in order
// (sequence, KV head, pair, unit), form one sequence of U units; cluster c
// of C takes units [floor(cU/C), floor((c+1)U/C)).  A row group that lies
// wholly inside one cluster's range is normalised and written out; the row
// groups cut by a range end leave partials (unnormalised O in bf16, running
// max in log2 units and row sum in float32) in workspace slot (c, first/
// last), merged by attn_tc2_combine_kernel.  Every cluster streams the same number of tiles
// whatever the prefix lengths.
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
//            it by 2^8 (then the sum and O are rescaled).  P = 2^(s - m) is
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
constexpr float kTau = 8.f;                  // running max moves only when a tile exceeds it by 2^8
constexpr uint16_t kBoth = 3;                // CTA mask of the pair
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
  float xm[128], xl[128];                      // per-row running max and sum at a row group's end
};
constexpr uint32_t kTileBytes = kQB * kQBytes + kKS * kKBytes + kVS * kVBytes;
constexpr uint32_t kSmemBytes = kTileBytes + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KB");

constexpr uint32_t kIdescS = idesc_bf16_f32(256, 128, 0, 0);   // Q, K both K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(256, 128, 0, 1);  // V MN-major (dims contiguous)

// ---------------------------------------------------------------------------
// Work schedule, shared by the main and combine kernels
// ---------------------------------------------------------------------------
struct Sched {
  const int32_t *prefix_len;
  int batch, hkv, pairs, n_nodes, s_max, max_prefix, n_clusters;
  __device__ int gpb() const { return hkv * pairs; }  // row groups per sequence
};

// Effective prefix of sequence b: its length, or 0 when out of bounds (the
// sequence is reported and its output left unwritten).
__device__ __forceinline__ int seq_prefix(const Sched &s, int b, bool *valid) {
  const int P = s.prefix_len[b];
  const bool ok = P >= 0 && P <= s.max_prefix && P <= s.s_max;
  *valid = ok;
  return ok ? P : 0;
}
__device__ __forceinline__ int seq_tiles(int P) { return 1 + (P + kBN - 1) / kBN; }

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Units of the row groups of sequences [0, b_end) (full warp).
__device__ long long warp_units_before(const Sched &s, int b_end) {
  const int lane = threadIdx.x & 31;
  long long acc = 0;
  for (int b0 = 0; b0 < b_end; b0 += 32) {
    long long v = 0;
    if (b0 + lane < b_end) {
      bool ok;
      v = seq_tiles(seq_prefix(s, b0 + lane, &ok));
    }
    acc += warp_sum_ll(v);
  }
  return acc * s.gpb();
}

// Sequence, row group and tile of unit u < U (full warp).
__device__ void warp_locate(const Sched &s, long long u, int *b_out, int *gi_out, int *t_out) {
  const int lane = threadIdx.x & 31;
  long long base = 0;
  for (int b0 = 0; b0 < s.batch; b0 += 32) {
    const int b = b0 + lane;
    int n = 0;
    if (b < s.batch) {
      bool ok;
      n = seq_tiles(seq_prefix(s, b, &ok));
    }
    const long long v = (long long)n * s.gpb();
    long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, b < s.batch && base + incl > u);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const long long before = base + __shfl_sync(0xffffffffu, incl - v, l);
      const int nl = __shfl_sync(0xffffffffu, n, l);
      const long long local = u - before;
      *b_out = b0 + l;
      *gi_out = (int)(local / nl);
      *t_out = (int)(local % nl);
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  *b_out = s.batch;
  *gi_out = 0;
  *t_out = 0;
}

// Tiles per row group of the lane's sequences b = 32 i + lane (B <= 128),
// loaded in one round; returns U, the units of all row groups (full warp).
constexpr int kLookupSeqs = 128;
__device__ long long warp_load_tiles(const Sched &s, int (&n)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b = 32 * i + lane;
    bool ok;
    n[i] = b < s.batch ? seq_tiles(seq_prefix(s, b, &ok)) : 0;
  }
  long long acc = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) acc += warp_sum_ll(n[i]);
  return acc * s.gpb();
}
// warp_locate with the tile counts already in registers (B <= 128).
__device__ void warp_locate_n(const Sched &s, const int (&n)[4], long long u, int *b_out, int *gi_out, int *t_out) {
  const int lane = threadIdx.x & 31;
  long long base = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long v = (long long)n[i] * s.gpb();
    long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, 32 * i + lane < s.batch && base + incl > u);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const long long before = base + __shfl_sync(0xffffffffu, incl - v, l);
      const int nl = __shfl_sync(0xffffffffu, n[i], l);
      const long long local = u - before;
      *b_out = 32 * i + l;
      *gi_out = (int)(local / nl);
      *t_out = (int)(local % nl);
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  *b_out = s.batch;
  *gi_out = 0;
  *t_out = 0;
}
// Total units U, and the sequence / row group / tile of unit u(U) (full
// warp; one round of loads when B <= 128).
template <typename UnitOf>
__device__ long long warp_find(const Sched &s, UnitOf unit_of, long long *u_out, int *b, int *gi, int *t) {
  long long U, u;
  if (s.batch <= kLookupSeqs) {
    int n[4];
    U = warp_load_tiles(s, n);
    u = unit_of(U);
    if (u >= 0) warp_locate_n(s, n, u, b, gi, t);
  } else {
    U = warp_units_before(s, s.batch);
    u = unit_of(U);
    if (u >= 0) warp_locate(s, u, b, gi, t);
  }
  *u_out = u;
  return U;
}

__device__ __forceinline__ long long range_start(long long c, long long U, long long C) { return c * U / C; }
// Cluster whose range holds unit u (the largest c with range_start(c) <= u).
__device__ __forceinline__ int cluster_of(long long u, long long U, long long C) {
  return (int)(((u + 1) * C - 1) / U);
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
  c.ok = raw >= 0 && raw <= s.max_prefix && raw <= s.s_max;
  c.P = c.ok ? raw : 0;
  c.n = seq_tiles(c.P);
}
__device__ __forceinline__ Cur cur_begin(const Bars *bars, const Sched &s) {
  Cur c;
  c.b = bars->start_b;
  c.gi = bars->start_gi;
  c.t = bars->start_t;
  cur_apply(c, s, load_prefix(s, c.b));
  c.raw_next = load_prefix(s, c.b + 1);
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
// Valid keys of a prefix tile (t >= 1).
__device__ __forceinline__ int tile_keys(const Cur &c) { return min(kBN, c.P - (c.t - 1) * kBN); }

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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_tc2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                    const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kt,
                    const __grid_constant__ CUtensorMap tm_vt, const Sched s, const uint64_t *__restrict__ anc,
                    __nv_bfloat16 *__restrict__ out, void *__restrict__ ws, int Hq, float scale_log2,
                    int32_t *status) {
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
  if (warp == 0) {
    // with C = min(clusters, U) every range below C holds at least one unit
    int b = s.batch, gi = 0, t = 0;
    long long u0;
    const long long U = warp_find(
        s, [&](long long U_) -> long long {
          const long long C = min((long long)s.n_clusters, U_);
          return cluster < C ? range_start(cluster, U_, C) : -1;
        },
        &u0, &b, &gi, &t);
    const long long C = min((long long)s.n_clusters, U);
    const long long u1 = cluster < C ? range_start(cluster + 1, U, C) : 0;
    if (lane == 0) {
      bars->start_b = b;
      bars->start_gi = gi;
      bars->start_t = t;
      bars->n_tiles = u0 >= 0 ? (int)(u1 - u0) : 0;
    }
  }
  __syncthreads();
  const int T = bars->n_tiles;
  if (T == 0) return;  // same range for both CTAs of the cluster

  if (threadIdx.x == 0) {
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
      mbar_init(&bars->qempty[i], 1);
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
  if (warp == 1) tmem_alloc_pair(&bars->tmem, 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the partner's barriers exist before any remote arrival or commit
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const int pairs = s.pairs;

  if (warp == 0 || warp == 10) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      const bool is_v = warp == 10;
      Cur c = cur_begin(bars, s);
      int seg = 0, issued = 0, q_issued = 0;
      if (!is_v) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_kc);
        tma_prefetch_desc(&tm_kt);
      } else {
        tma_prefetch_desc(&tm_vc);
        tma_prefetch_desc(&tm_vt);
      }
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
          const bool ptree = cpf.t == 0;
          const int prow = ptree ? pbh * N : pbh * s.s_max + (cpf.t - 1) * kBN;
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
          if (!mbar_wait_cluster(&bars->qempty[qb], ((seg / kQB) & 1) ^ 1, kWaitLimit) || bars->abort) {
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
        if (!mbar_wait_cluster(empty, (use & 1) ^ 1, kWaitLimit) || bars->abort) {
          give_up(bars, status);
          break;
        }
        const bool tree = c.t == 0;
        const int row0 = tree ? bh * N : bh * s.s_max + (c.t - 1) * kBN;
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
        const int nkeys = cp.t == 0 ? N : tile_keys(cp);
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
        if (!warp_wait(&bars->sfull[g % kSB], (g / kSB) & 1) || !v_ready(bars, sV, g, c.t == 0 ? N : tile_keys(c)) ||
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
    const uint32_t pair_bar = 1u + (uint32_t)quarter;
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
    const uint32_t pfull_even0 = mapa_cluster(&bars->pfull[0], 0);  // pfull[i] at + 8 i
    const float NEG_INF = -INFINITY;
    Cur c = cur_begin(bars, s);
    int seg = 0;
    bool from_start = c.t == 0;
    float ma = NEG_INF, mb = NEG_INF;  // running max of rows ra, rb (log2 units)
    float la = 0.f, lb_sum = 0.f;      // this thread's part of their sums
    // ancestor bits of a row in a row group (padding rows: all tree keys),
    // loaded one row group ahead so the tree tile never waits
    auto grow = [&](int gi, int lane_row) { return (gi % pairs) * kPairRows + (int)rank * 128 + lane_row; };
    auto load_mask = [&](int b, int gi, int lane_row) -> uint64_t {
      const int rr = grow(gi, lane_row);
      return rr < R ? anc[(int64_t)b * N + rr / G] : ~0ull;
    };
    uint64_t amask_a = c.t == 0 ? load_mask(c.b, c.gi, ra) : 0ull, amask_b = c.t == 0 ? load_mask(c.b, c.gi, rb) : 0ull;
    uint64_t next_a = 0ull, next_b = 0ull;
    bool ok = true;
    // A failed wait (timeout) or an abort turns the rest into a no-op that
    // still passes every pair barrier, so the two warps of a pair always
    // execute the same barriers.
    for (int g = 0; g < T; ++g) {
      const bool first = g == 0 || c.t == 0;
      if (first) {
        if (g > 0) {
          ++seg;
          from_start = true;
          amask_a = next_a;
          amask_b = next_b;
        }
        ma = mb = NEG_INF;
        la = lb_sum = 0.f;
      }
      if (c.t == c.n - 1 && g + 1 < T) {  // the next tile starts the next row group
        const bool same_b = c.gi + 1 < s.gpb();
        next_a = load_mask(same_b ? c.b : c.b + 1, same_b ? c.gi + 1 : 0, ra);
        next_b = load_mask(same_b ? c.b : c.b + 1, same_b ? c.gi + 1 : 0, rb);
      }
      if (ok && !warp_wait(&bars->sfull[g % kSB], (g / kSB) & 1)) ok = false;
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
      const bool tree = c.t == 0;
      const int nvalid = tree ? N : tile_keys(c);
      // The tile body comes in two instances so that full prefix tiles, the
      // steady state, carry no masking code: the masked one serves the tree
      // tile and the last, partial prefix tile.
      auto tile = [&](auto masked) {
        if constexpr (decltype(masked)::value) {
          // Visibility of this thread's keys 8j + 2 tq + e as bits 2j + e: the
          // keys below nvalid are a prefix of these bits (they increase with
          // the bit index); on the tree tile (N <= 64) also the ancestor bits.
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
            va &= mine(amask_a);
            vb &= mine(amask_b);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) {  // i = 2j + e: register 4j + e of row ra, 4j + 2 + e of row rb
            if (!((va >> i) & 1u)) sv[4 * (i >> 1) + (i & 1)] = __float_as_uint(NEG_INF);
            if (!((vb >> i) & 1u)) sv[4 * (i >> 1) + 2 + (i & 1)] = __float_as_uint(NEG_INF);
          }
        }
        // exact row max of the tile; every row sees a key in every tile
        // (itself on the tree tile), so it is finite
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
        if (ok) {
          // P = 2^(s * scale - m) as bf16 pairs: key pair 8j + 2 tq, +1 is P
          // column 4j + tq, written over the tile's first 64 S columns of this
          // warp's lanes (all of them were read above)
          const float2 sc2 = make_float2(scale_log2, scale_log2);
          const float2 na2 = make_float2(-ma, -ma), nb2 = make_float2(-mb, -mb);
          float2 sa2 = make_float2(0.f, 0.f), sb2 = make_float2(0.f, 0.f);
          uint32_t pk[32];
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
          tmem_st_16x128b_x16(s_addr, pk);
          la += sa2.x + sa2.y;
          lb_sum += sb2.x + sb2.y;
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(pfull_even0 + (uint32_t)(g % kSB) * (uint32_t)sizeof(uint64_t));
        }
      };
      if (tree || nvalid < kBN)
        tile(std::true_type{});
      else
        tile(std::false_type{});
      if (g == T - 1 || c.t == c.n - 1) {
        // ---------------------------------------------------- epilogue
        // Rows' running max and full sum through shared memory, then one row
        // per thread again (lanes of the quarter) for the O read-out: warp u
        // takes O columns [64 u, +64).
        if (ok && !warp_wait(&bars->ofull[g % kSB], (g / kSB) & 1)) ok = false;
        float sa = la + __shfl_xor_sync(0xffffffffu, la, 1);
        float sb = lb_sum + __shfl_xor_sync(0xffffffffu, lb_sum, 1);
        sa += __shfl_xor_sync(0xffffffffu, sa, 2);
        sb += __shfl_xor_sync(0xffffffffu, sb, 2);
        if (tq == 0) {
          bars->xm[ra] = ma;
          bars->xl[ra] = sa;
          bars->xm[rb] = mb;
          bars->xl[rb] = sb;
        }
        pair_sync();
        const int r = quarter * 32 + lane;  // the row this thread writes out
        const float m_row = bars->xm[r], l_row = bars->xl[r];
        pair_sync();  // read before either warp writes the next row group's
        const int rg = grow(c.gi, r);
        const bool complete = from_start && c.t == c.n - 1;
        const bool row_ok = rg < R;
        const int kvh = c.gi / pairs;
        const uint32_t q_off = (uint32_t)(quarter * 32) << 16;
        if (ok && !__any_sync(0xffffffffu, bars->abort != 0)) {
          tc_fence_after();
          if (complete) {
            const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
            __nv_bfloat16 *o = out + (((int64_t)c.b * N + rg / G) * Hq + kvh * G + rg % G) * kD + u * 64;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              uint32_t ov[32];
              tmem_ld32(tmem + q_off + kColO + u * 64 + cc * 32, ov);
              tmem_wait_ld();
              if (row_ok && c.ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(o + cc * 32);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  uint4 v;
                  v.x = pack_bf16(__uint_as_float(ov[8 * q4 + 0]) * inv, __uint_as_float(ov[8 * q4 + 1]) * inv);
                  v.y = pack_bf16(__uint_as_float(ov[8 * q4 + 2]) * inv, __uint_as_float(ov[8 * q4 + 3]) * inv);
                  v.z = pack_bf16(__uint_as_float(ov[8 * q4 + 4]) * inv, __uint_as_float(ov[8 * q4 + 5]) * inv);
                  v.w = pack_bf16(__uint_as_float(ov[8 * q4 + 6]) * inv, __uint_as_float(ov[8 * q4 + 7]) * inv);
                  dst[q4] = v;
                }
              }
            }
          } else {
            const int slot = cluster * 2 + (seg == 0 ? 0 : 1);
            uint8_t *w = reinterpret_cast<uint8_t *>(ws) +
                         ((int64_t)slot * kPairRows + (int)rank * 128 + r) * kPartialBytes;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              uint32_t ov[32];
              tmem_ld32(tmem + q_off + kColO + u * 64 + cc * 32, ov);
              tmem_wait_ld();
              if (row_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(w + u * 128 + cc * 64);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                  dst[q4] = make_uint4(pack_bf16(__uint_as_float(ov[8 * q4 + 0]), __uint_as_float(ov[8 * q4 + 1])),
                                       pack_bf16(__uint_as_float(ov[8 * q4 + 2]), __uint_as_float(ov[8 * q4 + 3])),
                                       pack_bf16(__uint_as_float(ov[8 * q4 + 4]), __uint_as_float(ov[8 * q4 + 5])),
                                       pack_bf16(__uint_as_float(ov[8 * q4 + 6]), __uint_as_float(ov[8 * q4 + 7])));
              }
            }
            if (row_ok && u == 0) *reinterpret_cast<float2 *>(w + kD * 2) = make_float2(m_row, l_row);
          }
        } else if (!ok) {
          give_up(bars, status);
        }
      }
      cur_next(c, s);
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

// Merges the partials of the row groups cut by cluster range ends.  At most
// C - 1 row groups are cut; a cut row group is merged by the blocks of the
// first range boundary inside it.  Block = (boundary k, 16 of the 256 rows);
// warp = 2 rows, lane = 4 head dims; all partials of a row are loaded at
// once (lane i: the i-th contributor's max and sum).
constexpr int kCombRows = 16;
__global__ void __launch_bounds__(256) attn_tc2_combine_kernel(const void *__restrict__ ws,
                                                               __nv_bfloat16 *__restrict__ out, const Sched s,
                                                               int Hq) {
  __shared__ int sh[7];  // usable, b, gi, c_lo, c_hi, c_lo's slot is its first
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = blockIdx.x + 1;  // boundary between clusters k-1 and k
  if (warp == 0) {
    int b = s.batch, gi = 0, t = 0;
    long long u;
    const long long U = warp_find(
        s, [&](long long U_) -> long long {
          const long long C = min((long long)s.n_clusters, U_);
          return k < C ? range_start(k, U_, C) : -1;
        },
        &u, &b, &gi, &t);
    const long long C = min((long long)s.n_clusters, U);
    int usable = 0, c_lo = 0, c_hi = 0, first = 0;
    if (u >= 0 && t != 0) {  // the boundary cuts row group (b, gi)
      bool ok;
      const int n = seq_tiles(seq_prefix(s, b, &ok));
      const long long ug = u - t;
      c_lo = cluster_of(ug, U, C);
      usable = ok && c_lo == k - 1;  // k is the first boundary inside it
      c_hi = cluster_of(ug + n - 1, U, C);
      first = range_start(c_lo, U, C) == ug;
    }
    if (lane == 0) {
      sh[0] = usable;
      sh[1] = b;
      sh[2] = gi;
      sh[3] = c_lo;
      sh[4] = c_hi;
      sh[5] = first;
    }
  }
  __syncthreads();
  if (!sh[0]) return;
  const int b = sh[1], gi = sh[2], c_lo = sh[3], c_hi = sh[4], first = sh[5];
  const int nc = c_hi - c_lo + 1;
  const int G = Hq / s.hkv, R = s.n_nodes * G;
  const int kvh = gi / s.pairs, pair = gi % s.pairs;
  auto row_of = [&](int c, int rr) -> const uint8_t * {
    const int slot = c * 2 + ((c == c_lo && !first) ? 1 : 0);
    return reinterpret_cast<const uint8_t *>(ws) + ((int64_t)slot * kPairRows + rr) * kPartialBytes;
  };
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int rr = blockIdx.y * kCombRows + warp * 2 + q;
    const int rg = pair * kPairRows + rr;
    if (rg >= R) continue;
    // the largest running max over the contributors
    float M = -INFINITY;
    for (int c0 = 0; c0 < nc; c0 += 32)
      if (c0 + lane < nc) M = fmaxf(M, reinterpret_cast<const float *>(row_of(c_lo + c0 + lane, rr) + kD * 2)[0]);
    M = sv::warp_max(M);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < nc; c0 += 32) {
      float f = 0.f;
      if (c0 + lane < nc) {
        const float2 ml = *reinterpret_cast<const float2 *>(row_of(c_lo + c0 + lane, rr) + kD * 2);
        f = exp2f(ml.x - M);
        L = fmaf(f, ml.y, L);
      }
      const int m = min(32, nc - c0);
      for (int i = 0; i < m; ++i) {
        const float fi = __shfl_sync(0xffffffffu, f, i);
        const uint2 o = reinterpret_cast<const uint2 *>(row_of(c_lo + c0 + i, rr))[lane];  // dims 4 lane .. +3
        acc.x = fmaf(fi, __uint_as_float(o.x << 16), acc.x);
        acc.y = fmaf(fi, __uint_as_float(o.x & 0xFFFF0000u), acc.y);
        acc.z = fmaf(fi, __uint_as_float(o.y << 16), acc.z);
        acc.w = fmaf(fi, __uint_as_float(o.y & 0xFFFF0000u), acc.w);
      }
    }
    L = sv::warp_sum(L);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16 *o = out + (((int64_t)b * s.n_nodes + rg / G) * Hq + kvh * G + rg % G) * kD + lane * 4;
    uint2 v;
    v.x = pack_bf16(acc.x * inv, acc.y * inv);
    v.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(o) = v;
  }
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
  if (cudaFuncSetAttribute(attn_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, attn_tc2_kernel, &cfg) != cudaSuccess || clusters < 1) return 0;
  g_clusters[dev].store(clusters);
  return clusters;
}

}  // namespace

bool sv_attn_tc2_supported(const SvAttnShape &s) {
  if (s.dtype != SPEC_BF16 || s.head_dim != kD || s.hkv < 1) return false;
  const int G = s.hq / s.hkv;
  return G <= 128 && (128 % G) == 0 && s.n_nodes * G > 128;
}

size_t sv_attn_tc2_ws_bytes() {
  const int c = tc2_clusters();
  return c > 0 ? (size_t)c * 2 * kPairRows * kPartialBytes : 0;
}

int sv_attn_tc2(const SvAttnShape &s, const void *q, const void *kc, const void *vc, const void *kt, const void *vt,
                const int32_t *prefix_len, const uint64_t *anc, void *out, float scale, void *ws, size_t ws_bytes,
                int32_t *status, cudaStream_t stream) {
  const int C = tc2_clusters();
  if (C < 1) return SPEC_ERR_CUDA;
  if (!ws || ws_bytes < sv_attn_tc2_ws_bytes()) return SPEC_ERR_CAPACITY;
  const int G = s.hq / s.hkv, R = s.n_nodes * G;
  CUtensorMap mq, mkc, mvc, mkt, mvt;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)G, (cuuint64_t)s.hkv, (cuuint64_t)s.batch * s.n_nodes};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)G * kD * 2, (cuuint64_t)s.hq * kD * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)(128 / G)};
    if (make_map(&mq, q, 4, dims, strides, box) != SPEC_OK) return SPEC_ERR_CUDA;
  }
  {
    // (at least one row so the map is valid when no prefix tile is ever loaded)
    const cuuint64_t rows = (cuuint64_t)s.batch * s.hkv * s.s_max;
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
  if (cudaFuncSetAttribute(attn_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  attn_tc2_kernel<<<2 * C, kThreads, kSmemBytes, stream>>>(mq, mkc, mvc, mkt, mvt, sc, anc, (__nv_bfloat16 *)out,
                                                          ws, s.hq, scale * 1.4426950408889634f, status);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (C > 1) {
    const dim3 cgrid(C - 1, kPairRows / kCombRows);
    attn_tc2_combine_kernel<<<cgrid, 256, 0, stream>>>(ws, (__nv_bfloat16 *)out, sc, s.hq);
  }
  return sv_launch_status();
}
