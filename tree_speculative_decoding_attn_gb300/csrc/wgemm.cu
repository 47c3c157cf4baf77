// Weight-streaming GEMM on the sm_103a tensor cores: the Medusa heads and
// the LM head over the tree nodes.
//
//   Y[r, g, m] = sum_k W[g, m, k] X[r, xg, k]     bf16 in, float32 accumulate
//
// "Medusa, explained", procedure step 1: head g computes W2_g (SiLU(W1_g h) +
// h); step 6: one pass of the base model scores every tree node, whose last
// contraction is the LM head.  Both are products of a large weight matrix
// (thousands to hundreds of thousands of rows) with a few activation rows
// (one hidden state per sequence, or one per tree node): the weights are read
// once per call and dominate the traffic.
//
// Layout of the work.  The product is computed transposed: W rows are the
// MMA's M dimension (tiles of kM = 128 * MT rows, MT MMAs of M = 128 per K
// step) and the activation rows its N dimension (NT = 16 .. 256, rows past
// the valid ones read as zeros).  A tile's K range is cut into chunks of 64
// (one 128-byte swizzle row of bf16).  Every (tile, chunk) is one unit; the
// units of all tiles, in order, are split into one contiguous range per CTA
// of a persistent grid (one CTA per SM), so every SM streams the same number
// of weight bytes whatever the tile count (stream-K).
//
// A tile whose chunks span several CTAs is "cut": each contributor writes its
// float32 partial accumulator to a workspace slot and takes a ticket from the
// tile's counter (one counter per epilogue warp, which owns 32 of every 128
// W rows); the last to arrive sums all contributors' slots in CTA order (so
// the result does not depend on arrival order) and runs the epilogue.  No
// CTA or warp ever waits for another.
//
// Roles (192 threads):
//   warp 0       TMA producer: W chunk (kM x 64) and X chunk (NT x 64) per
//                stage through a ring of kStages.  With `pdl_wait` the first
//                ring's W loads are issued before griddepcontrol.wait, so the
//                weight stream starts while the producing kernel of X drains.
//   warp 1       TMEM allocation and MMA issue (one lane), accumulating each
//                tile into one of two TMEM buffers (the epilogue of a tile
//                overlaps the next tile's MMAs).
//   warps 2-5    epilogue: TMEM -> registers -> output rows (a warp's 32
//                lanes hold 32 consecutive W rows, so every store of one
//                activation row is 32 consecutive elements).
// Epilogues: kEpiF32 stores Y as float32 [rows, G, M]; kEpiSiluRes stores
// bf16 z = res[r, m] + SiLU(Y + bias[g, m]) (the Medusa FC1 step).
// Every mbarrier wait is bounded (timeout -> SPEC_DEV_TIMEOUT, clean exit).
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace {

using namespace sv::ptx;

constexpr int kThreads = 192;
constexpr int kKC = 64;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint32_t kSmemBudget = 216 * 1024;
enum { kEpiF32 = 0, kEpiSiluRes = 1, kEpiStats = 2 };

template <int NT, int MT>
struct Cfg {
  static constexpr int kM = 128 * MT;
  static constexpr uint32_t kWBytes = kM * kKC * 2;
  static constexpr uint32_t kXBytes = NT * kKC * 2;
  static constexpr uint32_t kStage = kWBytes + kXBytes;
  static constexpr int kStages = kSmemBudget / kStage;
  static constexpr int kAccCols = MT * NT;  // one accumulator buffer
  static constexpr uint32_t kTmemCols = 2 * kAccCols < 32 ? 32 : 2 * kAccCols;
  static constexpr int kCW = NT < 32 ? 16 : 32;  // TMEM columns per epilogue load
  static constexpr uint32_t kSmem = kStages * kStage + 1024 + 256;
};

// One GEMM of a launch.  A launch runs one or two of them ("phases") over
// the same activation rows and reduction length; with two, every CTA first
// takes its share of phase 0, then its share of phase 1, and phase 1 reads
// phase 0's bf16 output as its X operand (the Medusa W1 -> W2 chain).
struct Phase {
  int M, tiles_pg, n_tiles, x_grouped, epi;
  long long units;             // n_tiles * nk
  float *out;                  // kEpiF32: [*, G, M] float32
  __nv_bfloat16 *zout;         // kEpiSiluRes: [*, G, M] bf16
  const __nv_bfloat16 *res;    // kEpiSiluRes: [*, M]
  const __nv_bfloat16 *bias;   // kEpiSiluRes: [G, M] or null
  float *partial;              // [2 * n_ctas][ceil(rows / 4)][kM][4] float32
  int *counters;               // [n_tiles * 4] (one per tile and epilogue warp), zero at launch
};

struct WArgs {
  Phase ph[2];
  int nphase;
  int K, G;                    // reduction length, groups (heads)
  int rows;                    // valid activation rows of this launch (<= NT)
  int r0;                      // first activation row of this launch
  int nk, n_ctas;
  int32_t *status;
  int pdl_wait;
  float inv_t;                 // kEpiStats: 1 / temperature
  float4 *stats;               // kEpiStats: [*, rec_stride] records of 32 W rows
  int rec_stride;              // kEpiStats: records per activation row (tiles * MT * 4)
  int *xready;                 // chained phases: count of phase-0 (tile, quarter) results stored
};

__device__ __forceinline__ long long range_start(long long c, long long units, long long ctas) {
  return c * units / ctas;
}
// CTA whose range holds unit x: the largest c with range_start(c) <= x.
__device__ __forceinline__ int cta_of_unit(long long x, long long units, long long ctas) {
  return (int)(((x + 1) * ctas - 1) / units);
}

// kEpiStats: softmax statistics of the 32 W rows a warp holds for activation
// row r (warp-collective: r is the same in every lane).  Record =
// (max logit, sum exp(z - zmax), sum exp(z - zmax) (z - zmax), argmax) with
// z = logit / T and zmax = max logit / T; argmax ties go to the lowest W row,
// -1 (and a zero sum) when none of the 32 rows exists.
// (kept out of line: it is warp-collective and called from several loops,
// and inlining it everywhere bloats the kernel's instruction footprint)
__device__ __noinline__ void store_stats(const WArgs &a, const Phase &ph, int m, int rec, int r, float acc) {
  if (r >= a.rows) return;
  const bool valid = m < ph.M;
  const unsigned long long best = sv::warp_max_u64_redux(valid ? sv::rank_key(acc, (uint32_t)m) : 0ull);
  const float mx = sv::key_value(best);
  const float zmax = mx * a.inv_t, z = acc * a.inv_t;
  const float e = valid ? __expf(z - zmax) : 0.f;
  const float S = sv::warp_sum(e), Q = sv::warp_sum(e * (z - zmax));
  if ((threadIdx.x & 31) == 0)
    a.stats[(long long)(a.r0 + r) * a.rec_stride + rec] =
        make_float4(mx, S, Q, __int_as_float(best ? (int)sv::key_index(best) : -1));
}

__device__ __forceinline__ void store_final(const WArgs &a, const Phase &ph, int g, int m, int r, float acc) {
  if (r >= a.rows || m >= ph.M) return;
  const long long o = ((long long)(a.r0 + r) * a.G + g) * ph.M + m;
  if (ph.epi == kEpiF32) {
    ph.out[o] = acc;
  } else {
    float x = acc + (ph.bias ? __bfloat162float(ph.bias[(long long)g * ph.M + m]) : 0.f);
    x = x / (1.f + __expf(-x));
    ph.zout[o] = __float2bfloat16_rn(__bfloat162float(ph.res[(long long)(a.r0 + r) * ph.M + m]) + x);
  }
}

// Store (or reduce into statistics) 4 consecutive rows of one W row.
__device__ __forceinline__ void store4(const WArgs &a, const Phase &ph, int g, int m, int rec, int r, float4 v) {
  if (ph.epi == kEpiStats) {
    store_stats(a, ph, m, rec, r, v.x);
    store_stats(a, ph, m, rec, r + 1, v.y);
    store_stats(a, ph, m, rec, r + 2, v.z);
    store_stats(a, ph, m, rec, r + 3, v.w);
  } else {
    store_final(a, ph, g, m, r, v.x);
    store_final(a, ph, g, m, r + 1, v.y);
    store_final(a, ph, g, m, r + 2, v.z);
    store_final(a, ph, g, m, r + 3, v.w);
  }
}

// The CTA's units of phase p: [lo, hi).
__device__ __forceinline__ void phase_range(const WArgs &a, int p, int c, long long &lo, long long &hi) {
  lo = range_start(c, a.ph[p].units, a.n_ctas);
  hi = range_start(c + 1, a.ph[p].units, a.n_ctas);
}

template <int NT, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    wgemm_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_x0,
                 const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_x1, const WArgs a) {
  using C = Cfg<NT, MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kStage);
  uint64_t *empty = full + C::kStages;
  uint64_t *acc_full = empty + C::kStages;   // [2]
  uint64_t *acc_empty = acc_full + 2;        // [2]
  uint64_t *done = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  long long lo0, hi0, lo1 = 0, hi1 = 0;
  phase_range(a, 0, c, lo0, hi0);
  if (a.nphase > 1) phase_range(a, 1, c, lo1, hi1);
  const long long n0 = hi0 - lo0, n_it = n0 + (hi1 - lo1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tm_w0);
    tma_prefetch_desc(&tm_x0);
    if (a.nphase > 1) {
      tma_prefetch_desc(&tm_w1);
      tma_prefetch_desc(&tm_x1);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // a dependent launch may be scheduled as soon as this grid's CTAs run
  grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      // item i of this CTA: phase 0 units first, then phase 1
      auto item = [&](long long i, int &p, int &t, int &k) {
        p = i < n0 ? 0 : 1;
        const long long u = p == 0 ? lo0 + i : lo1 + (i - n0);
        t = (int)(u / a.nk);
        k = (int)(u % a.nk);
      };
      auto load_w = [&](long long i) {
        int p, t, k;
        item(i, p, t, k);
        const int s = (int)(i % C::kStages);
        mbar_expect_tx(&full[s], C::kStage);
        tma_load_3d_hint(smem + s * C::kStage, p ? &tm_w1 : &tm_w0, k * kKC, (t % a.ph[p].tiles_pg) * C::kM,
                         t / a.ph[p].tiles_pg, &full[s], pol);
      };
      auto load_x = [&](long long i) {
        int p, t, k;
        item(i, p, t, k);
        const int s = (int)(i % C::kStages);
        tma_load_3d(smem + s * C::kStage + C::kWBytes, p ? &tm_x1 : &tm_x0, k * kKC,
                    a.ph[p].x_grouped ? t / a.ph[p].tiles_pg : 0, a.r0, &full[s]);
      };
      // the first ring's weight chunks do not depend on the previous kernel
      const long long pre = a.pdl_wait ? (n_it < C::kStages ? n_it : C::kStages) : 0;
      for (long long i = 0; i < pre; ++i) load_w(i);
      if (a.pdl_wait) grid_dep_wait();
      long long w_issued = pre, issued = 0;
      bool x_ok = a.nphase < 2;  // phase 1's X is phase 0's output
      for (long long i = 0; i < n_it; ++i) {
        if (i >= w_issued) {
          const int s = (int)(i % C::kStages);
          if (!mbar_wait(&empty[s], (uint32_t)((i / C::kStages) & 1) ^ 1u, kWaitLimit) || *abort_flag) {
            *abort_flag = 1;
            sv::report(a.status, SPEC_DEV_TIMEOUT);
            break;
          }
          load_w(i);
          w_issued = i + 1;
        }
        if (i >= n0 && !x_ok) {
          // first phase-1 chunk: wait (bounded) until every phase-0 result
          // is stored, meanwhile keeping the weight stream going into every
          // ring slot the MMAs free; then make those generic-proxy stores
          // visible to TMA
          const int target = a.ph[0].n_tiles * 4;
          uint32_t spins = 0;
          while (true) {
            while (w_issued < n_it && w_issued < i + C::kStages) {
              const long long j = w_issued;
              if (j >= C::kStages && !mbar_test(&empty[j % C::kStages], (uint32_t)((j / C::kStages) & 1) ^ 1u))
                break;
              load_w(j);
              w_issued = j + 1;
            }
            int v;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.xready) : "memory");
            if (v >= target || *abort_flag) break;
            if (++spins > kWaitLimit) break;
            __nanosleep(64);
          }
          if (spins > kWaitLimit || *abort_flag) {
            *abort_flag = 1;
            sv::report(a.status, SPEC_DEV_TIMEOUT);
            break;
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");
          x_ok = true;
        }
        load_x(i);
        issued = i + 1;
      }
      if (*abort_flag) {  // let this CTA's own copies land before it exits
        const long long last = w_issued > issued ? w_issued : issued;
        for (long long i = last > C::kStages ? last - C::kStages : 0; i < last; ++i) {
          // a stage whose X was never issued completes only its W bytes: give
          // it the missing transaction count so the wait can end
          if (i >= issued) mbar_complete_tx_local(&full[i % C::kStages], C::kXBytes);
          mbar_wait(&full[i % C::kStages], (uint32_t)((i / C::kStages) & 1), kWaitLimit);
        }
      }
    }
  } else if (warp == 1) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, NT, 0, 0);
    const uint32_t base = smem_u32(smem);
    bool ok = true;
    long long it = 0;
    int seg = 0;
    for (int p = 0; p < a.nphase && ok; ++p) {
      const long long ulo = p ? lo1 : lo0, uhi = p ? hi1 : hi0;
      for (long long u = ulo; u < uhi && ok; ++seg) {
        const int klo = (int)(u % a.nk);
        const int khi = (int)((uhi - u) < (long long)(a.nk - klo) ? klo + (uhi - u) : a.nk);
        const int buf = seg & 1;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&acc_empty[buf], ((seg >> 1) & 1) ^ 1, kWaitLimit)))) break;
        tc_fence_after();
        const uint32_t dacc = tmem + (uint32_t)(buf * C::kAccCols);
        for (int k = klo; k < khi; ++k, ++it) {
          const int s = (int)(it % C::kStages);
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (uint32_t)((it / C::kStages) & 1), kWaitLimit)) &&
                     !*abort_flag))
            break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t wa = base + (uint32_t)s * C::kStage, xa = wa + C::kWBytes;
#pragma unroll
            for (int kk = 0; kk < kKC / 16; ++kk)
#pragma unroll
              for (int j = 0; j < MT; ++j)
                mma_ss(dacc + j * NT, smem_desc_sw128(wa + j * (128 * kKC * 2) + kk * 32, 16, 1024),
                       smem_desc_sw128(xa + kk * 32, 16, 1024), idesc, (k > klo || kk > 0));
            mma_commit(&empty[s]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) mma_commit(&acc_full[buf]);
        __syncwarp();
        u += khi - klo;
      }
    }
    if (!ok) {
      *abort_flag = 1;
      sv::report(a.status, SPEC_DEV_TIMEOUT);
    }
    if (lane == 0) mma_commit(done);  // also drains whatever was issued
    __syncwarp();
    mbar_wait(done, 0, kWaitLimit);
  } else {
    const int quarter = warp & 3;
    const int ml = quarter * 32 + lane;  // W row within a 128-row sub-tile
    const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);
    const int rows4 = (a.rows + 3) >> 2;
    int seg = 0;
    bool live = true;
    for (int p = 0; p < a.nphase && live; ++p) {
      const Phase &ph = a.ph[p];
      const long long ulo = p ? lo1 : lo0, uhi = p ? hi1 : hi0;
      // this quarter's results of phase 0 count toward phase 1's X readiness
      const bool feeds = p == 0 && a.nphase > 1;
      for (long long u = ulo; u < uhi; ++seg) {
        const int t = (int)(u / a.nk), klo = (int)(u % a.nk);
        const int khi = (int)((uhi - u) < (long long)(a.nk - klo) ? klo + (uhi - u) : a.nk);
        const int g = t / ph.tiles_pg, mt = t % ph.tiles_pg;
        const bool whole = klo == 0 && khi == a.nk;
        const int buf = seg & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (seg >> 1) & 1, kWaitLimit)) ||
            __any_sync(0xffffffffu, *abort_flag != 0)) {
          *abort_flag = 1;
          sv::report(a.status, SPEC_DEV_TIMEOUT);
          live = false;
          break;
        }
        tc_fence_after();
        // partial slot layout: [rows / 4][kM][4] floats, so four rows of one
        // W row are one 16-byte vector (for the reducer's loads)
        float4 *slot = reinterpret_cast<float4 *>(ph.partial) + (long long)(2 * c + (u == ulo ? 0 : 1)) * rows4 * C::kM;
#pragma unroll 1
        for (int j = 0; j < MT; ++j) {
#pragma unroll 1
          for (int cc = 0; cc < NT / C::kCW; ++cc) {
            if (cc * C::kCW >= a.rows) break;  // warp-uniform
            const uint32_t ta = tq + (uint32_t)(buf * C::kAccCols + j * NT + cc * C::kCW);
            if (whole && ph.epi == kEpiStats) {
              // statistics: one TMEM column (activation row) at a time, a
              // rolled loop (small code; this path is not bandwidth-bound)
              const int m = mt * C::kM + j * 128 + ml;
              const int rec = (mt * MT + j) * 4 + quarter;
#pragma unroll 1
              for (int i = 0; i < C::kCW && cc * C::kCW + i < a.rows; ++i) {
                uint32_t v;
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(ta + (uint32_t)i));
                tmem_wait_ld();
                store_stats(a, ph, m, rec, cc * C::kCW + i, __uint_as_float(v));
              }
              continue;
            }
            uint32_t acc[32];
            if constexpr (C::kCW == 32) {
              tmem_ld32(ta, acc);
            } else {
              tmem_ld16(ta, *reinterpret_cast<uint32_t(*)[16]>(acc));
            }
            tmem_wait_ld();
            const int m = mt * C::kM + j * 128 + ml;
            if (whole) {
              const int rec = (mt * MT + j) * 4 + quarter;
#pragma unroll
              for (int i = 0; i < C::kCW; i += 4)
                store4(a, ph, g, m, rec, cc * C::kCW + i,
                       make_float4(__uint_as_float(acc[i]), __uint_as_float(acc[i + 1]), __uint_as_float(acc[i + 2]),
                                   __uint_as_float(acc[i + 3])));
            } else {
#pragma unroll
              for (int i = 0; i < C::kCW; i += 4) {
                const int r = cc * C::kCW + i;
                if (r < a.rows)
                  slot[(long long)(r >> 2) * C::kM + j * 128 + ml] =
                      make_float4(__uint_as_float(acc[i]), __uint_as_float(acc[i + 1]), __uint_as_float(acc[i + 2]),
                                  __uint_as_float(acc[i + 3]));
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        bool stored = whole;
        if (!whole) {
          // ticket per (tile, quarter): the warp that brings the last
          // contributor's rows of this quarter reduces them; no warp waits
          __threadfence();
          __syncwarp();
          int ticket = 0;
          if (lane == 0) ticket = atomicAdd(&ph.counters[4 * t + quarter], 1);
          ticket = __shfl_sync(0xffffffffu, ticket, 0);
          const long long tu = (long long)t * a.nk;
          const int c_first = cta_of_unit(tu, ph.units, a.n_ctas);
          const int c_last = cta_of_unit(tu + a.nk - 1, ph.units, a.n_ctas);
          if (ticket == c_last - c_first) {
            stored = true;
            __threadfence();
            // Entries (sub-tile j, 4 rows) x contributors in one index space,
            // 16 loads in flight per round; each entry's contributions are
            // summed in CTA order.  Only the first contributor can have
            // started before the tile (slot 2c + 1); the others start inside
            // it (2c).
            const float4 *part = reinterpret_cast<const float4 *>(ph.partial);
            const int nc = c_last - c_first + 1;
            const int slot_first = 2 * c_first + (range_start(c_first, ph.units, a.n_ctas) >= tu ? 0 : 1);
            const int n_ent = MT * rows4;
            const int per = nc >= 16 ? 1 : 16 / nc;
#pragma unroll 1
            for (int e0 = 0; e0 < n_ent; e0 += per) {
              float4 sum[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
              for (int k0 = 0; k0 < per * nc; k0 += 16) {  // more than one round only when nc > 16
                float4 v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const int k = k0 + i, e = e0 + k / nc, cq = k % nc;
                  v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                  if (k < per * nc && e < n_ent) {
                    const int sl = cq == 0 ? slot_first : 2 * (c_first + cq);
                    const int j = e / rows4, q = e % rows4;
                    v[i] = __ldcg(part + ((long long)sl * rows4 + q) * C::kM + j * 128 + ml);
                  }
                }
                // (static register indices only: entry t takes the loads with k / nc == t)
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const int k = k0 + i, el = k / nc;
#pragma unroll
                  for (int tt = 0; tt < 16; ++tt)
                    if (el == tt && k < per * nc) {
                      sum[tt].x += v[i].x;
                      sum[tt].y += v[i].y;
                      sum[tt].z += v[i].z;
                      sum[tt].w += v[i].w;
                    }
                }
              }
#pragma unroll
              for (int el = 0; el < 16; ++el) {
                if (el >= per || e0 + el >= n_ent) break;
                const int e = e0 + el, j = e / rows4;
                store4(a, ph, g, mt * C::kM + j * 128 + ml, (mt * MT + j) * 4 + quarter, (e % rows4) * 4, sum[el]);
              }
            }
          }
        }
        if (feeds && stored) {  // this (tile, quarter) of phase 0 is final
          __threadfence();
          __syncwarp();
          if (lane == 0) atomicAdd(a.xready, 1);
        }
        u += khi - klo;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D bf16 map (K, d1, d2) with row pitch K and plane pitch d1 * K elements;
// box (64, box1, 1-or-box2), 128-byte swizzle; out-of-range rows read as 0.
int map3(CUtensorMap *m, const void *base, int K, int d1, int d2, int box1, int box2) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return SPEC_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)d1, (cuuint64_t)d2};
  const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)K * 2 * (cuuint64_t)d1};
  const cuuint32_t box[3] = {(cuuint32_t)kKC, (cuuint32_t)box1, (cuuint32_t)box2};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

inline int pick_nt(int rows) { return rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : rows <= 128 ? 128 : 256; }
inline int pick_mt(int nt) { return nt <= 128 ? 2 : 1; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// One GEMM's launch geometry and workspace: counters (4 per tile) then the
// partial slots (two per CTA).
SvGemmPlan sv_wgemm_plan(int M, int K, int G, int rows) {
  SvGemmPlan p{};
  const int rl = rows < 256 ? rows : 256;  // rows per launch
  p.nt = pick_nt(rl);
  p.mt = pick_mt(p.nt);
  const int km = 128 * p.mt;
  p.nk = K / kKC;
  p.tiles_pg = (M + km - 1) / km;
  p.n_tiles = p.tiles_pg * G;
  p.units = (long long)p.n_tiles * p.nk;
  const int sms = sm_count();
  p.n_ctas = (int)(p.units < sms ? p.units : sms);
  p.rows_per_launch = rl;
  p.counter_bytes = align256((size_t)p.n_tiles * 16);
  p.partial_bytes = align256((size_t)2 * p.n_ctas * ((rl + 3) / 4 * 4) * km * 4);
  return p;
}

namespace {

template <int NT, int MT>
int launch_t(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream) {
  using C = Cfg<NT, MT>;
  auto kern = wgemm_kernel<NT, MT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], a) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

int launch_nt(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream) {
  switch (p.nt) {
    case 16: return launch_t<16, 2>(p, maps, a, pdl, stream);
    case 32: return launch_t<32, 2>(p, maps, a, pdl, stream);
    case 64: return launch_t<64, 2>(p, maps, a, pdl, stream);
    case 128: return launch_t<128, 2>(p, maps, a, pdl, stream);
    default: return launch_t<256, 1>(p, maps, a, pdl, stream);
  }
}

Phase make_phase(const SvGemmPlan &p, int M, int x_grouped, int epi, float *out, void *zout, const void *res,
                 const void *bias, int *counters, float *partial) {
  Phase ph{};
  ph.M = M;
  ph.tiles_pg = p.tiles_pg;
  ph.n_tiles = p.n_tiles;
  ph.x_grouped = x_grouped;
  ph.epi = epi;
  ph.units = p.units;
  ph.out = out;
  ph.zout = reinterpret_cast<__nv_bfloat16 *>(zout);
  ph.res = reinterpret_cast<const __nv_bfloat16 *>(res);
  ph.bias = reinterpret_cast<const __nv_bfloat16 *>(bias);
  ph.counters = counters;
  ph.partial = partial;
  return ph;
}

}  // namespace

// One weight-streaming GEMM over all activation rows (one launch per block of
// up to 256 rows).  x: [rows, Gx, K] bf16 (Gx = G when x_grouped, else 1).
// `counters` (p.counter_bytes) must be zero for the first launch when
// `counters_clear`; otherwise they are cleared here, as they are before every
// later row block.  `pdl`: the first launch may overlap the previous kernel
// on the stream (only its X loads wait for that kernel).
int sv_wgemm(const SvGemmPlan &p, const void *w, const void *x, int x_grouped, int M, int K, int G, int rows,
             int epi, float *out, void *zout, const void *res, const void *bias, int *counters, float *partial,
             bool counters_clear, bool pdl, int32_t *status, cudaStream_t stream, float inv_t, void *stats) {
  const int km = 128 * p.mt;
  if (p.n_ctas < 1) return SPEC_ERR_CUDA;
  CUtensorMap maps[4];
  if (map3(&maps[0], w, K, M, G, km, 1) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map3(&maps[1], x, K, x_grouped ? G : 1, rows, 1, p.nt) != SPEC_OK) return SPEC_ERR_CUDA;
  maps[2] = maps[0];
  maps[3] = maps[1];
  for (int r0 = 0; r0 < rows; r0 += p.rows_per_launch) {
    if (r0 > 0 || !counters_clear)
      if (cudaMemsetAsync(counters, 0, p.counter_bytes, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    WArgs a{};
    a.ph[0] = make_phase(p, M, x_grouped, epi, out, zout, res, bias, counters, partial);
    a.nphase = 1;
    a.K = K;
    a.G = G;
    a.rows = rows - r0 < p.rows_per_launch ? rows - r0 : p.rows_per_launch;
    a.r0 = r0;
    a.nk = p.nk;
    a.n_ctas = p.n_ctas;
    a.status = status;
    const bool dep = pdl && r0 == 0 && counters_clear;
    a.pdl_wait = dep ? 1 : 0;
    a.inv_t = inv_t;
    a.stats = reinterpret_cast<float4 *>(stats);
    a.rec_stride = p.tiles_pg * p.mt * 4;
    const int rc = launch_nt(p, maps, a, dep, stream);
    if (rc != SPEC_OK) return rc;
  }
  return sv_launch_status();
}

// Medusa heads: z = h + SiLU(W1 h + b1) (bf16), then logits = W2 z (float32),
// in one persistent launch per block of up to 256 rows: every CTA streams its
// share of W1, then its share of W2; a CTA's first W2 chunks are in flight
// while the last W1 results are stored, and its first z load waits (bounded)
// until all of them are.  Workspace: both phases' counters and the readiness
// count side by side (one memset clears them), then each phase's partial
// slots.
namespace {
struct HeadsLayout {
  SvGemmPlan p1, p2;
  size_t c1, c2, ready, pa1, pa2, total;
};
HeadsLayout heads_layout(int batch, int n_heads, int hidden, int vocab) {
  HeadsLayout l{};
  l.p1 = sv_wgemm_plan(hidden, hidden, n_heads, batch);
  l.p2 = sv_wgemm_plan(vocab, hidden, n_heads, batch);
  l.c1 = 0;
  l.c2 = l.p1.counter_bytes;
  l.ready = l.c2 + l.p2.counter_bytes;
  l.pa1 = l.ready + 256;
  l.pa2 = l.pa1 + l.p1.partial_bytes;
  l.total = l.pa2 + l.p2.partial_bytes;
  return l;
}
}  // namespace

size_t sv_medusa_heads_ws_bytes(int batch, int n_heads, int hidden, int vocab) {
  return heads_layout(batch, n_heads, hidden, vocab).total;
}

int sv_medusa_heads(const void *h, const void *w1, const void *b1, const void *w2, int batch, int n_heads,
                    int hidden, int vocab, void *z, float *logits, void *ws, int32_t *status, cudaStream_t stream) {
  const HeadsLayout l = heads_layout(batch, n_heads, hidden, vocab);
  if (l.p1.n_ctas < 1 || l.p2.n_ctas < 1) return SPEC_ERR_CUDA;
  if (l.p1.nt != l.p2.nt) return SPEC_ERR_CUDA;  // same rows: same tile shape
  uint8_t *base = reinterpret_cast<uint8_t *>(ws);
  if (l.p1.n_ctas != l.p2.n_ctas) {
    // fewer W1 chunks than CTAs: one grid would leave CTAs without W1 work
    // (stream-K assumes none); two launches, the second dependent on the first
    if (cudaMemsetAsync(base, 0, l.ready, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    int rc = sv_wgemm(l.p1, w1, h, 0, hidden, hidden, n_heads, batch, kEpiSiluRes, nullptr, z, h, b1,
                      reinterpret_cast<int *>(base + l.c1), reinterpret_cast<float *>(base + l.pa1), true, false,
                      status, stream);
    if (rc != SPEC_OK) return rc;
    return sv_wgemm(l.p2, w2, z, 1, vocab, hidden, n_heads, batch, kEpiF32, logits, nullptr, nullptr, nullptr,
                    reinterpret_cast<int *>(base + l.c2), reinterpret_cast<float *>(base + l.pa2), true, true, status,
                    stream);
  }
  const int km = 128 * l.p1.mt;
  CUtensorMap maps[4];
  if (map3(&maps[0], w1, hidden, hidden, n_heads, km, 1) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map3(&maps[1], h, hidden, 1, batch, 1, l.p1.nt) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map3(&maps[2], w2, hidden, vocab, n_heads, km, 1) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map3(&maps[3], z, hidden, n_heads, batch, 1, l.p1.nt) != SPEC_OK) return SPEC_ERR_CUDA;
  const int n_ctas = l.p2.n_ctas;  // both phases are split over the whole grid
  const SvGemmPlan &p = l.p2;
  for (int r0 = 0; r0 < batch; r0 += l.p1.rows_per_launch) {
    if (cudaMemsetAsync(base, 0, l.pa1, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    WArgs a{};
    a.ph[0] = make_phase(l.p1, hidden, 0, kEpiSiluRes, nullptr, z, h, b1, reinterpret_cast<int *>(base + l.c1),
                         reinterpret_cast<float *>(base + l.pa1));
    a.ph[1] = make_phase(l.p2, vocab, 1, kEpiF32, logits, nullptr, nullptr, nullptr,
                         reinterpret_cast<int *>(base + l.c2), reinterpret_cast<float *>(base + l.pa2));
    a.nphase = 2;
    a.K = hidden;
    a.G = n_heads;
    a.rows = batch - r0 < l.p1.rows_per_launch ? batch - r0 : l.p1.rows_per_launch;
    a.r0 = r0;
    a.nk = l.p1.nk;
    a.n_ctas = n_ctas;
    a.status = status;
    a.xready = reinterpret_cast<int *>(base + l.ready);
    a.inv_t = 1.f;
    const int rc = launch_nt(p, maps, a, false, stream);
    if (rc != SPEC_OK) return rc;
  }
  return sv_launch_status();
}

size_t sv_lm_head_ws_bytes(int rows, int hidden, int vocab) {
  const SvGemmPlan p = sv_wgemm_plan(vocab, hidden, 1, rows);
  return p.counter_bytes + p.partial_bytes;
}

int sv_lm_head(const void *hid, const void *w, int rows, int hidden, int vocab, float *logits, void *ws,
               int32_t *status, cudaStream_t stream) {
  const SvGemmPlan p = sv_wgemm_plan(vocab, hidden, 1, rows);
  uint8_t *base = reinterpret_cast<uint8_t *>(ws);
  return sv_wgemm(p, w, hid, 0, vocab, hidden, 1, rows, kEpiF32, logits, nullptr, nullptr, nullptr,
                  reinterpret_cast<int *>(base), reinterpret_cast<float *>(base + p.counter_bytes), false, false,
                  status, stream);
}
