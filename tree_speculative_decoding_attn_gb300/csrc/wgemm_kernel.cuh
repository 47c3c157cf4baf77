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
// A tile whose chunks span several CTAs is "cut": each contributor writes
// its float32 partial accumulator to a workspace slot (2c for the first
// segment of CTA c's range, 2c + 1 for a later one) and the launch's
// dependent, wgemm_fixup_kernel or wgemm_fixup_stats_kernel in wgemm.cu,
// sums the slots of every cut tile in CTA order over the whole GPU and runs
// the epilogue.  Whole tiles run it here.  No CTA or warp ever waits for
// another.  (A reduction by the last contributor to arrive was measured
// slower at every shape: one warp then reads every partial of its tile.)
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
#pragma once
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace sv {
namespace wg {

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

// The GEMM of a launch: its weight matrix, tiles, units and outputs.
struct Phase {
  int M, tiles_pg, n_tiles, x_grouped, epi;  // epi: the launched kernel's epilogue
  long long units;             // n_tiles * nk
  float *out;                  // kEpiF32: [*, G, M] float32
  __nv_bfloat16 *zout;         // kEpiSiluRes: [*, G, M] bf16
  const __nv_bfloat16 *res;    // kEpiSiluRes: [*, M]
  const __nv_bfloat16 *bias;   // kEpiSiluRes: [G, M] or null
  float *partial;              // [2 * n_ctas][ceil(rows / 4)][kM][4] float32
};

struct WArgs {
  Phase ph;
  int K, G;                    // reduction length, groups (heads)
  int rows;                    // valid activation rows of this launch (<= NT)
  int r0;                      // first activation row of this launch
  int nk, n_ctas;
  int32_t *status;
  int pdl_wait;
  float inv_t;                 // kEpiStats: 1 / temperature
  float4 *stats;               // kEpiStats: [*, rec_stride] records (one per tile and epilogue warp)
  int rec_stride;              // kEpiStats: records per activation row (tiles * 4)
};

__device__ __forceinline__ long long range_start(long long c, long long units, long long ctas) {
  return c * units / ctas;
}
// CTA whose range holds unit x: the largest c with range_start(c) <= x.
__device__ __forceinline__ int cta_of_unit(long long x, long long units, long long ctas) {
  return (int)(((x + 1) * ctas - 1) / units);
}

// kEpiStats: softmax statistics over W rows.  A statistic of a set of
// logits: m = max z (z = logit / T), S = sum exp(z - m), Q = sum exp(z - m)
// (z - m), and k = the (logit, lowest W row) maximum key of the argmax.
struct St {
  float m, S, Q;
  unsigned long long k;
};
__device__ __forceinline__ St st_one(float logit, int m, bool valid, float inv_t) {
  return valid ? St{logit * inv_t, 1.f, 0.f, sv::rank_key(logit, (uint32_t)m)} : St{-INFINITY, 0.f, 0.f, 0ull};
}
// Union of two disjoint sets (both brought to the larger max).
__device__ __forceinline__ St st_merge(St a, St b) {
  if (!(b.S > 0.f)) return a;
  if (!(a.S > 0.f)) return b;
  const float mn = fmaxf(a.m, b.m), da = a.m - mn, db = b.m - mn;
  const float ea = __expf(da), eb = __expf(db);
  return St{mn, fmaf(ea, a.S, eb * b.S), fmaf(ea, fmaf(da, a.S, a.Q), eb * fmaf(db, b.S, b.Q)), a.k > b.k ? a.k : b.k};
}
__device__ __forceinline__ St st_shfl(St v, int o) {
  return St{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.S, o),
            __shfl_xor_sync(0xffffffffu, v.Q, o), __shfl_xor_sync(0xffffffffu, v.k, o)};
}
// Transpose-reduction over the warp: e[i] holds this lane's statistic of
// activation row i (16 rows); afterwards lanes l and l + 16 return the union
// over all 32 lanes of row l % 16.  At each stage a lane keeps half of its
// rows (by one bit of its lane index), sends the other half to the partner
// lane and merges what it receives (8 + 4 + 2 + 1 merges), then the two
// half-warps merge: 16 merges per lane instead of 16 full warp reductions.
__device__ __forceinline__ St st_transpose_reduce16(St (&e)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool hi = lane & o;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const St send = hi ? e[i] : e[i + o];
      const St own = hi ? e[i + o] : e[i];
      e[i] = st_merge(own, st_shfl(send, o));
    }
  }
  return st_merge(e[0], st_shfl(e[0], 16));
}
// Lane l < 16 writes the record of activation row r0 + l: (max logit, S, Q,
// argmax) with S and Q relative to max logit / T; argmax -1 and S = 0 when
// none of the record's W rows exists.
__device__ __forceinline__ void put_record(const WArgs &a, int rec, int r0, const St &t) {
  const int r = r0 + (int)(threadIdx.x & 31);
  if ((threadIdx.x & 31) >= 16 || r >= a.rows) return;
  a.stats[(long long)(a.r0 + r) * a.rec_stride + rec] =
      make_float4(t.k ? sv::key_value(t.k) : 0.f, t.S, t.Q, __int_as_float(t.k ? (int)sv::key_index(t.k) : -1));
}

template <int EPI>
__device__ __forceinline__ void store_final(const WArgs &a, const Phase &ph, int g, int m, int r, float acc) {
  if (r >= a.rows || m >= ph.M) return;
  const long long o = ((long long)(a.r0 + r) * a.G + g) * ph.M + m;
  if constexpr (EPI == kEpiF32) {
    ph.out[o] = acc;
  } else {
    float x = acc + (ph.bias ? __bfloat162float(ph.bias[(long long)g * ph.M + m]) : 0.f);
    x = x / (1.f + __expf(-x));
    ph.zout[o] = __float2bfloat16_rn(__bfloat162float(ph.res[(long long)(a.r0 + r) * ph.M + m]) + x);
  }
}

// Store (or reduce into statistics) 4 consecutive rows of one W row.
template <int EPI>
__device__ __forceinline__ void store4(const WArgs &a, const Phase &ph, int g, int m, int rec, int r, float4 v) {
  if constexpr (EPI == kEpiStats) {
    static_assert(EPI != kEpiStats, "statistics are written by the transpose-reduction paths");
  } else {
    store_final<EPI>(a, ph, g, m, r, v.x);
    store_final<EPI>(a, ph, g, m, r + 1, v.y);
    store_final<EPI>(a, ph, g, m, r + 2, v.z);
    store_final<EPI>(a, ph, g, m, r + 3, v.w);
  }
}

template <int NT, int MT, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    wgemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x, const WArgs a) {
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
  const Phase &ph = a.ph;
  const long long lo = range_start(c, ph.units, a.n_ctas), hi = range_start(c + 1, ph.units, a.n_ctas);
  const long long n_it = hi - lo;  // this CTA's units

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
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
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
      // item i of this CTA: unit lo + i = (tile t, K chunk k)
      auto item = [&](long long i, int &t, int &k) {
        const long long u = lo + i;
        t = (int)(u / a.nk);
        k = (int)(u % a.nk);
      };
      auto load_w = [&](long long i) {
        int t, k;
        item(i, t, k);
        const int s = (int)(i % C::kStages);
        mbar_expect_tx(&full[s], C::kStage);
        tma_load_3d_hint(smem + s * C::kStage, &tm_w, k * kKC, (t % ph.tiles_pg) * C::kM, t / ph.tiles_pg, &full[s],
                         pol);
      };
      auto load_x = [&](long long i) {
        int t, k;
        item(i, t, k);
        const int s = (int)(i % C::kStages);
        tma_load_3d(smem + s * C::kStage + C::kWBytes, &tm_x, k * kKC, ph.x_grouped ? t / ph.tiles_pg : 0, a.r0,
                    &full[s]);
      };
      // the first ring's weight chunks do not depend on the previous kernel
      const long long pre = a.pdl_wait ? (n_it < C::kStages ? n_it : C::kStages) : 0;
      for (long long i = 0; i < pre; ++i) load_w(i);
      if (a.pdl_wait) grid_dep_wait();
      long long w_issued = pre, issued = 0;
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
    for (long long u = lo; u < hi && ok; ++seg) {
      const int klo = (int)(u % a.nk);
      const int khi = (int)((hi - u) < (long long)(a.nk - klo) ? klo + (hi - u) : a.nk);
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
    for (long long u = lo; u < hi; ++seg) {
      const int t = (int)(u / a.nk), klo = (int)(u % a.nk);
      const int khi = (int)((hi - u) < (long long)(a.nk - klo) ? klo + (hi - u) : a.nk);
      const int g = t / ph.tiles_pg, mt = t % ph.tiles_pg;
      const bool whole = klo == 0 && khi == a.nk;
      const int buf = seg & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (seg >> 1) & 1, kWaitLimit)) ||
          __any_sync(0xffffffffu, *abort_flag != 0)) {
        *abort_flag = 1;
        sv::report(a.status, SPEC_DEV_TIMEOUT);
        break;
      }
      tc_fence_after();
      // partial slot layout: [rows / 4][kM][4] floats, so four rows of one
      // W row are one 16-byte vector (for the reducer's loads)
      float4 *slot = reinterpret_cast<float4 *>(ph.partial) + (long long)(2 * c + (u == lo ? 0 : 1)) * rows4 * C::kM;
      if constexpr (EPI == kEpiStats) {
        if (whole) {
          // 16 activation rows at a time: each lane merges its MT W rows
          // of a row, then the transpose-reduction over the warp; one
          // record per (row, tile, quarter) covering 32 * MT W rows
#pragma unroll 1
          for (int c0 = 0; c0 < a.rows && c0 < NT; c0 += 16) {
            St e[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) e[i] = St{-INFINITY, 0.f, 0.f, 0ull};
#pragma unroll
            for (int j = 0; j < MT; ++j) {
              const int m = mt * C::kM + j * 128 + ml;
              uint32_t acc[16];
              tmem_ld16(tq + (uint32_t)(buf * C::kAccCols + j * NT + c0), acc);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i)
                e[i] = st_merge(e[i], st_one(__uint_as_float(acc[i]), m, m < ph.M, a.inv_t));
            }
            put_record(a, mt * 4 + quarter, c0, st_transpose_reduce16(e));
          }
        }
      }
#pragma unroll 1
      for (int j = 0; j < MT; ++j) {
        if (EPI == kEpiStats && whole) break;
#pragma unroll 1
        for (int cc = 0; cc < NT / C::kCW; ++cc) {
          if (cc * C::kCW >= a.rows) break;  // warp-uniform
          const uint32_t ta = tq + (uint32_t)(buf * C::kAccCols + j * NT + cc * C::kCW);
          uint32_t acc[32];
          if constexpr (C::kCW == 32) {
            tmem_ld32(ta, acc);
          } else {
            tmem_ld16(ta, *reinterpret_cast<uint32_t(*)[16]>(acc));
          }
          tmem_wait_ld();
          const int m = mt * C::kM + j * 128 + ml;
          if constexpr (EPI != kEpiStats) {
            if (whole) {
              const int rec = 0;
#pragma unroll
              for (int i = 0; i < C::kCW; i += 4)
                store4<EPI>(a, ph, g, m, rec, cc * C::kCW + i,
                       make_float4(__uint_as_float(acc[i]), __uint_as_float(acc[i + 1]),
                                   __uint_as_float(acc[i + 2]), __uint_as_float(acc[i + 3])));
              continue;
            }
          }
          {
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
      u += khi - klo;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Launch one kernel instance over p.n_ctas CTAs (PDL attribute when `pdl`).
template <int NT, int MT, int EPI>
int launch_t(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream) {
  using C = Cfg<NT, MT>;
  auto kern = wgemm_kernel<NT, MT, EPI>;
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
  if (cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], a) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

template <int EPI>
int launch_nt(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream) {
  switch (p.nt) {
    case 16: return launch_t<16, 2, EPI>(p, maps, a, pdl, stream);
    case 32: return launch_t<32, 2, EPI>(p, maps, a, pdl, stream);
    case 64: return launch_t<64, 2, EPI>(p, maps, a, pdl, stream);
    case 128: return launch_t<128, 2, EPI>(p, maps, a, pdl, stream);
    default: return launch_t<256, 1, EPI>(p, maps, a, pdl, stream);
  }
}

// One translation unit per epilogue family (compiled in parallel).
int launch_f32(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream);
int launch_silu(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream);
int launch_stats(const SvGemmPlan &p, const CUtensorMap *maps, const WArgs &a, bool pdl, cudaStream_t stream);

}  // namespace wg
}  // namespace sv
