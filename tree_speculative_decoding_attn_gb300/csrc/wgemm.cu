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
enum { kEpiF32 = 0, kEpiSiluRes = 1 };

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

struct WArgs {
  int M, K, G;           // W rows per group, reduction length, groups
  int rows;              // valid activation rows of this launch (<= NT)
  int r0;                // first activation row of this launch
  int x_grouped;         // 1: group g reads X group g; 0: X group 0
  int nk, tiles_pg, n_tiles, n_ctas;
  long long units;       // n_tiles * nk
  float *out;            // kEpiF32: [*, G, M] float32
  __nv_bfloat16 *zout;   // kEpiSiluRes: [*, G, M] bf16
  const __nv_bfloat16 *res;   // kEpiSiluRes: [*, M]
  const __nv_bfloat16 *bias;  // kEpiSiluRes: [G, M] or null
  float *partial;        // [2 * n_ctas][rows][kM] float32
  int *counters;         // [n_tiles * 4] (one per tile and epilogue warp), zero at launch
  int32_t *status;
  int pdl_wait;
};

__device__ __forceinline__ long long range_start(long long c, long long units, long long ctas) {
  return c * units / ctas;
}
// CTA whose range holds unit x: the largest c with range_start(c) <= x.
__device__ __forceinline__ int cta_of_unit(long long x, long long units, long long ctas) {
  return (int)(((x + 1) * ctas - 1) / units);
}

template <int NT, int MT, int EPI>
__device__ __forceinline__ void store_final(const WArgs &a, int g, int m, int r, float acc) {
  if (r >= a.rows || m >= a.M) return;
  const long long o = ((long long)(a.r0 + r) * a.G + g) * a.M + m;
  if constexpr (EPI == kEpiF32) {
    a.out[o] = acc;
  } else {
    float x = acc + (a.bias ? __bfloat162float(a.bias[(long long)g * a.M + m]) : 0.f);
    x = x / (1.f + __expf(-x));
    a.zout[o] = __float2bfloat16_rn(__bfloat162float(a.res[(long long)(a.r0 + r) * a.M + m]) + x);
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
  const long long u0 = range_start(c, a.units, a.n_ctas), u1 = range_start(c + 1, a.units, a.n_ctas);

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
      const long long n_it = u1 - u0;
      const long long pre = a.pdl_wait ? (n_it < C::kStages ? n_it : C::kStages) : 0;
      // the first ring's weight chunks do not depend on the previous kernel
      for (long long i = 0; i < pre; ++i) {
        const long long u = u0 + i;
        const int t = (int)(u / a.nk), k = (int)(u % a.nk);
        uint8_t *st = smem + i * C::kStage;
        mbar_expect_tx(&full[i], C::kStage);
        tma_load_3d_hint(st, &tm_w, k * kKC, (t % a.tiles_pg) * C::kM, t / a.tiles_pg, &full[i], pol);
      }
      if (a.pdl_wait) grid_dep_wait();
      long long issued = 0;
      for (long long i = 0; i < n_it; ++i) {
        const int s = (int)(i % C::kStages);
        if (i >= pre) {
          if (!mbar_wait(&empty[s], (uint32_t)((i / C::kStages) & 1) ^ 1u, kWaitLimit) || *abort_flag) {
            *abort_flag = 1;
            sv::report(a.status, SPEC_DEV_TIMEOUT);
            break;
          }
        }
        const long long u = u0 + i;
        const int t = (int)(u / a.nk), k = (int)(u % a.nk);
        const int g = t / a.tiles_pg;
        uint8_t *st = smem + s * C::kStage;
        if (i >= pre) {
          mbar_expect_tx(&full[s], C::kStage);
          tma_load_3d_hint(st, &tm_w, k * kKC, (t % a.tiles_pg) * C::kM, g, &full[s], pol);
        }
        tma_load_3d(st + C::kWBytes, &tm_x, k * kKC, a.x_grouped ? g : 0, a.r0, &full[s]);
        issued = i + 1;
      }
      if (*abort_flag)  // let this CTA's own copies land before it exits
        for (long long i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i)
          mbar_wait(&full[i % C::kStages], (uint32_t)((i / C::kStages) & 1), kWaitLimit);
    }
  } else if (warp == 1) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, NT, 0, 0);
    const uint32_t base = smem_u32(smem);
    bool ok = true;
    long long it = 0;
    int seg = 0;
    for (long long u = u0; u < u1 && ok; ++seg) {
      const int klo = (int)(u % a.nk);
      const int khi = (int)((u1 - u) < (long long)(a.nk - klo) ? klo + (u1 - u) : a.nk);
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
    int seg = 0;
    for (long long u = u0; u < u1; ++seg) {
      const int t = (int)(u / a.nk), klo = (int)(u % a.nk);
      const int khi = (int)((u1 - u) < (long long)(a.nk - klo) ? klo + (u1 - u) : a.nk);
      const int g = t / a.tiles_pg, mt = t % a.tiles_pg;
      const bool whole = klo == 0 && khi == a.nk;
      const int buf = seg & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (seg >> 1) & 1, kWaitLimit)) ||
          __any_sync(0xffffffffu, *abort_flag != 0)) {
        *abort_flag = 1;
        sv::report(a.status, SPEC_DEV_TIMEOUT);
        break;
      }
      tc_fence_after();
      float *slot = a.partial + (long long)(2 * c + (u == u0 ? 0 : 1)) * a.rows * C::kM;
#pragma unroll 1
      for (int j = 0; j < MT; ++j) {
#pragma unroll 1
        for (int cc = 0; cc < NT / C::kCW; ++cc) {
          if (cc * C::kCW >= a.rows) break;  // warp-uniform
          uint32_t acc[32];
          const uint32_t ta = tq + (uint32_t)(buf * C::kAccCols + j * NT + cc * C::kCW);
          if constexpr (C::kCW == 32) {
            tmem_ld32(ta, acc);
          } else {
            tmem_ld16(ta, *reinterpret_cast<uint32_t(*)[16]>(acc));
          }
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < C::kCW; ++i) {
            const int r = cc * C::kCW + i;
            if (whole) {
              store_final<NT, MT, EPI>(a, g, mt * C::kM + j * 128 + ml, r, __uint_as_float(acc[i]));
            } else if (r < a.rows) {
              slot[(long long)r * C::kM + j * 128 + ml] = __uint_as_float(acc[i]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
      if (!whole) {
        // ticket per (tile, quarter): the warp that brings the last
        // contributor's rows of this quarter reduces them; no warp waits
        __threadfence();
        __syncwarp();
        int ticket = 0;
        if (lane == 0) ticket = atomicAdd(&a.counters[4 * t + quarter], 1);
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        const long long tu = (long long)t * a.nk;
        const int c_first = cta_of_unit(tu, a.units, a.n_ctas);
        const int c_last = cta_of_unit(tu + a.nk - 1, a.units, a.n_ctas);
        if (ticket == c_last - c_first) {
          __threadfence();
          // 16 rows at a time, each contributor's 16 loads issued together
#pragma unroll 1
          for (int j = 0; j < MT; ++j) {
#pragma unroll 1
            for (int r0 = 0; r0 < a.rows; r0 += 16) {
              float sum[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) sum[i] = 0.f;
#pragma unroll 1
              for (int cq = c_first; cq <= c_last; ++cq) {
                const int sl = 2 * cq + (range_start(cq, a.units, a.n_ctas) >= tu ? 0 : 1);
                const float *src = a.partial + ((long long)sl * a.rows + r0) * C::kM + j * 128 + ml;
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = r0 + i < a.rows ? __ldcg(src + (long long)i * C::kM) : 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) sum[i] += v[i];
              }
#pragma unroll
              for (int i = 0; i < 16; ++i) store_final<NT, MT, EPI>(a, g, mt * C::kM + j * 128 + ml, r0 + i, sum[i]);
            }
          }
        }
      }
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
  p.partial_bytes = align256((size_t)2 * p.n_ctas * rl * km * 4);
  return p;
}

namespace {

template <int NT, int MT, int EPI>
int launch_t(const SvGemmPlan &p, const CUtensorMap &mw, const CUtensorMap &mx, const WArgs &a, bool pdl,
             cudaStream_t stream) {
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
  if (cudaLaunchKernelEx(&cfg, kern, mw, mx, a) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

template <int EPI>
int launch_nt(const SvGemmPlan &p, const CUtensorMap &mw, const CUtensorMap &mx, const WArgs &a, bool pdl,
              cudaStream_t stream) {
  switch (p.nt) {
    case 16: return launch_t<16, 2, EPI>(p, mw, mx, a, pdl, stream);
    case 32: return launch_t<32, 2, EPI>(p, mw, mx, a, pdl, stream);
    case 64: return launch_t<64, 2, EPI>(p, mw, mx, a, pdl, stream);
    case 128: return launch_t<128, 2, EPI>(p, mw, mx, a, pdl, stream);
    default: return launch_t<256, 1, EPI>(p, mw, mx, a, pdl, stream);
  }
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
             bool counters_clear, bool pdl, int32_t *status, cudaStream_t stream) {
  const int km = 128 * p.mt;
  if (p.n_ctas < 1) return SPEC_ERR_CUDA;
  CUtensorMap mw, mx;
  if (map3(&mw, w, K, M, G, km, 1) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map3(&mx, x, K, x_grouped ? G : 1, rows, 1, p.nt) != SPEC_OK) return SPEC_ERR_CUDA;
  for (int r0 = 0; r0 < rows; r0 += p.rows_per_launch) {
    if (r0 > 0 || !counters_clear)
      if (cudaMemsetAsync(counters, 0, p.counter_bytes, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    WArgs a{};
    a.M = M; a.K = K; a.G = G;
    a.rows = rows - r0 < p.rows_per_launch ? rows - r0 : p.rows_per_launch;
    a.r0 = r0; a.x_grouped = x_grouped;
    a.nk = p.nk; a.tiles_pg = p.tiles_pg; a.n_tiles = p.n_tiles; a.n_ctas = p.n_ctas; a.units = p.units;
    a.out = out; a.zout = reinterpret_cast<__nv_bfloat16 *>(zout);
    a.res = reinterpret_cast<const __nv_bfloat16 *>(res);
    a.bias = reinterpret_cast<const __nv_bfloat16 *>(bias);
    a.partial = partial; a.counters = counters; a.status = status;
    const bool dep = pdl && r0 == 0 && counters_clear;
    a.pdl_wait = dep ? 1 : 0;
    const int rc = epi == kEpiF32 ? launch_nt<kEpiF32>(p, mw, mx, a, dep, stream)
                                  : launch_nt<kEpiSiluRes>(p, mw, mx, a, dep, stream);
    if (rc != SPEC_OK) return rc;
  }
  return sv_launch_status();
}

// Medusa heads: z = h + SiLU(W1 h + b1) (bf16), then logits = W2 z (float32).
// Workspace: both GEMMs' counters side by side (one memset clears them),
// then each GEMM's partial slots.  With a single row block the second GEMM
// launches as a programmatic dependent of the first: its weight stream starts
// while the first drains, and only its z loads wait.
size_t sv_medusa_heads_ws_bytes(int batch, int n_heads, int hidden, int vocab) {
  const SvGemmPlan p1 = sv_wgemm_plan(hidden, hidden, n_heads, batch);
  const SvGemmPlan p2 = sv_wgemm_plan(vocab, hidden, n_heads, batch);
  return p1.counter_bytes + p2.counter_bytes + p1.partial_bytes + p2.partial_bytes;
}

int sv_medusa_heads(const void *h, const void *w1, const void *b1, const void *w2, int batch, int n_heads,
                    int hidden, int vocab, void *z, float *logits, void *ws, int32_t *status, cudaStream_t stream) {
  const SvGemmPlan p1 = sv_wgemm_plan(hidden, hidden, n_heads, batch);
  const SvGemmPlan p2 = sv_wgemm_plan(vocab, hidden, n_heads, batch);
  uint8_t *base = reinterpret_cast<uint8_t *>(ws);
  int *c1 = reinterpret_cast<int *>(base), *c2 = reinterpret_cast<int *>(base + p1.counter_bytes);
  float *pa1 = reinterpret_cast<float *>(base + p1.counter_bytes + p2.counter_bytes);
  float *pa2 = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(pa1) + p1.partial_bytes);
  const bool single = batch <= p1.rows_per_launch;
  if (single && cudaMemsetAsync(base, 0, p1.counter_bytes + p2.counter_bytes, stream) != cudaSuccess)
    return SPEC_ERR_CUDA;
  int rc = sv_wgemm(p1, w1, h, 0, hidden, hidden, n_heads, batch, kEpiSiluRes, nullptr, z, h, b1, c1, pa1, single,
                    false, status, stream);
  if (rc != SPEC_OK) return rc;
  return sv_wgemm(p2, w2, z, 1, vocab, hidden, n_heads, batch, kEpiF32, logits, nullptr, nullptr, nullptr, c2, pa2,
                  single, single, status, stream);
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
