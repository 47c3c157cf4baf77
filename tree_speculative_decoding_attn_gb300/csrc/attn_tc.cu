// Tree attention on the sm_103a tensor cores (bf16 in, float32 softmax and
// accumulation, head_dim 128).
//
// "5.3 Medusa、EAGLE 与 MTP" (infra-guide), sections 3.1 and 8: every node
// attends to the shared prefix and to its ancestors-or-self; "Medusa,
// explained", step 6: all nodes are scored in one pass.
//
// One CTA per (256 query rows, KV split, sequence x KV head).  Query row r
// of a (sequence, KV head) is node r / G, head kvh*G + r % G, so the G heads
// of a GQA group and all tree nodes share every K/V tile: the tile is read
// from HBM once and feeds up to two 128-row query tiles.
//
//   warp 0      TMA producer: Q once, then K and V tiles (128 keys x 128
//               dims, 128-byte swizzle) through a two-stage ring each
//   warp 1      TMEM allocation and the MMA issuer (one lane):
//                 S_t = Q_t K^T        (A, B from shared memory)
//                 O_t += P_t V         (A = P from TMEM, B = V, MN-major)
//               issued in the order S0 S1 | PV0 S0' PV1 S1' | ... so the
//               tensor core works on one query tile while the other's
//               softmax runs
//   warps 2-9   two softmax warpgroups, one per query tile; thread = row:
//               S from TMEM, scale and mask (prefix range; ancestor bits on
//               the tree tile), P = 2^(s - m) written back as bf16 into the
//               S columns, one read of S per tile: the running max only
//               moves when a 64-column group exceeds it by more than 2^64
//               (then the sum, O and the tile's earlier P are rescaled in
//               place), which keeps every value in float32 / bf16 range.
//
// TMEM: S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512) columns.
// Every mbarrier wait is bounded; on a timeout the CTA reports
// SPEC_DEV_TIMEOUT, waits (bounded) for its own loads and MMAs, frees TMEM
// and returns.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace {

using namespace sv::ptx;

constexpr int kBN = 128;               // keys per K/V tile
constexpr int kD = 128;                // head_dim
constexpr int kStages = 2;             // K and V ring depth
constexpr int kQT = 2;                 // 128-row query tiles per CTA
constexpr int kThreads = 320;
constexpr uint32_t kTile = 128 * 128 * 2;  // bytes of one 128 x 128 bf16 tile
constexpr uint32_t kHalf = kTile / 2;      // 128 rows x 64 dims (one swizzle column)
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kGrow = 64.0f;         // log2 headroom above the running max before it is raised
constexpr int kSms = 152;

struct Bars {
  uint64_t q;
  uint64_t kfull[kStages], kempty[kStages], vfull[kStages], vempty[kStages];
  uint64_t s[kQT], p[kQT];
  uint64_t done, drain;
  uint32_t tmem;
  volatile int abort;
};
constexpr uint32_t kSmemBytes = (kQT + 2 * kStages) * kTile + sizeof(Bars) + 1024;

__device__ __forceinline__ uint32_t s_col(int t) { return (uint32_t)t * 128u; }
__device__ __forceinline__ uint32_t o_col(int t) { return 256u + (uint32_t)t * 128u; }

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);  // Q, K both K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1);  // V is MN-major (dims contiguous)

__device__ __forceinline__ void give_up(Bars *bars, int32_t *status) {
  bars->abort = 1;
  sv::report(status, SPEC_DEV_TIMEOUT);
}

// Bounded wait whose outcome is the same for every lane of the warp (so the
// warp-collective tcgen05 instructions that follow never run diverged).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, kWaitLimit));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                   const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kt,
                   const __grid_constant__ CUtensorMap tm_vt, const int32_t *__restrict__ prefix_len,
                   const uint64_t *__restrict__ anc, __nv_bfloat16 *__restrict__ out, float *__restrict__ ws,
                   int N, int Hq, int Hkv, int s_max, int max_prefix, int splits, int chunk, float scale_log2,
                   int32_t *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + kQT * kTile;
  uint8_t *sV = sK + kStages * kTile;
  Bars *bars = reinterpret_cast<Bars *>(sV + kStages * kTile);

  const int G = Hq / Hkv, R = N * G;
  const int qg = blockIdx.x, split = blockIdx.y, bh = blockIdx.z;
  const int b = bh / Hkv, kvh = bh % Hkv;
  const int row0 = qg * (kQT * 128);
  const int nq = min(kQT, (R - row0 + 127) / 128);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int P = prefix_len[b];
  if (P < 0 || P > max_prefix || P > s_max) {
    if (threadIdx.x == 0) sv::report(status, SPEC_DEV_CAPACITY);
    return;
  }
  const int k0 = split * chunk;
  const int k1 = min(P, k0 + chunk);
  const int n_pref = k1 > k0 ? (k1 - k0 + kBN - 1) / kBN : 0;
  const bool with_tree = split == splits - 1;
  const int n_tiles = n_pref + (with_tree ? 1 : 0);
  if (n_tiles == 0) {  // empty split: neutral partials (only when splits > 1)
    for (int e = threadIdx.x; e < nq * 128; e += kThreads) {
      const int rg = row0 + e;
      if (rg >= R) continue;
      float *w = ws + (((int64_t)bh * splits + split) * R + rg) * sv_partial_stride(kD);
      for (int d = 0; d < kD; ++d) w[d] = 0.f;
      w[kD] = -INFINITY;
      w[kD + 1] = 0.f;
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars->q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kfull[s], 1);
      mbar_init(&bars->vfull[s], 1);
      mbar_init(&bars->kempty[s], 1);
      mbar_init(&bars->vempty[s], 1);
    }
    for (int t = 0; t < kQT; ++t) {
      mbar_init(&bars->s[t], 1);
      mbar_init(&bars->p[t], 128);
    }
    mbar_init(&bars->done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_kc);
      tma_prefetch_desc(&tm_vc);
      mbar_expect_tx(&bars->q, nq * kTile);
      for (int t = 0; t < nq; ++t) {
        const int node0 = b * N + (row0 + t * 128) / G;
        tma_load_4d(sQ + t * kTile, &tm_q, 0, 0, kvh, node0, &bars->q);
        tma_load_4d(sQ + t * kTile + kHalf, &tm_q, 64, 0, kvh, node0, &bars->q);
      }
      int nk = 0, nv = 0;  // tiles whose K / V loads were issued
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        const bool tree = with_tree && j == n_tiles - 1;
        const CUtensorMap *mk = tree ? &tm_kt : &tm_kc;
        const CUtensorMap *mv = tree ? &tm_vt : &tm_vc;
        const int row = tree ? bh * N : bh * s_max + k0 + j * kBN;
        if (!mbar_wait(&bars->kempty[s], ph ^ 1, kWaitLimit) || bars->abort) {
          give_up(bars, status);
          break;
        }
        mbar_expect_tx(&bars->kfull[s], kTile);
        tma_load_2d(sK + s * kTile, mk, 0, row, &bars->kfull[s]);
        tma_load_2d(sK + s * kTile + kHalf, mk, 64, row, &bars->kfull[s]);
        ++nk;
        if (!mbar_wait(&bars->vempty[s], ph ^ 1, kWaitLimit) || bars->abort) {
          give_up(bars, status);
          break;
        }
        mbar_expect_tx(&bars->vfull[s], kTile);
        tma_load_2d(sV + s * kTile, mv, 0, row, &bars->vfull[s]);
        tma_load_2d(sV + s * kTile + kHalf, mv, 64, row, &bars->vfull[s]);
        ++nv;
      }
      if (bars->abort) {  // let this CTA's own copies land before it exits
        mbar_wait(&bars->q, 0, kWaitLimit);
        for (int j = nk > 2 ? nk - 2 : 0; j < nk; ++j) mbar_wait(&bars->kfull[j & 1], (j >> 1) & 1, kWaitLimit);
        for (int j = nv > 2 ? nv - 2 : 0; j < nv; ++j) mbar_wait(&bars->vfull[j & 1], (j >> 1) & 1, kWaitLimit);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV);
    auto issue_s = [&](int t, int j) {
      const uint32_t kb = ka + (uint32_t)(j & 1) * kTile, qb = qa + (uint32_t)t * kTile;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t off = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32u;
        mma_ss(tmem + s_col(t), smem_desc_sw128(qb + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024),
               kIdescQK, kk > 0);
      }
      mma_commit(&bars->s[t]);
    };
    auto issue_pv = [&](int t, int j) {
      const uint32_t vb = va + (uint32_t)(j & 1) * kTile;
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)
        mma_ts(tmem + o_col(t), tmem + s_col(t) + (uint32_t)kk * 8u,
               smem_desc_sw128(vb + (uint32_t)kk * 2048u, kHalf, 1024), kIdescPV, (j > 0 || kk > 0));
    };
    bool ok = warp_wait(&bars->q, 0) && warp_wait(&bars->kfull[0], 0);
    if (ok) {
      tc_fence_after();
      if (lane == 0) {
        for (int t = 0; t < nq; ++t) issue_s(t, 0);
        mma_commit(&bars->kempty[0]);
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!(ok = warp_wait(&bars->vfull[s], ph))) break;
      // the last prefix tile of a split may run past the split's keys: zero
      // those V rows so that stale cache rows (possibly not finite) never
      // meet the zero probabilities of masked keys
      const bool tree = with_tree && j == n_tiles - 1;
      const int nvalid = tree ? kBN : min(kBN, k1 - (k0 + j * kBN));
      if (nvalid < kBN) {
        uint4 *vs = reinterpret_cast<uint4 *>(sV + s * kTile);
        const int first = nvalid * 8, count = (kBN - nvalid) * 8;  // 16-byte chunks per half
        for (int e = lane; e < 2 * count; e += 32) {
          const int h = e / count, c = e % count;
          vs[h * (kHalf / 16) + first + c] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (!(ok = warp_wait(&bars->p[0], j & 1))) break;
      tc_fence_after();
      if (lane == 0) issue_pv(0, j);
      const bool more = j + 1 < n_tiles;
      if (more) {
        if (!(ok = warp_wait(&bars->kfull[(j + 1) & 1], ((j + 1) >> 1) & 1))) break;
        tc_fence_after();
        if (lane == 0) issue_s(0, j + 1);
      }
      if (nq > 1) {
        if (!(ok = warp_wait(&bars->p[1], j & 1))) break;
        tc_fence_after();
        if (lane == 0) issue_pv(1, j);
      }
      if (lane == 0) mma_commit(&bars->vempty[s]);
      if (more && lane == 0) {
        if (nq > 1) issue_s(1, j + 1);
        mma_commit(&bars->kempty[(j + 1) & 1]);
      }
      __syncwarp();
    }
    if (ok) {
      if (lane == 0) mma_commit(&bars->done);
    } else {
      give_up(bars, status);
      if (lane == 0) mma_commit(&bars->drain);  // let issued MMAs finish before TMEM is freed
      mbar_wait(&bars->drain, 0, kWaitLimit);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 2) >> 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int rg = row0 + t * 128 + r;
    const bool row_ok = rg < R;
    const int node = rg / G;
    const uint64_t amask = row_ok ? anc[(int64_t)b * N + node] : 0ull;
    if (t < nq) {
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < n_tiles; ++j) {
        if (!warp_wait(&bars->s[t], j & 1) || __any_sync(0xffffffffu, bars->abort != 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool tree = with_tree && j == n_tiles - 1;
        const int nvalid = tree ? N : min(kBN, k1 - (k0 + j * kBN));
        const bool masked = tree || nvalid < kBN;  // full prefix tiles need no mask
        // column `col` visible to this row (tree: col < N <= 64)
        auto visible = [&](int col) {
          return col < nvalid && (!tree || ((amask >> (col & 63)) & 1ull));
        };
        const float NEG_INF = -INFINITY;
        const uint32_t s_addr = tmem + lane_off + s_col(t);
        float2 acc2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
        // Two groups of 64 S columns; each is read into registers, then P =
        // 2^(s * scale - m) goes as bf16 pairs into 32 P columns (P columns
        // of group g only cover S columns already read).  The running max m
        // moves only when a group's max exceeds it by more than 2^kGrow (the
        // first visible scores, or inputs of extraordinary range): the row
        // sum, O and the group already written are then rescaled in place.
        // Otherwise every P stays within [0, 2^kGrow], far inside float32 and
        // bf16 range, and the normalisation by the row sum is unchanged.
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t sv2[2][32];
          tmem_ld32(s_addr + g * 64, sv2[0]);
          tmem_ld32(s_addr + g * 64 + 32, sv2[1]);
          tmem_wait_ld();
          float mx[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (masked) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (!visible(g * 64 + h * 32 + i)) sv2[h][i] = __float_as_uint(NEG_INF);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
              mx[i & 3] = fmax3(mx[i & 3], __uint_as_float(sv2[h][2 * i]), __uint_as_float(sv2[h][2 * i + 1]));
          }
          const float m_g = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
          const bool need = m_g > m_used + kGrow;  // true for the first visible scores
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? ex2(m_used - m_g) : 1.f;  // 0 when m was -inf
            if (need) {
              m_used = m_g;
              l *= alpha;
#pragma unroll
              for (int k = 0; k < 4; ++k) acc2[k] = make_float2(acc2[k].x * alpha, acc2[k].y * alpha);
            }
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
              if (j > 0) {  // the S commit this tile waited on covered every earlier PV
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                  uint32_t o[16];
                  tmem_ld16(tmem + lane_off + o_col(t) + c * 16, o);
                  tmem_wait_ld();
#pragma unroll
                  for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                  tmem_st16(tmem + lane_off + o_col(t) + c * 16, o);
                }
              }
              if (g == 1) {  // group 0 of this tile was written with the old max
                tmem_wait_st();
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                  uint32_t pw[16];
                  tmem_ld16(s_addr + c * 16, pw);
                  tmem_wait_ld();
#pragma unroll
                  for (int i = 0; i < 16; ++i) {
                    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&pw[i]);
                    pw[i] = pack_bf16(__low2float(v) * alpha, __high2float(v) * alpha);
                  }
                  tmem_st16(s_addr + c * 16, pw);
                }
              }
            }
          }
          const bool live = m_used != NEG_INF;
          const float2 sc2 = make_float2(scale_log2, scale_log2);
          const float2 nm2 = make_float2(live ? -m_used : 0.f, live ? -m_used : 0.f);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x = fma2(make_float2(__uint_as_float(sv2[h][2 * i]), __uint_as_float(sv2[h][2 * i + 1])),
                                    sc2, nm2);
              const float2 pp = live ? make_float2(ex2(x.x), ex2(x.y)) : make_float2(0.f, 0.f);
              acc2[i & 3] = add2(acc2[i & 3], pp);
              pk[i] = pack_bf16(pp.x, pp.y);
            }
            tmem_st16(s_addr + g * 32 + h * 16, pk);
          }
        }
        const float2 st2 = add2(add2(acc2[0], acc2[1]), add2(acc2[2], acc2[3]));
        const float lsum = st2.x + st2.y;
        l += lsum;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p[t]);
      }
      if (ok && !warp_wait(&bars->done, 0)) ok = false;
      if (ok && !__any_sync(0xffffffffu, bars->abort != 0)) {
        tc_fence_after();
        const int g = rg % G;
        if (splits == 1) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          __nv_bfloat16 *o = out + (((int64_t)b * N + node) * Hq + kvh * G + g) * kD;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_off + o_col(t) + c * 32, ov);
            tmem_wait_ld();
            if (row_ok) {
              uint4 *dst = reinterpret_cast<uint4 *>(o + c * 32);
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
          float *w = ws + (((int64_t)bh * splits + split) * R + rg) * sv_partial_stride(kD);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_off + o_col(t) + c * 32, ov);
            tmem_wait_ld();
            if (row_ok) {
              float4 *dst = reinterpret_cast<float4 *>(w + c * 32);
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4)
                dst[q4] = make_float4(__uint_as_float(ov[4 * q4]), __uint_as_float(ov[4 * q4 + 1]),
                                      __uint_as_float(ov[4 * q4 + 2]), __uint_as_float(ov[4 * q4 + 3]));
            }
          }
          if (row_ok) {
            w[kD] = m_used;
            w[kD + 1] = l;
          }
        }
      } else if (!ok) {
        give_up(bars, status);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda); resolved once per process.
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

}  // namespace

SvAttnPlan sv_attn_tc_plan(const SvAttnShape &s, int num_splits, bool *ok) {
  *ok = false;
  SvAttnPlan p{};
  if (s.dtype != SPEC_BF16 || s.head_dim != kD) return p;
  const int G = s.hq / s.hkv;
  if (G > 128 || (128 % G) != 0) return p;
  const int R = s.n_nodes * G;
  const int qgroups = (R + kQT * 128 - 1) / (kQT * 128);
  const int base = qgroups * s.batch * s.hkv;
  const int max_useful = s.max_prefix > 0 ? (s.max_prefix + kBN - 1) / kBN : 1;
  int splits = num_splits > 0 ? num_splits : (2 * kSms + base - 1) / base;
  if (splits > max_useful) splits = max_useful;
  if (splits > 64) splits = 64;
  if (splits < 1) splits = 1;
  int chunk = (s.max_prefix + splits - 1) / splits;
  chunk = (chunk + kBN - 1) / kBN * kBN;
  p.use_tc = 1;
  p.splits = splits;
  p.chunk = chunk;
  p.ws_bytes = splits > 1 ? (size_t)s.batch * s.hkv * splits * R * sv_partial_stride(kD) * sizeof(float) : 0;
  *ok = true;
  return p;
}

int sv_attn_tc(const SvAttnShape &s, const SvAttnPlan &p, const void *q, const void *kc, const void *vc,
               const void *kt, const void *vt, const int32_t *prefix_len, const uint64_t *anc, void *out,
               float scale, void *ws, int32_t *status, cudaStream_t stream) {
  const int G = s.hq / s.hkv;
  CUtensorMap mq, mkc, mvc, mkt, mvt;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)G, (cuuint64_t)s.hkv,
                                (cuuint64_t)s.batch * s.n_nodes};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)G * kD * 2, (cuuint64_t)s.hq * kD * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)(128 / G)};
    if (make_map(&mq, q, 4, dims, strides, box) != SPEC_OK) return SPEC_ERR_CUDA;
  }
  {
    // (at least one row so the map is valid when no prefix tile is ever loaded)
    const cuuint64_t rows = (cuuint64_t)s.batch * s.hkv * s.s_max;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, rows > 0 ? rows : 1};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBN};
    if (make_map(&mkc, kc, 2, dims, strides, box) != SPEC_OK) return SPEC_ERR_CUDA;
    if (make_map(&mvc, vc, 2, dims, strides, box) != SPEC_OK) return SPEC_ERR_CUDA;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)s.batch * s.hkv * s.n_nodes};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBN};
    if (make_map(&mkt, kt, 2, dims, strides, box) != SPEC_OK) return SPEC_ERR_CUDA;
    if (make_map(&mvt, vt, 2, dims, strides, box) != SPEC_OK) return SPEC_ERR_CUDA;
  }
  if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  const int R = s.n_nodes * G;
  dim3 grid((R + kQT * 128 - 1) / (kQT * 128), p.splits, s.batch * s.hkv);
  attn_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(
      mq, mkc, mvc, mkt, mvt, prefix_len, anc, (__nv_bfloat16 *)out, (float *)ws, s.n_nodes, s.hq, s.hkv, s.s_max,
      s.max_prefix, p.splits, p.chunk, scale * 1.4426950408889634f, status);
  return sv_launch_status();
}
