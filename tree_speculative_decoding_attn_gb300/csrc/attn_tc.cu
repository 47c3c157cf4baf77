// Tree attention on the sm_103a tensor cores (bf16 in, float32 softmax and
// accumulation, head_dim 128).
//
// "5.3 Medusa、EAGLE 与 MTP" (infra-guide), sections 3.1 and 8: every node
// attends to the shared prefix and to its ancestors-or-self; "Medusa,
// explained", step 6: all nodes are scored in one pass.
//
// Query row r of a (sequence, KV head) is node r / G, head kvh*G + r % G, so
// the G heads of a GQA group and all tree nodes share every K/V tile.  One
// CTA owns the (at most 128) query rows of a (sequence, KV head, split);
// more rows per KV head are served by the SM-pair kernel (attn_tc2.cu).
//
//   warp 0      TMA producers, lane 0: Q once, then K; lane 1: V.  Tiles of
//               128 keys x 128 dims, 128-byte swizzle, through two rings
//               that refill independently
//   warp 1      TMEM allocation and the MMA issuer (one lane):
//                 S(j) = Q K(j)^T     into TMEM buffer j % 2 (A, B in smem)
//                 O   += P(j) V(j)    (A = P in TMEM, B = V, MN-major)
//               S(j+2) is issued right after PV(j), so S for the next tile
//               is ready while the softmax of the current one runs
//   warps 2-9   softmax: two warps per TMEM lane quarter, one per half of the
//               tile's columns; thread = (row, column half).  S from TMEM,
//               scale and mask (prefix range; ancestor bits on the tree
//               tile), P = 2^(s - m) written as bf16 to a P buffer.  The first
//               tile of a row takes the exact max (shared by the pair through
//               shared memory); later tiles exponentiate against the running
//               max m in one pass and are redone exactly only if their row sum
//               leaves [0, 2^64] (a score far above m, rescaling the sum and O
//               in place), so every P stays far within float32 / bf16 range.
//
// TMEM columns: S0 [0,128)  S1 [128,256)  O [256,384)  P0 [384,448)
// P1 [448,512).
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
constexpr int kKStages = 3;            // K ring depth
constexpr int kVStages = 3;            // V ring depth
constexpr int kThreads = 320;
constexpr uint32_t kTile = 128 * 128 * 2;  // bytes of one 128 x 128 bf16 tile
constexpr uint32_t kHalf = kTile / 2;      // 128 rows x 64 dims (one swizzle column)
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kMaxTileSum = 18446744073709551616.0f;  // 2^64: bound on a tile's row sum against the running max
constexpr int kSms = 152;
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;        // two P buffers of 64 columns (128 bf16 per row)

struct Bars {
  uint64_t q;
  uint64_t kfull[kKStages], kempty[kKStages], vfull[kVStages], vempty[kVStages];
  uint64_t sfull[2], ofull[2], pfull[2], done, drain;
  uint32_t tmem;
  volatile int abort;
  float xmax[2][128];  // per-row partial maxima (then sums) of the two softmax column halves
  unsigned char xflag[2][2][128];  // per-row "tile needs the exact max" flags, by tile parity
};
constexpr uint32_t kSmemBytes = (1 + kKStages + kVStages) * kTile + sizeof(Bars) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KB");

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
                   int32_t *status, const sv::KvPages pg) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + kTile;
  uint8_t *sV = sK + kKStages * kTile;
  Bars *bars = reinterpret_cast<Bars *>(sV + kVStages * kTile);

  const int G = Hq / Hkv, R = N * G;
  const int qt = blockIdx.x, split = blockIdx.y, bh = blockIdx.z;
  const int b = bh / Hkv, kvh = bh % Hkv;
  const int row0 = qt * 128;
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
    for (int e = threadIdx.x; e < 128; e += kThreads) {
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
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars->kfull[s], 1);
      mbar_init(&bars->kempty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars->vfull[s], 1);
      mbar_init(&bars->vempty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->sfull[i], 1);
      mbar_init(&bars->ofull[i], 1);
      // one P barrier per S buffer: the softmax may finish tiles j and j+1
      // before the MMA warp observes tile j, but never tile j+2 (it needs
      // S(j+2), issued after PV(j)), so neither barrier can run two phases
      // ahead of its waiter
      mbar_init(&bars->pfull[i], 256);
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
    // ------------------------------------------------------------ producers
    // lane 0 streams Q then K, lane 1 streams V: the two rings refill
    // independently (K is released by S, V only after the softmax and PV)
    // (a 128-key tile lies inside one cache block: block sizes are multiples
    // of 128; a bad block id gives row -1, which TMA reads as zeros)
    auto tile_row = [&](int j, bool &tree) {
      tree = with_tree && j == n_tiles - 1;
      return tree ? bh * N : sv::kv_row(pg, b, Hkv, kvh, s_max, k0 + j * kBN, status);
    };
    auto stream_ring = [&](bool is_v) {
      const int n_st = is_v ? kVStages : kKStages;
      uint64_t *full = is_v ? bars->vfull : bars->kfull;
      uint64_t *empty = is_v ? bars->vempty : bars->kempty;
      uint8_t *ring = is_v ? sV : sK;
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % n_st;
        bool tree;
        const int row = tile_row(j, tree);
        const CUtensorMap *m = is_v ? (tree ? &tm_vt : &tm_vc) : (tree ? &tm_kt : &tm_kc);
        if (!mbar_wait(&empty[s], ((j / n_st) & 1) ^ 1, kWaitLimit) || bars->abort) {
          give_up(bars, status);
          break;
        }
        mbar_expect_tx(&full[s], kTile);
        tma_load_2d(ring + s * kTile, m, 0, row, &full[s]);
        tma_load_2d(ring + s * kTile + kHalf, m, 64, row, &full[s]);
        ++issued;
      }
      if (bars->abort)  // let the copies into this CTA land before it exits
        for (int j = issued > n_st ? issued - n_st : 0; j < issued; ++j)
          mbar_wait(&full[j % n_st], (j / n_st) & 1, kWaitLimit);
    };
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_kc);
      tma_prefetch_desc(&tm_vc);
      mbar_expect_tx(&bars->q, kTile);
      const int node0 = b * N + row0 / G;
      tma_load_4d(sQ, &tm_q, 0, 0, kvh, node0, &bars->q);
      tma_load_4d(sQ + kHalf, &tm_q, 64, 0, kvh, node0, &bars->q);
      stream_ring(false);
      if (bars->abort) mbar_wait(&bars->q, 0, kWaitLimit);
    } else if (lane == 1) {
      stream_ring(true);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV);
    auto release = [&](uint64_t *bar) { mma_commit(bar); };
    // S(j) = Q K(j)^T into S buffer j % 2
    auto issue_s = [&](int j) -> bool {
      const int s = j % kKStages;
      if (!warp_wait(&bars->kfull[s], (j / kKStages) & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t kb = ka + (uint32_t)s * kTile;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32u;
          mma_ss(tmem + (uint32_t)(j & 1) * 128u, smem_desc_sw128(qa + off, 16, 1024),
                 smem_desc_sw128(kb + off, 16, 1024), kIdescQK, kk > 0);
        }
        mma_commit(&bars->sfull[j & 1]);
        release(&bars->kempty[s]);
      }
      __syncwarp();
      return true;
    };
    bool ok = warp_wait(&bars->q, 0) && issue_s(0) && (n_tiles < 2 || issue_s(1));
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int s = j % kVStages;
      if (!(ok = warp_wait(&bars->vfull[s], (j / kVStages) & 1))) break;
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
      if (!(ok = warp_wait(&bars->pfull[j & 1], (j >> 1) & 1))) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t vb = va + (uint32_t)s * kTile;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(tmem + kColO, tmem + kColP + (uint32_t)(j & 1) * 64u + (uint32_t)kk * 8u,
                 smem_desc_sw128(vb + (uint32_t)kk * 2048u, kHalf, 1024), kIdescPV, (j > 0 || kk > 0));
        mma_commit(&bars->ofull[j & 1]);
        release(&bars->vempty[s]);
      }
      __syncwarp();
      if (j + 2 < n_tiles && !(ok = issue_s(j + 2))) break;
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
    // Warps 2-9: warp w reads TMEM lane quarter w % 4 (32 rows) and column
    // half h = (w - 2) / 4 of each tile; the two warps of a quarter exchange
    // their partial row maxima through shared memory (named barrier 1 + q).
    const int quarter = warp & 3;
    const int h = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t pair_bar = 1u + (uint32_t)quarter;
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
    const int rg = row0 + r;
    const bool row_ok = rg < R;
    const int node = rg / G;
    const uint64_t amask = row_ok ? anc[(int64_t)b * N + node] : 0ull;
    const float NEG_INF = -INFINITY;
    float m_used = NEG_INF, l = 0.f;  // l: this warp's half of the row sum
    bool ok = true;
    // A failed wait (timeout) or an abort turns the rest of the loop into a
    // no-op that still passes every pair barrier, so the two warps of a pair
    // always execute the same barriers.
    for (int j = 0; j < n_tiles; ++j) {
      if (ok && (!warp_wait(&bars->sfull[j & 1], (j >> 1) & 1) || __any_sync(0xffffffffu, bars->abort != 0)))
        ok = false;
      const uint32_t s_addr = tmem + lane_off + (uint32_t)(j & 1) * 128u;
      uint32_t sv[2][32];
      if (ok) {
        tc_fence_after();
        tmem_ld32(s_addr + h * 64, sv[0]);
        tmem_ld32(s_addr + h * 64 + 32, sv[1]);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[0][i] = sv[1][i] = __float_as_uint(NEG_INF);
      }
      const bool tree = with_tree && j == n_tiles - 1;
      const int nvalid = tree ? N : min(kBN, k1 - (k0 + j * kBN));
      if (tree || nvalid < kBN) {  // full prefix tiles need no mask
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const int col = h * 64 + i;
          const bool vis = col < nvalid && (!tree || ((amask >> (col & 63)) & 1ull));  // tree: col < N <= 64
          if (!vis) sv[i >> 5][i & 31] = __float_as_uint(NEG_INF);
        }
      }
      // P goes to its own TMEM buffer (P(j+2) reuses it once S(j+2),
      // issued after PV(j), has completed), so it may be written as soon as
      // it is computed
      const uint32_t p_addr = tmem + lane_off + kColP + (uint32_t)(j & 1) * 64u + (uint32_t)h * 32u;
      // P = 2^(s * scale - m) of this warp's 64 columns; returns their sum
      auto exp_write = [&](float m) -> float {
        if (!ok) return 0.f;
        const bool live = m != NEG_INF;
        const float2 sc2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(live ? -m : 0.f, live ? -m : 0.f);
        float2 acc2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x =
                fma2(make_float2(__uint_as_float(sv[c][2 * i]), __uint_as_float(sv[c][2 * i + 1])), sc2, nm2);
            const float2 pp = live ? make_float2(ex2(x.x), ex2(x.y)) : make_float2(0.f, 0.f);
            acc2[i & 3] = add2(acc2[i & 3], pp);
            pk[i] = pack_bf16(pp.x, pp.y);
          }
          tmem_st16(p_addr + c * 16, pk);
        }
        const float2 st2 = add2(add2(acc2[0], acc2[1]), add2(acc2[2], acc2[3]));
        return st2.x + st2.y;
      };
      // Exact step: the tile's row max over both column halves; a larger max
      // rescales the running sum and (from the second tile on) O, then P.
      auto exact = [&]() -> float {
        float mx[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
        for (int i = 0; i < 32; ++i)
          mx[i & 3] = fmax3(mx[i & 3], __uint_as_float(sv[i >> 4][(2 * i) & 31]),
                            __uint_as_float(sv[i >> 4][(2 * i + 1) & 31]));
        bars->xmax[h][r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        pair_sync();
        const float m_t = fmaxf(bars->xmax[0][r], bars->xmax[1][r]) * scale_log2;
        pair_sync();  // both maxima read before they are overwritten
        const bool need = m_t > m_used;
        if (ok && __any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2(m_used - m_t) : 1.f;  // 0 when m was -inf
          if (need) {
            m_used = m_t;
            l *= alpha;
          }
          // O holds PV(j-1) once that MMA completes: wait for it, then scale
          // this warp's half of the O columns
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f) &&
              (ok = warp_wait(&bars->ofull[(j - 1) & 1], ((j - 1) >> 1) & 1))) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t o[16];
              const uint32_t oa = tmem + lane_off + kColO + h * 64 + c * 16;
              tmem_ld16(oa, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st16(oa, o);
            }
          }
        }
        return exp_write(m_used);
      };
      // Both warps of a pair hold the same running max, so these decisions
      // are the same in both and the pair barriers stay matched.
      float tsum;
      if (__any_sync(0xffffffffu, m_used == NEG_INF)) {
        tsum = exact();  // first visible scores of the row
      } else {
        // later tiles: against the running max in one pass; a row whose
        // tile sum leaves [0, 2^kGrow] (a score far above the running max,
        // or an overflow) is redone exactly by both warps of the pair
        tsum = exp_write(m_used);
        bars->xflag[j & 1][h][r] = !(tsum <= kMaxTileSum);
        pair_sync();
        const bool redo = bars->xflag[j & 1][0][r] | bars->xflag[j & 1][1][r];
        if (__any_sync(0xffffffffu, redo)) tsum = exact();
      }
      if (!ok) continue;
      l += tsum;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->pfull[j & 1]);
    }
    // full row sum: both halves (same running max on both warps)
    bars->xmax[h][r] = l;
    pair_sync();
    const float l_row = bars->xmax[0][r] + bars->xmax[1][r];
    if (ok && !warp_wait(&bars->done, 0)) ok = false;
    if (ok && !__any_sync(0xffffffffu, bars->abort != 0)) {
      tc_fence_after();
      const int g = rg % G;
      if (splits == 1) {
        const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
        __nv_bfloat16 *o = out + (((int64_t)b * N + node) * Hq + kvh * G + g) * kD + h * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_off + kColO + h * 64 + c * 32, ov);
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
        for (int c = 0; c < 2; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_off + kColO + h * 64 + c * 32, ov);
          tmem_wait_ld();
          if (row_ok) {
            float4 *dst = reinterpret_cast<float4 *>(w + h * 64 + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(ov[4 * q4]), __uint_as_float(ov[4 * q4 + 1]),
                                    __uint_as_float(ov[4 * q4 + 2]), __uint_as_float(ov[4 * q4 + 3]));
          }
        }
        if (row_ok && h == 0) {
          w[kD] = m_used;
          w[kD + 1] = l_row;
        }
      }
    } else if (!ok) {
      give_up(bars, status);
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

int launch_tc(dim3 grid, cudaStream_t stream, const CUtensorMap &mq, const CUtensorMap &mkc, const CUtensorMap &mvc,
              const CUtensorMap &mkt, const CUtensorMap &mvt, const int32_t *prefix_len, const uint64_t *anc,
              void *out, void *ws, const SvAttnShape &s, const SvAttnPlan &p, float scale, int32_t *status) {
  if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  attn_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(
      mq, mkc, mvc, mkt, mvt, prefix_len, anc, (__nv_bfloat16 *)out, (float *)ws, s.n_nodes, s.hq, s.hkv, s.s_max,
      s.max_prefix, p.splits, p.chunk, scale * 1.4426950408889634f, status,
      sv::KvPages{s.block_table, s.block_size, s.max_blocks, s.num_blocks});
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Modelled time of one split count, in units of one K/V tile streamed by
// one SM: CTAs are dispatched in launch order (split fastest, then
// sequence x KV head) onto the free SMs;
// each streams its prefix chunk, the tree tile on the last split, and about
// one tile's worth of set-up.  Split partials cost their write and re-read
// plus a combine launch.  `prefix` holds each sequence's prefix length, or
// is null for "every sequence at max_prefix".
double tc_split_cost(const SvAttnShape &s, const int32_t *prefix, int splits) {
  const int G = s.hq / s.hkv, R = s.n_nodes * G;
  const int slots = kSms;
  int chunk = (s.max_prefix + splits - 1) / splits;
  chunk = (chunk + kBN - 1) / kBN * kBN;
  // min-heap of slot finish times (small arrays: slots <= 152)
  double finish[kSms];
  for (int i = 0; i < slots; ++i) finish[i] = 0.0;
  for (int bh = 0; bh < s.batch * s.hkv; ++bh) {
    const int P = prefix ? prefix[bh / s.hkv] : s.max_prefix;
    for (int sp = 0; sp < splits; ++sp) {
      const int k0 = sp * chunk, k1 = P < k0 + chunk ? P : k0 + chunk;
      const int tiles = k1 > k0 ? (k1 - k0 + kBN - 1) / kBN : 0;
      const double work = tiles + (sp == splits - 1 ? 2.0 : (tiles ? 1.0 : 0.1));
      int best = 0;
      for (int i = 1; i < slots; ++i)
        if (finish[i] < finish[best]) best = i;
      finish[best] += work;
    }
  }
  double makespan = 0.0;
  for (int i = 0; i < slots; ++i) makespan = finish[i] > makespan ? finish[i] : makespan;
  if (splits > 1) {
    const double tile_bytes = (double)kBN * kD * 2 * 2 * slots;  // bytes moved per unit of time
    const double partial = 2.0 * s.batch * s.hkv * splits * R * sv_partial_stride(kD) * 4.0;
    // the combine launch, plus about one tile per split for the partial rows'
    // write-back and merge (measured on the 32-head, 2048-key shape: three
    // splits beat four)
    makespan += partial / tile_bytes + 4.0 + splits;
  }
  return makespan;
}

int tc_best_splits(const SvAttnShape &s, const int32_t *prefix) {
  const int max_useful = s.max_prefix > 0 ? (s.max_prefix + kBN - 1) / kBN : 1;
  int best = 1;
  double best_cost = tc_split_cost(s, prefix, 1);
  for (int c = 2; c <= 64 && c <= max_useful; ++c) {
    const double cost = tc_split_cost(s, prefix, c);
    if (cost < best_cost) {
      best_cost = cost;
      best = c;
    }
  }
  return best;
}

}  // namespace

bool sv_attn_tc_supported(const SvAttnShape &s) {
  if (s.dtype != SPEC_BF16 || s.head_dim != kD) return false;
  const int G = s.hq / s.hkv;
  return s.n_nodes <= 64 && G <= 128 && (128 % G) == 0 && s.n_nodes * G <= 128;
}

int sv_attn_tc_ragged_splits(const SvAttnShape &s, const int32_t *host_prefix) {
  return tc_best_splits(s, host_prefix);
}

SvAttnPlan sv_attn_tc_plan(const SvAttnShape &s, int num_splits, bool *ok) {
  *ok = false;
  SvAttnPlan p{};
  if (!sv_attn_tc_supported(s)) return p;
  const int R = s.n_nodes * (s.hq / s.hkv);
  const int max_useful = s.max_prefix > 0 ? (s.max_prefix + kBN - 1) / kBN : 1;
  int splits = num_splits > 0 ? num_splits : tc_best_splits(s, nullptr);
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
    // (at least one row so the map is valid when no prefix tile is ever
    // loaded; a paged cache is one pool of blocks)
    const cuuint64_t rows = s.block_table ? (cuuint64_t)s.num_blocks * s.hkv * s.block_size
                                          : (cuuint64_t)s.batch * s.hkv * s.s_max;
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
  const dim3 grid(1, p.splits, s.batch * s.hkv);  // at most 128 query rows: one query tile
  return launch_tc(grid, stream, mq, mkc, mvc, mkt, mvt, prefix_len, anc, out, ws, s, p, scale, status);
}
