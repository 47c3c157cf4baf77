// LM head over the tree nodes on the sm_103a tensor cores:
// logits[r, v] = sum_i hid[r, i] W[v, i]  (bf16 in, float32 accumulate/out).
//
// "Medusa, explained", step 6: one forward pass of the base model scores
// every tree node; the LM head is that pass's last contraction.
//
// With tens of tree rows against a vocabulary of tens of thousands, the
// product is computed transposed: the vocabulary is the MMA's M dimension
// (128-row tiles of W, one per CTA) and the tree rows its N dimension, so
// each CTA streams its 128 W rows once while the small hidden-state matrix
// is re-read from L2.
//   warp 0      TMA producer: K chunks of 64 (W 128 x 64, hid N x 64, 128-byte
//               swizzle) through a ring of kStages
//   warp 1      TMEM allocation and MMA issue (one lane): D[128 x N] +=
//               W_chunk . hid_chunk^T, four K=16 steps per chunk
//   warps 2-5   epilogue: TMEM -> registers -> logits (each warp its 32 vocab
//               rows; a warp's stores for one tree row are 32 consecutive
//               floats)
// Every mbarrier wait is bounded (timeout -> SPEC_DEV_TIMEOUT, clean exit).
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace {

using namespace sv::ptx;

constexpr int kThreads = 192;
constexpr int kKC = 64;                     // K elements per chunk (one 128-byte swizzle row)
constexpr uint32_t kWTile = 128 * kKC * 2;  // 16 KB
constexpr uint32_t kWaitLimit = 1u << 22;

// With up to 64 tree rows two CTAs share an SM (half the ring each, the
// same bytes in flight per SM), so a vocabulary of a few hundred tiles is
// resident in one wave instead of running 1.6 waves of one CTA per SM.
template <int NT>
struct GemmCfg {
  static constexpr uint32_t kHTile = NT * kKC * 2;
  static constexpr uint32_t kStage = kWTile + kHTile;
  static constexpr int kCtasPerSm = NT <= 64 ? 2 : 1;
  static constexpr int kStages = ((kCtasPerSm == 2 ? 104 : 192) * 1024) / kStage;
  static constexpr uint32_t kSmem = kStages * kStage + 256 + 1024;
};

template <int NT>
__global__ void __launch_bounds__(kThreads, GemmCfg<NT>::kCtasPerSm)
    lm_head_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h, int R, int V,
                      int hidden, float *__restrict__ out, int32_t *status) {
  using C = GemmCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kStage);
  uint64_t *empty = full + C::kStages;
  uint64_t *done = empty + C::kStages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v0 = blockIdx.x * 128, r0 = blockIdx.y * NT;
  const int nk = hidden / kKC;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, NT < 32 ? 32 : NT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int k = 0; k < nk; ++k) {
        const int s = k % C::kStages;
        if (!mbar_wait(&empty[s], ((k / C::kStages) & 1) ^ 1, kWaitLimit) || *abort_flag) {
          *abort_flag = 1;
          sv::report(status, SPEC_DEV_TIMEOUT);
          break;
        }
        uint8_t *st = smem + s * C::kStage;
        mbar_expect_tx(&full[s], C::kStage);
        tma_load_2d(st, &tm_w, k * kKC, v0, &full[s]);
        tma_load_2d(st + kWTile, &tm_h, k * kKC, r0, &full[s]);
        ++issued;
      }
      if (*abort_flag)  // let this CTA's own copies land before it exits
        for (int k = issued > C::kStages ? issued - C::kStages : 0; k < issued; ++k)
          mbar_wait(&full[k % C::kStages], (k / C::kStages) & 1, kWaitLimit);
    }
  } else if (warp == 1) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, NT, 0, 0);
    const uint32_t base = smem_u32(smem);
    bool ok = true;
    for (int k = 0; k < nk; ++k) {
      const int s = k % C::kStages;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (k / C::kStages) & 1, kWaitLimit)))) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t wa = base + (uint32_t)s * C::kStage, ha = wa + kWTile;
#pragma unroll
        for (int kk = 0; kk < kKC / 16; ++kk)
          mma_ss(tmem, smem_desc_sw128(wa + kk * 32, 16, 1024), smem_desc_sw128(ha + kk * 32, 16, 1024), idesc,
                 (k > 0 || kk > 0));
        mma_commit(&empty[s]);
      }
      __syncwarp();
    }
    if (!ok) {
      *abort_flag = 1;
      sv::report(status, SPEC_DEV_TIMEOUT);
    }
    if (lane == 0) mma_commit(done);  // also drains whatever was issued
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int v = v0 + quarter * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
    if (__all_sync(0xffffffffu, mbar_wait(done, 0, kWaitLimit)) && !__any_sync(0xffffffffu, *abort_flag != 0)) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < NT / 32; ++c) {
        uint32_t acc[32];
        tmem_ld32(taddr + c * 32, acc);
        tmem_wait_ld();
        if (v < V) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int r = r0 + c * 32 + j;
            if (r < R) out[(int64_t)r * V + v] = __uint_as_float(acc[j]);
          }
        }
      }
    } else {
      sv::report(status, SPEC_DEV_TIMEOUT);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, NT < 32 ? 32 : NT);
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

int map_rows(CUtensorMap *m, const void *base, int cols, int rows, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return SPEC_ERR_CUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kKC, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

template <int NT>
int launch(const void *hid, const void *w, int rows, int hidden, int vocab, float *logits, int32_t *status,
           cudaStream_t stream) {
  CUtensorMap mw, mh;
  if (map_rows(&mw, w, hidden, vocab, 128) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map_rows(&mh, hid, hidden, rows, NT) != SPEC_OK) return SPEC_ERR_CUDA;
  if (cudaFuncSetAttribute(lm_head_tc_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)GemmCfg<NT>::kSmem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  const dim3 grid((vocab + 127) / 128, (rows + NT - 1) / NT);
  lm_head_tc_kernel<NT><<<grid, kThreads, GemmCfg<NT>::kSmem, stream>>>(mw, mh, rows, vocab, hidden, logits, status);
  return sv_launch_status();
}

}  // namespace

int sv_lm_head_tc(const void *hid, const void *w, int rows, int hidden, int vocab, float *logits, int32_t *status,
                  cudaStream_t stream) {
  if (rows <= 64) return launch<64>(hid, w, rows, hidden, vocab, logits, status, stream);
  if (rows <= 128) return launch<128>(hid, w, rows, hidden, vocab, logits, status, stream);
  return launch<256>(hid, w, rows, hidden, vocab, logits, status, stream);
}
