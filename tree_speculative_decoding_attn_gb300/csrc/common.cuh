// Internal helpers shared by the sm_103a kernels of the verify step.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "specverify.h"

namespace sv {

// Record the first device-side error (0 -> code); never traps.
__device__ __forceinline__ void report(int32_t *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t ptx_smem(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// 16-byte read-only streaming load (bypasses L1 allocation).
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Unpack 8 bf16 held in a uint4 into floats (exact widening).
__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float *f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}
// The same by two single-instruction 32-bit warp reductions: the largest
// high word, then the largest low word among the lanes holding it.
__device__ __forceinline__ unsigned long long warp_max_u64_redux(unsigned long long v) {
  const unsigned hi = __reduce_max_sync(0xffffffffu, (unsigned)(v >> 32));
  const unsigned lo = __reduce_max_sync(0xffffffffu, (unsigned)(v >> 32) == hi ? (unsigned)v : 0u);
  return ((unsigned long long)hi << 32) | lo;
}

// Total order key for "larger value first, then lower index first":
// maximising the key selects the larger value, and among equal values the
// lower index.  Values are finite floats; -0 and +0 compare equal, so -0 is
// mapped to +0 before its bits are used.
__device__ __forceinline__ unsigned long long rank_key(float v, uint32_t idx) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t key_index(unsigned long long k) {
  return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull);
}
__device__ __forceinline__ float key_value(unsigned long long k) {
  uint32_t u = (uint32_t)(k >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 multiplies with the Philox multipliers, key advanced by the
// Weyl increments between rounds.
struct u32x4 {
  uint32_t x, y, z, w;
};
__device__ __forceinline__ u32x4 philox4x32_10(u32x4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = u32x4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}

// Prefix cache addressing.  Contiguous: [batch, hkv, s_max, D], row
// (b * hkv + h) * s_max + key.  Paged: blocks [num_blocks, hkv, block_size,
// D] and a block table [batch, max_blocks]; key k of sequence b lives in
// block table[b][k / block_size] at row k % block_size, i.e. at row
// (block * hkv + h) * block_size + k % block_size of the pool.
struct KvPages {
  const int32_t *table;  // null: contiguous cache
  int block_size, max_blocks, num_blocks;
};
// Row of (sequence b, KV head h, prefix key `key`), or -1 for a block id
// outside the pool (reported as SPEC_DEV_BAD_BLOCK; callers read zeros).
__device__ __forceinline__ int kv_row(const KvPages &pg, int b, int hkv, int h, int s_max, int key,
                                      int32_t *status) {
  if (!pg.table) return (b * hkv + h) * s_max + key;
  const int blk = __ldg(pg.table + (int64_t)b * pg.max_blocks + key / pg.block_size);
  if (blk < 0 || blk >= pg.num_blocks) {
    report(status, SPEC_DEV_BAD_BLOCK);
    return -1;
  }
  return (blk * hkv + h) * pg.block_size + key % pg.block_size;
}

}  // namespace sv

// Launch wrapper status helper (host).
static inline int sv_launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
