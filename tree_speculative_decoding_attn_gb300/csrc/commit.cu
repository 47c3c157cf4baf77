// Commit of the accepted path's K/V: "5.3 Medusa、EAGLE 与 MTP"
// (infra-guide), section 3.2 -- all nodes share the prefix KV; only the
// accepted path is committed and the other branches' temporary KV is
// discarded.  The tree K/V live in their own buffer, so the copy never
// overlaps its source and needs no in-place compaction.
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ bool commit_ok(int P, int L, int s_max, int path_cap, int N,
                                          const int32_t *path, int *code) {
  if (P < 0 || L < 0 || L + 1 > path_cap || P + L + 1 > s_max) {
    *code = SPEC_DEV_CAPACITY;
    return false;
  }
  for (int j = 0; j <= L; ++j)
    if (path[j] < 0 || path[j] >= N) {
      *code = SPEC_DEV_BAD_PATH;
      return false;
    }
  return true;
}

// grid: (layer * batch * hkv); each CTA copies rows 0..L of one
// (layer, sequence, KV head) for K and V with 16-byte vectors.
__global__ void __launch_bounds__(kThreads)
    commit_copy_kernel(uint4 *kc, uint4 *vc, const uint4 *__restrict__ kt,
                       const uint4 *__restrict__ vt, int batch, int hkv, int s_max, int N,
                       int vec_per_row, const int32_t *__restrict__ acc_len,
                       const int32_t *__restrict__ acc_path, int path_cap,
                       const int32_t *__restrict__ prefix_len, int32_t *status) {
  __shared__ int s_path[SPEC_MAX_NODES + 1];
  __shared__ int s_ok;
  const int lbh = blockIdx.x;
  const int h = lbh % hkv, b = (lbh / hkv) % batch;
  const int64_t layer = lbh / (hkv * batch);
  const int P = prefix_len[b], L = acc_len[b];
  if (threadIdx.x == 0) {
    int code = 0;
    const int32_t *path = acc_path + (int64_t)b * path_cap;
    s_ok = commit_ok(P, L, s_max, path_cap, N, path, &code);
    if (!s_ok) sv::report(status, code);
    else
      for (int j = 0; j <= L; ++j) s_path[j] = path[j];
  }
  __syncthreads();
  if (!s_ok) return;
  const int64_t lb = (layer * batch + b) * hkv + h;
  const int64_t cache_row0 = (lb * s_max + P) * vec_per_row;
  const int64_t tree_row0 = lb * N * vec_per_row;
  const int total = (L + 1) * vec_per_row;
  for (int e = threadIdx.x; e < 2 * total; e += kThreads) {
    const bool is_v = e >= total;
    const int f = is_v ? e - total : e;
    const int j = f / vec_per_row, c = f % vec_per_row;
    const int64_t src = tree_row0 + (int64_t)s_path[j] * vec_per_row + c;
    const int64_t dst = cache_row0 + (int64_t)j * vec_per_row + c;
    if (is_v) vc[dst] = vt[src];
    else kc[dst] = kt[src];
  }
}

__global__ void commit_len_kernel(int batch, int s_max, int N, const int32_t *__restrict__ acc_len,
                                  const int32_t *__restrict__ acc_path, int path_cap,
                                  const int32_t *prefix_len, int32_t *prefix_len_out) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int P = prefix_len[b], L = acc_len[b];
  int code = 0;
  const bool ok = commit_ok(P, L, s_max, path_cap, N, acc_path + (int64_t)b * path_cap, &code);
  prefix_len_out[b] = ok ? P + L + 1 : P;
}

}  // namespace

int sv_kv_commit(void *kc, void *vc, const void *kt, const void *vt, int elem_bytes, int n_layers,
                 int batch, int hkv, int s_max, int n_nodes, int head_dim, const int32_t *acc_len,
                 const int32_t *acc_path, int path_cap, const int32_t *prefix_len,
                 int32_t *prefix_len_out, int32_t *status, cudaStream_t stream) {
  const int vec_per_row = head_dim * elem_bytes / 16;
  commit_copy_kernel<<<n_layers * batch * hkv, kThreads, 0, stream>>>(
      (uint4 *)kc, (uint4 *)vc, (const uint4 *)kt, (const uint4 *)vt, batch, hkv, s_max, n_nodes,
      vec_per_row, acc_len, acc_path, path_cap, prefix_len, status);
  int rc = sv_launch_status();
  if (rc != SPEC_OK || prefix_len_out == nullptr) return rc;
  commit_len_kernel<<<(batch + 127) / 128, 128, 0, stream>>>(batch, s_max, n_nodes, acc_len, acc_path,
                                                             path_cap, prefix_len, prefix_len_out);
  return sv_launch_status();
}
