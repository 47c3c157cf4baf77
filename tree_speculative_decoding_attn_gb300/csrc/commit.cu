// Commit of the accepted path's K/V: "5.3 Medusa、EAGLE 与 MTP"
// (infra-guide), section 3.2 -- all nodes share the prefix KV; only the
// accepted path is committed and the other branches' temporary KV is
// discarded.  The tree K/V live in their own buffer, so the copy never
// overlaps its source and needs no in-place compaction.
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kThreads = 512;

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

// One CTA per sequence: copies rows 0..L of every (layer, KV head) for K and
// V with 16-byte vectors, then advances that sequence's prefix length.  No
// other CTA reads or writes the sequence's entry, so the update may be in
// place (prefix_len_out == prefix_len) without a second launch.
__global__ void __launch_bounds__(kThreads)
    commit_kernel(uint4 *kc, uint4 *vc, const uint4 *__restrict__ kt, const uint4 *__restrict__ vt, int n_layers,
                  int batch, int hkv, int s_max, int N, int vec_per_row, const int32_t *__restrict__ acc_len,
                  const int32_t *__restrict__ acc_path, int path_cap, const int32_t *prefix_len,
                  int32_t *prefix_len_out, int32_t *status) {
  __shared__ int s_path[SPEC_MAX_NODES + 1];
  __shared__ int s_ok, s_P, s_L;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    const int P = prefix_len[b], L = acc_len[b];
    int code = 0;
    const int32_t *path = acc_path + (int64_t)b * path_cap;
    s_ok = commit_ok(P, L, s_max, path_cap, N, path, &code);
    if (!s_ok) sv::report(status, code);
    else
      for (int j = 0; j <= L; ++j) s_path[j] = path[j];
    s_P = P;
    s_L = L;
  }
  __syncthreads();
  const int P = s_P, L = s_L;
  if (s_ok) {
    const int per_head = (L + 1) * vec_per_row;  // vectors of one (layer, head) for K or V
    const int64_t total = (int64_t)n_layers * hkv * per_head;
    for (int64_t e = threadIdx.x; e < 2 * total; e += kThreads) {
      const bool is_v = e >= total;
      const int64_t f = is_v ? e - total : e;
      const int64_t lh = f / per_head;  // layer * hkv + head
      const int rem = (int)(f % per_head);
      const int j = rem / vec_per_row, c = rem % vec_per_row;
      const int64_t lb = ((lh / hkv) * batch + b) * hkv + lh % hkv;
      const int64_t src = (lb * N + s_path[j]) * vec_per_row + c;
      const int64_t dst = (lb * s_max + P + j) * vec_per_row + c;
      if (is_v) vc[dst] = vt[src];
      else kc[dst] = kt[src];
    }
  }
  if (prefix_len_out && threadIdx.x == 0) prefix_len_out[b] = s_ok ? P + L + 1 : P;
}

}  // namespace

int sv_kv_commit(void *kc, void *vc, const void *kt, const void *vt, int elem_bytes, int n_layers,
                 int batch, int hkv, int s_max, int n_nodes, int head_dim, const int32_t *acc_len,
                 const int32_t *acc_path, int path_cap, const int32_t *prefix_len,
                 int32_t *prefix_len_out, int32_t *status, cudaStream_t stream) {
  const int vec_per_row = head_dim * elem_bytes / 16;
  commit_kernel<<<batch, kThreads, 0, stream>>>((uint4 *)kc, (uint4 *)vc, (const uint4 *)kt, (const uint4 *)vt,
                                                n_layers, batch, hkv, s_max, n_nodes, vec_per_row, acc_len,
                                                acc_path, path_cap, prefix_len, prefix_len_out, status);
  return sv_launch_status();
}
