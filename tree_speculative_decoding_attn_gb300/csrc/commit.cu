// Commit of the accepted path's K/V: "5.3 Medusa、EAGLE 与 MTP"
// (infra-guide), section 3.2 -- all nodes share the prefix KV; only the
// accepted path is committed and the other branches' temporary KV is
// discarded.  The tree K/V live in their own buffer, so the copy never
// overlaps its source and needs no in-place compaction.
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kThreads = 512;

// One CTA per sequence: checks the accepted path (one thread per entry),
// copies rows 0..L of every (layer, KV head) for K and V with 16-byte
// vectors, then advances that sequence's prefix length.  No other CTA reads
// or writes the sequence's entry, so the update may be in place
// (prefix_len_out == prefix_len) without a second launch.  With a paged
// cache every destination block is checked before anything is copied.
__global__ void __launch_bounds__(kThreads)
    commit_kernel(uint4 *kc, uint4 *vc, const uint4 *__restrict__ kt, const uint4 *__restrict__ vt, int n_layers,
                  int batch, int hkv, int s_max, int N, int vec_per_row, const int32_t *__restrict__ acc_len,
                  const int32_t *__restrict__ acc_path, int path_cap, const int32_t *prefix_len,
                  int32_t *prefix_len_out, int32_t *status, const SvPages pg) {
  __shared__ int s_path[SPEC_MAX_NODES + 1];
  __shared__ int s_row[SPEC_MAX_NODES + 1];  // destination row of entry j within a layer
  __shared__ int s_bad;
  const int b = blockIdx.x;
  const int P = prefix_len[b], L = acc_len[b];
  const bool fits = P >= 0 && L >= 0 && L + 1 <= path_cap && P + L + 1 <= s_max;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  if (fits && (int)threadIdx.x <= L) {
    const int j = threadIdx.x;
    const int v = acc_path[(int64_t)b * path_cap + j];
    s_path[j] = v;
    if (v < 0 || v >= N) atomicOr(&s_bad, 1);
    // row of (layer 0, head 0); heads are block_size (or s_max) rows apart
    int row = b * hkv * s_max + P + j;
    if (pg.table) {
      const int key = P + j;
      const int blk = pg.table[(int64_t)b * pg.max_blocks + key / pg.block_size];
      if (blk < 0 || blk >= pg.num_blocks) atomicOr(&s_bad, 2);
      row = blk * hkv * pg.block_size + key % pg.block_size;
    }
    s_row[j] = row;
  }
  __syncthreads();
  const bool ok = fits && !s_bad;
  if (threadIdx.x == 0 && !ok)
    sv::report(status, !fits ? SPEC_DEV_CAPACITY : (s_bad & 2) ? SPEC_DEV_BAD_BLOCK : SPEC_DEV_BAD_PATH);
  if (ok) {
    // rows apart of consecutive KV heads, and of consecutive layers
    const int64_t head_rows = pg.table ? pg.block_size : s_max;
    const int64_t layer_rows = pg.table ? (int64_t)pg.num_blocks * hkv * pg.block_size : (int64_t)batch * hkv * s_max;
    // every (K or V, layer, head, row, vector) in one index space, so all
    // of a thread's copies are in flight together
    const int n = (L + 1) * vec_per_row;  // vectors of one (layer, head) for K or V
    const int total = 2 * n_layers * hkv * n;
#pragma unroll 4
    for (int idx = threadIdx.x; idx < total; idx += kThreads) {
      const int it = idx / n, e = idx - it * n;
      const int j = e / vec_per_row, c = e - j * vec_per_row;
      const int lh = it >> 1;  // layer * hkv + head
      const int layer = lh / hkv, h = lh % hkv;
      const int64_t lb = ((int64_t)layer * batch + b) * hkv + h;
      const uint4 v = ((it & 1) ? vt : kt)[(lb * N + s_path[j]) * vec_per_row + c];
      const int64_t dst = layer * layer_rows + s_row[j] + h * head_rows;
      ((it & 1) ? vc : kc)[dst * vec_per_row + c] = v;
    }
  }
  if (prefix_len_out && threadIdx.x == 0) prefix_len_out[b] = ok ? P + L + 1 : P;
}

}  // namespace

int sv_kv_commit(void *kc, void *vc, const void *kt, const void *vt, int elem_bytes, int n_layers,
                 int batch, int hkv, int s_max, int n_nodes, int head_dim, const int32_t *acc_len,
                 const int32_t *acc_path, int path_cap, const int32_t *prefix_len,
                 int32_t *prefix_len_out, int32_t *status, cudaStream_t stream, SvPages pages) {
  const int vec_per_row = head_dim * elem_bytes / 16;
  commit_kernel<<<batch, kThreads, 0, stream>>>((uint4 *)kc, (uint4 *)vc, (const uint4 *)kt, (const uint4 *)vt,
                                                n_layers, batch, hkv, s_max, n_nodes, vec_per_row, acc_len,
                                                acc_path, path_cap, prefix_len, prefix_len_out, status, pages);
  return sv_launch_status();
}
