// tree_attn_verify_noalloc: tree attention for callers that cannot allocate
// device memory.
//
// Some callers of this library are handed only their input and output
// buffers: a plugin inside a host runtime that owns every device byte and
// exposes no allocator, or a serving loop that bans cudaMalloc/cudaFree after
// start-up because those calls synchronise the device and stall every stream
// in flight.  Such a caller cannot provide the split-KV workspace that
// tree_attn_verify needs.  This entry point runs the same kernels with the
// partials held in a fixed, library-owned device array instead.
//
// The array (SPEC_NOALLOC_SCRATCH_BYTES) lives in every GPU that loads the
// library until the process exits.  All calls share it: two calls that
// overlap on the GPU (different streams, no ordering between them) race on
// it.  Nothing in it has to start at zero: every partial a launch reads was
// written by the same launch's main kernel first.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "specverify.h"

namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];  // device address of g_attn_scratch, per device
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device; looked up once
// per device (cudaGetSymbolAddress with that device current).
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return SPEC_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" int tree_attn_verify_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                        const void *k_tree, const void *v_tree,
                                        const int32_t *prefix_len, const uint64_t *anc_mask,
                                        void *out, int dtype, int batch, int n_nodes, int hq,
                                        int hkv, int head_dim, int s_max, int max_prefix,
                                        float scale, int num_splits, int32_t *dev_status,
                                        spec_stream_t stream) {
  const size_t need = tree_attn_workspace_bytes(dtype, batch, n_nodes, hq, hkv, head_dim,
                                                max_prefix, num_splits);
  if (need > SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_CAPACITY;
  void *ws = nullptr;
  if (need > 0) {
    const int rc = scratch_address(&ws);
    if (rc != SPEC_OK) return rc;
  }
  return tree_attn_verify(q, k_cache, v_cache, k_tree, v_tree, prefix_len, anc_mask, out, dtype,
                          batch, n_nodes, hq, hkv, head_dim, s_max, max_prefix, scale, num_splits,
                          ws, need, dev_status, stream);
}
