// Internal launchers (host functions) implemented by the kernel files and
// called by the C-ABI layer in spec_api.cu.  Arguments are validated there.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "specverify.h"

int sv_build_static(const int32_t *parents, const int32_t *rank, const int32_t *cand_tok,
                    int cand_levels, int cand_s, const int32_t *root_tok, const int32_t *prefix_len,
                    int batch, int n, int32_t *tok, int32_t *depth, int32_t *pos, uint64_t *anc,
                    int32_t *first_child, int32_t *next_sibling, int32_t *status, cudaStream_t stream);

int sv_build_batch(const int32_t *parents, int par_stride, const int32_t *n_valid, const int32_t *tok_in,
                   const int32_t *rank, const int32_t *cand_tok, int cand_levels, int cand_s,
                   const int32_t *root_tok, const int32_t *prefix_len, int batch, int n, int32_t *tok,
                   int32_t *depth, int32_t *pos, uint64_t *anc, int32_t *first_child, int32_t *next_sibling,
                   int32_t *status, cudaStream_t stream);

int sv_build_dynamic(const int32_t *pool_parent, const int32_t *pool_tok, const float *pool_conf,
                     int M, const int32_t *prefix_len, int batch, int n, int32_t *tok,
                     int32_t *parents_out, int32_t *depth, int32_t *pos, uint64_t *anc,
                     int32_t *first_child, int32_t *next_sibling, int32_t *pool_index, float *val,
                     int32_t *status, cudaStream_t stream);

// Tree attention.  `plan` picks the kernel family and split count; the
// workspace size follows from it.  Split-KV partials: one row per (sequence,
// KV head, split, query row) of head_dim unnormalised accumulators, then the
// running max (log2 units) and the running sum, padded to a 16-byte multiple.
inline constexpr int sv_partial_stride(int head_dim) { return head_dim + 4; }
struct SvAttnShape {
  int dtype, batch, n_nodes, hq, hkv, head_dim, s_max, max_prefix;
  // paged prefix cache (block_table null: contiguous [batch, hkv, s_max, D];
  // paged: s_max = max_blocks * block_size is each sequence's capacity)
  const int32_t *block_table;
  int block_size, max_blocks, num_blocks;
};
struct SvAttnPlan {
  int use_tc;        // 2 = pair (cta_group::2) kernel, 1 = tcgen05 kernel, 0 = CUDA-core kernel
  int splits;        // KV splits per (sequence, KV head)
  int chunk;         // prefix keys per split (multiple of the key tile)
  size_t ws_bytes;   // partials (0 when splits == 1)
};
SvAttnPlan sv_attn_plan(const SvAttnShape &s, int num_splits);
bool sv_attn_tc_supported(const SvAttnShape &s);
int sv_attn_tc_ragged_splits(const SvAttnShape &s, const int32_t *host_prefix);
int sv_attn_simt(const SvAttnShape &s, const SvAttnPlan &p, const void *q, const void *kc,
                 const void *vc, const void *kt, const void *vt, const int32_t *prefix_len,
                 const uint64_t *anc, void *out, float scale, void *ws, int32_t *status,
                 cudaStream_t stream);
int sv_attn_tc(const SvAttnShape &s, const SvAttnPlan &p, const void *q, const void *kc,
               const void *vc, const void *kt, const void *vt, const int32_t *prefix_len,
               const uint64_t *anc, void *out, float scale, void *ws, int32_t *status,
               cudaStream_t stream);
// Pair kernel (bf16, head_dim 128, more than 128 query rows per KV head):
// persistent, stream-K; launches its own combine.  Workspace: a fixed
// number of partial slots per cluster of the grid.
bool sv_attn_tc2_supported(const SvAttnShape &s);
size_t sv_attn_tc2_ws_bytes();
int sv_attn_tc2(const SvAttnShape &s, const void *q, const void *kc, const void *vc, const void *kt,
                const void *vt, const int32_t *prefix_len, const uint64_t *anc, void *out,
                float scale, void *ws, size_t ws_bytes, int32_t *status, cudaStream_t stream);
int sv_attn_run(const SvAttnShape &s, const SvAttnPlan &p, const void *q, const void *kc, const void *vc,
                const void *kt, const void *vt, const int32_t *prefix_len, const uint64_t *anc, void *out,
                float scale, void *ws, size_t ws_bytes, int32_t *status, cudaStream_t stream);
int sv_attn_combine(const SvAttnShape &s, const SvAttnPlan &p, const void *ws, void *out,
                    const int32_t *prefix_len, cudaStream_t stream);

// Weight-streaming tensor-core GEMM (Medusa heads, LM head): launch
// geometry and workspace share of one GEMM.
struct SvGemmPlan {
  int nt, mt;              // activation rows per MMA (N), 128-row MMAs per tile
  int nk, tiles_pg, n_tiles, n_ctas, rows_per_launch;
  long long units;         // (tile, 64-wide K chunk) pairs
  size_t partial_bytes;
  bool any_cut;            // some tile is cut: the fixup launch sums its partials
};
SvGemmPlan sv_wgemm_plan(int M, int K, int G, int rows);
// One weight-streaming GEMM (all row blocks).  epi: 0 float32 logits, 1
// bf16 SiLU + residual, 2 softmax statistics records (float4 per 32 W rows
// and activation row: max logit, sum exp, first moment, argmax).
int sv_wgemm(const SvGemmPlan &p, const void *w, const void *x, int x_grouped, int M, int K, int G, int rows,
             int epi, float *out, void *zout, const void *res, const void *bias, float *partial, bool pdl,
             int32_t *status, cudaStream_t stream, float inv_t = 1.f,
             void *stats = nullptr);
size_t sv_medusa_heads_ws_bytes(int batch, int n_heads, int hidden, int vocab);
int sv_medusa_heads(const void *h, const void *w1, const void *b1, const void *w2, int batch,
                    int n_heads, int hidden, int vocab, void *z, float *logits, void *ws,
                    int32_t *status, cudaStream_t stream);
size_t sv_lm_head_ws_bytes(int rows, int hidden, int vocab);
int sv_lm_head(const void *hid, const void *w, int rows, int hidden, int vocab, float *logits,
               void *ws, int32_t *status, cudaStream_t stream);
size_t sv_lm_head_accept_ws_bytes(int batch, int n_nodes, int hidden, int vocab);
int sv_lm_head_accept(int mode, const void *hid, const void *w, int batch, int n_nodes, int hidden, int vocab,
                      const int32_t *tok, const int32_t *parents, const int32_t *first_child,
                      const int32_t *next_sibling, float temperature, float eps, float delta, int path_cap,
                      int32_t *acc_len, int32_t *acc_path, int32_t *bonus, void *ws, int32_t *status,
                      cudaStream_t stream);
typedef spec_eagle_weights SvEagleWeights;
size_t sv_eagle_round_ws_bytes(int batch, int n_front, int hidden, int hq, int hkv, int head_dim, int ffn,
                               int vocab, int s_max, int max_prefix);
int sv_eagle_round(const SvEagleWeights &w, int batch, int hidden, int hq, int hkv, int head_dim, int ffn, int vocab,
                   const void *k_prefix, const void *v_prefix, int s_max, const int32_t *prefix_len, int max_prefix,
                   void *k_nodes, void *v_nodes, void *feat, const int32_t *frontier, int n_front, int depth, int k,
                   float temperature, int32_t *pool_parent, int32_t *pool_tok, float *pool_conf, float *pool_val,
                   int32_t *pool_count, int pool_cap, int32_t *next_frontier, int n_next, float *logits_out,
                   void *ws, int32_t *status, cudaStream_t stream);
int sv_topk(const void *rows, int dtype, int n_rows, int row_len, int row_stride, int s,
            int32_t *idx, float *val, cudaStream_t stream);
int sv_tree_expand(const void *logits, int dtype, int batch, int n_front, int vocab,
                   const int32_t *frontier, int k, float temperature, int32_t *pool_parent,
                   int32_t *pool_tok, float *pool_conf, float *pool_val, int32_t *pool_count,
                   int pool_cap, int32_t *next_frontier, int n_next, int32_t *status,
                   cudaStream_t stream);
// The commit fused into the acceptance launch (contiguous cache; kc null:
// no commit).  Layouts as kv_commit; vec_per_row = head_dim * elem_bytes / 16.
struct SvCommit {
  uint4 *kc, *vc;
  const uint4 *kt, *vt;
  int n_layers, hkv, s_max, vec_per_row;
  const int32_t *prefix_len;
  int32_t *prefix_len_out;
};
int sv_accept(int mode, const void *logits, const void *draft, int dtype, int batch, int n_nodes, int vocab,
              const int32_t *tok, const int32_t *parents, const int32_t *first_child,
              const int32_t *next_sibling, float temperature, float eps, float delta,
              uint64_t seed, uint64_t step, int path_cap, int32_t *acc_len, int32_t *acc_path,
              int32_t *bonus, int32_t *status, cudaStream_t stream, SvCommit commit = SvCommit{});
// kv_commit; `pages` (table null: contiguous) addresses a paged cache
// [n_layers, num_blocks, hkv, block_size, D] with s_max = max_blocks *
// block_size.
struct SvPages {
  const int32_t *table;
  int block_size, max_blocks, num_blocks;
};
int sv_kv_commit(void *kc, void *vc, const void *kt, const void *vt, int elem_bytes, int n_layers,
                 int batch, int hkv, int s_max, int n_nodes, int head_dim, const int32_t *acc_len,
                 const int32_t *acc_path, int path_cap, const int32_t *prefix_len,
                 int32_t *prefix_len_out, int32_t *status, cudaStream_t stream, SvPages pages = SvPages{});
