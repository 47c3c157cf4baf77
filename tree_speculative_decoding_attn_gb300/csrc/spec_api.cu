// C-ABI entry points of libspecverify: argument validation, kernel choice,
// launch.  Stateless; every call enqueues on the caller's stream.
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "specverify.h"

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t cs(spec_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

SvAttnPlan sv_attn_simt_plan(const SvAttnShape &s, int num_splits);
SvAttnPlan sv_attn_tc_plan(const SvAttnShape &s, int num_splits, bool *ok);

SvAttnPlan sv_attn_plan(const SvAttnShape &s, int num_splits) {
  if (sv_attn_tc2_supported(s)) {
    SvAttnPlan p{};
    p.use_tc = 2;
    p.splits = 1;  // the pair kernel balances its own work
    p.ws_bytes = sv_attn_tc2_ws_bytes();
    return p;
  }
  bool ok = false;
  SvAttnPlan p = sv_attn_tc_plan(s, num_splits, &ok);
  if (ok) return p;
  return sv_attn_simt_plan(s, num_splits);
}

// Run the planned attention kernel (and its combine) for shape s.
int sv_attn_run(const SvAttnShape &s, const SvAttnPlan &p, const void *q, const void *kc, const void *vc,
                const void *kt, const void *vt, const int32_t *prefix_len, const uint64_t *anc, void *out,
                float scale, void *ws, size_t ws_bytes, int32_t *status, cudaStream_t stream) {
  if (p.use_tc == 2) {
    if (p.ws_bytes == 0) return SPEC_ERR_CUDA;
    return sv_attn_tc2(s, q, kc, vc, kt, vt, prefix_len, anc, out, scale, ws, ws_bytes, status, stream);
  }
  const int rc = p.use_tc ? sv_attn_tc(s, p, q, kc, vc, kt, vt, prefix_len, anc, out, scale, ws, status, stream)
                          : sv_attn_simt(s, p, q, kc, vc, kt, vt, prefix_len, anc, out, scale, ws, status, stream);
  if (rc != SPEC_OK || p.splits == 1) return rc;
  return sv_attn_combine(s, p, ws, out, prefix_len, stream);
}

extern "C" {

const char *spec_status_string(int status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or size";
    case SPEC_ERR_CAPACITY: return "size exceeds a buffer's capacity";
    case SPEC_ERR_CUDA: return "CUDA launch error";
    default: return "unknown status";
  }
}

int spec_abi_version(void) { return 2; }

static bool gemm_shape_ok(int rows, int groups, int hidden, int m) {
  return rows >= 1 && groups >= 1 && m >= 1 && hidden >= 64 && hidden % 64 == 0;
}

size_t spec_medusa_heads_workspace_bytes(int batch, int n_heads, int hidden, int vocab) {
  if (!gemm_shape_ok(batch, n_heads, hidden, vocab)) return 0;
  return sv_medusa_heads_ws_bytes(batch, n_heads, hidden, vocab);
}

int spec_medusa_heads(const void *h, const void *w1, const void *b1, const void *w2, int batch,
                      int n_heads, int hidden, int vocab, void *z, float *logits, void *workspace,
                      size_t workspace_bytes, int32_t *dev_status, spec_stream_t stream) {
  if (!h || !w1 || !w2 || !z || !logits || !workspace) return SPEC_ERR_INVALID_ARG;
  if (!gemm_shape_ok(batch, n_heads, hidden, vocab)) return SPEC_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w1) || !aligned16(w2) || !aligned16(z) || !aligned16(workspace) ||
      (b1 && !aligned16(b1)))
    return SPEC_ERR_INVALID_ARG;
  if (workspace_bytes < sv_medusa_heads_ws_bytes(batch, n_heads, hidden, vocab)) return SPEC_ERR_CAPACITY;
  return sv_medusa_heads(h, w1, b1, w2, batch, n_heads, hidden, vocab, z, logits, workspace, dev_status,
                         cs(stream));
}

int spec_topk(const void *rows, int dtype, int n_rows, int row_len, int row_stride, int s,
              int32_t *idx_out, float *val_out, spec_stream_t stream) {
  if (!rows || !idx_out) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (n_rows < 1 || row_len < 1 || row_stride < row_len || s < 1 || s > row_len) return SPEC_ERR_INVALID_ARG;
  if (s > 16) return SPEC_ERR_UNSUPPORTED;
  return sv_topk(rows, dtype, n_rows, row_len, row_stride, s, idx_out, val_out, cs(stream));
}

int spec_build_tree(const int32_t *parents, const int32_t *rank, const int32_t *cand_tok,
                    int cand_levels, int cand_s, const int32_t *root_tok,
                    const int32_t *prefix_len, int batch, int n_nodes, int32_t *tok,
                    int32_t *depth, int32_t *pos_ids, uint64_t *anc_mask, int32_t *first_child,
                    int32_t *next_sibling, int32_t *dev_status, spec_stream_t stream) {
  if (!parents || !prefix_len || !depth || !pos_ids || !anc_mask || !first_child || !next_sibling)
    return SPEC_ERR_INVALID_ARG;
  if (batch < 1 || n_nodes < 1) return SPEC_ERR_INVALID_ARG;
  if (n_nodes > SPEC_MAX_NODES) return SPEC_ERR_UNSUPPORTED;
  if (cand_tok && (!rank || !root_tok || !tok || cand_levels < 0 || cand_s < 1)) return SPEC_ERR_INVALID_ARG;
  return sv_build_static(parents, rank, cand_tok, cand_levels, cand_s, root_tok, prefix_len, batch,
                         n_nodes, cand_tok ? tok : nullptr, depth, pos_ids, anc_mask, first_child,
                         next_sibling, dev_status, cs(stream));
}

int spec_build_tree_dynamic(const int32_t *pool_parent, const int32_t *pool_tok,
                            const float *pool_conf, int pool_size, const int32_t *prefix_len,
                            int batch, int n_nodes, int32_t *tok, int32_t *parents_out,
                            int32_t *depth, int32_t *pos_ids, uint64_t *anc_mask,
                            int32_t *first_child, int32_t *next_sibling, int32_t *pool_index,
                            float *val, int32_t *dev_status, spec_stream_t stream) {
  if (!pool_parent || !pool_tok || !pool_conf || !prefix_len || !tok || !parents_out || !depth ||
      !pos_ids || !anc_mask || !first_child || !next_sibling)
    return SPEC_ERR_INVALID_ARG;
  if (batch < 1 || n_nodes < 1 || pool_size < n_nodes) return SPEC_ERR_INVALID_ARG;
  if (n_nodes > SPEC_MAX_NODES || pool_size > 4096) return SPEC_ERR_UNSUPPORTED;
  return sv_build_dynamic(pool_parent, pool_tok, pool_conf, pool_size, prefix_len, batch, n_nodes,
                          tok, parents_out, depth, pos_ids, anc_mask, first_child, next_sibling,
                          pool_index, val, dev_status, cs(stream));
}

int spec_tree_expand(const void *draft_logits, int dtype, int batch, int n_front, int vocab,
                     const int32_t *frontier, int k, float temperature, int32_t *pool_parent,
                     int32_t *pool_tok, float *pool_conf, float *pool_val, int32_t *pool_count,
                     int pool_cap, int32_t *next_frontier, int n_next, int32_t *dev_status,
                     spec_stream_t stream) {
  if (!draft_logits || !frontier || !pool_parent || !pool_tok || !pool_conf || !pool_val ||
      !pool_count || !next_frontier)
    return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (batch < 1 || n_front < 1 || vocab < k || k < 1 || n_next < 1 || pool_cap < 1 ||
      !(temperature > 0.f))
    return SPEC_ERR_INVALID_ARG;
  if (k > 16 || n_front * k > 1024) return SPEC_ERR_UNSUPPORTED;
  return sv_tree_expand(draft_logits, dtype, batch, n_front, vocab, frontier, k, temperature,
                        pool_parent, pool_tok, pool_conf, pool_val, pool_count, pool_cap,
                        next_frontier, n_next, dev_status, cs(stream));
}

static int attn_check(int dtype, int batch, int n_nodes, int hq, int hkv, int head_dim, int s_max,
                      int max_prefix) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (batch < 1 || n_nodes < 1 || hq < 1 || hkv < 1 || s_max < 0 || max_prefix < 0)
    return SPEC_ERR_INVALID_ARG;
  if (hq % hkv) return SPEC_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SPEC_ERR_UNSUPPORTED;
  if (n_nodes > SPEC_MAX_NODES || (hq / hkv) * n_nodes > (n_nodes <= 64 ? 512 : 2048))
    return SPEC_ERR_UNSUPPORTED;
  if (max_prefix > s_max) return SPEC_ERR_CAPACITY;
  return SPEC_OK;
}

size_t tree_attn_workspace_bytes(int dtype, int batch, int n_nodes, int hq, int hkv, int head_dim,
                                 int max_prefix, int num_splits) {
  if (attn_check(dtype, batch, n_nodes, hq, hkv, head_dim, max_prefix, max_prefix) != SPEC_OK) return 0;
  const SvAttnShape s{dtype, batch, n_nodes, hq, hkv, head_dim, max_prefix, max_prefix};
  return sv_attn_plan(s, num_splits).ws_bytes;
}

int tree_attn_plan_splits(int dtype, int batch, int n_nodes, int hq, int hkv, int head_dim,
                          const int32_t *host_prefix_len) {
  if (!host_prefix_len) return 0;
  int max_prefix = 0;
  for (int b = 0; b < batch; ++b) {
    if (host_prefix_len[b] < 0) return 0;
    max_prefix = host_prefix_len[b] > max_prefix ? host_prefix_len[b] : max_prefix;
  }
  if (attn_check(dtype, batch, n_nodes, hq, hkv, head_dim, max_prefix, max_prefix) != SPEC_OK) return 0;
  const SvAttnShape s{dtype, batch, n_nodes, hq, hkv, head_dim, max_prefix, max_prefix};
  if (sv_attn_tc2_supported(s)) return 1;
  if (sv_attn_tc_supported(s)) return sv_attn_tc_ragged_splits(s, host_prefix_len);
  return sv_attn_plan(s, 0).splits;
}

int tree_attn_verify(const void *q, const void *k_cache, const void *v_cache, const void *k_tree,
                     const void *v_tree, const int32_t *prefix_len, const uint64_t *anc_mask,
                     void *out, int dtype, int batch, int n_nodes, int hq, int hkv, int head_dim,
                     int s_max, int max_prefix, float scale, int num_splits, void *workspace,
                     size_t workspace_bytes, int32_t *dev_status, spec_stream_t stream) {
  if (!q || !k_cache || !v_cache || !k_tree || !v_tree || !prefix_len || !anc_mask || !out)
    return SPEC_ERR_INVALID_ARG;
  int rc = attn_check(dtype, batch, n_nodes, hq, hkv, head_dim, s_max, max_prefix);
  if (rc != SPEC_OK) return rc;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_tree) ||
      !aligned16(v_tree) || !aligned16(out))
    return SPEC_ERR_INVALID_ARG;
  const SvAttnShape s{dtype, batch, n_nodes, hq, hkv, head_dim, s_max, max_prefix};
  const SvAttnPlan p = sv_attn_plan(s, num_splits);
  if (p.ws_bytes > 0 && (!workspace || workspace_bytes < p.ws_bytes || !aligned16(workspace)))
    return SPEC_ERR_CAPACITY;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)head_dim);
  return sv_attn_run(s, p, q, k_cache, v_cache, k_tree, v_tree, prefix_len, anc_mask, out, scale, workspace,
                     workspace_bytes, dev_status, cs(stream));
}

size_t spec_lm_head_workspace_bytes(int rows, int hidden, int vocab) {
  if (!gemm_shape_ok(rows, 1, hidden, vocab)) return 0;
  return sv_lm_head_ws_bytes(rows, hidden, vocab);
}

int tree_attn_verify_paged(const void *q, const void *k_pages, const void *v_pages, const int32_t *block_table,
                           int block_size, int num_blocks, int max_blocks, const void *k_tree, const void *v_tree,
                           const int32_t *prefix_len, const uint64_t *anc_mask, void *out, int dtype, int batch,
                           int n_nodes, int hq, int hkv, int head_dim, int max_prefix, float scale, int num_splits,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status, spec_stream_t stream) {
  if (!q || !k_pages || !v_pages || !block_table || !k_tree || !v_tree || !prefix_len || !anc_mask || !out)
    return SPEC_ERR_INVALID_ARG;
  if (block_size < 128 || block_size % 128 || num_blocks < 1 || max_blocks < 1) return SPEC_ERR_INVALID_ARG;
  if ((long long)max_blocks * block_size > (1 << 30) || (long long)num_blocks * hkv * block_size > (1 << 30))
    return SPEC_ERR_UNSUPPORTED;
  const int s_max = max_blocks * block_size;
  int rc = attn_check(dtype, batch, n_nodes, hq, hkv, head_dim, s_max, max_prefix);
  if (rc != SPEC_OK) return rc;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(k_tree) || !aligned16(v_tree) ||
      !aligned16(out))
    return SPEC_ERR_INVALID_ARG;
  SvAttnShape s{dtype, batch, n_nodes, hq, hkv, head_dim, s_max, max_prefix};
  s.block_table = block_table;
  s.block_size = block_size;
  s.max_blocks = max_blocks;
  s.num_blocks = num_blocks;
  const SvAttnPlan p = sv_attn_plan(s, num_splits);
  if (p.ws_bytes > 0 && (!workspace || workspace_bytes < p.ws_bytes || !aligned16(workspace)))
    return SPEC_ERR_CAPACITY;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)head_dim);
  return sv_attn_run(s, p, q, k_pages, v_pages, k_tree, v_tree, prefix_len, anc_mask, out, scale, workspace,
                     workspace_bytes, dev_status, cs(stream));
}

static bool eagle_shape_ok(int batch, int n_front, int hidden, int hq, int hkv, int head_dim, int ffn, int vocab) {
  return batch >= 1 && n_front >= 1 && hidden >= 64 && hidden % 64 == 0 && hidden <= 8192 && hq >= 1 && hkv >= 1 && hq % hkv == 0 &&
         (head_dim == 64 || head_dim == 128) && (hq * head_dim) % 64 == 0 && ffn >= 64 && ffn % 64 == 0 &&
         vocab >= 1;
}

size_t spec_eagle_round_workspace_bytes(int batch, int n_front, int hidden, int hq, int hkv, int head_dim, int ffn,
                                        int vocab, int s_max, int max_prefix) {
  if (!eagle_shape_ok(batch, n_front, hidden, hq, hkv, head_dim, ffn, vocab) || max_prefix < 0 || s_max < max_prefix)
    return 0;
  return sv_eagle_round_ws_bytes(batch, n_front, hidden, hq, hkv, head_dim, ffn, vocab, s_max, max_prefix);
}

int spec_eagle_round(const spec_eagle_weights *w, int batch, int hidden, int hq, int hkv, int head_dim, int ffn,
                     int vocab, const void *k_prefix, const void *v_prefix, int s_max, const int32_t *prefix_len,
                     int max_prefix, void *k_nodes, void *v_nodes, void *feat, const int32_t *frontier, int n_front,
                     int depth, int k, float temperature, int32_t *pool_parent, int32_t *pool_tok,
                     float *pool_conf, float *pool_val, int32_t *pool_count, int pool_cap, int32_t *next_frontier,
                     int n_next, float *draft_logits, void *workspace, size_t workspace_bytes,
                     int32_t *dev_status, spec_stream_t stream) {
  if (!w || !w->fc || !w->ln1 || !w->qkv || !w->o || !w->ln2 || !w->gate_up || !w->down || !w->lnf || !w->lm ||
      !w->emb || !k_prefix || !v_prefix || !prefix_len || !k_nodes || !v_nodes || !feat || !frontier ||
      !pool_parent || !pool_tok || !pool_conf || !pool_val || !pool_count || !next_frontier || !workspace)
    return SPEC_ERR_INVALID_ARG;
  if (!eagle_shape_ok(batch, n_front, hidden, hq, hkv, head_dim, ffn, vocab)) return SPEC_ERR_INVALID_ARG;
  if (depth < 0 || max_prefix < 0 || s_max < max_prefix || pool_cap < 1 || n_next < 1 || k < 1 || vocab < k ||
      !(temperature > 0.f))
    return SPEC_ERR_INVALID_ARG;
  if ((long long)n_front * (depth + 1) > 64 || k > 16 || n_front * k > 1024 || pool_cap > 4000)
    return SPEC_ERR_UNSUPPORTED;
  const void *ptrs[] = {w->fc, w->ln1, w->qkv, w->o, w->ln2, w->gate_up, w->down, w->lnf, w->lm, w->emb,
                        k_prefix, v_prefix, k_nodes, v_nodes, feat, workspace};
  for (const void *q : ptrs)
    if (!aligned16(q)) return SPEC_ERR_INVALID_ARG;
  if (workspace_bytes <
      sv_eagle_round_ws_bytes(batch, n_front, hidden, hq, hkv, head_dim, ffn, vocab, s_max, max_prefix))
    return SPEC_ERR_CAPACITY;
  return sv_eagle_round(*w, batch, hidden, hq, hkv, head_dim, ffn, vocab, k_prefix, v_prefix, s_max, prefix_len,
                        max_prefix, k_nodes, v_nodes, feat, frontier, n_front, depth, k, temperature, pool_parent,
                        pool_tok, pool_conf, pool_val, pool_count, pool_cap, next_frontier, n_next, draft_logits,
                        workspace, dev_status, cs(stream));
}

int spec_lm_head(const void *hid, const void *w, int rows, int hidden, int vocab, float *logits,
                 void *workspace, size_t workspace_bytes, int32_t *dev_status, spec_stream_t stream) {
  if (!hid || !w || !logits || !workspace) return SPEC_ERR_INVALID_ARG;
  if (!gemm_shape_ok(rows, 1, hidden, vocab)) return SPEC_ERR_INVALID_ARG;
  if (!aligned16(hid) || !aligned16(w) || !aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  if (workspace_bytes < sv_lm_head_ws_bytes(rows, hidden, vocab)) return SPEC_ERR_CAPACITY;
  return sv_lm_head(hid, w, rows, hidden, vocab, logits, workspace, dev_status, cs(stream));
}

size_t spec_lm_head_accept_workspace_bytes(int batch, int n_nodes, int hidden, int vocab) {
  if (batch < 1 || n_nodes < 1 || n_nodes > SPEC_MAX_NODES || !gemm_shape_ok(batch * n_nodes, 1, hidden, vocab))
    return 0;
  return sv_lm_head_accept_ws_bytes(batch, n_nodes, hidden, vocab);
}

int spec_lm_head_accept(int mode, const void *hid, const void *w, int batch, int n_nodes, int hidden, int vocab,
                        const int32_t *tok, const int32_t *parents, const int32_t *first_child,
                        const int32_t *next_sibling, float temperature, float eps, float delta, int path_cap,
                        int32_t *acc_len, int32_t *acc_path, int32_t *bonus, void *workspace,
                        size_t workspace_bytes, int32_t *dev_status, spec_stream_t stream) {
  if (!hid || !w || !tok || !parents || !first_child || !next_sibling || !acc_len || !acc_path || !bonus ||
      !workspace)
    return SPEC_ERR_INVALID_ARG;
  if (mode == SPEC_ACCEPT_REJECT || mode == SPEC_ACCEPT_REJECT_STOCHASTIC) return SPEC_ERR_UNSUPPORTED;
  if (mode != SPEC_ACCEPT_GREEDY && mode != SPEC_ACCEPT_TYPICAL) return SPEC_ERR_INVALID_ARG;
  if (batch < 1 || n_nodes < 1 || path_cap < 1) return SPEC_ERR_INVALID_ARG;
  if (n_nodes > SPEC_MAX_NODES || path_cap > SPEC_MAX_NODES + 1) return SPEC_ERR_UNSUPPORTED;
  if (!gemm_shape_ok(batch * n_nodes, 1, hidden, vocab)) return SPEC_ERR_INVALID_ARG;
  if (!aligned16(hid) || !aligned16(w) || !aligned16(workspace)) return SPEC_ERR_INVALID_ARG;
  if (mode == SPEC_ACCEPT_TYPICAL && !(temperature > 0.f)) return SPEC_ERR_INVALID_ARG;
  if (mode == SPEC_ACCEPT_GREEDY) temperature = 1.f;
  if (workspace_bytes < sv_lm_head_accept_ws_bytes(batch, n_nodes, hidden, vocab)) return SPEC_ERR_CAPACITY;
  return sv_lm_head_accept(mode, hid, w, batch, n_nodes, hidden, vocab, tok, parents, first_child, next_sibling,
                           temperature, eps, delta, path_cap, acc_len, acc_path, bonus, workspace, dev_status,
                           cs(stream));
}

int spec_accept(int mode, const void *logits, const void *draft_logits, int dtype, int batch,
                int n_nodes, int vocab, const int32_t *tok, const int32_t *parents, const int32_t *first_child,
                const int32_t *next_sibling, float temperature, float eps, float delta,
                uint64_t seed, uint64_t step, int path_cap, int32_t *acc_len, int32_t *acc_path,
                int32_t *bonus, int32_t *dev_status, spec_stream_t stream) {
  if (!logits || !tok || !parents || !first_child || !next_sibling || !acc_len || !acc_path || !bonus)
    return SPEC_ERR_INVALID_ARG;
  if (mode != SPEC_ACCEPT_GREEDY && mode != SPEC_ACCEPT_TYPICAL && mode != SPEC_ACCEPT_REJECT &&
      mode != SPEC_ACCEPT_REJECT_STOCHASTIC)
    return SPEC_ERR_INVALID_ARG;
  if ((mode == SPEC_ACCEPT_REJECT_STOCHASTIC) != (draft_logits != nullptr)) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (batch < 1 || n_nodes < 1 || vocab < 1 || path_cap < 1) return SPEC_ERR_INVALID_ARG;
  if (n_nodes > SPEC_MAX_NODES) return SPEC_ERR_UNSUPPORTED;
  if (mode != SPEC_ACCEPT_GREEDY && !(temperature > 0.f)) return SPEC_ERR_INVALID_ARG;
  if (mode == SPEC_ACCEPT_GREEDY) temperature = 1.f;
  return sv_accept(mode, logits, draft_logits, dtype, batch, n_nodes, vocab, tok, parents, first_child,
                   next_sibling, temperature, eps, delta, seed, step, path_cap, acc_len, acc_path,
                   bonus, dev_status, cs(stream));
}

int spec_accept_commit(int mode, const void *logits, const void *draft_logits, int dtype, int batch,
                       int n_nodes, int vocab, const int32_t *tok, const int32_t *parents,
                       const int32_t *first_child, const int32_t *next_sibling, float temperature,
                       float eps, float delta, uint64_t seed, uint64_t step, int path_cap,
                       int32_t *acc_len, int32_t *acc_path, int32_t *bonus, void *k_cache,
                       void *v_cache, const void *k_tree, const void *v_tree, int elem_bytes,
                       int n_layers, int hkv, int s_max, int head_dim, const int32_t *prefix_len,
                       int32_t *prefix_len_out, int32_t *dev_status, spec_stream_t stream) {
  if (!logits || !tok || !parents || !first_child || !next_sibling || !acc_len || !acc_path || !bonus)
    return SPEC_ERR_INVALID_ARG;
  if (mode != SPEC_ACCEPT_GREEDY && mode != SPEC_ACCEPT_TYPICAL && mode != SPEC_ACCEPT_REJECT &&
      mode != SPEC_ACCEPT_REJECT_STOCHASTIC)
    return SPEC_ERR_INVALID_ARG;
  if ((mode == SPEC_ACCEPT_REJECT_STOCHASTIC) != (draft_logits != nullptr)) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (batch < 1 || n_nodes < 1 || vocab < 1 || path_cap < 1) return SPEC_ERR_INVALID_ARG;
  if (n_nodes > SPEC_MAX_NODES) return SPEC_ERR_UNSUPPORTED;
  if (mode != SPEC_ACCEPT_GREEDY && !(temperature > 0.f)) return SPEC_ERR_INVALID_ARG;
  if (mode == SPEC_ACCEPT_GREEDY) temperature = 1.f;
  // the commit's arguments, as kv_commit
  if (!k_cache || !v_cache || !k_tree || !v_tree || !prefix_len) return SPEC_ERR_INVALID_ARG;
  if (elem_bytes != 2 && elem_bytes != 4) return SPEC_ERR_UNSUPPORTED;
  if (n_layers < 1 || hkv < 1 || s_max < 1 || head_dim < 1) return SPEC_ERR_INVALID_ARG;
  if (path_cap > SPEC_MAX_NODES + 1) return SPEC_ERR_UNSUPPORTED;
  if ((head_dim * elem_bytes) % 16) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_tree) || !aligned16(v_tree))
    return SPEC_ERR_INVALID_ARG;
  SvCommit cm{};
  cm.kc = static_cast<uint4 *>(k_cache);
  cm.vc = static_cast<uint4 *>(v_cache);
  cm.kt = static_cast<const uint4 *>(k_tree);
  cm.vt = static_cast<const uint4 *>(v_tree);
  cm.n_layers = n_layers;
  cm.hkv = hkv;
  cm.s_max = s_max;
  cm.vec_per_row = head_dim * elem_bytes / 16;
  cm.prefix_len = prefix_len;
  cm.prefix_len_out = prefix_len_out;
  return sv_accept(mode, logits, draft_logits, dtype, batch, n_nodes, vocab, tok, parents, first_child,
                   next_sibling, temperature, eps, delta, seed, step, path_cap, acc_len, acc_path, bonus,
                   dev_status, cs(stream), cm);
}

int spec_build_tree_batch(const int32_t *parents, const int32_t *n_valid, const int32_t *tok_in,
                          const int32_t *prefix_len, int batch, int n_nodes, int32_t *tok, int32_t *depth,
                          int32_t *pos_ids, uint64_t *anc_mask, int32_t *first_child, int32_t *next_sibling,
                          int32_t *dev_status, spec_stream_t stream) {
  if (!parents || !prefix_len || !depth || !pos_ids || !anc_mask || !first_child || !next_sibling)
    return SPEC_ERR_INVALID_ARG;
  if (batch < 1 || n_nodes < 1 || (tok_in && !tok)) return SPEC_ERR_INVALID_ARG;
  if (n_nodes > SPEC_MAX_NODES) return SPEC_ERR_UNSUPPORTED;
  return sv_build_batch(parents, n_nodes, n_valid, tok_in, nullptr, nullptr, 0, 1, nullptr, prefix_len, batch,
                        n_nodes, tok_in ? tok : nullptr, depth, pos_ids, anc_mask, first_child, next_sibling,
                        dev_status, cs(stream));
}

int kv_commit_paged(void *k_pages, void *v_pages, const int32_t *block_table, int block_size, int num_blocks,
                    int max_blocks, const void *k_tree, const void *v_tree, int elem_bytes, int n_layers,
                    int batch, int hkv, int n_nodes, int head_dim, const int32_t *acc_len,
                    const int32_t *acc_path, int path_cap, const int32_t *prefix_len, int32_t *prefix_len_out,
                    int32_t *dev_status, spec_stream_t stream) {
  if (!k_pages || !v_pages || !block_table || !k_tree || !v_tree || !acc_len || !acc_path || !prefix_len)
    return SPEC_ERR_INVALID_ARG;
  if (elem_bytes != 2 && elem_bytes != 4) return SPEC_ERR_UNSUPPORTED;
  if (block_size < 1 || num_blocks < 1 || max_blocks < 1 || n_layers < 1 || batch < 1 || hkv < 1 ||
      n_nodes < 1 || head_dim < 1 || path_cap < 1)
    return SPEC_ERR_INVALID_ARG;
  if (n_nodes > SPEC_MAX_NODES || path_cap > SPEC_MAX_NODES + 1) return SPEC_ERR_UNSUPPORTED;
  if ((head_dim * elem_bytes) % 16) return SPEC_ERR_UNSUPPORTED;
  if ((long long)max_blocks * block_size > (1 << 30) || (long long)num_blocks * hkv * block_size > (1 << 30))
    return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(k_pages) || !aligned16(v_pages) || !aligned16(k_tree) || !aligned16(v_tree))
    return SPEC_ERR_INVALID_ARG;
  return sv_kv_commit(k_pages, v_pages, k_tree, v_tree, elem_bytes, n_layers, batch, hkv, max_blocks * block_size,
                      n_nodes, head_dim, acc_len, acc_path, path_cap, prefix_len, prefix_len_out, dev_status,
                      cs(stream), SvPages{block_table, block_size, max_blocks, num_blocks});
}

int kv_commit(void *k_cache, void *v_cache, const void *k_tree, const void *v_tree, int elem_bytes,
              int n_layers, int batch, int hkv, int s_max, int n_nodes, int head_dim,
              const int32_t *acc_len, const int32_t *acc_path, int path_cap,
              const int32_t *prefix_len, int32_t *prefix_len_out, int32_t *dev_status,
              spec_stream_t stream) {
  if (!k_cache || !v_cache || !k_tree || !v_tree || !acc_len || !acc_path || !prefix_len)
    return SPEC_ERR_INVALID_ARG;
  if (elem_bytes != 2 && elem_bytes != 4) return SPEC_ERR_UNSUPPORTED;
  if (n_layers < 1 || batch < 1 || hkv < 1 || s_max < 1 || n_nodes < 1 || head_dim < 1 || path_cap < 1)
    return SPEC_ERR_INVALID_ARG;
  if (n_nodes > SPEC_MAX_NODES || path_cap > SPEC_MAX_NODES + 1) return SPEC_ERR_UNSUPPORTED;
  if ((head_dim * elem_bytes) % 16) return SPEC_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_tree) || !aligned16(v_tree))
    return SPEC_ERR_INVALID_ARG;
  return sv_kv_commit(k_cache, v_cache, k_tree, v_tree, elem_bytes, n_layers, batch, hkv, s_max,
                      n_nodes, head_dim, acc_len, acc_path, path_cap, prefix_len, prefix_len_out,
                      dev_status, cs(stream));
}

}  // extern "C"
