/*
 * specverify.h -- C ABI of the tree-verification step of Medusa/EAGLE
 * self-speculative decoding, for NVIDIA GB300 (sm_103a).
 *
 * The step, as the pages state it:
 *   - Medusa residual heads propose candidates: head k computes
 *     softmax(W2_k (SiLU(W1_k h) + h)) and offers its top s_k tokens
 *     ("Medusa, explained", procedure step 1 and step 5; "Medusa and EAGLE:
 *     self-speculative decoding heads, explained", section "Medusa: heads,
 *     losses and trees").
 *   - The candidates form a tree, flattened in node order with an
 *     ancestor mask and depth-based position ids ("5.3 Medusa、EAGLE 与 MTP",
 *     sections 3.1, 3.2 and 8).  EAGLE-2 picks the nodes by the product of
 *     draft confidences along their path (same page, section 5.2).
 *   - One target pass scores every node (tree attention over the shared
 *     prefix KV plus each node's own ancestors).
 *   - The longest target-agreeing path is accepted: greedy match, typical
 *     acceptance, or min(1, p/q) rejection with residual resampling
 *     ("Drafters: draft models, Medusa, EAGLE, MTP, DFlash, DSpark", section
 *     "Why the answer does not change"; "Medusa, explained", section
 *     "Typical acceptance").
 *   - Only the accepted path's KV is committed to the cache; sibling
 *     branches are discarded ("5.3 Medusa、EAGLE 与 MTP", section 3.2).
 *
 * General rules for every entry point
 *   - Every pointer argument is a DEVICE pointer to caller-owned memory
 *     unless stated otherwise.  The library allocates nothing, keeps no
 *     state between calls, and never frees caller memory.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL
 *     means the legacy default stream).  Calls are capturable in CUDA
 *     graphs and are thread-safe (they share nothing).
 *   - The return value is a host-side status (SPEC_OK, or an SPEC_ERR_*
 *     code when an argument is invalid or a launch failed).  On an
 *     argument error nothing is launched.
 *   - Errors that only the device can see (a malformed parents array, a
 *     commit past the cache capacity, a bad accepted path) are written to
 *     the optional `dev_status` word (int32, device memory; the first
 *     error wins, via atomicCAS from 0).  The kernel then skips the
 *     offending work item; it never traps.  Pass NULL to not report.
 *   - Layouts are dense row-major with the last index contiguous.
 *     Dtype codes: SPEC_F32 (float) and SPEC_BF16 (__nv_bfloat16).
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *spec_stream_t; /* same handle as cudaStream_t */

/* host-side return codes */
enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent shapes */
  SPEC_ERR_UNSUPPORTED = 2, /* dtype / head_dim / node count not built    */
  SPEC_ERR_CAPACITY = 3,    /* a host-known size exceeds a buffer         */
  SPEC_ERR_CUDA = 4         /* a kernel launch reported an error          */
};

/* device status codes written to dev_status */
enum {
  SPEC_DEV_OK = 0,
  SPEC_DEV_BAD_PARENTS = 1,  /* parents[0] != -1 or not 0 <= parents[i] < i */
  SPEC_DEV_CAPACITY = 2,     /* prefix_len + rows > s_max (or > max_prefix) */
  SPEC_DEV_BAD_PATH = 3,     /* accepted path entry out of [0, n_nodes)     */
  SPEC_DEV_BAD_POOL = 4,     /* pool parent not earlier / confidence > 1    */
  SPEC_DEV_BAD_TOKEN = 5,    /* token id outside [0, vocab)                 */
  SPEC_DEV_TIMEOUT = 6,      /* a bounded device-side wait gave up          */
  SPEC_DEV_INTERNAL = 7,     /* a kernel's own layout precondition failed   */
  SPEC_DEV_BAD_BLOCK = 8     /* a block-table entry outside the block pool  */
};

/* dtype codes */
enum { SPEC_F32 = 0, SPEC_BF16 = 1 };

/* acceptance modes */
enum {
  SPEC_ACCEPT_GREEDY = 0,
  SPEC_ACCEPT_TYPICAL = 1,
  SPEC_ACCEPT_REJECT = 2,           /* siblings are deterministic drafts */
  SPEC_ACCEPT_REJECT_STOCHASTIC = 3 /* siblings drawn from the drafter's q */
};

/* Largest tree (nodes, root included).  The ancestor bitmask of a node is
 * SPEC_MASK_WORDS(n_nodes) uint64 words: bit j % 64 of word j / 64 stands
 * for node j.  Trees of up to 64 nodes therefore use one word per node. */
#define SPEC_MAX_NODES 256
#define SPEC_MASK_WORDS(n) (((n) + 63) / 64)

/* Text for a host or device status code (static string, never NULL). */
const char *spec_status_string(int status);

/* ABI version of this header (bumped on any signature change). */
int spec_abi_version(void);

/* --------------------------------------------------------------------
 * spec_medusa_heads -- Medusa residual heads (candidate proposal).
 * "Medusa, explained", procedure step 1: head k maps the last hidden
 * state h to W2_k (SiLU(W1_k h) + h); "Medusa and EAGLE ... explained",
 * section "Implementation sketch": W1 may carry a bias, W2 has none.
 *
 *   h      [batch, hidden]               bf16
 *   w1     [n_heads, hidden, hidden]     bf16, nn.Linear layout [out, in]
 *   b1     [n_heads, hidden]             bf16, or NULL for no bias
 *   w2     [n_heads, vocab, hidden]      bf16
 *   z      [batch, n_heads, hidden]      bf16 out: h + SiLU(W1 h + b1),
 *                                        rounded to bf16 (the W2 operand)
 *   logits [batch, n_heads, vocab]       f32 out: W2 z (softmax omitted:
 *                                        it does not change the top-s)
 *   workspace  device scratch of spec_medusa_heads_workspace_bytes()
 *              bytes (16-byte aligned; contents need not be initialised;
 *              calls that may overlap on the GPU need separate ones)
 * Both products run on the tensor cores with float32 accumulation; every
 * SM streams an equal share of the weights, and the sum over hidden is
 * taken in a fixed order, so results repeat bit for bit across calls.
 * Requires hidden % 64 == 0; any batch >= 1 (blocks of 256 rows).  A
 * device-side timeout (never expected) sets SPEC_DEV_TIMEOUT in dev_status
 * (optional).  SPEC_ERR_CAPACITY: workspace too small.
 * ------------------------------------------------------------------ */
size_t spec_medusa_heads_workspace_bytes(int batch, int n_heads, int hidden, int vocab);
int spec_medusa_heads(const void *h, const void *w1, const void *b1, const void *w2,
                      int batch, int n_heads, int hidden, int vocab,
                      void *z, float *logits, void *workspace, size_t workspace_bytes,
                      int32_t *dev_status, spec_stream_t stream);

/* --------------------------------------------------------------------
 * spec_topk -- top-s candidates per row ("Medusa and EAGLE ...
 * explained", section "Medusa: heads, losses and trees": head k
 * contributes its top s_k tokens).
 *
 *   rows     [n_rows, row_stride] (f32 or bf16 per `dtype`); the first
 *            row_len entries of each row are ranked
 *   idx_out  [n_rows, s] int32: column indices, by value descending;
 *            equal values -> lower index first
 *   val_out  [n_rows, s] f32: the values (may be NULL)
 * Requires 1 <= s <= 16 and s <= row_len.
 * ------------------------------------------------------------------ */
int spec_topk(const void *rows, int dtype, int n_rows, int row_len, int row_stride, int s,
              int32_t *idx_out, float *val_out, spec_stream_t stream);

/* --------------------------------------------------------------------
 * spec_build_tree -- static (Medusa) tree for a batch.
 * "5.3 Medusa、EAGLE 与 MTP", section 8: node 0 is the root, parents[i] < i;
 * a node sees its ancestors and itself (section 3.1); position id =
 * prefix length + depth, siblings share a position (section 3.2).
 * "Medusa, explained", step 5-6: node at depth d >= 1 carries candidate
 * rank[i] of head d.
 *
 *   parents    [n_nodes] int32 (shared by the batch); parents[0] = -1
 *   rank       [n_nodes] int32: candidate rank of node i (rank[0] unused)
 *   cand_tok   [batch, cand_levels, cand_s] int32: cand_tok[b, d-1, r] is
 *              head d's rank-r candidate; may be NULL (then `tok` is not
 *              written)
 *   root_tok   [batch] int32: token the target already chose (node 0)
 *   prefix_len [batch] int32: committed cache length of each sequence
 * Outputs, all [batch, n_nodes]:
 *   tok (int32, may be NULL), depth (int32), pos_ids (int32) = prefix_len
 *   + depth, anc_mask ([batch, n_nodes, SPEC_MASK_WORDS(n_nodes)] uint64:
 *   the bit of node j in node i's words is set iff node j is node i or an
 *   ancestor of it), first_child / next_sibling (int32, -1 = none;
 *   children in node order).
 * n_nodes <= SPEC_MAX_NODES.  A malformed parents array or a depth beyond
 * cand_levels sets SPEC_DEV_BAD_PARENTS.
 * ------------------------------------------------------------------ */
int spec_build_tree(const int32_t *parents, const int32_t *rank, const int32_t *cand_tok,
                    int cand_levels, int cand_s, const int32_t *root_tok,
                    const int32_t *prefix_len, int batch, int n_nodes,
                    int32_t *tok, int32_t *depth, int32_t *pos_ids, uint64_t *anc_mask,
                    int32_t *first_child, int32_t *next_sibling, int32_t *dev_status,
                    spec_stream_t stream);

/* --------------------------------------------------------------------
 * spec_build_tree_batch -- one tree per sequence, of up to n_nodes nodes
 * each, in one launch (ragged multi-tree batching of serving: requests with
 * different tree budgets and shapes; "5.3 Medusa、EAGLE 与 MTP", section 8,
 * closing remarks on batching trees of different requests).
 *   parents  [batch, n_nodes] int32: sequence b's parents array (rules of
 *            spec_build_tree) over its first n_valid[b] entries
 *   n_valid  [batch] int32 (1 .. n_nodes), or NULL for all n_nodes: entries
 *            at and past it are absent nodes (padding)
 *   tok_in   [batch, n_nodes] int32 tokens copied to `tok`, or NULL (then
 *            `tok` is not written)
 * Outputs as spec_build_tree.  An absent node is nobody's child, has depth
 * 0, position prefix_len, a mask of itself only and no child links, so
 * attention, acceptance and commit never reach it (its attention output is
 * computed but meaningless).
 * ------------------------------------------------------------------ */
int spec_build_tree_batch(const int32_t *parents, const int32_t *n_valid, const int32_t *tok_in,
                          const int32_t *prefix_len, int batch, int n_nodes, int32_t *tok,
                          int32_t *depth, int32_t *pos_ids, uint64_t *anc_mask,
                          int32_t *first_child, int32_t *next_sibling, int32_t *dev_status,
                          spec_stream_t stream);

/* --------------------------------------------------------------------
 * spec_build_tree_dynamic -- EAGLE-2 style tree from a drafted pool.
 * "5.3 Medusa、EAGLE 与 MTP", section 5.2: a node's value is the product of
 * the draft confidences along its path; the highest-value nodes go to
 * verification; confidence never enters acceptance (section 5.3).
 *
 *   pool_parent [batch, pool_size] int32: pool_parent[b,0] = -1 (root),
 *               0 <= pool_parent[b,i] < i otherwise
 *   pool_tok    [batch, pool_size] int32
 *   pool_conf   [batch, pool_size] f32 in [0, 1] (entry 0 ignored)
 * val[i] = val[parent] * conf[i] (one float32 multiply each, root-to-node
 * order, root 1).  Kept: the root and the n_nodes-1 nodes of highest value
 * (ties: smaller depth, then lower pool index).  Emitted breadth-first:
 * by depth, then new parent index, then value descending, then pool index.
 * Outputs [batch, n_nodes]: tok, parents_out, depth, pos_ids, anc_mask,
 * first_child, next_sibling (as spec_build_tree), pool_index (int32, may
 * be NULL), val (f32, may be NULL).  pool_size <= 4096.
 * ------------------------------------------------------------------ */
int spec_build_tree_dynamic(const int32_t *pool_parent, const int32_t *pool_tok,
                            const float *pool_conf, int pool_size, const int32_t *prefix_len,
                            int batch, int n_nodes, int32_t *tok, int32_t *parents_out,
                            int32_t *depth, int32_t *pos_ids, uint64_t *anc_mask,
                            int32_t *first_child, int32_t *next_sibling, int32_t *pool_index,
                            float *val, int32_t *dev_status, spec_stream_t stream);

/* --------------------------------------------------------------------
 * spec_tree_expand -- one confidence-product expansion round of the
 * draft tree ("5.3 Medusa、EAGLE 与 MTP", section 5.2; "Medusa and EAGLE
 * ... explained", section "EAGLE: autoregression over features").
 *
 *   draft_logits [batch, n_front, vocab] (f32 or bf16): draft distribution
 *                of each frontier node (softmax of logits / temperature)
 *   frontier     [batch, n_front] int32 pool indices (all valid)
 *   pool_parent, pool_tok [batch, pool_cap] int32, pool_conf, pool_val
 *                [batch, pool_cap] f32: the pool, appended to in place
 *   pool_count   [batch] int32, in/out: entries in use
 * Frontier node f gets its k most probable tokens (ties: lower id) as
 * children at pool positions count + f*k + j, with conf = probability and
 * val = val(f) * conf (float32).  next_frontier [batch, n_next] receives
 * the n_next new children of highest value (ties: lower pool index),
 * highest first.  pool_val[b, 0] (the root) must hold 1.  Requires
 * 1 <= k <= 16, n_front * k <= 1024, and pool_count + n_front * k <=
 * pool_cap (else SPEC_DEV_CAPACITY).
 * ------------------------------------------------------------------ */
int spec_tree_expand(const void *draft_logits, int dtype, int batch, int n_front, int vocab,
                     const int32_t *frontier, int k, float temperature, int32_t *pool_parent,
                     int32_t *pool_tok, float *pool_conf, float *pool_val, int32_t *pool_count,
                     int pool_cap, int32_t *next_frontier, int n_next, int32_t *dev_status,
                     spec_stream_t stream);

/* --------------------------------------------------------------------
 * spec_eagle_round -- one drafting round of an EAGLE-2 style draft: the
 * draft layer applied to the frontier nodes, then spec_tree_expand on its
 * distributions ("Medusa and EAGLE ... explained", section "EAGLE:
 * autoregression over features": [feature ; embedding of the next token]
 * -> FC (2d -> d) -> one decoder layer -> next feature -> the target's LM
 * head; "5.3 Medusa、EAGLE 与 MTP", sections 4.1 and 5.2).
 *
 * Weights (bf16, nn.Linear layout [out, in]):
 *   fc [hidden, 2*hidden]; ln1, ln2, lnf [hidden] (RMSNorm gains);
 *   qkv [(hq + 2*hkv) * head_dim, hidden]; o [hidden, hq * head_dim];
 *   gate_up [2, ffn, hidden]; down [hidden, ffn]; lm [vocab, hidden] (the
 *   target's LM head); emb [vocab, hidden] (the target's embedding).
 * The decoder layer is a pre-norm block: x1 = x + W_o attn(RMSNorm(x)),
 * out = x1 + W_down(SiLU(W_gate n) * W_up n), n = RMSNorm(x1), RMSNorm eps
 * 1e-6; rotary embedding rotate-half, base 10000, position = prefix_len +
 * depth; the predicted feature passes RMSNorm(lnf) before the LM head.
 *
 *   k_prefix, v_prefix [batch, hkv, s_max, head_dim]: the draft layer's cache
 *            of the verified prefix (rotary applied), prefix_len [batch]
 *   k_nodes, v_nodes  [batch, hkv, pool_cap, head_dim]: draft K/V of pool
 *            nodes; this round writes its frontier nodes' rows
 *   feat     [batch, pool_cap + 1, hidden]: node features; slot pool_cap is
 *            the target's feature of the last verified position (the root's
 *            parent); this round writes its frontier nodes' rows
 *   frontier [batch, n_front] pool indices (all at depth `depth`; round 1:
 *            the root alone at depth 0)
 *   pool_*, pool_count, next_frontier, k, temperature: as spec_tree_expand
 *   draft_logits  [batch, n_front, vocab] f32 out (may be NULL: kept in the
 *            workspace)
 *   workspace  spec_eagle_round_workspace_bytes() bytes
 * A frontier node attends to the prefix cache and to its ancestors and
 * itself in the draft tree (at most 64 nodes per round: n_front * (depth +
 * 1) <= 64).  Requires hidden (at most 8192), hq * head_dim and ffn
 * multiples of 64, head_dim 64 or 128, hq % hkv == 0, pool_cap <= 4000
 * (else SPEC_ERR_UNSUPPORTED).  Malformed pools or frontiers set
 * SPEC_DEV_BAD_POOL.
 * ------------------------------------------------------------------ */
typedef struct spec_eagle_weights {
  const void *fc, *ln1, *qkv, *o, *ln2, *gate_up, *down, *lnf, *lm, *emb;
} spec_eagle_weights;
size_t spec_eagle_round_workspace_bytes(int batch, int n_front, int hidden, int hq, int hkv,
                                        int head_dim, int ffn, int vocab, int s_max,
                                        int max_prefix);
int spec_eagle_round(const spec_eagle_weights *w, int batch, int hidden, int hq, int hkv,
                     int head_dim, int ffn, int vocab, const void *k_prefix, const void *v_prefix,
                     int s_max, const int32_t *prefix_len, int max_prefix, void *k_nodes,
                     void *v_nodes, void *feat, const int32_t *frontier, int n_front, int depth,
                     int k, float temperature, int32_t *pool_parent, int32_t *pool_tok,
                     float *pool_conf, float *pool_val, int32_t *pool_count, int pool_cap,
                     int32_t *next_frontier, int n_next, float *draft_logits, void *workspace,
                     size_t workspace_bytes, int32_t *dev_status, spec_stream_t stream);

/* --------------------------------------------------------------------
 * tree_attn_verify -- attention of every tree node over the shared prefix
 * KV and its own ancestors ("5.3 Medusa、EAGLE 与 MTP", sections 3.1 and 8;
 * "Medusa, explained", step 6; "Medusa and EAGLE ... explained", section
 * "Medusa: heads, losses and trees").
 *
 * For node i of sequence b and query head h (KV head h / (hq/hkv)):
 *   out[b,i,h] = softmax_j(scale * q[b,i,h] . k_j) v_j over
 *   j in { cache rows 0 .. prefix_len[b]-1 } U { tree rows t : bit t of
 *   anc_mask[b,i] }.
 *
 *   q        [batch, n_nodes, hq, head_dim]       dtype
 *   k_cache, v_cache [batch, hkv, s_max, head_dim] dtype (rows at and past
 *            prefix_len are ignored)
 *   k_tree, v_tree   [batch, hkv, n_nodes, head_dim] dtype: this pass's
 *            K/V of the tree nodes (position ids already applied)
 *   prefix_len [batch] int32 (device), each <= max_prefix (host bound)
 *   anc_mask   [batch, n_nodes, SPEC_MASK_WORDS(n_nodes)] uint64 (from
 *            spec_build_tree*)
 *   out      [batch, n_nodes, hq, head_dim]       dtype
 *   scale    softmax scale; <= 0 selects 1/sqrt(head_dim)
 *   num_splits  KV splits per (sequence, KV head); 0 = automatic
 *   workspace   device scratch of tree_attn_workspace_bytes() bytes
 *               (may be NULL when that size is 0)
 * dtype SPEC_F32 or SPEC_BF16; head_dim 64 or 128; n_nodes <= 256;
 * hq % hkv == 0; (hq / hkv) * n_nodes <= 512 for trees of up to 64 nodes,
 * <= 2048 above.  Softmax and accumulation are float32.  A prefix_len above
 * max_prefix sets SPEC_DEV_CAPACITY and that sequence's output is left
 * unwritten.
 * bf16 with head_dim 128 (hq / hkv dividing 128) and either more than 128
 * query rows per KV head ((hq / hkv) * n_nodes > 128) or more than 64
 * nodes runs on pairs of SMs with a persistent grid that balances its own
 * work: num_splits is ignored there (tree_attn_plan_splits returns 1) and
 * the workspace holds the partial rows of the row groups cut between SM
 * pairs.  f32 and head_dim 64 run on CUDA cores.  Calls that may overlap
 * on the GPU need separate workspaces.
 * ------------------------------------------------------------------ */
size_t tree_attn_workspace_bytes(int dtype, int batch, int n_nodes, int hq, int hkv,
                                 int head_dim, int max_prefix, int num_splits);
/* tree_attn_plan_splits -- KV split count for a batch whose prefix lengths
 * the host knows (HOST pointer, [batch] int32).  num_splits = 0 in
 * tree_attn_verify plans for every sequence at max_prefix; with ragged
 * prefixes this planner (a simulation of the kernel's work distribution
 * over the SMs) usually finds a better count.  Pass the result as
 * num_splits to tree_attn_workspace_bytes and tree_attn_verify.  Returns
 * >= 1, or 0 on invalid arguments. */
int tree_attn_plan_splits(int dtype, int batch, int n_nodes, int hq, int hkv, int head_dim,
                          const int32_t *host_prefix_len);
int tree_attn_verify(const void *q, const void *k_cache, const void *v_cache,
                     const void *k_tree, const void *v_tree, const int32_t *prefix_len,
                     const uint64_t *anc_mask, void *out, int dtype, int batch, int n_nodes,
                     int hq, int hkv, int head_dim, int s_max, int max_prefix, float scale,
                     int num_splits, void *workspace, size_t workspace_bytes,
                     int32_t *dev_status, spec_stream_t stream);

/* --------------------------------------------------------------------
 * tree_attn_verify_paged -- tree_attn_verify over a paged prefix cache
 * (block tables of paged KV: "5.3 Medusa、EAGLE 与 MTP", section 8, closing
 * remarks).
 *   k_pages, v_pages [num_blocks, hkv, block_size, head_dim]: the block pool
 *   block_table [batch, max_blocks] int32: prefix positions
 *            [j * block_size, (j + 1) * block_size) of sequence b are rows of
 *            block block_table[b, j]; entries past the prefix are not read
 *   block_size  a multiple of 128 (one 128-key tile never spans blocks)
 * Everything else as tree_attn_verify, with each sequence's capacity
 * max_blocks * block_size in place of s_max; the workspace size is
 * tree_attn_workspace_bytes() of the same shape.  A block id outside
 * [0, num_blocks) sets SPEC_DEV_BAD_BLOCK (those keys read as zeros).
 * ------------------------------------------------------------------ */
int tree_attn_verify_paged(const void *q, const void *k_pages, const void *v_pages,
                           const int32_t *block_table, int block_size, int num_blocks,
                           int max_blocks, const void *k_tree, const void *v_tree,
                           const int32_t *prefix_len, const uint64_t *anc_mask, void *out,
                           int dtype, int batch, int n_nodes, int hq, int hkv, int head_dim,
                           int max_prefix, float scale, int num_splits, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status, spec_stream_t stream);

/* --------------------------------------------------------------------
 * tree_attn_verify_noalloc -- tree_attn_verify without a caller workspace.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory: a plugin inside a host runtime that
 * owns all device memory and hands it only its input and output buffers,
 * or a serving loop that bans cudaMalloc/cudaFree after start-up because
 * they synchronise the device.
 *
 * Arguments and results are those of tree_attn_verify, minus the workspace:
 * the split-KV partials go to a library-owned device array of
 * SPEC_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library keeps
 * until the process exits.  Allocates nothing.  Returns SPEC_ERR_CAPACITY
 * (nothing launched) when tree_attn_workspace_bytes() for these arguments
 * exceeds SPEC_NOALLOC_SCRATCH_BYTES.  The first call on each device looks
 * up the array's device address; make that first call before any stream
 * capture.  All calls share the one array: calls that overlap on the GPU
 * (unordered streams) race on it.  Nothing in it needs to start at zero.
 * ------------------------------------------------------------------ */
#define SPEC_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB */
int tree_attn_verify_noalloc(const void *q, const void *k_cache, const void *v_cache,
                             const void *k_tree, const void *v_tree, const int32_t *prefix_len,
                             const uint64_t *anc_mask, void *out, int dtype, int batch,
                             int n_nodes, int hq, int hkv, int head_dim, int s_max, int max_prefix,
                             float scale, int num_splits, int32_t *dev_status,
                             spec_stream_t stream);

/* --------------------------------------------------------------------
 * spec_lm_head -- target logits of every tree node ("Medusa, explained",
 * step 6: one forward pass scores every node).
 *   hid    [rows, hidden] bf16
 *   w      [vocab, hidden] bf16 (LM head weight)
 *   logits [rows, vocab]   f32 out = hid . w^T (float32 accumulation)
 *   workspace  device scratch of spec_lm_head_workspace_bytes() bytes
 *              (as spec_medusa_heads)
 * Requires hidden % 64 == 0; any rows >= 1 (blocks of 256 rows).  Runs on
 * the tensor cores; a device-side timeout (never expected) sets
 * SPEC_DEV_TIMEOUT in dev_status (optional).
 * ------------------------------------------------------------------ */
size_t spec_lm_head_workspace_bytes(int rows, int hidden, int vocab);
int spec_lm_head(const void *hid, const void *w, int rows, int hidden, int vocab, float *logits,
                 void *workspace, size_t workspace_bytes, int32_t *dev_status, spec_stream_t stream);

/* --------------------------------------------------------------------
 * spec_lm_head_accept -- LM head over the tree nodes fused with greedy or
 * typical acceptance: the target logits never reach device memory.
 * "Medusa, explained", step 6 (one pass scores every node) and step 7 /
 * section "Typical acceptance"; "Drafters: ...", section "Why the answer
 * does not change".
 *
 *   hid    [batch, n_nodes, hidden] bf16: the final hidden state of every
 *          tree node
 *   w      [vocab, hidden] bf16: LM-head weight
 *   tok, parents, first_child, next_sibling [batch, n_nodes] int32 (as
 *          spec_accept)
 *   mode   SPEC_ACCEPT_GREEDY or SPEC_ACCEPT_TYPICAL with the rules of
 *          spec_accept applied to logits = hid . w^T (float32 accumulation
 *          on the tensor cores).  The rejection modes need the full
 *          residual row: use spec_lm_head + spec_accept
 *          (SPEC_ERR_UNSUPPORTED here).
 *   workspace  device scratch of spec_lm_head_accept_workspace_bytes()
 *          bytes (16-byte aligned, uninitialised; separate per overlapping
 *          call): per (node, 32 vocabulary rows) softmax statistics
 *          records, about hidden / 256 times smaller than the logits.
 * The greedy argmax is taken over the same float32 values spec_lm_head
 * would write, so greedy results equal spec_lm_head + spec_accept bit for
 * bit.  Typical: a child's probability uses its own logit recomputed as a
 * float32 dot product; entropy and normaliser come from the records.
 * Outputs as spec_accept.  dev_status: SPEC_DEV_BAD_TOKEN,
 * SPEC_DEV_BAD_PARENTS, SPEC_DEV_CAPACITY (path_cap), SPEC_DEV_TIMEOUT.
 * ------------------------------------------------------------------ */
size_t spec_lm_head_accept_workspace_bytes(int batch, int n_nodes, int hidden, int vocab);
int spec_lm_head_accept(int mode, const void *hid, const void *w, int batch, int n_nodes, int hidden,
                        int vocab, const int32_t *tok, const int32_t *parents,
                        const int32_t *first_child, const int32_t *next_sibling,
                        float temperature, float eps, float delta, int path_cap,
                        int32_t *acc_len, int32_t *acc_path, int32_t *bonus, void *workspace,
                        size_t workspace_bytes, int32_t *dev_status, spec_stream_t stream);

/* --------------------------------------------------------------------
 * spec_accept -- accept the longest target-agreeing path.
 *
 *   logits  [batch, n_nodes, vocab] (f32 or bf16): target logits at each
 *           node (distribution of the token after it)
 *   draft_logits [batch, n_nodes, vocab] (same dtype): the drafter's
 *           logits at each node (SPEC_ACCEPT_REJECT_STOCHASTIC only; NULL
 *           otherwise)
 *   tok, parents, first_child, next_sibling [batch, n_nodes] int32
 * Modes (p_v = softmax(logits[b,v] / temperature)):
 *   SPEC_ACCEPT_GREEDY  child c of v is accepted iff tok[c] == argmax
 *       logits[b,v] (ties: lowest id); walk from the root, stop when no
 *       child agrees; bonus = that argmax ("Drafters: ...", section "Why
 *       the answer does not change"; "Medusa, explained", step 7).
 *   SPEC_ACCEPT_TYPICAL node c is valid iff p_parent(tok[c]) >
 *       min(eps, delta * exp(-H(p_parent))), natural-log entropy; the
 *       accepted path ends at the deepest node whose whole path is valid
 *       (ties: lowest node index); bonus = greedy token there ("Medusa,
 *       explained", section "Typical acceptance").
 *   SPEC_ACCEPT_REJECT  at node v with residual r (= p_v on arrival),
 *       children in node order: accept c iff u < r(tok[c]) (min(1, p/q)
 *       with the point-mass proposal of a deterministic draft); otherwise
 *       r <- r with tok[c] removed, renormalised.  If no child is
 *       accepted the bonus is a sample of r ("Drafters: ...", section "Why
 *       the answer does not change").  Uniforms: Philox4x32-10 with key
 *       `seed`; accept draw counter (c, 0, b, step), u = (word0 >> 8) *
 *       2^-24.  Sampling is the exponential race argmax_x (logits/T +
 *       Gumbel(u'_x)) over the tokens not removed, u' = ((w >> 9) + 0.5) *
 *       2^-23 with w = word (x mod 4) of counter (x div 4, 256 + v, b,
 *       step).
 *   SPEC_ACCEPT_REJECT_STOCHASTIC  the children of v are independent
 *       draws from the drafter's q_v = softmax(draft_logits[b,v] / T)
 *       (SpecInfer-style multi-draft; "Medusa and EAGLE ... explained",
 *       section "Medusa: heads, losses and trees"; "Drafters: ...", section
 *       "Why the answer does not change"): child c is accepted iff u <
 *       r(tok[c]) / q_v(tok[c]) (always when q_v(tok[c]) = 0); a rejection
 *       sets r <- norm(max(0, r - q_v)); if no child is accepted the bonus
 *       is the race over log r(x) + Gumbel(u'_x) for r(x) > 0.  Same draws
 *       as SPEC_ACCEPT_REJECT.
 *       REJECT modes require temperature > 0.
 * Outputs: acc_len [batch] (accepted nodes, root excluded), acc_path
 * [batch, path_cap] (node ids root first, -1 after), bonus [batch].
 * path_cap must exceed the tree depth.  Decisions use float32.
 * dev_status: SPEC_DEV_BAD_TOKEN (a child token outside [0, vocab): never
 * accepted), SPEC_DEV_CAPACITY (path longer than path_cap), and in typical
 * mode SPEC_DEV_BAD_PARENTS when parents[] disagrees with the child links
 * (that sequence accepts the root alone).
 * ------------------------------------------------------------------ */
int spec_accept(int mode, const void *logits, const void *draft_logits, int dtype, int batch,
                int n_nodes, int vocab,
                const int32_t *tok, const int32_t *parents, const int32_t *first_child,
                const int32_t *next_sibling, float temperature, float eps, float delta,
                uint64_t seed, uint64_t step, int path_cap, int32_t *acc_len, int32_t *acc_path,
                int32_t *bonus, int32_t *dev_status, spec_stream_t stream);

/* --------------------------------------------------------------------
 * spec_accept_commit -- spec_accept and kv_commit (contiguous cache) in one
 * launch: each sequence's cluster, once it has taken its path, copies that
 * path's K/V rows into the cache and advances prefix_len.  The pages'
 * steps 7 and 8 of "Medusa, explained" / section 3.2 of "5.3 Medusa、EAGLE
 * 与 MTP"; the arguments, results and device errors are those of the two
 * calls (acc_len and acc_path are still written).  prefix_len_out may equal
 * prefix_len; a path that would pass s_max sets SPEC_DEV_CAPACITY and that
 * sequence is neither copied nor advanced.
 * ------------------------------------------------------------------ */
int spec_accept_commit(int mode, const void *logits, const void *draft_logits, int dtype, int batch,
                       int n_nodes, int vocab, const int32_t *tok, const int32_t *parents,
                       const int32_t *first_child, const int32_t *next_sibling, float temperature,
                       float eps, float delta, uint64_t seed, uint64_t step, int path_cap,
                       int32_t *acc_len, int32_t *acc_path, int32_t *bonus, void *k_cache,
                       void *v_cache, const void *k_tree, const void *v_tree, int elem_bytes,
                       int n_layers, int hkv, int s_max, int head_dim, const int32_t *prefix_len,
                       int32_t *prefix_len_out, int32_t *dev_status, spec_stream_t stream);

/* --------------------------------------------------------------------
 * kv_commit -- append the accepted path's K/V rows to the cache and
 * discard the rest ("5.3 Medusa、EAGLE 与 MTP", section 3.2).
 *
 * For every layer l, sequence b, KV head h and j = 0 .. acc_len[b]:
 *   k_cache[l,b,h,prefix_len[b]+j,:] = k_tree[l,b,h,acc_path[b,j],:]
 *   (same for v), then prefix_len_out[b] = prefix_len[b] + acc_len[b] + 1.
 *   k_cache, v_cache  [n_layers, batch, hkv, s_max, head_dim]
 *   k_tree,  v_tree   [n_layers, batch, hkv, n_nodes, head_dim]
 *   elem_bytes        2 (bf16) or 4 (f32); head_dim * elem_bytes % 16 == 0
 *   prefix_len_out    may equal prefix_len (each sequence's entry is
 *                     updated in place after its copies); may be NULL
 * A row past s_max or a path entry outside [0, n_nodes) sets a device
 * status and that sequence is neither copied nor advanced.
 * ------------------------------------------------------------------ */
int kv_commit(void *k_cache, void *v_cache, const void *k_tree, const void *v_tree,
              int elem_bytes, int n_layers, int batch, int hkv, int s_max, int n_nodes,
              int head_dim, const int32_t *acc_len, const int32_t *acc_path, int path_cap,
              const int32_t *prefix_len, int32_t *prefix_len_out, int32_t *dev_status,
              spec_stream_t stream);

/* --------------------------------------------------------------------
 * kv_commit_paged -- kv_commit into a paged cache: the accepted path is an
 * append to each sequence's block list (block tables of paged KV: "5.3
 * Medusa、EAGLE 与 MTP", section 8).
 *   k_pages, v_pages [n_layers, num_blocks, hkv, block_size, head_dim]
 *   block_table [batch, max_blocks] int32 (one table for every layer); the
 *            blocks holding positions prefix_len .. prefix_len + acc_len
 *            must already be assigned (the caller's allocator)
 * Row prefix_len[b] + j of sequence b is row (prefix_len[b] + j) %
 * block_size of block block_table[b, (prefix_len[b] + j) / block_size].
 * Every destination block is checked first: a block id outside
 * [0, num_blocks) sets SPEC_DEV_BAD_BLOCK and that sequence is neither
 * copied nor advanced.  Otherwise as kv_commit.
 * ------------------------------------------------------------------ */
int kv_commit_paged(void *k_pages, void *v_pages, const int32_t *block_table, int block_size,
                    int num_blocks, int max_blocks, const void *k_tree, const void *v_tree,
                    int elem_bytes, int n_layers, int batch, int hkv, int n_nodes, int head_dim,
                    const int32_t *acc_len, const int32_t *acc_path, int path_cap,
                    const int32_t *prefix_len, int32_t *prefix_len_out, int32_t *dev_status,
                    spec_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */
