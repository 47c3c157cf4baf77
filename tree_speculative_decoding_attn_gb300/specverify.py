"""Python binding of libspecverify (the C ABI in ``include/specverify.h``).

Argument marshalling only: every function takes torch CUDA tensors (caller
owned), checks their dtype/device/contiguity, passes raw device pointers
and sizes to the C entry point of the same name on the current torch
stream, and raises ``SpecError`` on a non-zero status.  No step of the
method runs here.  There is no fallback: if the library is missing or a
tensor is not on a CUDA device, the call fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CAPACITY, ERR_CUDA = range(5)
(DEV_OK, DEV_BAD_PARENTS, DEV_CAPACITY, DEV_BAD_PATH, DEV_BAD_POOL, DEV_BAD_TOKEN, DEV_TIMEOUT, DEV_INTERNAL,
 DEV_BAD_BLOCK) = range(9)
F32, BF16 = 0, 1
GREEDY, TYPICAL, REJECT, REJECT_STOCHASTIC = 0, 1, 2, 3
MAX_NODES = 256


def mask_words(n_nodes):
    """uint64 words of one node's ancestor mask."""
    return (n_nodes + 63) // 64

_lib = None

_vp, _i, _f, _u64, _sz = C.c_void_p, C.c_int, C.c_float, C.c_uint64, C.c_size_t
_SIGS = {
    "spec_status_string": ([_i], C.c_char_p),
    "spec_abi_version": ([], _i),
    "spec_medusa_heads_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "spec_medusa_heads": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp, _vp], _i),
    "spec_topk": ([_vp, _i, _i, _i, _i, _i, _vp, _vp, _vp], _i),
    "spec_build_tree": ([_vp, _vp, _vp, _i, _i, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _i),
    "spec_build_tree_dynamic": ([_vp, _vp, _vp, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                 _vp, _vp, _vp], _i),
    "spec_build_tree_batch": ([_vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _i),
    "spec_tree_expand": ([_vp, _i, _i, _i, _i, _vp, _i, _f, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _vp], _i),
    "spec_eagle_round_workspace_bytes": ([_i] * 10, _sz),
    "spec_eagle_round": ([_vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _f,
                          _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _vp, _sz, _vp, _vp], _i),
    "tree_attn_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i, _i], _sz),
    "tree_attn_plan_splits": ([_i, _i, _i, _i, _i, _i, _vp], _i),
    "tree_attn_verify": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i,
                          _vp, _sz, _vp, _vp], _i),
    "tree_attn_verify_paged": ([_vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                _i, _f, _i, _vp, _sz, _vp, _vp], _i),
    "tree_attn_verify_noalloc": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f,
                                  _i, _vp, _vp], _i),
    "spec_lm_head_workspace_bytes": ([_i, _i, _i], _sz),
    "spec_lm_head": ([_vp, _vp, _i, _i, _i, _vp, _vp, _sz, _vp, _vp], _i),
    "spec_lm_head_accept_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "spec_lm_head_accept": ([_i, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _f, _f, _i, _vp, _vp, _vp, _vp, _sz,
                             _vp, _vp], _i),
    "spec_accept": ([_i, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _f, _f, _u64, _u64, _i, _vp, _vp,
                     _vp, _vp, _vp], _i),
    "kv_commit_paged": ([_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _i, _vp, _vp, _vp,
                         _vp], _i),
    "kv_commit": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp], _i),
    "spec_accept_commit": ([_i, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _f, _f, _u64, _u64, _i, _vp, _vp,
                            _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp], _i),
}


class SpecError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn}: status {code} ({spec_status_string(code)})")
        self.code = code


def load(path: str | None = None):
    """Load the shared library once (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or os.environ.get("SPECVERIFY_LIB", LIB_PATH)
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = C.CDLL(p)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res
    _lib = lib
    return lib


def exported_symbols():
    return sorted(_SIGS)


# ---------------------------------------------------------------- helpers

_DT = {torch.float32: F32, torch.bfloat16: BF16}


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return C.c_void_p(t.data_ptr())


def _want(t, *dtypes):
    if t is not None and t.dtype not in dtypes:
        raise TypeError(f"dtype {t.dtype} not in {dtypes}")
    return t


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn, code):
    if code != OK:
        raise SpecError(fn, code)


def spec_status_string(code: int) -> str:
    return load().spec_status_string(int(code)).decode()


def spec_abi_version() -> int:
    return int(load().spec_abi_version())


# ---------------------------------------------------------------- entry points


def spec_medusa_heads_workspace_bytes(batch, n_heads, hidden, vocab):
    return int(load().spec_medusa_heads_workspace_bytes(batch, n_heads, hidden, vocab))


def _scratch(nbytes, like):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=like.device)


def spec_medusa_heads(h, w1, b1, w2, z, logits, workspace=None, dev_status=None):
    """z (bf16) and logits (float32) of every head; ``workspace`` (uint8,
    at least spec_medusa_heads_workspace_bytes) is allocated per call when
    not given."""
    B, d = h.shape
    K, V = w2.shape[0], w2.shape[1]
    for t in (h, w1, w2, z):
        _want(t, torch.bfloat16)
    _want(b1, torch.bfloat16)
    _want(logits, torch.float32)
    if workspace is None:
        workspace = _scratch(spec_medusa_heads_workspace_bytes(B, K, d, V), h)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("spec_medusa_heads", load().spec_medusa_heads(_p(h), _p(w1), _p(b1), _p(w2), B, K, d, V, _p(z),
                                                         _p(logits), _p(workspace), ws_bytes, _p(dev_status),
                                                         _stream()))


def spec_topk(rows, s, idx_out, val_out=None, row_len=None):
    _want(rows, torch.float32, torch.bfloat16)
    _want(idx_out, torch.int32); _want(val_out, torch.float32)
    n_rows, stride = rows.reshape(-1, rows.shape[-1]).shape
    _check("spec_topk", load().spec_topk(_p(rows), _DT[rows.dtype], n_rows, row_len or stride, stride, s,
                                         _p(idx_out), _p(val_out), _stream()))


def spec_build_tree(parents, rank, cand_tok, root_tok, prefix_len, tok, depth, pos_ids, anc_mask,
                    first_child, next_sibling, dev_status=None):
    B, N = depth.shape
    levels = cand_tok.shape[1] if cand_tok is not None else 0
    s = cand_tok.shape[2] if cand_tok is not None else 0
    for t in (parents, rank, cand_tok, root_tok, prefix_len, tok, depth, pos_ids, first_child, next_sibling,
              dev_status):
        _want(t, torch.int32)
    _want(anc_mask, torch.int64)
    _check("spec_build_tree", load().spec_build_tree(
        _p(parents), _p(rank), _p(cand_tok), levels, s, _p(root_tok), _p(prefix_len), B, N, _p(tok),
        _p(depth), _p(pos_ids), _p(anc_mask), _p(first_child), _p(next_sibling), _p(dev_status), _stream()))


def spec_build_tree_batch(parents, prefix_len, depth, pos_ids, anc_mask, first_child, next_sibling, n_valid=None,
                          tok_in=None, tok=None, dev_status=None):
    """One tree per sequence: parents [B, N] (first n_valid[b] entries
    valid), tokens copied from tok_in when given."""
    B, N = parents.shape
    for t in (parents, n_valid, tok_in, tok, prefix_len, depth, pos_ids, first_child, next_sibling, dev_status):
        _want(t, torch.int32)
    _want(anc_mask, torch.int64)
    _check("spec_build_tree_batch", load().spec_build_tree_batch(
        _p(parents), _p(n_valid), _p(tok_in), _p(prefix_len), B, N, _p(tok), _p(depth), _p(pos_ids), _p(anc_mask),
        _p(first_child), _p(next_sibling), _p(dev_status), _stream()))


def spec_build_tree_dynamic(pool_parent, pool_tok, pool_conf, prefix_len, tok, parents_out, depth, pos_ids,
                            anc_mask, first_child, next_sibling, pool_index=None, val=None, dev_status=None):
    B, M = pool_parent.shape
    N = tok.shape[1]
    _want(pool_conf, torch.float32); _want(val, torch.float32); _want(anc_mask, torch.int64)
    _check("spec_build_tree_dynamic", load().spec_build_tree_dynamic(
        _p(pool_parent), _p(pool_tok), _p(pool_conf), M, _p(prefix_len), B, N, _p(tok), _p(parents_out),
        _p(depth), _p(pos_ids), _p(anc_mask), _p(first_child), _p(next_sibling), _p(pool_index), _p(val),
        _p(dev_status), _stream()))


def spec_tree_expand(draft_logits, frontier, k, temperature, pool_parent, pool_tok, pool_conf, pool_val,
                     pool_count, next_frontier, dev_status=None):
    B, F, V = draft_logits.shape
    _check("spec_tree_expand", load().spec_tree_expand(
        _p(draft_logits), _DT[draft_logits.dtype], B, F, V, _p(frontier), k, float(temperature),
        _p(pool_parent), _p(pool_tok), _p(pool_conf), _p(pool_val), _p(pool_count), pool_parent.shape[1],
        _p(next_frontier), next_frontier.shape[1], _p(dev_status), _stream()))


EAGLE_WEIGHTS = ("fc", "ln1", "qkv", "o", "ln2", "gate_up", "down", "lnf", "lm", "emb")


class _EagleWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in EAGLE_WEIGHTS]


def spec_eagle_round_workspace_bytes(batch, n_front, hidden, hq, hkv, head_dim, ffn, vocab, s_max, max_prefix):
    return int(load().spec_eagle_round_workspace_bytes(batch, n_front, hidden, hq, hkv, head_dim, ffn, vocab, s_max,
                                                       max_prefix))


def spec_eagle_round(weights, k_prefix, v_prefix, prefix_len, max_prefix, k_nodes, v_nodes, feat, frontier, depth, k,
                     temperature, pool_parent, pool_tok, pool_conf, pool_val, pool_count, next_frontier,
                     draft_logits=None, workspace=None, dev_status=None):
    """One EAGLE drafting round; ``weights`` maps the names in EAGLE_WEIGHTS
    to bf16 tensors (layouts in the C header)."""
    B, _, d = feat.shape
    hkv, S, D = k_prefix.shape[1], k_prefix.shape[2], k_prefix.shape[3]
    hq = weights["o"].shape[1] // D
    ffn = weights["down"].shape[1]
    V = weights["lm"].shape[0]
    F = frontier.shape[1]
    for n in EAGLE_WEIGHTS:
        _want(weights[n], torch.bfloat16)
    for t in (k_prefix, v_prefix, k_nodes, v_nodes, feat):
        _want(t, torch.bfloat16)
    _want(draft_logits, torch.float32)
    w = _EagleWeights(*[_p(weights[n]).value for n in EAGLE_WEIGHTS])
    if workspace is None:
        workspace = _scratch(spec_eagle_round_workspace_bytes(B, F, d, hq, hkv, D, ffn, V, S, int(max_prefix)), feat)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("spec_eagle_round", load().spec_eagle_round(
        C.c_void_p(C.addressof(w)), B, d, hq, hkv, D, ffn, V, _p(k_prefix), _p(v_prefix), S, _p(prefix_len),
        int(max_prefix), _p(k_nodes), _p(v_nodes), _p(feat), _p(frontier), F, int(depth), int(k), float(temperature),
        _p(pool_parent), _p(pool_tok), _p(pool_conf), _p(pool_val), _p(pool_count), pool_parent.shape[1],
        _p(next_frontier), next_frontier.shape[1], _p(draft_logits), _p(workspace), ws_bytes, _p(dev_status),
        _stream()))


def tree_attn_workspace_bytes(dtype, batch, n_nodes, hq, hkv, head_dim, max_prefix, num_splits=0):
    code = _DT[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().tree_attn_workspace_bytes(code, batch, n_nodes, hq, hkv, head_dim, max_prefix, num_splits))


def tree_attn_plan_splits(dtype, batch, n_nodes, hq, hkv, head_dim, host_prefix_len):
    """Split count for a batch whose prefix lengths the host knows (a
    sequence of ints); pass it as num_splits."""
    import numpy as np
    code = _DT[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    arr = np.ascontiguousarray(np.asarray(host_prefix_len, dtype=np.int32))
    n = int(load().tree_attn_plan_splits(code, batch, n_nodes, hq, hkv, head_dim,
                                         arr.ctypes.data_as(C.c_void_p)))
    if n <= 0:
        raise SpecError("tree_attn_plan_splits", ERR_INVALID_ARG)
    return n


def tree_attn_verify(q, k_cache, v_cache, k_tree, v_tree, prefix_len, anc_mask, out, max_prefix,
                     scale=0.0, num_splits=0, workspace=None, dev_status=None):
    B, N, Hq, D = q.shape
    Hkv, S = k_cache.shape[1], k_cache.shape[2]
    _want(q, torch.float32, torch.bfloat16)
    for t in (k_cache, v_cache, k_tree, v_tree, out):
        if t.dtype != q.dtype:
            raise TypeError("q, caches, tree K/V and out must share one dtype")
    _want(anc_mask, torch.int64); _want(prefix_len, torch.int32)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("tree_attn_verify", load().tree_attn_verify(
        _p(q), _p(k_cache), _p(v_cache), _p(k_tree), _p(v_tree), _p(prefix_len), _p(anc_mask), _p(out),
        _DT[q.dtype], B, N, Hq, Hkv, D, S, int(max_prefix), float(scale), int(num_splits), _p(workspace),
        ws_bytes, _p(dev_status), _stream()))


def tree_attn_verify_paged(q, k_pages, v_pages, block_table, k_tree, v_tree, prefix_len, anc_mask, out, max_prefix,
                           scale=0.0, num_splits=0, workspace=None, dev_status=None):
    """tree_attn_verify over a paged prefix cache: k_pages/v_pages
    [num_blocks, Hkv, block_size, D], block_table [B, max_blocks] int32."""
    B, N, Hq, D = q.shape
    nb, Hkv, bs = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    _want(q, torch.float32, torch.bfloat16)
    for t in (k_pages, v_pages, k_tree, v_tree, out):
        if t.dtype != q.dtype:
            raise TypeError("q, pages, tree K/V and out must share one dtype")
    _want(anc_mask, torch.int64); _want(prefix_len, torch.int32); _want(block_table, torch.int32)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("tree_attn_verify_paged", load().tree_attn_verify_paged(
        _p(q), _p(k_pages), _p(v_pages), _p(block_table), bs, nb, block_table.shape[1], _p(k_tree), _p(v_tree),
        _p(prefix_len), _p(anc_mask), _p(out), _DT[q.dtype], B, N, Hq, Hkv, D, int(max_prefix), float(scale),
        int(num_splits), _p(workspace), ws_bytes, _p(dev_status), _stream()))


NOALLOC_SCRATCH_BYTES = 32 << 20


def tree_attn_verify_noalloc(q, k_cache, v_cache, k_tree, v_tree, prefix_len, anc_mask, out, max_prefix,
                             scale=0.0, num_splits=0, dev_status=None):
    """tree_attn_verify for callers that cannot allocate: the split-KV
    partials live in the library's own fixed device array (32 MiB, shared by
    every call; calls that overlap on the GPU race on it)."""
    B, N, Hq, D = q.shape
    Hkv, S = k_cache.shape[1], k_cache.shape[2]
    _want(q, torch.float32, torch.bfloat16)
    for t in (k_cache, v_cache, k_tree, v_tree, out):
        if t.dtype != q.dtype:
            raise TypeError("q, caches, tree K/V and out must share one dtype")
    _want(anc_mask, torch.int64); _want(prefix_len, torch.int32)
    _check("tree_attn_verify_noalloc", load().tree_attn_verify_noalloc(
        _p(q), _p(k_cache), _p(v_cache), _p(k_tree), _p(v_tree), _p(prefix_len), _p(anc_mask), _p(out),
        _DT[q.dtype], B, N, Hq, Hkv, D, S, int(max_prefix), float(scale), int(num_splits), _p(dev_status),
        _stream()))


def spec_lm_head_workspace_bytes(rows, hidden, vocab):
    return int(load().spec_lm_head_workspace_bytes(rows, hidden, vocab))


def spec_lm_head(hid, w, logits, dev_status=None, workspace=None):
    R, d = hid.shape
    V = w.shape[0]
    _want(hid, torch.bfloat16); _want(w, torch.bfloat16); _want(logits, torch.float32)
    if workspace is None:
        workspace = _scratch(spec_lm_head_workspace_bytes(R, d, V), hid)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("spec_lm_head", load().spec_lm_head(_p(hid), _p(w), R, d, V, _p(logits), _p(workspace), ws_bytes,
                                               _p(dev_status), _stream()))


def spec_lm_head_accept_workspace_bytes(batch, n_nodes, hidden, vocab):
    return int(load().spec_lm_head_accept_workspace_bytes(batch, n_nodes, hidden, vocab))


def spec_lm_head_accept(mode, hid, w, tok, parents, first_child, next_sibling, acc_len, acc_path, bonus,
                        temperature=1.0, eps=0.0, delta=0.0, dev_status=None, workspace=None):
    """LM head fused with greedy / typical acceptance.  hid [B, N, hidden]
    bf16, w [V, hidden] bf16; outputs as spec_accept."""
    B, N, d = hid.shape
    V = w.shape[0]
    _want(hid, torch.bfloat16); _want(w, torch.bfloat16)
    if workspace is None:
        workspace = _scratch(spec_lm_head_accept_workspace_bytes(B, N, d, V), hid)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("spec_lm_head_accept", load().spec_lm_head_accept(
        int(mode), _p(hid), _p(w), B, N, d, V, _p(tok), _p(parents), _p(first_child), _p(next_sibling),
        float(temperature), float(eps), float(delta), acc_path.shape[1], _p(acc_len), _p(acc_path), _p(bonus),
        _p(workspace), ws_bytes, _p(dev_status), _stream()))


def spec_accept(mode, logits, tok, parents, first_child, next_sibling, acc_len, acc_path, bonus,
                temperature=1.0, eps=0.0, delta=0.0, seed=0, step=0, dev_status=None, draft_logits=None):
    B, N, V = logits.shape
    _want(logits, torch.float32, torch.bfloat16)
    if draft_logits is not None and (draft_logits.dtype != logits.dtype or draft_logits.shape != logits.shape):
        raise TypeError("draft_logits must match logits in dtype and shape")
    _check("spec_accept", load().spec_accept(
        int(mode), _p(logits), _p(draft_logits), _DT[logits.dtype], B, N, V, _p(tok), _p(parents), _p(first_child),
        _p(next_sibling), float(temperature), float(eps), float(delta), int(seed), int(step),
        acc_path.shape[1], _p(acc_len), _p(acc_path), _p(bonus), _p(dev_status), _stream()))


def spec_accept_commit(mode, logits, tok, parents, first_child, next_sibling, acc_len, acc_path, bonus, k_cache,
                       v_cache, k_tree, v_tree, prefix_len, prefix_len_out=None, temperature=1.0, eps=0.0,
                       delta=0.0, seed=0, step=0, dev_status=None, draft_logits=None):
    """spec_accept and kv_commit (contiguous cache) in one launch."""
    B, N, V = logits.shape
    _want(logits, torch.float32, torch.bfloat16)
    if draft_logits is not None and (draft_logits.dtype != logits.dtype or draft_logits.shape != logits.shape):
        raise TypeError("draft_logits must match logits in dtype and shape")
    if k_cache.dim() == 4:
        L, (_, Hkv, S, D) = 1, k_cache.shape
    else:
        L, _, Hkv, S, D = k_cache.shape
    _check("spec_accept_commit", load().spec_accept_commit(
        int(mode), _p(logits), _p(draft_logits), _DT[logits.dtype], B, N, V, _p(tok), _p(parents), _p(first_child),
        _p(next_sibling), float(temperature), float(eps), float(delta), int(seed), int(step), acc_path.shape[1],
        _p(acc_len), _p(acc_path), _p(bonus), _p(k_cache), _p(v_cache), _p(k_tree), _p(v_tree),
        k_cache.element_size(), L, Hkv, S, D, _p(prefix_len), _p(prefix_len_out), _p(dev_status), _stream()))


def kv_commit(k_cache, v_cache, k_tree, v_tree, acc_len, acc_path, prefix_len, prefix_len_out=None,
              dev_status=None):
    if k_cache.dim() == 4:
        L, (B, Hkv, S, D) = 1, k_cache.shape
    else:
        L, B, Hkv, S, D = k_cache.shape
    N = k_tree.shape[-2]
    _check("kv_commit", load().kv_commit(
        _p(k_cache), _p(v_cache), _p(k_tree), _p(v_tree), k_cache.element_size(), L, B, Hkv, S, N, D,
        _p(acc_len), _p(acc_path), acc_path.shape[1], _p(prefix_len), _p(prefix_len_out), _p(dev_status),
        _stream()))


def kv_commit_paged(k_pages, v_pages, block_table, k_tree, v_tree, acc_len, acc_path, prefix_len,
                    prefix_len_out=None, dev_status=None):
    """kv_commit into a paged cache [L, num_blocks, Hkv, block_size, D] (or
    without the layer axis) addressed by block_table [B, max_blocks]."""
    if k_pages.dim() == 4:
        L, (nb, Hkv, bs, D) = 1, k_pages.shape
    else:
        L, nb, Hkv, bs, D = k_pages.shape
    B, N = block_table.shape[0], k_tree.shape[-2]
    _want(block_table, torch.int32)
    _check("kv_commit_paged", load().kv_commit_paged(
        _p(k_pages), _p(v_pages), _p(block_table), bs, nb, block_table.shape[1], _p(k_tree), _p(v_tree),
        k_pages.element_size(), L, B, Hkv, N, D, _p(acc_len), _p(acc_path), acc_path.shape[1], _p(prefix_len),
        _p(prefix_len_out), _p(dev_status), _stream()))
