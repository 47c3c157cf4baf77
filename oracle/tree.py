"""Tree bookkeeping of the verify pass (oracle; test infrastructure only).

Follows "5.3 Medusa、EAGLE 与 MTP" (infra-guide), section 3.1 (every node
sees the shared prefix and its own ancestors, never a sibling branch),
section 3.2 (position ids set by depth; siblings share a position) and the
worked example of section 8 (a parents array with parent < node; walk each
node's ancestor chain to mark what it may see).  "Medusa, explained",
procedure steps 5-6: the tree is flattened into one sequence with that mask
and depth positions.  EAGLE-2 rerank: section 5.2 of the same infra-guide
page (node value = product of draft confidences along its path; the top
nodes by value go to verification).
"""
from __future__ import annotations

import numpy as np


def check_parents(parents) -> None:
    """parents[0] == -1 and 0 <= parents[i] < i for i >= 1 (section 8's
    requirement that a parent precedes its child)."""
    p = [int(x) for x in parents]
    if not p or p[0] != -1:
        raise ValueError("node 0 must be the root (parent -1)")
    for i in range(1, len(p)):
        if not (0 <= p[i] < i):
            raise ValueError(f"parents[{i}]={p[i]} must satisfy 0 <= parent < node")


def depth_and_mask(parents):
    """depth[i] and the boolean ancestor-or-self matrix mask[i][j].

    Section 8's procedure: depth = depth(parent) + 1 (root 0); for each node
    walk parent links up to the root, marking every node met (itself first).
    """
    check_parents(parents)
    n = len(parents)
    mask = np.zeros((n, n), dtype=bool)
    depth = np.zeros(n, dtype=np.int64)
    for node in range(n):
        parent = int(parents[node])
        depth[node] = 0 if parent == -1 else depth[parent] + 1
        cursor = node
        while cursor != -1:
            mask[node, cursor] = True
            cursor = int(parents[cursor])
    return depth, mask


def mask_words(mask: np.ndarray) -> np.ndarray:
    """Pack mask rows into uint64 words: bit j of word i = mask[i][j] (N <= 64)."""
    n = mask.shape[-1]
    assert n <= 64
    w = np.zeros(mask.shape[:-1], dtype=np.uint64)
    for j in range(n):
        w |= mask[..., j].astype(np.uint64) << np.uint64(j)
    return w


def mask_words_multi(mask: np.ndarray) -> np.ndarray:
    """Pack mask rows into ceil(N / 64) uint64 words per row: node j is bit
    j % 64 of word j // 64.  Shape [..., N, words]."""
    n = mask.shape[-1]
    nw = (n + 63) // 64
    w = np.zeros(mask.shape[:-1] + (nw,), dtype=np.uint64)
    for j in range(n):
        w[..., j // 64] |= mask[..., j].astype(np.uint64) << np.uint64(j % 64)
    return w


def child_links(parents):
    """first_child[v] and next_sibling[c] in node order (-1 = none)."""
    n = len(parents)
    first = np.full(n, -1, np.int64)
    nxt = np.full(n, -1, np.int64)
    last = {}
    for c in range(1, n):
        p = int(parents[c])
        if first[p] == -1:
            first[p] = c
        else:
            nxt[last[p]] = c
        last[p] = c
    return first, nxt


def build_tree(parents, prefix_len: int) -> dict:
    """Everything the verify pass needs from one tree's parents array."""
    depth, mask = depth_and_mask(parents)
    first, nxt = child_links(parents)
    return dict(parent=np.asarray(parents, np.int64), depth=depth, mask=mask,
                anc=mask_words(mask) if len(parents) <= 64 else mask_words_multi(mask), pos=prefix_len + depth,
                first_child=first, next_sibling=nxt)


def build_tree_static(parents, rank, cand_tok, root_tok, prefix_len) -> dict:
    """Medusa static tree for a batch ("Medusa, explained", steps 5-6;
    "Medusa and EAGLE ... explained", section "Medusa: heads, losses and
    trees"): the shape (parents, rank) is shared; node i at depth d >= 1
    carries the rank[i]-th candidate of head d, cand_tok[b, d-1, rank[i]];
    the root carries the token the target already chose."""
    B = len(root_tok)
    t = build_tree(parents, 0)
    n = len(parents)
    tok = np.empty((B, n), np.int64)
    for b in range(B):
        tok[b, 0] = root_tok[b]
        for i in range(1, n):
            tok[b, i] = cand_tok[b, t["depth"][i] - 1, rank[i]]
    out = {k: np.broadcast_to(v, (B,) + v.shape).copy() for k, v in t.items() if k != "pos"}
    out["tok"] = tok
    out["pos"] = np.asarray(prefix_len, np.int64)[:, None] + t["depth"][None, :]
    return out


def path_values_f32(pool_parent, pool_conf):
    """val[i] = val[parent] * conf[i], root value 1, each product one IEEE
    float32 multiply taken in root-to-node order (section 5.2's path
    product).  Requires pool_parent[i] < i."""
    m = len(pool_parent)
    val = np.zeros(m, np.float32)
    val[0] = np.float32(1.0)
    for i in range(1, m):
        p = int(pool_parent[i])
        assert 0 <= p < i
        val[i] = np.float32(val[p] * np.float32(pool_conf[i]))
    return val


def rerank_dynamic(pool_parent, pool_tok, pool_conf, n: int, prefix_len: int) -> dict:
    """Keep the root and the n-1 pool nodes of highest path value (ties:
    shallower first, then lower pool index), then re-emit them breadth-first
    (by depth, then parent's new index, then value descending, then pool
    index).  Section 5.2: expansion picks nodes by path value, the rerank
    sends the highest-value nodes of the whole tree to verification.

    With confidences in [0, 1] a child's value never exceeds its parent's,
    and the tie order puts the parent first, so the kept set contains every
    kept node's parent."""
    m = len(pool_parent)
    val = path_values_f32(pool_parent, pool_conf)
    depth = np.zeros(m, np.int64)
    for i in range(1, m):
        depth[i] = depth[pool_parent[i]] + 1
    others = sorted(range(1, m), key=lambda i: (-float(val[i]), depth[i], i))
    keep = [0] + others[: n - 1]
    kept = set(keep)
    for i in keep[1:]:
        if int(pool_parent[i]) not in kept:
            raise ValueError("kept set is not closed under parents (confidence > 1?)")
    # breadth-first re-emission
    order = [0]
    new_index = {0: 0}
    for d in range(1, int(depth[keep].max()) + 1 if len(keep) > 1 else 1):
        level = [i for i in keep if depth[i] == d]
        level.sort(key=lambda i: (new_index[int(pool_parent[i])], -float(val[i]), i))
        for i in level:
            new_index[i] = len(order)
            order.append(i)
    parents = [-1] + [new_index[int(pool_parent[i])] for i in order[1:]]
    t = build_tree(parents, prefix_len)
    t["tok"] = np.array([pool_tok[i] for i in order], np.int64)
    t["pool_index"] = np.array(order, np.int64)
    t["val"] = np.array([val[i] for i in order], np.float32)
    return t
