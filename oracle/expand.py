"""One confidence-product expansion round (oracle; test infrastructure only).

"5.3 Medusa、EAGLE 与 MTP" (infra-guide), section 5.2: a node's value is the
product of the draft's confidences along its path; the expansion phase grows
the nodes of highest value.  "Medusa and EAGLE ... explained", section
"EAGLE: autoregression over features": the draft runs step by step to build
a tree of depth m.

One round: every frontier node f gets the k tokens of highest draft
probability (softmax(draft_logits[f] / T), ties to the lower token id) as
children, with confidence = that probability and value = value(f) *
confidence (one float32 multiply); the next frontier is the F_next new
children of highest value (ties: lower pool index), highest first.
Probabilities are computed in float32 as the kernel does; value ties closer
than ``NEAR`` (relative) are counted as near ties.
"""
from __future__ import annotations

import numpy as np

NEAR = 1e-5


def expand_round(draft_logits, frontier, pool_parent, pool_tok, pool_conf, pool_val, pool_count,
                 k, T, f_next):
    """Arrays are modified copies; returns (pool_parent, pool_tok, pool_conf,
    pool_val, pool_count, next_frontier, near_ties)."""
    pool_parent, pool_tok = pool_parent.copy(), pool_tok.copy()
    pool_conf, pool_val = pool_conf.copy(), pool_val.copy()
    pool_count = np.array(pool_count).copy()
    B, F, V = draft_logits.shape
    nxt = np.full((B, f_next), -1, np.int64)
    near = 0
    for b in range(B):
        base = int(pool_count[b])
        new = []
        for f in range(F):
            src = int(frontier[b, f])
            z = np.asarray(draft_logits[b, f], np.float32) / np.float32(T)
            e = np.exp(z - z.max())
            p = e / e.sum(dtype=np.float32)
            order = np.lexsort((np.arange(V), -np.asarray(draft_logits[b, f], np.float64)))[:k]
            for j, x in enumerate(order):
                m = base + f * k + j
                pool_parent[b, m] = src
                pool_tok[b, m] = x
                pool_conf[b, m] = p[x]
                pool_val[b, m] = np.float32(pool_val[b, src] * p[x])
                new.append(m)
        pool_count[b] = base + F * k
        ranked = sorted(new, key=lambda m: (-float(pool_val[b, m]), m))
        nxt[b, : min(f_next, len(ranked))] = ranked[:f_next]
        if f_next < len(ranked):
            a, c = float(pool_val[b, ranked[f_next - 1]]), float(pool_val[b, ranked[f_next]])
            if abs(a - c) <= NEAR * max(a, 1e-30):
                near += 1
    return pool_parent, pool_tok, pool_conf, pool_val, pool_count, nxt, near
