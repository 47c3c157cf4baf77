"""One confidence-product expansion round (oracle; test infrastructure only).

"5.3 Medusa、EAGLE 与 MTP" (infra-guide), section 5.2: a node's value is the
product of the draft's confidences along its path; the expansion phase grows
the nodes of highest value.  "Medusa and EAGLE ... explained", section
"EAGLE: autoregression over features": the draft runs step by step to build
a tree of depth m.

One round: every frontier node f gets the k tokens of highest draft
probability (softmax(draft_logits[f] / T), ties to the lower token id) as
children, with confidence = that probability and value = value(f) *
confidence; the next frontier is the F_next new children of highest value
(ties: lower pool index), highest first.  Probabilities and values are
computed in float64 (the pool's stored confidences and values are read
exactly); frontier slots whose value is within ``NEAR`` (relative) of a
neighbour in the ranking are reported as near ties, since a kernel working in
float32 may order those two the other way.
"""
from __future__ import annotations

import numpy as np

NEAR = 1e-5


def expand_round(draft_logits, frontier, pool_parent, pool_tok, pool_conf, pool_val, pool_count,
                 k, T, f_next):
    """Returns modified copies (pool_parent, pool_tok, pool_conf, pool_val,
    pool_count, next_frontier, near) with float64 confidences and values;
    ``near`` lists the (sequence, frontier slot) pairs whose entry is within
    rounding of a neighbour in the value ranking."""
    pool_parent, pool_tok = pool_parent.copy(), pool_tok.copy()
    pool_conf = np.asarray(pool_conf, np.float64).copy()
    pool_val = np.asarray(pool_val, np.float64).copy()
    pool_count = np.array(pool_count).copy()
    B, F, V = draft_logits.shape
    nxt = np.full((B, f_next), -1, np.int64)
    near = []
    for b in range(B):
        base = int(pool_count[b])
        new = []
        for f in range(F):
            src = int(frontier[b, f])
            z = np.asarray(draft_logits[b, f], np.float64) / T
            e = np.exp(z - z.max())
            p = e / e.sum()
            order = np.lexsort((np.arange(V), -np.asarray(draft_logits[b, f], np.float64)))[:k]
            for j, x in enumerate(order):
                m = base + f * k + j
                pool_parent[b, m] = src
                pool_tok[b, m] = x
                pool_conf[b, m] = p[x]
                pool_val[b, m] = pool_val[b, src] * p[x]
                new.append(m)
        pool_count[b] = base + F * k
        ranked = sorted(new, key=lambda m: (-float(pool_val[b, m]), m))
        nxt[b, : min(f_next, len(ranked))] = ranked[:f_next]
        for j in range(min(f_next, len(ranked) - 1)):
            a, c = float(pool_val[b, ranked[j]]), float(pool_val[b, ranked[j + 1]])
            if abs(a - c) <= NEAR * max(a, 1e-30):
                near += [(b, j)] + ([(b, j + 1)] if j + 1 < f_next else [])
    return pool_parent, pool_tok, pool_conf, pool_val, pool_count, nxt, sorted(set(near))
