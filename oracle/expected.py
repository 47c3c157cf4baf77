"""Expected accepted length (oracle; test infrastructure only).

"Medusa and EAGLE ... explained", section "Medusa: heads, losses and trees":
if head k holds the target's token among its top s_k with probability
h_k(s_k), independently across heads, a step yields 1 + sum_k prod_{j<=k}
h_j(s_j) tokens on average (the worked example gives 1.91 for a chain of
top-1 guesses with rates 0.6/0.4/0.3 and 2.37 for a 15-node tree).
"Medusa, explained": one guess accepted with probability a, s guesses with
1 - (1 - a)^s; four heads at 0.8/0.65/0.5/0.35 give about 2.7 tokens per pass.
"""
from __future__ import annotations

import numpy as np


def expected_len_chain(hit):
    """1 + sum_k prod_{j<=k} hit[j]."""
    total, run = 1.0, 1.0
    for h in hit:
        run *= h
        total += run
    return total


def hit_with_candidates(a, s):
    """Probability that at least one of s independent guesses is right."""
    return 1.0 - (1.0 - a) ** s


def expected_len_tree(parents, rank, depth, p_rank):
    """Tree form: 1 + sum over non-root nodes of the probability that every
    node on its root path is the target's token, where p_rank[d-1][r] is the
    probability that head d's rank-r candidate is the target's token (ranks
    are disjoint events).  Equals the chain formula for a full Cartesian tree
    with h_d = sum of its first s_d rank probabilities."""
    n = len(parents)
    pa = np.ones(n)
    total = 1.0
    for i in range(1, n):
        pa[i] = pa[parents[i]] * p_rank[depth[i] - 1][rank[i]]
        total += pa[i]
    return total
