"""Tree attention (oracle; test infrastructure only).

"5.3 Medusa、EAGLE 与 MTP" (infra-guide), sections 3.1 and 8: each flattened
tree node attends to the shared prefix and to its own ancestors (itself
included), never to another branch; "Medusa, explained", step 6 and
"Medusa and EAGLE ... explained", section "Medusa: heads, losses and
trees": all nodes are scored in one pass with that mask.  Scores use the
usual softmax(q.k * scale) with scale = 1/sqrt(head_dim) unless given.

For node i of sequence b and query head h the key list is written out
explicitly: cache rows 0..prefix_len[b]-1 of KV head h // (Hq/Hkv), then the
tree rows of i's ancestors-or-self in ascending node order.  Float64, two
passes (max, then sum of exponentials), then the weighted value sum.
"""
from __future__ import annotations

import numpy as np


def node_keys(kc, vc, kt, vt, b, kvh, prefix, anc_nodes):
    """The explicit (K, V) rows node attention reads, in order."""
    k = np.concatenate([kc[b, kvh, :prefix], kt[b, kvh, anc_nodes]], axis=0)
    v = np.concatenate([vc[b, kvh, :prefix], vt[b, kvh, anc_nodes]], axis=0)
    return np.asarray(k, np.float64), np.asarray(v, np.float64)


def softmax_weighted_sum(q, k, v, scale):
    """softmax(k q * scale) . v for one query vector, float64, two passes."""
    s = (k @ np.asarray(q, np.float64)) * scale
    m = s.max()
    e = np.exp(s - m)
    return (e @ v) / e.sum()


def tree_attention(q, kc, vc, kt, vt, prefix_len, mask, scale=None, nodes=None, heads=None):
    """q [B,N,Hq,D]; kc/vc [B,Hkv,S,D]; kt/vt [B,Hkv,N,D]; prefix_len [B];
    mask [B,N,N] bool (or [N,N] shared) ancestor-or-self matrix.
    Returns o [B,N,Hq,D] float64 (only the listed ``nodes``/``heads`` are
    filled when given; others are NaN)."""
    B, N, Hq, D = q.shape
    Hkv = kc.shape[1]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    mask = np.broadcast_to(mask, (B, N, N))
    out = np.full((B, N, Hq, D), np.nan)
    for b in range(B):
        for i in (range(N) if nodes is None else nodes):
            anc_nodes = np.nonzero(mask[b, i])[0]
            for h in (range(Hq) if heads is None else heads):
                k, v = node_keys(kc, vc, kt, vt, b, h // G, int(prefix_len[b]), anc_nodes)
                out[b, i, h] = softmax_weighted_sum(q[b, i, h], k, v, scale)
    return out
