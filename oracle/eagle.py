"""EAGLE draft layer, one drafting round (oracle; test infrastructure only).

"Medusa and EAGLE: self-speculative decoding heads, explained", section
"EAGLE: autoregression over features": the draft concatenates the feature of
a position with the embedding of the token that follows it, reduces the
2d-dimensional vector to d with a fully connected layer, and passes it
through one decoder layer to predict the next feature; the target's frozen
embedding and LM head turn features into tokens.  "5.3 Medusa、EAGLE 与 MTP",
section 4.1 (one fully connected layer plus one decoder layer, the top-layer
feature before the LM head) and section 5.2 (the tree grows at the nodes of
highest path value, the product of draft confidences).

Readings where the pages are silent (each is listed in the design notes):

* The decoder layer has the target's architecture, a LLaMA-style pre-norm
  block: x1 = x + O(attn(RMSNorm(x) W_qkv)); out = x1 + W_down(SiLU(W_gate
  n) * W_up n) with n = RMSNorm(x1).  RMSNorm(x) = x / sqrt(mean(x^2) +
  1e-6) * w.  Attention uses rotary position embedding in the rotate-half
  form (dims i and i + D/2 rotated by pos * base^(-2i/D)), base 10000.
* A drafted node's position is prefix length + its depth, as in the
  verification pass; it attends to the draft layer's own cache of the prefix
  and to the draft K/V of its ancestors and itself in the draft tree.
* The node's input is [feature of its parent ; embedding of its own token];
  the root's parent feature is the target's feature of the last verified
  position (an input).  The predicted feature passes the target's final
  RMSNorm before the LM head; the draft distribution at the node is the
  softmax of those logits / T, expanded by expand_round.
"""
from __future__ import annotations

import numpy as np

from . import attention as A
from . import tree as T

EPS = 1e-6
ROPE_BASE = 10000.0


def rmsnorm(x, w):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + EPS) * np.asarray(w, np.float64)


def rope(x, pos):
    """Rotate-half rotary embedding of x [..., D] at integer positions pos
    (broadcast over the leading axes of x but the head axis)."""
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    half = D // 2
    inv = ROPE_BASE ** (-np.arange(half, dtype=np.float64) * 2.0 / D)
    ang = np.asarray(pos, np.float64)[..., None] * inv            # [..., half]
    c, s = np.cos(ang), np.sin(ang)
    c, s = c[..., None, :], s[..., None, :]                        # broadcast over heads
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


def draft_round(wts, feat, tok_emb, pool_parent, pool_tok, frontier, depth, prefix_len, k_prefix, v_prefix,
                k_nodes, v_nodes, hq, hkv):
    """One drafting round for a batch.

    wts: dict of float arrays: fc [d, 2d], ln1 [d], qkv [(hq + 2 hkv) D, d],
    o [d, hq D], ln2 [d], gate [f, d], up [f, d], down [d, f], lnf [d],
    lm [V, d]; tok_emb [V, d]; feat [B, M + 1, d] node features (slot M: the
    root's parent feature); frontier [B, F] pool indices at depth ``depth``;
    k_prefix/v_prefix [B, hkv, S, D] the draft layer's prefix cache; k_nodes /
    v_nodes [B, hkv, M, D] draft K/V of earlier rounds' nodes (rotary applied).

    Returns (new features [B, F, d], new node K and V [B, hkv, F, D] (rotary
    applied), draft logits [B, F, V]), all float64."""
    B, F = frontier.shape
    M = pool_parent.shape[1]
    d = feat.shape[-1]
    D = wts["qkv"].shape[0] // (hq + 2 * hkv)
    out_f = np.zeros((B, F, d))
    out_k = np.zeros((B, hkv, F, D))
    out_v = np.zeros((B, hkv, F, D))
    logits = np.zeros((B, F, wts["lm"].shape[0]))
    for b in range(B):
        fr = [int(x) for x in frontier[b]]
        par = [int(pool_parent[b, v]) for v in fr]
        x = np.concatenate([np.asarray(feat[b, [p if p >= 0 else M for p in par]], np.float64),
                            np.asarray(tok_emb[[int(pool_tok[b, v]) for v in fr]], np.float64)], axis=-1)
        h0 = x @ np.asarray(wts["fc"], np.float64).T
        n1 = rmsnorm(h0, wts["ln1"])
        qkv = n1 @ np.asarray(wts["qkv"], np.float64).T
        pos = np.full(F, int(prefix_len[b]) + depth)
        q = rope(qkv[:, : hq * D].reshape(F, hq, D), pos)
        kk = rope(qkv[:, hq * D:(hq + hkv) * D].reshape(F, hkv, D), pos)
        vv = qkv[:, (hq + hkv) * D:].reshape(F, hkv, D)
        out_k[b] = kk.transpose(1, 0, 2)
        out_v[b] = vv.transpose(1, 0, 2)
        # the draft tree seen by this round: the frontier and all its
        # ancestors, in pool order (a parent precedes its child)
        nodes = set()
        for v in fr:
            u = v
            while u >= 0:
                nodes.add(u)
                u = int(pool_parent[b, u])
        nodes = sorted(nodes)
        idx = {u: i for i, u in enumerate(nodes)}
        cpar = np.array([-1 if u == nodes[0] else idx[int(pool_parent[b, u])] for u in nodes])
        mask = T.depth_and_mask(cpar)[1]
        kt = np.zeros((1, hkv, len(nodes), D))
        vt = np.zeros((1, hkv, len(nodes), D))
        qq = np.zeros((1, len(nodes), hq, D))
        for i, u in enumerate(nodes):
            if u in fr:
                j = fr.index(u)
                kt[0, :, i], vt[0, :, i], qq[0, i] = out_k[b, :, j], out_v[b, :, j], q[j]
            else:
                kt[0, :, i], vt[0, :, i] = k_nodes[b, :, u], v_nodes[b, :, u]
        att = A.tree_attention(qq, k_prefix[b:b + 1], v_prefix[b:b + 1], kt, vt, np.array([int(prefix_len[b])]),
                               mask, nodes=[idx[v] for v in fr])
        a = att[0, [idx[v] for v in fr]].reshape(F, hq * D)
        h1 = h0 + a @ np.asarray(wts["o"], np.float64).T
        n2 = rmsnorm(h1, wts["ln2"])
        act = silu(n2 @ np.asarray(wts["gate"], np.float64).T) * (n2 @ np.asarray(wts["up"], np.float64).T)
        f = h1 + act @ np.asarray(wts["down"], np.float64).T
        out_f[b] = f
        logits[b] = rmsnorm(f, wts["lnf"]) @ np.asarray(wts["lm"], np.float64).T
    return out_f, out_k, out_v, logits
