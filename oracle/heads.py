"""Medusa heads, LM head and top-s selection (oracle; test infrastructure only).

"Medusa, explained", procedure step 1 and the symbol list: head k computes
softmax(W2_k (SiLU(W1_k h) + h)), W1 d x d, W2 d x vocabulary.  "Medusa and
EAGLE: self-speculative decoding heads, explained", section "Implementation
sketch": the first linear layer may carry a bias (zero-initialised), the
vocabulary projection has none.  Section "Medusa: heads, losses and trees":
head k contributes its top s_k candidates to the tree.
"""
from __future__ import annotations

import numpy as np


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x) = x / (1 + exp(-x))."""
    return x / (1.0 + np.exp(-x))


def medusa_heads(h, w1, b1, w2):
    """h [B,d]; w1 [K,d,d] (nn.Linear [out,in]); b1 [K,d] or None;
    w2 [K,V,d].  Returns z [B,K,d] = h + SiLU(W1 h + b1) and the head logits
    [B,K,V] = W2 z, float64 throughout (softmax is monotone, so top-s on the
    logits equals top-s on the probabilities)."""
    h = np.asarray(h, np.float64)
    K = w1.shape[0]
    B, d = h.shape
    z = np.empty((B, K, d))
    logits = np.empty((B, K, w2.shape[1]))
    for k in range(K):
        a = h @ np.asarray(w1[k], np.float64).T
        if b1 is not None:
            a = a + np.asarray(b1[k], np.float64)
        z[:, k] = h + silu(a)
        logits[:, k] = z[:, k] @ np.asarray(w2[k], np.float64).T
    return z, logits


def lm_head(hid, w):
    """logits [R,V] = hid [R,d] . W[V,d]^T in float64 ("Medusa, explained",
    step 6: one pass of the base model scores every tree node)."""
    return np.asarray(hid, np.float64) @ np.asarray(w, np.float64).T


def topk(rows, s: int):
    """Top-s per row by value, descending; equal values -> lower index
    first.  A full stable sort is the definition.  Returns (idx, val)."""
    rows = np.asarray(rows)
    flat = rows.reshape(-1, rows.shape[-1])
    idx = np.empty((flat.shape[0], s), np.int64)
    for r in range(flat.shape[0]):
        order = sorted(range(flat.shape[1]), key=lambda x: (-float(flat[r, x]), x)) if flat.shape[1] <= 64 \
            else np.lexsort((np.arange(flat.shape[1]), -flat[r].astype(np.float64)))
        idx[r] = np.asarray(order[:s])
    val = np.take_along_axis(flat, idx, axis=1)
    return idx.reshape(rows.shape[:-1] + (s,)), val.reshape(rows.shape[:-1] + (s,))
