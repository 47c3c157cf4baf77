"""Commit of the accepted path's K/V (oracle; test infrastructure only).

"5.3 Medusa、EAGLE 与 MTP" (infra-guide), section 3.2: all nodes share the
prefix KV; after verification only the one accepted path is committed and the
other branches' temporary KV is discarded.  The accepted path (root first,
acc_len + 1 nodes) is appended to each sequence's cache right after its
prefix, and the prefix grows by acc_len + 1.
"""
from __future__ import annotations

import numpy as np


def kv_commit(kc, vc, kt, vt, prefix_len, acc_len, acc_path):
    """kc/vc [L,B,Hkv,S,D] (or [B,Hkv,S,D]) and kt/vt [L,B,Hkv,N,D] (or
    [B,Hkv,N,D]); returns the updated copies and the new prefix lengths.
    Row prefix_len[b] + j receives tree row acc_path[b, j], j = 0..acc_len[b]."""
    kc, vc = kc.copy(), vc.copy()
    layered = kc.ndim == 5
    if not layered:
        kc, vc, kt, vt = kc[None], vc[None], kt[None], vt[None]
    L, B, Hkv = kc.shape[:3]
    for layer in range(L):
        for b in range(B):
            for h in range(Hkv):
                for j in range(int(acc_len[b]) + 1):
                    src = int(acc_path[b, j])
                    kc[layer, b, h, int(prefix_len[b]) + j] = kt[layer, b, h, src]
                    vc[layer, b, h, int(prefix_len[b]) + j] = vt[layer, b, h, src]
    new_len = np.asarray(prefix_len) + np.asarray(acc_len) + 1
    if not layered:
        kc, vc = kc[0], vc[0]
    return kc, vc, new_len
