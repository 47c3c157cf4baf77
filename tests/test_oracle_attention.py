"""Pins for the oracle's tree attention (no GPU).

Textbook special cases computed with PyTorch's own scaled-dot-product
attention on the CPU in float64 (a library routine independent of the
oracle): a chain tree is ordinary causal attention; every tree node equals
ordinary causal attention over the sequence prefix ++ (root-to-node path),
read at its last position; one node is plain decode attention.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as A
from oracle import tree as T
from tree_speculative_decoding_attn_gb300 import synth


def _inputs(seed, B, Hq, Hkv, D, P, N, smax=None):
    g = np.random.default_rng(seed)
    smax = smax or P + N + 3
    q = g.standard_normal((B, N, Hq, D)) * 2.0
    kc = g.standard_normal((B, Hkv, smax, D))
    vc = g.standard_normal((B, Hkv, smax, D))
    kt = g.standard_normal((B, Hkv, N, D))
    vt = g.standard_normal((B, Hkv, N, D))
    return q, kc, vc, kt, vt


def _sdpa_causal(q_seq, k_seq, v_seq):
    """q/k/v [H, L, D] float64 -> causal attention [H, L, D] via torch."""
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x))
    return F.scaled_dot_product_attention(t(q_seq), t(k_seq), t(v_seq), is_causal=True).numpy()


@pytest.mark.parametrize("G", [1, 4])
def test_chain_tree_equals_causal_attention(G):
    B, Hkv, D, P, N = 2, 2, 16, 9, 6
    Hq = Hkv * G
    q, kc, vc, kt, vt = _inputs(1, B, Hq, Hkv, D, P, N)
    mask = T.depth_and_mask(synth.chain(N).parents)[1]
    prefix = np.array([P, P - 4])
    o = A.tree_attention(q, kc, vc, kt, vt, prefix, mask)
    for b in range(B):
        p = prefix[b]
        for h in range(Hq):
            kv = h // G
            k_seq = np.concatenate([kc[b, kv, :p], kt[b, kv]])[None]
            v_seq = np.concatenate([vc[b, kv, :p], vt[b, kv]])[None]
            # queries for prefix positions are irrelevant: use zeros there
            q_seq = np.concatenate([np.zeros((p, D)), q[b, :, h]])[None]
            ref = _sdpa_causal(q_seq, k_seq, v_seq)[0, p:]
            np.testing.assert_allclose(o[b, :, h], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed,n,caps", [(2, 5, None), (3, 24, (4, 3, 2)), (4, 40, (6, 3, 2, 2)),
                                         (5, 256, (8, 8, 4, 2))])
def test_every_node_equals_attention_over_its_path(seed, n, caps):
    shape = synth.p4_example() if caps is None else synth.random_tree(seed, n, caps)
    B, Hkv, G, D, P = 2, 2, 2, 8, 11
    q, kc, vc, kt, vt = _inputs(seed, B, Hkv * G, Hkv, D, P, n)
    depth, mask = T.depth_and_mask(shape.parents)
    prefix = np.array([P, 3])
    o = A.tree_attention(q, kc, vc, kt, vt, prefix, mask)
    for b in range(B):
        p = prefix[b]
        for i in range(n):
            path = [i]
            while shape.parents[path[-1]] >= 0:
                path.append(int(shape.parents[path[-1]]))
            path = path[::-1]
            for h in range(Hkv * G):
                kv = h // G
                k_seq = np.concatenate([kc[b, kv, :p], kt[b, kv, path]])[None]
                v_seq = np.concatenate([vc[b, kv, :p], vt[b, kv, path]])[None]
                q_seq = np.zeros((1, p + len(path), D))
                q_seq[0, -1] = q[b, i, h]
                ref = _sdpa_causal(q_seq, k_seq, v_seq)[0, -1]
                np.testing.assert_allclose(o[b, i, h], ref, rtol=1e-12, atol=1e-12)


def test_single_node_is_decode_attention():
    q, kc, vc, kt, vt = _inputs(5, 1, 4, 1, 32, 50, 1)
    o = A.tree_attention(q, kc, vc, kt, vt, np.array([50]), np.ones((1, 1), bool))
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x))
    k = np.concatenate([kc[0, 0, :50], kt[0, 0]])
    v = np.concatenate([vc[0, 0, :50], vt[0, 0]])
    ref = F.scaled_dot_product_attention(t(q[0, 0][:, None]), t(k)[None], t(v)[None])[:, 0].numpy()
    np.testing.assert_allclose(o[0, 0], ref, rtol=1e-12, atol=1e-12)


def test_gqa_head_mapping_matches_library():
    B, Hkv, G, D, P, N = 1, 2, 4, 8, 13, 5
    q, kc, vc, kt, vt = _inputs(6, B, Hkv * G, Hkv, D, P, N)
    mask = T.depth_and_mask(synth.P4_PARENTS)[1]
    o = A.tree_attention(q, kc, vc, kt, vt, np.array([P]), mask)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x))
    k = np.concatenate([kc[0, :, :P], kt[0]], axis=1)          # [Hkv, P+N, D]
    v = np.concatenate([vc[0, :, :P], vt[0]], axis=1)
    allowed = np.concatenate([np.ones((N, P), bool), mask], axis=1)  # [N, P+N]
    qh = t(q[0].transpose(1, 0, 2))                               # [Hq, N, D]
    ref = F.scaled_dot_product_attention(qh, t(k).repeat_interleave(G, 0), t(v).repeat_interleave(G, 0),
                                         attn_mask=t(allowed)).numpy()
    np.testing.assert_allclose(o[0].transpose(1, 0, 2), ref, rtol=1e-12, atol=1e-12)


def test_prefix_order_does_not_matter_and_stale_rows_are_ignored():
    B, Hkv, D, P, N = 1, 1, 16, 20, 5
    q, kc, vc, kt, vt = _inputs(7, B, 2, Hkv, D, P, N, smax=40)
    mask = T.depth_and_mask(synth.P4_PARENTS)[1]
    o = A.tree_attention(q, kc, vc, kt, vt, np.array([P]), mask)
    perm = np.random.default_rng(0).permutation(P)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[0, 0, :P] = kc[0, 0, perm]
    vc2[0, 0, :P] = vc[0, 0, perm]
    kc2[0, 0, P:] = 1e3                                          # rows past the prefix
    vc2[0, 0, P:] = -1e3
    o2 = A.tree_attention(q, kc2, vc2, kt, vt, np.array([P]), mask)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)


def test_sibling_branch_kv_is_invisible():
    B, Hkv, D, P, N = 1, 1, 8, 6, 5
    q, kc, vc, kt, vt = _inputs(8, B, 1, Hkv, D, P, N)
    mask = T.depth_and_mask(synth.P4_PARENTS)[1]
    o = A.tree_attention(q, kc, vc, kt, vt, np.array([P]), mask)
    kt2, vt2 = kt.copy(), vt.copy()
    kt2[0, 0, [1, 3]] += 5.0                                     # the "return" branch
    vt2[0, 0, [1, 3]] -= 5.0
    o2 = A.tree_attention(q, kc, vc, kt2, vt2, np.array([P]), mask)
    np.testing.assert_array_equal(o[0, [0, 2, 4]], o2[0, [0, 2, 4]])
    assert np.abs(o[0, [1, 3]] - o2[0, [1, 3]]).max() > 1e-3
