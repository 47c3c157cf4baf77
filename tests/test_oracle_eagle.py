"""Pins of the EAGLE draft-round oracle against facts it does not compute
itself: properties of rotary embedding and RMSNorm, and special weights under
which the layer reduces to a closed form ("Medusa and EAGLE ... explained",
section "EAGLE: autoregression over features": FC over [feature ; token
embedding], one decoder layer, the target's LM head)."""
import numpy as np

from oracle import eagle as E


def test_rope_is_a_rotation_with_relative_positions():
    g = np.random.default_rng(0)
    q = g.standard_normal((3, 64))
    k = g.standard_normal((3, 64))
    # position 0 is the identity; every position keeps the norm
    np.testing.assert_allclose(E.rope(q[None], np.array([0]))[0], q, atol=1e-12)
    qr = E.rope(q[None], np.array([37]))[0]
    np.testing.assert_allclose(np.linalg.norm(qr, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-12)
    # the score of a rotated pair depends only on the position difference
    s1 = (E.rope(q[None], np.array([100]))[0] * E.rope(k[None], np.array([90]))[0]).sum(-1)
    s2 = (E.rope(q[None], np.array([1010]))[0] * E.rope(k[None], np.array([1000]))[0]).sum(-1)
    np.testing.assert_allclose(s1, s2, rtol=1e-9, atol=1e-9)


def test_rmsnorm_closed_forms():
    w = np.array([1.0, 2.0, 3.0, 4.0])
    x = np.array([[3.0, 3.0, 3.0, 3.0], [1.0, -1.0, 1.0, -1.0]])
    y = E.rmsnorm(x, w)
    np.testing.assert_allclose(y[0], w * 3.0 / np.sqrt(9.0 + E.EPS), rtol=1e-14)
    np.testing.assert_allclose(y[1], w * np.array([1, -1, 1, -1]) / np.sqrt(1.0 + E.EPS), rtol=1e-14)
    np.testing.assert_allclose(E.rmsnorm(5.0 * x, w), E.rmsnorm(x, w), rtol=1e-6)   # scale invariance (up to eps)


def _weights(g, d, hq, hkv, D, f, V, zero_o=False, zero_mlp=False):
    n = lambda *s: g.standard_normal(s) * 0.05
    w = dict(fc=n(d, 2 * d), ln1=1 + n(d), qkv=n((hq + 2 * hkv) * D, d), o=n(d, hq * D), ln2=1 + n(d),
             gate=n(f, d), up=n(f, d), down=n(d, f), lnf=1 + n(d), lm=n(V, d))
    if zero_o:
        w["o"] = np.zeros_like(w["o"])
    if zero_mlp:
        w["down"] = np.zeros_like(w["down"])
    return w


def _pool():
    # root 0; children 1, 2; node 3 under 1
    par = np.array([[-1, 0, 0, 1]])
    tok = np.array([[5, 7, 9, 11]])
    return par, tok


def test_identity_layer_reduces_to_the_fc_of_parent_feature_and_token_embedding():
    g = np.random.default_rng(1)
    d, hq, hkv, D, f, V = 16, 2, 1, 8, 24, 13
    w = _weights(g, d, hq, hkv, D, f, V, zero_o=True, zero_mlp=True)
    emb = g.standard_normal((V, d))
    par, tok = _pool()
    feat = g.standard_normal((1, 5, d))               # slot 4: the root's parent feature
    S = 6
    kp, vp = g.standard_normal((1, hkv, S, D)), g.standard_normal((1, hkv, S, D))
    kn, vn = g.standard_normal((1, hkv, 4, D)), g.standard_normal((1, hkv, 4, D))
    fr = np.array([[2, 3]])
    out_f, _, _, logits = E.draft_round(w, feat, emb, par, tok, fr, 2, np.array([4]), kp, vp, kn, vn, hq, hkv)
    # node 2: parent 0, token 9; node 3: parent 1, token 11
    x = np.stack([np.concatenate([feat[0, 0], emb[9]]), np.concatenate([feat[0, 1], emb[11]])])
    np.testing.assert_allclose(out_f[0], x @ w["fc"].T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(logits[0], E.rmsnorm(out_f[0], w["lnf"]) @ w["lm"].T, rtol=1e-12, atol=1e-12)


def test_lone_root_with_empty_prefix_attends_to_itself_only():
    """Prefix length 0 and the root alone: softmax over one key is 1, so the
    attention output is the node's own V and x1 = h0 + V W_o."""
    g = np.random.default_rng(2)
    d, hq, hkv, D, f, V = 16, 2, 1, 8, 24, 13
    w = _weights(g, d, hq, hkv, D, f, V, zero_mlp=True)
    emb = g.standard_normal((V, d))
    par, tok = _pool()
    feat = g.standard_normal((1, 5, d))
    kp = vp = np.zeros((1, hkv, 4, D))
    kn = vn = np.zeros((1, hkv, 4, D))
    out_f, out_k, out_v, _ = E.draft_round(w, feat, emb, par, tok, np.array([[0]]), 0, np.array([0]), kp, vp, kn, vn,
                                           hq, hkv)
    h0 = np.concatenate([feat[0, 4], emb[5]]) @ w["fc"].T
    qkv = E.rmsnorm(h0, w["ln1"]) @ w["qkv"].T
    v = qkv[(hq + hkv) * D:]
    np.testing.assert_allclose(out_v[0, 0, 0], v, rtol=1e-12)
    a = np.tile(v, hq)                                   # every query head of the group reads the same V
    np.testing.assert_allclose(out_f[0, 0], h0 + a @ w["o"].T, rtol=1e-10, atol=1e-12)
    # the root sits at position 0: its K carries no rotation
    np.testing.assert_allclose(out_k[0, 0, 0], qkv[hq * D:(hq + hkv) * D], rtol=1e-12)


def test_node_attends_to_prefix_and_its_own_path_only():
    """Brute force: node 3's output equals attention over the explicit key
    list prefix ++ (root, node 1, node 3) in root-to-node order; node 2 is
    not on that path and changing its K/V leaves node 3 unchanged."""
    g = np.random.default_rng(3)
    d, hq, hkv, D, f, V = 16, 2, 1, 8, 24, 13
    w = _weights(g, d, hq, hkv, D, f, V)
    emb = g.standard_normal((V, d))
    par, tok = _pool()
    feat = g.standard_normal((1, 5, d))
    S = 7
    kp, vp = g.standard_normal((1, hkv, S, D)), g.standard_normal((1, hkv, S, D))
    kn, vn = g.standard_normal((1, hkv, 4, D)), g.standard_normal((1, hkv, 4, D))
    r1 = E.draft_round(w, feat, emb, par, tok, np.array([[3]]), 2, np.array([5]), kp, vp, kn, vn, hq, hkv)
    kn2, vn2 = kn.copy(), vn.copy()
    kn2[0, :, 2] += 7.0
    vn2[0, :, 2] -= 3.0
    r2 = E.draft_round(w, feat, emb, par, tok, np.array([[3]]), 2, np.array([5]), kp, vp, kn2, vn2, hq, hkv)
    np.testing.assert_allclose(r1[0], r2[0], rtol=1e-12)
    # explicit keys: prefix rows, then nodes 0 and 1 (earlier rounds), then node 3 itself
    h0 = np.concatenate([feat[0, 1], emb[11]]) @ w["fc"].T
    qkv = E.rmsnorm(h0, w["ln1"]) @ w["qkv"].T
    q = E.rope(qkv[: hq * D].reshape(1, hq, D), np.array([7]))[0]
    keys = np.concatenate([kp[0, 0, :5], kn[0, 0, [0, 1]], r1[1][0, 0]], axis=0)
    vals = np.concatenate([vp[0, 0, :5], vn[0, 0, [0, 1]], r1[2][0, 0]], axis=0)
    outs = []
    for h in range(hq):
        s = keys @ q[h] / np.sqrt(D)
        p = np.exp(s - s.max())
        outs.append(p @ vals / p.sum())
    h1 = h0 + np.concatenate(outs) @ w["o"].T
    n2 = E.rmsnorm(h1, w["ln2"])
    fexp = h1 + (E.silu(n2 @ w["gate"].T) * (n2 @ w["up"].T)) @ w["down"].T
    np.testing.assert_allclose(r1[0][0, 0], fexp, rtol=1e-10, atol=1e-12)
