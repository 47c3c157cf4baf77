"""Pins for the oracle's Medusa heads, LM head and top-s (no GPU)."""
import numpy as np
import pytest
import torch

from oracle import heads as H


def test_zero_w1_heads_reproduce_lm_head():
    """With W1 = 0 (and bias 0) and W2 = a copy of the LM head, every head
    predicts exactly the LM head's next token ("Medusa, explained", step 1;
    "Medusa and EAGLE ... explained", section "Medusa: heads, losses and
    trees")."""
    g = np.random.default_rng(0)
    B, K, d, V = 3, 4, 32, 200
    h = g.standard_normal((B, d))
    wlm = g.standard_normal((V, d)) * 0.1
    w1 = np.zeros((K, d, d))
    z, logits = H.medusa_heads(h, w1, np.zeros((K, d)), np.broadcast_to(wlm, (K, V, d)))
    lm = H.lm_head(h, wlm)
    for k in range(K):
        np.testing.assert_array_equal(z[:, k], h)
        np.testing.assert_allclose(logits[:, k], lm, rtol=1e-13, atol=1e-13)
        assert (H.topk(logits[:, k], 10)[0] == H.topk(lm, 10)[0]).all()


def test_silu_residual_and_weight_orientation():
    """A one-entry W1 (row 0, column 1) and an identity W2 give
    z = h + SiLU(W1 h) in closed form: SiLU(ln 3) = (3/4) ln 3 because the
    logistic function at ln 3 is 3/4.  A transposed W1/W2 or a dropped
    residual breaks it."""
    d = 4
    h = np.array([[0.5, 2.0, -1.0, 0.25]])
    w1 = np.zeros((1, d, d))
    w1[0, 0, 1] = np.log(3.0) / 2.0            # (W1 h)_0 = ln 3, all other outputs 0
    b1 = np.array([[0.0, 0.0, 0.0, np.log(3.0)]])  # bias reaches output 3 only
    w2 = np.zeros((1, 6, d))
    w2[0, :d, :d] = np.eye(d)
    w2[0, 5, 2] = 1.0                           # logit 5 reads z_2
    z, logits = H.medusa_heads(h, w1, b1, w2)
    s = 0.75 * np.log(3.0)
    expect = h[0] + np.array([s, 0.0, 0.0, s])
    np.testing.assert_allclose(z[0, 0], expect, rtol=1e-15)
    np.testing.assert_allclose(logits[0, 0], list(expect) + [0.0, expect[2]], rtol=1e-15)
    np.testing.assert_allclose(H.silu(np.array([0.0, -np.log(3.0)])), [0.0, -0.25 * np.log(3.0)])


def test_lm_head_orientation():
    hid = np.arange(12, dtype=float).reshape(3, 4)
    w = np.zeros((5, 4))
    w[2, 3] = 1.0
    w[4, 0] = -2.0
    out = H.lm_head(hid, w)
    assert out.shape == (3, 5)
    np.testing.assert_array_equal(out[:, 2], hid[:, 3])
    np.testing.assert_array_equal(out[:, 4], -2 * hid[:, 0])


def test_medusa_heads_match_torch_modules_float64():
    """The head as two torch.nn.Linear layers (library matmuls)."""
    g = np.random.default_rng(1)
    B, K, d, V = 2, 3, 24, 50
    h = g.standard_normal((B, d))
    w1 = g.standard_normal((K, d, d)) * 0.2
    b1 = g.standard_normal((K, d)) * 0.1
    w2 = g.standard_normal((K, V, d)) * 0.2
    z, logits = H.medusa_heads(h, w1, b1, w2)
    th = torch.from_numpy(h)
    for k in range(K):
        l1 = torch.nn.Linear(d, d).double()
        l2 = torch.nn.Linear(d, V, bias=False).double()
        with torch.no_grad():
            l1.weight.copy_(torch.from_numpy(w1[k])); l1.bias.copy_(torch.from_numpy(b1[k]))
            l2.weight.copy_(torch.from_numpy(w2[k]))
            ref = l2(torch.nn.functional.silu(l1(th)) + th).numpy()
        np.testing.assert_allclose(logits[:, k], ref, rtol=1e-12, atol=1e-12)


def test_topk_order_and_ties():
    row = np.array([1.0, 3.0, 3.0, -1.0, 3.0, 2.0, 2.0])
    idx, val = H.topk(row[None], 5)
    assert idx[0].tolist() == [1, 2, 4, 5, 6]
    assert val[0].tolist() == [3.0, 3.0, 3.0, 2.0, 2.0]


@pytest.mark.parametrize("V", [7, 1000, 32000])
def test_topk_matches_brute_force_sort(V):
    g = np.random.default_rng(V)
    rows = np.round(g.standard_normal((3, V)) * 4) / 4   # many exact ties
    idx, _ = H.topk(rows, 10 if V > 10 else 3)
    for r in range(3):
        brute = sorted(range(V), key=lambda x: (-rows[r, x], x))[: idx.shape[1]]
        assert idx[r].tolist() == brute
    distinct = g.permutation(V).astype(float)[None]
    assert H.topk(distinct, 3)[0][0].tolist() == torch.topk(torch.from_numpy(distinct[0]), 3).indices.tolist()
