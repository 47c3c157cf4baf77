"""Pins for the expected-length closed forms, the generator and the expansion round (no GPU)."""
import itertools
import os

import numpy as np
import pytest
from scipy import stats

from oracle import expand as X
from oracle import expected as E
from oracle import rng as R
from oracle import tree as T

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lengths():
    rows = []
    for line in open(os.path.join(GOLDEN, "expected_length_worked.txt"), encoding="utf-8"):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        eq = f.index("=")
        rows.append((f[0], f[1:eq], float(f[eq + 1]), int(f[eq + 3])))
    return rows


def test_worked_expected_lengths():
    rows = _golden_lengths()
    assert len(rows) == 3
    for kind, terms, value, nodes in rows:
        if kind == "chain":
            hit = [float(x) for x in terms]
            got = E.expected_len_chain(hit)
            assert len(hit) == nodes
        else:
            s = [int(x.split(":")[0]) for x in terms]
            hit = [float(x.split(":")[1]) for x in terms]
            got = E.expected_len_chain(hit)
            assert sum(np.prod(s[: k + 1]) for k in range(len(s))) == nodes   # 3 + 3*2 + 3*2*1
        # the pages print the value rounded (2 decimals, or "~2.7")
        assert abs(got - value) <= (0.05 if value == 2.7 else 0.005)
    assert E.expected_len_chain([0.6, 0.4, 0.3]) == pytest.approx(1.912)
    assert E.expected_len_chain([0.8, 0.55, 0.3]) == pytest.approx(2.372)
    assert E.expected_len_chain([0.8, 0.65, 0.5, 0.35]) == pytest.approx(2.671)
    assert E.expected_len_chain([1, 1, 1, 1]) == 5                           # perfect heads: K + 1


def test_tree_form_equals_chain_form_on_cartesian_tree():
    """Cartesian tree 3 x 2 x 1 with per-rank probabilities summing to the
    worked example's 0.8 / 0.55 / 0.3."""
    p_rank = [[0.5, 0.2, 0.1], [0.4, 0.15], [0.3]]
    parents, rank, depth = [-1], [0], [0]
    level = [0]
    for d, s in enumerate([3, 2, 1], start=1):
        nxt = []
        for v in level:
            for r in range(s):
                parents.append(v); rank.append(r); depth.append(d); nxt.append(len(parents) - 1)
        level = nxt
    assert len(parents) == 1 + 15
    got = E.expected_len_tree(parents, rank, depth, p_rank)
    assert got == pytest.approx(E.expected_len_chain([0.8, 0.55, 0.3]), rel=1e-12)


def test_hit_with_candidates_by_enumeration():
    for a, s in [(0.3, 1), (0.3, 3), (0.65, 2), (0.1, 10)]:
        brute = sum(np.prod([a if h else 1 - a for h in hits])
                    for hits in itertools.product([0, 1], repeat=s) if any(hits))
        assert E.hit_with_candidates(a, s) == pytest.approx(brute, rel=1e-12)


def _kat():
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt"), encoding="utf-8"):
        f = line.split()
        if f and not f[0].startswith("#"):
            v = [int(x, 16) for x in f]
            yield v[:4], v[4:6], v[6:]


def test_philox_known_answers():
    for ctr, key, out in _kat():
        got = R.philox4x32_10(ctr, key)
        assert [int(x) for x in got] == out


def test_uniforms_range_and_uniformity():
    u = R.uniform_accept(123, 0, 0, np.arange(200000))
    assert u.min() >= 0.0 and u.max() < 1.0
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    w = R.uniform_race(123, 1, 2, 3, np.arange(200000))
    assert w.min() > 0.0 and w.max() < 1.0
    assert not np.array_equal(u[:100], R.uniform_accept(123, 0, 1, np.arange(100)))   # step matters


def test_expand_round_hand_worked_example():
    """A round computed by hand ("5.3 Medusa、EAGLE 与 MTP", section 5.2:
    value = product of confidences along the path; the best-valued nodes
    are expanded next).  Rows with equal maxima and entries of -200
    (exp(-200) is negligible against 1) give exact probabilities 1/2 and
    1/4, so every value below is exact:
      frontier node 1 (value 1/2): probabilities (1/2, 1/2, 0, 0, 0) ->
        children tokens 0, 1 (equal -> lower id first), value 1/4 each;
      frontier node 2 (value 1/4): probabilities (0, 1/4, 1/4, 1/4, 1/4) ->
        children tokens 1, 2, value 1/16 each.
    Children go to pool slots 3, 4 (node 1) and 5, 6 (node 2); the next
    frontier of three is 3, 4, 5 (equal values -> lower pool index)."""
    logits = np.array([[[0, 0, -200, -200, -200], [-200, 0, 0, 0, 0]]], np.float64)
    par = np.array([[-1, 0, 0, -1, -1, -1, -1]]); tok = np.array([[7, 3, 4, 0, 0, 0, 0]])
    conf = np.array([[1.0, 0.5, 0.25, 0, 0, 0, 0]]); val = conf.copy()
    p2, t2, c2, v2, cnt, nxt, near = X.expand_round(logits, np.array([[1, 2]]), par, tok, conf, val,
                                                     np.array([3]), 2, 1.0, 3)
    assert cnt.tolist() == [7]
    assert p2[0].tolist() == [-1, 0, 0, 1, 1, 2, 2]
    assert t2[0].tolist() == [7, 3, 4, 0, 1, 1, 2]
    assert c2[0, 3:].tolist() == [0.5, 0.5, 0.25, 0.25]
    assert v2[0, 3:].tolist() == [0.25, 0.25, 0.0625, 0.0625]
    assert nxt[0].tolist() == [3, 4, 5]
    assert (0, 2) in near and (0, 0) in near          # the exact ties are flagged
    # temperature 2 halves the logits: probabilities unchanged for rows of 0 / -200 (to rounding)
    _, _, c3, _, _, nxt3, _ = X.expand_round(logits, np.array([[1, 2]]), par, tok, conf, val, np.array([3]), 2,
                                             2.0, 3)
    np.testing.assert_allclose(c3[0, 3:], [0.5, 0.5, 0.25, 0.25], rtol=1e-12)
    assert nxt3[0].tolist() == [3, 4, 5]


def test_expand_round_brute_force():
    g = np.random.default_rng(0)
    B, F, V, k, M = 2, 3, 30, 4, 1 + 3 + 12
    logits = np.round(g.standard_normal((B, F, V)) * 3, 1).astype(np.float32)
    par = np.full((B, M), -1); tok = np.zeros((B, M), np.int64)
    conf = np.zeros((B, M), np.float32); val = np.zeros((B, M), np.float32)
    for b in range(B):                              # root with three children already in the pool
        val[b, 0] = 1.0
        for j in range(1, 4):
            par[b, j] = 0; tok[b, j] = j; conf[b, j] = val[b, j] = 0.25 * j
    front = np.array([[1, 2, 3], [3, 1, 2]])
    p2, t2, c2, v2, cnt, nxt, near = X.expand_round(logits, front, par, tok, conf, val, np.array([4, 4]), k, 1.0, 5)
    assert cnt.tolist() == [16, 16]
    for b in range(B):
        for f in range(F):
            z = logits[b, f].astype(np.float64)
            prob = np.exp(z - z.max()) / np.exp(z - z.max()).sum()
            order = sorted(range(V), key=lambda x: (-z[x], x))[:k]
            for j in range(k):
                m = 4 + f * k + j
                assert p2[b, m] == front[b, f] and t2[b, m] == order[j]
                assert c2[b, m] == pytest.approx(prob[order[j]], rel=1e-5)
                assert v2[b, m] == pytest.approx(float(val[b, front[b, f]]) * prob[order[j]], rel=1e-12)
        new = list(range(4, 16))
        best = sorted(new, key=lambda m: (-float(v2[b, m]), m))[:5]
        assert nxt[b].tolist() == best
    # the expanded pool reranks into a valid tree
    t = T.rerank_dynamic(p2[0], t2[0], c2[0], 8, 0)
    assert all(0 <= t["parent"][i] < i for i in range(1, 8))
