"""Pins for the oracle's tree bookkeeping (no GPU)."""
import itertools
import os

import networkx as nx
import numpy as np
import pytest

from oracle import tree as T
from tree_speculative_decoding_attn_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_p4():
    out = {"mask_row": {}, "depth": {}, "leak": {}}
    for line in open(os.path.join(GOLDEN, "p4_worked_example.txt"), encoding="utf-8"):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "parents":
            out["parents"] = [int(x) for x in f[1:]]
        elif f[0] == "mask_row":
            out["mask_row"][int(f[1])] = [int(x) for x in f[2:]]
        elif f[0] == "depth":
            out["depth"][int(f[1])] = int(f[2])
        elif f[0] == "causal_leak":
            out["leak"][int(f[1])] = [int(x) for x in f[2:]]
    return out


def test_worked_example_values():
    g = _golden_p4()
    depth, mask = T.depth_and_mask(g["parents"])
    for i, row in g["mask_row"].items():
        assert mask[i].astype(int).tolist() == row
    for i, d in g["depth"].items():
        assert depth[i] == d
    n = len(g["parents"])
    for i, leak in g["leak"].items():
        causal = [j for j in range(n) if j <= i]
        assert [j for j in causal if not mask[i, j]] == leak


def test_worked_example_siblings_invisible_and_positions():
    depth, mask = T.depth_and_mask(synth.P4_PARENTS)
    assert not mask[1, 2] and not mask[2, 1]            # siblings never see each other
    assert not mask[3, 2] and not mask[4, 1] and not mask[4, 3]
    t = T.build_tree(synth.P4_PARENTS, prefix_len=128)
    assert t["pos"][1] == t["pos"][2] == 129             # siblings share a position id
    assert t["pos"].tolist() == [128, 129, 129, 130, 130]


@pytest.mark.parametrize("seed,n,caps", [(1, 64, (10, 10, 10, 10)), (2, 32, (4, 3, 2)),
                                         (3, 64, (8, 4, 3, 2, 2)), (4, 7, (2, 2)), (5, 256, (8, 8, 4, 2))])
def test_mask_is_ancestor_relation(seed, n, caps):
    """Ancestor-or-self sets against networkx's graph ancestors; up to 64
    nodes also the one-word-per-node packing (256 nodes: the pages' dense
    tree size, beyond one word)."""
    shape = synth.random_tree(seed, n, caps)
    depth, mask = T.depth_and_mask(shape.parents)
    g = nx.DiGraph()
    g.add_nodes_from(range(n))
    g.add_edges_from((int(p), i) for i, p in enumerate(shape.parents) if p >= 0)
    for i in range(n):
        assert set(np.nonzero(mask[i])[0]) == nx.ancestors(g, i) | {i}
        assert mask[i].sum() == depth[i] + 1                        # popcount = depth + 1
        assert depth[i] == nx.shortest_path_length(g, 0, i)
        if i:
            p = shape.parents[i]
            assert set(np.nonzero(mask[i])[0]) == set(np.nonzero(mask[p])[0]) | {i}
    if n > 64:
        return
    words = T.mask_words(mask)
    for i in range(n):
        for j in range(n):
            assert bool((int(words[i]) >> j) & 1) == mask[i, j]


def test_chain_mask_is_lower_triangular():
    depth, mask = T.depth_and_mask(synth.chain(9).parents)
    assert (mask == np.tril(np.ones((9, 9), bool))).all()
    assert depth.tolist() == list(range(9))


@pytest.mark.parametrize("bad", [[0, 0], [-1, 1], [-1, 0, 2], [-1, -1], []])
def test_bad_parents_rejected(bad):
    with pytest.raises(ValueError):
        T.depth_and_mask(bad)


def test_child_links_enumerate_children_in_order():
    shape = synth.random_tree(5, 40, (6, 4, 3))
    first, nxt = T.child_links(shape.parents)
    for v in range(40):
        kids, c = [], first[v]
        while c != -1:
            kids.append(int(c))
            c = nxt[c]
        assert kids == [i for i in range(40) if shape.parents[i] == v]


def test_static_tokens_follow_head_rank():
    shape = synth.random_tree(7, 20, (5, 4, 3))
    cand = synth.candidate_tokens(7, 3, shape.n_levels, 5, 1000)
    root = np.array([11, 22, 33])
    t = T.build_tree_static(shape.parents, shape.rank, cand, root, np.array([10, 20, 30]))
    for b in range(3):
        assert t["tok"][b, 0] == root[b]
        for i in range(1, 20):
            d = int(t["depth"][b, i])
            assert d == shape.level[i]
            assert t["tok"][b, i] == cand[b, d - 1, shape.rank[i]]
        # siblings carry distinct tokens (distinct ranks of one head's top-s)
        for v in range(20):
            kids = [i for i in range(20) if shape.parents[i] == v]
            assert len(set(t["tok"][b, kids].tolist())) == len(kids)
    assert (t["pos"][1] == 20 + t["depth"][1]).all()


def test_path_value_products_exact_on_powers_of_two():
    par = np.array([-1, 0, 0, 1, 3, 2])
    conf = np.array([1.0, 0.5, 0.25, 0.125, 0.5, 0.0625], np.float32)
    val = T.path_values_f32(par, conf)
    assert val.tolist() == [1.0, 0.5, 0.25, 0.0625, 0.03125, 0.015625]


def _prefix_closed_subsets(par, n):
    m = len(par)
    for comb in itertools.combinations(range(1, m), n - 1):
        s = set(comb) | {0}
        if all(int(par[i]) in s for i in comb):
            yield s


@pytest.mark.parametrize("seed", range(6))
def test_rerank_is_best_prefix_closed_set(seed):
    """Brute force over every parent-closed node set of the budget: the kept
    set has the lexicographically largest sorted value vector (hence the
    largest value sum)."""
    g = np.random.default_rng(seed)
    m = 11
    par = np.array([-1] + [int(g.integers(0, i)) for i in range(1, m)])
    conf = g.uniform(0.05, 0.95, m).astype(np.float32)
    conf[0] = 1
    n = 6
    val = T.path_values_f32(par, conf)
    t = T.rerank_dynamic(par, np.arange(m) + 100, conf, n, prefix_len=7)
    kept = set(t["pool_index"].tolist())
    best = max(_prefix_closed_subsets(par, n), key=lambda s: sorted((float(val[i]) for i in s), reverse=True))
    assert kept == best
    sums = [sum(float(val[i]) for i in s) for s in _prefix_closed_subsets(par, n)]
    assert sum(float(val[i]) for i in kept) == pytest.approx(max(sums))
    # breadth-first re-emission: parents before children, depth non-decreasing
    assert t["parent"][0] == -1 and all(0 <= t["parent"][i] < i for i in range(1, n))
    assert np.all(np.diff(t["depth"]) >= 0)
    for i in range(1, n):
        assert t["pool_index"][t["parent"][i]] == par[t["pool_index"][i]]
        assert t["tok"][i] == t["pool_index"][i] + 100
    assert t["pos"].tolist() == (7 + t["depth"]).tolist()


def test_rerank_rejects_confidence_above_one():
    par = np.array([-1, 0, 1])
    conf = np.array([1.0, 0.1, 5.0], np.float32)   # child worth more than its parent
    with pytest.raises(ValueError):
        T.rerank_dynamic(par, np.arange(3), conf, 2, 0)
