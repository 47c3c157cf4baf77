"""Pins for the oracle's acceptance rules, commit and the whole greedy step (no GPU)."""
import itertools
import math

import numpy as np
import pytest
from scipy import stats

from oracle import accept as ACC
from oracle import attention as A
from oracle import commit as C
from oracle import expected as E
from oracle import tree as T
from tree_speculative_decoding_attn_gb300 import synth


def _tree_arrays(parents, B=1):
    t = T.build_tree(parents, 0)
    rep = lambda x: np.broadcast_to(x, (B,) + x.shape).copy()
    return rep(t["parent"]), rep(t["first_child"]), rep(t["next_sibling"]), t


# ---------------------------------------------------------------- greedy


@pytest.mark.parametrize("target_path", [[0], [0, 1], [0, 1, 3], [0, 2], [0, 2, 4]])
def test_greedy_every_path_of_the_worked_tree(target_path):
    """Plant the argmax so that exactly ``target_path`` agrees; the bonus
    is the argmax at its last node."""
    par, fc, ns, _ = _tree_arrays(synth.P4_PARENTS)
    V = 20
    tok = np.array([[5, 6, 7, 8, 9]])
    logits = np.zeros((1, 5, V))
    for v in range(5):
        logits[0, v, 15 + v] = 1.0                  # default argmax: a token no child has
    for a, b in zip(target_path, target_path[1:]):
        logits[0, a, tok[0, b]] = 2.0
    acc_len, acc_path, bonus = ACC.accept_greedy(logits, tok, fc, ns, path_cap=3)
    assert acc_len[0] == len(target_path) - 1
    assert acc_path[0, : len(target_path)].tolist() == target_path
    assert (acc_path[0, len(target_path):] == -1).all()
    assert bonus[0] == 15 + target_path[-1]


def test_greedy_argmax_ties_go_to_lowest_id():
    par, fc, ns, _ = _tree_arrays([-1, 0, 0])
    logits = np.zeros((1, 3, 10))
    logits[0, 0, [3, 7]] = 4.0                      # tie between tokens 3 and 7
    tok = np.array([[0, 7, 3]])
    acc_len, acc_path, bonus = ACC.accept_greedy(logits, tok, fc, ns, 2)
    assert acc_path[0, :2].tolist() == [0, 2]       # the child holding token 3


def test_greedy_mean_length_under_planted_agreement_matches_the_tree_form():
    """Cartesian tree 3 x 2 x 2 with distinct sibling tokens, float32 target
    logits N(0, 2) and planted agreement: at a node on level l the
    generator raises one uniformly chosen child's token above the row max
    with probability r_l; otherwise the argmax is uniform over the V tokens.
    So the child of rank r is the argmax with probability r_l / n_l +
    (1 - r_l) / V, and the mean accepted length (root excluded) over many
    seeded sequences must match the tree form of the expected length minus
    the root, within a 99% interval."""
    branching, V, B = (3, 2, 2), 64, 10000
    parents, rank, depth, level = [-1], [0], [0], [0]
    for d, s in enumerate(branching, start=1):
        nxt = []
        for v in level:
            for r in range(s):
                parents.append(v); rank.append(r); depth.append(d); nxt.append(len(parents) - 1)
        level = nxt
    parents, rank, depth = np.array(parents), np.array(rank), np.array(depth)
    N = len(parents)
    cand = synth.candidate_tokens(11, B, len(branching) + 1, max(branching), V)
    tok = np.empty((B, N), np.int64)
    tok[:, 0] = 0
    for i in range(1, N):
        tok[:, i] = cand[:, depth[i] - 1, rank[i]]
    lg = synth.target_logits(12, B, N, V, 2.0, bf16=False)
    synth.plant_agreement(13, lg, parents, depth, tok, bf16=False)
    _, fc, ns, _ = _tree_arrays(parents, B)
    acc_len, _, _ = ACC.accept_greedy(lg, tok, fc, ns, path_cap=len(branching) + 1)
    rates = synth.PLANT_RATES
    p_rank = [[rates[d] / s + (1 - rates[d]) / V] * s for d, s in enumerate(branching)]
    want = E.expected_len_tree(parents, rank, depth, p_rank) - 1.0
    half = 2.576 * acc_len.std(ddof=1) / math.sqrt(B)
    assert abs(acc_len.mean() - want) <= half, (acc_len.mean(), want, half)
    # and the process is not degenerate: every length 0..3 occurs
    assert set(np.unique(acc_len).tolist()) == {0, 1, 2, 3}


def _tiny_model(seed, V=40, d=32, Hq=4, Hkv=2, Dh=8):
    g = np.random.default_rng(seed)
    return dict(E=g.standard_normal((V, d)), Wq=g.standard_normal((Hq * Dh, d)) / np.sqrt(d),
                Wk=g.standard_normal((Hkv * Dh, d)) / np.sqrt(d),
                Wv=g.standard_normal((Hkv * Dh, d)) / np.sqrt(d),
                Wo=g.standard_normal((d, Hq * Dh)) / np.sqrt(Hq * Dh),
                Wlm=g.standard_normal((V, d)) * 2.0, Hq=Hq, Hkv=Hkv, Dh=Dh, V=V)


def _rope(x, pos):
    """Rotary position embedding on the last axis (pairs (2i, 2i+1))."""
    Dh = x.shape[-1]
    inv = 1.0 / (10000 ** (np.arange(0, Dh, 2) / Dh))
    ang = np.asarray(pos, float)[..., None] * inv
    c, s = np.cos(ang), np.sin(ang)
    out = x.copy()
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
    return out


def _qkv(m, tokens, pos):
    """q [n,Hq,Dh], k/v [n,Hkv,Dh] with rotary positions ``pos``."""
    h = m["E"][tokens]
    q = (h @ m["Wq"].T).reshape(len(tokens), m["Hq"], m["Dh"])
    k = (h @ m["Wk"].T).reshape(len(tokens), m["Hkv"], m["Dh"])
    v = (h @ m["Wv"].T).reshape(len(tokens), m["Hkv"], m["Dh"])
    return _rope(q, pos[:, None]), _rope(k, pos[:, None]), v, h


def _logits(m, attn, h):
    return (h + attn.reshape(len(h), -1) @ m["Wo"].T) @ m["Wlm"].T


def _sequential_greedy(m, prompt, n_new):
    """Ordinary decoding, one token per pass, causal attention written
    directly (no tree code)."""
    toks = list(prompt)
    K, Vv = [], []
    out = []
    for t in range(len(prompt) + n_new - 1):
        q, k, v, h = _qkv(m, np.array([toks[t]]), np.array([t]))
        K.append(k[0]); Vv.append(v[0])
        Ks, Vs = np.stack(K), np.stack(Vv)              # [t+1, Hkv, Dh]
        G = m["Hq"] // m["Hkv"]
        att = np.zeros((m["Hq"], m["Dh"]))
        for hq in range(m["Hq"]):
            s = Ks[:, hq // G] @ q[0, hq] / np.sqrt(m["Dh"])
            e = np.exp(s - s.max())
            att[hq] = e @ Vs[:, hq // G] / e.sum()
        nxt = int(np.argmax(_logits(m, att[None], h)[0]))
        if t >= len(prompt) - 1:
            toks.append(nxt)
            out.append(nxt)
    return out


def test_tree_greedy_steps_reproduce_sequential_greedy_decoding():
    """Greedy tree verification emits exactly the ordinary greedy stream
    ("Medusa, explained", step 7; "Drafters: ...", section "Why the answer
    does not change").  Exercises depth positions (through rotary
    embeddings), the ancestor mask, tree attention, greedy acceptance, the
    bonus token and the KV commit together."""
    m = _tiny_model(3)
    prompt = [1, 5, 9, 2, 7]
    n_new = 30
    ref = _sequential_greedy(m, prompt, n_new)
    g = np.random.default_rng(11)
    shape = synth.random_tree(4, 12, (3, 2, 2))
    S = len(prompt) + n_new + 16
    kc = np.zeros((1, m["Hkv"], S, m["Dh"]))
    vc = np.zeros_like(kc)
    # prefill the prompt except its last token (the first root)
    _, k, v, _ = _qkv(m, np.array(prompt[:-1]), np.arange(len(prompt) - 1))
    kc[0, :, : len(prompt) - 1] = k.transpose(1, 0, 2)
    vc[0, :, : len(prompt) - 1] = v.transpose(1, 0, 2)
    prefix = np.array([len(prompt) - 1])
    root = prompt[-1]
    emitted, steps = [], 0
    while len(emitted) < n_new:
        steps += 1
        # drafter: random distinct sibling tokens, and with some probability
        # the true continuation along the rank-0 chain
        n = shape.n
        tok = np.zeros(n, np.int64)
        tok[0] = root
        truth = ref[len(emitted):] + [0] * 8
        for v_ in range(n):
            kids = [i for i in range(n) if shape.parents[i] == v_]
            choice = g.choice(m["V"], size=len(kids), replace=False)
            for c, x in zip(kids, choice):
                tok[c] = x
        chain = [0]
        while True:
            kids = [i for i in range(n) if shape.parents[i] == chain[-1]]
            if not kids or g.random() > 0.7:
                break
            c = kids[int(g.integers(len(kids)))]
            want = truth[len(chain) - 1]
            for s in kids:                              # keep siblings distinct
                if tok[s] == want:
                    tok[s] = tok[c]
            tok[c] = want
            chain.append(c)
        t = T.build_tree(shape.parents, int(prefix[0]))
        q, kt, vt, h = _qkv(m, tok, t["pos"])
        o = A.tree_attention(q[None], kc, vc, kt.transpose(1, 0, 2)[None], vt.transpose(1, 0, 2)[None],
                             prefix, t["mask"])
        logits = _logits(m, o[0], h)[None]
        acc_len, acc_path, bonus = ACC.accept_greedy(logits, tok[None], t["first_child"][None],
                                                     t["next_sibling"][None], path_cap=4)
        emitted += [int(tok[i]) for i in acc_path[0, 1: acc_len[0] + 1]] + [int(bonus[0])]
        kc, vc, prefix = C.kv_commit(kc, vc, kt.transpose(1, 0, 2)[None], vt.transpose(1, 0, 2)[None],
                                     prefix, acc_len, acc_path)
        root = int(bonus[0])
    assert emitted[:n_new] == ref
    assert steps < n_new                                  # some steps accepted drafts


# ---------------------------------------------------------------- typical


def test_typical_threshold_closed_form_on_uniform_rows():
    """Uniform target over V: H = ln V, p = 1/V, threshold
    min(eps, delta / V)."""
    V = 64
    p, thr = ACC.typical_threshold(np.zeros(V), eps=0.3, delta=0.5, T=1.0, dtype=np.float64)
    assert thr == pytest.approx(0.5 / V, rel=1e-12)
    np.testing.assert_allclose(p, 1.0 / V, rtol=1e-12)
    p, thr = ACC.typical_threshold(np.zeros(V), eps=0.001, delta=0.5, T=1.0, dtype=np.float64)
    assert thr == 0.001
    # a one-hot-like row has near-zero entropy: threshold -> min(eps, delta)
    row = np.full(V, -200.0); row[3] = 0.0
    p, thr = ACC.typical_threshold(row, eps=0.3, delta=0.09, T=1.0, dtype=np.float64)
    assert thr == pytest.approx(0.09, rel=1e-9)
    # entropy of a two-point distribution (1/2, 1/2): ln 2
    row = np.full(V, -1e4); row[[1, 2]] = 0.0
    p, thr = ACC.typical_threshold(row, eps=1.0, delta=1.0, T=1.0, dtype=np.float64)
    assert thr == pytest.approx(0.5, rel=1e-12)


def _rand_tree_logits(seed, n=24, V=50, B=3):
    shape = synth.random_tree(seed, n, (4, 3, 2))
    g = np.random.default_rng(seed)
    logits = g.standard_normal((B, n, V)) * 2.0
    tok = np.stack([np.concatenate([[0], g.integers(0, V, n - 1)]) for _ in range(B)])
    for b in range(B):                                    # distinct sibling tokens
        for v in range(n):
            kids = [i for i in range(n) if shape.parents[i] == v]
            tok[b, kids] = g.choice(V, size=len(kids), replace=False)
    par, fc, ns, t = _tree_arrays(shape.parents, B)
    return shape, logits, tok, par, fc, ns, t


def test_typical_eps_delta_zero_accepts_deepest_node():
    shape, logits, tok, par, fc, ns, t = _rand_tree_logits(1)
    acc_len, acc_path, bonus, near = ACC.accept_typical(logits, tok, par, fc, ns, 0.0, 0.0, 1.0, 4,
                                                        dtype=np.float64)
    deepest = t["depth"].max()
    first_deepest = int(np.nonzero(t["depth"] == deepest)[0][0])
    assert (acc_len == deepest).all()
    for b in range(3):
        assert acc_path[b, deepest] == first_deepest
        assert bonus[b] == np.argmax(logits[b, first_deepest])


def test_typical_high_threshold_is_a_prefix_of_the_greedy_path():
    for seed in range(5):
        shape, logits, tok, par, fc, ns, t = _rand_tree_logits(seed)
        # plant argmax agreement on a few branches so greedy paths are long
        g = np.random.default_rng(seed + 100)
        for b in range(3):
            for v in range(shape.n):
                kids = [i for i in range(shape.n) if shape.parents[i] == v]
                if kids and g.random() < 0.8:
                    logits[b, v, tok[b, kids[int(g.integers(len(kids)))]]] += 10.0
        gl, gp, gb = ACC.accept_greedy(logits, tok, fc, ns, 4)
        tl, tp, tb, _ = ACC.accept_typical(logits, tok, par, fc, ns, 0.5, 10.0, 1.0, 4, dtype=np.float64)
        for b in range(3):
            assert tl[b] <= gl[b]
            assert tp[b, : tl[b] + 1].tolist() == gp[b, : tl[b] + 1].tolist()
            last = tp[b, tl[b]]
            assert tb[b] == np.argmax(logits[b, last])      # first token is the greedy one


# ---------------------------------------------------------------- rejection


def _target_table(seed, V, depth):
    """A seeded 'target model': logits for every context of length <= depth."""
    g = np.random.default_rng(seed)
    table = {}
    for L in range(depth + 2):
        for ctx in itertools.product(range(V), repeat=L):
            table[ctx] = g.standard_normal(V) * 1.5
    return table


def _softmax64(x):
    e = np.exp(x - x.max())
    return e / e.sum()


@pytest.mark.parametrize("V,parents", [(3, [-1, 0, 0]), (4, [-1, 0, 0, 1, 2]), (5, [-1, 0, 0, 0, 1, 1, 4]),
                                       (3, [-1, 0, 1, 2]), (4, [-1, 0, 0, 0, 0])])
def test_rejection_preserves_the_target_distribution_exactly(V, parents):
    """Exact enumeration: (accepted tokens + bonus) extended by target
    sampling to a fixed length has exactly the target's autoregressive
    joint distribution ("Drafters: ...", section "Why the answer does not
    change")."""
    n = len(parents)
    _, fc, ns, t = _tree_arrays(parents)
    depth = t["depth"]
    Lmax = int(depth.max()) + 1
    table = _target_table(V + n, V, Lmax)
    g = np.random.default_rng(V * 10 + n)
    for trial in range(3):
        tok = np.zeros(n, np.int64)
        for v in range(n):
            kids = [i for i in range(n) if parents[i] == v]
            tok[kids] = g.choice(V, size=len(kids), replace=len(kids) > V)
        ctx_of = {}
        for i in range(n):                      # context of node i = tokens on its path after the root
            path = []
            u = i
            while u > 0:
                path.append(int(tok[u])); u = parents[u]
            ctx_of[i] = tuple(path[::-1])
        probs = {i: _softmax64(table[ctx_of[i]]) for i in range(n)}
        outcomes = ACC.reject_outcome_probs(probs, tok, fc[0], ns[0])
        assert sum(outcomes.values()) == pytest.approx(1.0, abs=1e-12)
        joint = {}
        for (path, bonus), pr in outcomes.items():
            seq = tuple(int(tok[i]) for i in path[1:]) + (bonus,)
            # extend with target sampling to length Lmax
            frontier = {seq: pr}
            while len(next(iter(frontier))) < Lmax:
                nf = {}
                for s, p in frontier.items():
                    q = _softmax64(table[s])
                    for x in range(V):
                        nf[s + (x,)] = nf.get(s + (x,), 0.0) + p * q[x]
                frontier = nf
            for s, p in frontier.items():
                joint[s] = joint.get(s, 0.0) + p
        for s in itertools.product(range(V), repeat=Lmax):
            ref = 1.0
            for j in range(Lmax):
                ref *= _softmax64(table[s[:j]])[s[j]]
            assert joint.get(s, 0.0) == pytest.approx(ref, abs=1e-12)


@pytest.mark.slow
def test_rejection_walk_frequencies_match_exact_enumeration():
    """The RNG-driven walk (float32 decisions, Philox draws) against the
    exact outcome distribution, chi-square over many steps."""
    parents = [-1, 0, 0, 1, 2]
    V = 4
    _, fc, ns, t = _tree_arrays(parents)
    tok = np.array([[2, 0, 1, 3, 0]])
    g = np.random.default_rng(5)
    logits = (g.standard_normal((1, 5, V)) * 1.2).astype(np.float32)
    probs = {i: _softmax64(logits[0, i].astype(np.float64)) for i in range(5)}
    exact = ACC.reject_outcome_probs(probs, tok[0], fc[0], ns[0])
    keys = sorted(exact)
    counts = dict.fromkeys(keys, 0)
    n_draws = 20000
    for step in range(n_draws):
        acc_len, acc_path, bonus, _ = ACC.accept_reject(logits, tok, fc, ns, seed=77, step=step, T=1.0, path_cap=3)
        key = (tuple(int(x) for x in acc_path[0, : acc_len[0] + 1]), int(bonus[0]))
        counts[key] += 1
    obs = np.array([counts[k] for k in keys], float)
    exp_ = np.array([exact[k] for k in keys]) * n_draws
    chi2 = ((obs - exp_) ** 2 / exp_).sum()
    assert stats.chi2.sf(chi2, len(keys) - 1) > 1e-3


@pytest.mark.parametrize("V", [2, 3])
def test_rejection_children_covering_the_vocabulary_always_accept_one(V):
    """Exact arithmetic: after every other token is removed, the last child
    holds the whole residual and is accepted with probability 1, so the walk
    never samples an empty residual; the first child's acceptance frequency
    is p(tok 0) (here checked against its exact value over many steps)."""
    parents = [-1] + [0] * V
    _, fc, ns, _ = _tree_arrays(parents)
    tok = np.array([[0] + list(range(V))])
    logits = np.array([[[0.3, -0.2, 0.9][:V]] * (V + 1)], np.float32)
    p = _softmax64(logits[0, 0].astype(np.float64))
    first = 0
    n = 4000
    for step in range(n):
        acc_len, acc_path, bonus, _ = ACC.accept_reject(logits, tok, fc, ns, seed=3, step=step, T=1.0, path_cap=2)
        assert acc_len[0] == 1 and 0 <= bonus[0] < V
        first += int(acc_path[0, 1] == 1)
    assert abs(first / n - p[0]) < 4 * np.sqrt(p[0] * (1 - p[0]) / n)


def _contexts(parents, tok):
    """Tokens on each node's path after the root."""
    ctx = {}
    for i in range(len(parents)):
        path, u = [], i
        while u > 0:
            path.append(int(tok[u])); u = parents[u]
        ctx[i] = tuple(path[::-1])
    return ctx


@pytest.mark.parametrize("V,parents", [(3, [-1, 0, 0]), (3, [-1, 0, 0, 1, 2]), (3, [-1, 0, 0, 0, 1, 1, 4]),
                                       (4, [-1, 0, 1, 2]), (3, [-1, 0, 0, 0, 0])])
def test_stochastic_sibling_rejection_preserves_the_target_distribution_exactly(V, parents):
    """Siblings drawn independently from the drafter's q at their parent's
    context, each tested against the residual the earlier rejections left:
    averaged over every draw and every accept/reject branch, (accepted
    tokens + bonus) extended by target sampling has exactly the target's
    joint distribution ("Drafters: ...", section "Why the answer does not
    change": min(1, p/q), then the target minus the drafter)."""
    n = len(parents)
    _, fc, ns, t = _tree_arrays(parents)
    Lmax = int(t["depth"].max()) + 1
    ptab = _target_table(10 * V + n, V, Lmax)
    qtab = _target_table(10 * V + n + 1, V, Lmax)        # the drafter: another seeded model
    joint = {}
    for toks in itertools.product(range(V), repeat=n - 1):
        tok = np.array((0,) + toks)
        ctx = _contexts(parents, tok)
        weight = 1.0
        for i in range(1, n):
            weight *= _softmax64(qtab[ctx[parents[i]]])[tok[i]]
        probs = {i: _softmax64(ptab[ctx[i]]) for i in range(n)}
        qprobs = {i: _softmax64(qtab[ctx[i]]) for i in range(n)}
        out = ACC.reject_stochastic_outcome_probs(probs, qprobs, tok, fc[0], ns[0])
        assert sum(out.values()) == pytest.approx(1.0, abs=1e-12)
        for (path, bonus), pr in out.items():
            frontier = {tuple(int(tok[i]) for i in path[1:]) + (bonus,): weight * pr}
            while len(next(iter(frontier))) < Lmax:
                nf = {}
                for sq, pq in frontier.items():
                    tp = _softmax64(ptab[sq])
                    for x in range(V):
                        nf[sq + (x,)] = nf.get(sq + (x,), 0.0) + pq * tp[x]
                frontier = nf
            for sq, pq in frontier.items():
                joint[sq] = joint.get(sq, 0.0) + pq
    for sq in itertools.product(range(V), repeat=Lmax):
        ref = 1.0
        for j in range(Lmax):
            ref *= _softmax64(ptab[sq[:j]])[sq[j]]
        assert joint.get(sq, 0.0) == pytest.approx(ref, abs=1e-12)


@pytest.mark.parametrize("length", [1, 2, 3])
def test_stochastic_rule_with_a_point_mass_drafter_is_the_deterministic_rule(length):
    """On a chain, a drafter certain of each drafted token (q = point mass)
    turns min(1, r/q) into r(x) and norm(max(0, r - q)) into r with x
    removed: the two rules give the same outcome distribution."""
    parents = list(range(-1, length))
    V = 4
    _, fc, ns, _t = _tree_arrays(parents)
    g = np.random.default_rng(length)
    for trial in range(5):
        tok = np.concatenate([[0], g.integers(0, V, length)])
        probs = {i: _softmax64(g.standard_normal(V) * 1.5) for i in range(length + 1)}
        qprobs = {}
        for i in range(length + 1):
            q = np.full(V, 0.25)
            if i < length:
                q = np.zeros(V); q[tok[i + 1]] = 1.0
            qprobs[i] = q
        a = ACC.reject_stochastic_outcome_probs(probs, qprobs, tok, fc[0], ns[0])
        b = ACC.reject_outcome_probs(probs, tok, fc[0], ns[0])
        for k in set(a) | set(b):
            assert a.get(k, 0.0) == pytest.approx(b.get(k, 0.0), abs=1e-12)


@pytest.mark.slow
def test_stochastic_rejection_walk_frequencies_match_exact_enumeration():
    """The RNG-driven walk (float32 decisions, Philox draws) against the
    exact outcome distribution for fixed drafted tokens, chi-square."""
    parents = [-1, 0, 0, 1, 2]
    V = 4
    _, fc, ns, t = _tree_arrays(parents)
    tok = np.array([[2, 0, 0, 3, 1]])                    # two siblings drew the same token
    g = np.random.default_rng(6)
    logits = (g.standard_normal((1, 5, V)) * 1.2).astype(np.float32)
    draft = (g.standard_normal((1, 5, V)) * 1.2).astype(np.float32)
    probs = {i: _softmax64(logits[0, i].astype(np.float64)) for i in range(5)}
    qprobs = {i: _softmax64(draft[0, i].astype(np.float64)) for i in range(5)}
    exact = ACC.reject_stochastic_outcome_probs(probs, qprobs, tok[0], fc[0], ns[0])
    keys = sorted(k for k, v in exact.items() if v > 0)
    counts = dict.fromkeys(keys, 0)
    n_draws = 20000
    for step in range(n_draws):
        acc_len, acc_path, bonus, _ = ACC.accept_reject_stochastic(logits, draft, tok, fc, ns, seed=78, step=step,
                                                                   T=1.0, path_cap=3)
        key = (tuple(int(x) for x in acc_path[0, : acc_len[0] + 1]), int(bonus[0]))
        counts[key] += 1
    obs = np.array([counts[k] for k in keys], float)
    exp_ = np.array([exact[k] for k in keys]) * n_draws
    assert obs.sum() == n_draws
    chi2 = ((obs - exp_) ** 2 / exp_).sum()
    assert stats.chi2.sf(chi2, len(keys) - 1) > 1e-3


def test_rejection_with_certain_target_accepts_and_leaf_bonus_is_target_sample():
    parents = [-1, 0, 1]
    _, fc, ns, t = _tree_arrays(parents)
    V = 6
    logits = np.full((1, 3, V), -1e9, np.float32)
    tok = np.array([[0, 2, 4]])
    logits[0, 0, 2] = 0.0       # target is certain of token 2 after the root
    logits[0, 1, 4] = 0.0       # and of token 4 after that
    logits[0, 2, 5] = 0.0       # and of 5 at the leaf
    acc_len, acc_path, bonus, near = ACC.accept_reject(logits, tok, fc, ns, seed=3, step=0, T=1.0, path_cap=3)
    assert acc_len[0] == 2 and acc_path[0].tolist() == [0, 1, 2] and bonus[0] == 5
    logits[0, 0, 2] = -1e9
    logits[0, 0, 1] = 0.0       # now the draft is certainly wrong
    acc_len, acc_path, bonus, near = ACC.accept_reject(logits, tok, fc, ns, seed=3, step=0, T=1.0, path_cap=3)
    assert acc_len[0] == 0 and bonus[0] == 1


# ---------------------------------------------------------------- commit


def test_commit_copies_path_rows_and_leaves_everything_else():
    g = np.random.default_rng(9)
    L, B, Hkv, S, N, D = 2, 3, 2, 20, 5, 4
    kc = g.standard_normal((L, B, Hkv, S, D)); vc = g.standard_normal((L, B, Hkv, S, D))
    kt = g.standard_normal((L, B, Hkv, N, D)); vt = g.standard_normal((L, B, Hkv, N, D))
    prefix = np.array([3, 10, 0])
    acc_len = np.array([2, 0, 1])
    acc_path = np.array([[0, 2, 4], [0, -1, -1], [0, 1, -1]])
    k2, v2, new = C.kv_commit(kc, vc, kt, vt, prefix, acc_len, acc_path)
    assert new.tolist() == [6, 11, 2]
    for b in range(B):
        rows = list(range(prefix[b], prefix[b] + acc_len[b] + 1))
        for j, r in enumerate(rows):
            np.testing.assert_array_equal(k2[:, b, :, r], kt[:, b, :, acc_path[b, j]])
            np.testing.assert_array_equal(v2[:, b, :, r], vt[:, b, :, acc_path[b, j]])
        other = [r for r in range(S) if r not in rows]
        np.testing.assert_array_equal(k2[:, b, :, other], kc[:, b, :, other])
        np.testing.assert_array_equal(v2[:, b, :, other], vc[:, b, :, other])
