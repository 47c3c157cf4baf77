"""Acceptance of the longest target-agreeing path (oracle; test infrastructure only).

Rules, as the pages state them:

* Greedy -- "Drafters: ..." (robertz.co), section "Why the answer does not
  change": a drafted token is kept only if it is the target's own pick; at
  the first disagreement the target's choice is used.  "Medusa, explained",
  step 7: a node is valid when its token equals the target's argmax at its
  parent; the longest valid path is accepted.
* Typical -- "Medusa and EAGLE ... explained", section "Medusa: heads,
  losses and trees" and "Medusa, explained", section "Typical acceptance":
  keep x when p(x) > min(eps, delta * exp(-H(p))), H the entropy of the
  target's distribution; the step's first token is always the target's
  greedy choice.
* Rejection -- "Drafters: ...", section "Why the answer does not change":
  keep a drafted token with probability min(1, p/q); on rejection draw from
  the target's distribution with the drafter's probabilities subtracted.
  "5.3 Medusa、EAGLE 与 MTP", section 9.2: token-level verification from
  left to right, stopping at the first rejection.

Readings where the pages leave a step open (each is listed in the design
notes):

* Tree siblings are deterministic top-ranked drafts, so the proposal q of
  a sibling is a point mass on its token: min(1, p/q) = r(x), and "target
  minus drafter" renormalised is r with x removed.  Siblings are tried in
  node order; the next sibling is tested against that residual.
* Argmax ties go to the lowest token id.  Typical: natural-log entropy;
  among several valid branches the deepest valid node wins, ties to the
  lowest node index; the bonus is the greedy token at the stop node.
* Decisions that compare floats (typical threshold, accept draw, sampling
  race) are taken in ``dtype``, float64 by default.  Every decision whose
  margin is below ``NEAR`` (relative) is reported by name in ``near``: a
  kernel that takes it in float32 may take it the other way and still follow
  the rule within rounding.  ``flip`` names decisions to take the other way,
  so a test can check that a divergence sits exactly at a flagged decision.
  Decision names: ("valid", c) typical validity of child c; ("accept", c)
  the accept draw of child c; ("race", v) the sampling race at stop node v
  (flipped: the runner-up wins).
* Sampling from the residual uses the exponential race in its log form:
  argmax over non-removed x of z_x + G_x, z = logits / T and
  G_x = -log(-log u'_x) with u'_x from the counter-based generator.
"""
from __future__ import annotations

import numpy as np

from . import rng

NEAR_REJECT = 1e-5
NEAR_TYPICAL = 1e-4


def _children(first_child, next_sibling, v):
    out = []
    c = int(first_child[v])
    while c != -1:
        out.append(c)
        c = int(next_sibling[c])
    return out


def _pack(paths, bonus, path_cap):
    B = len(paths)
    acc_len = np.array([len(p) - 1 for p in paths], np.int64)
    acc_path = np.full((B, path_cap), -1, np.int64)
    for b, p in enumerate(paths):
        acc_path[b, : len(p)] = p
    return acc_len, acc_path, np.asarray(bonus, np.int64)


def accept_greedy(logits, tok, first_child, next_sibling, path_cap):
    """Walk from the root; descend into the first child (node order) whose
    token is the argmax of the current node's logits; stop when none is.
    Bonus = that argmax at the stop node."""
    B = logits.shape[0]
    paths, bonus = [], []
    for b in range(B):
        v, path = 0, [0]
        while True:
            a = int(np.argmax(np.asarray(logits[b, v], np.float64)))  # first max = lowest id
            nxt = [c for c in _children(first_child[b], next_sibling[b], v) if int(tok[b, c]) == a]
            if not nxt:
                bonus.append(a)
                break
            v = nxt[0]
            path.append(v)
        paths.append(path)
    return _pack(paths, bonus, path_cap)


def typical_threshold(row, eps, delta, T, dtype=np.float64):
    """(p, thr) for one logits row: p = softmax(row / T) and
    thr = min(eps, delta * exp(-H)) with the entropy H = -sum_x p(x) ln p(x)
    (natural log; a zero probability contributes nothing)."""
    z = np.asarray(row, dtype) / dtype(T)
    e = np.exp(z - z.max())
    p = e / e.sum(dtype=dtype)
    nz = p > 0
    H = -np.sum(p[nz] * np.log(p[nz]), dtype=dtype)
    thr = min(dtype(eps), dtype(delta) * np.exp(-H))
    return p, thr


def _race(z_or_logr, g, excluded_mask, flipped):
    """Winner of the exponential race (lowest id among equal keys), the
    runner-up when ``flipped``; also the top-two gap."""
    key = z_or_logr + g
    key[excluded_mask] = -np.inf
    x = int(np.argmax(key))
    k1 = key[x]
    key2 = key.copy()
    key2[x] = -np.inf
    y = int(np.argmax(key2))
    gap = float(k1 - key2[y])
    near = gap <= NEAR_REJECT * max(1.0, abs(float(k1)))
    return (y if flipped else x), near


def accept_typical(logits, tok, parents, first_child, next_sibling, eps, delta, T, path_cap,
                   dtype=np.float64, flip=()):
    """Node c (non-root) is valid iff p_parent(tok_c) > thr_parent; the
    accepted path is the root path of the deepest node whose whole path is
    valid (ties: lowest node index); bonus = argmax at that node.
    Returns (acc_len, acc_path, bonus, near) with near[b] the list of
    near-tie decisions of sequence b; ``flip`` holds (b, decision) pairs to
    take the other way."""
    B, N, _ = logits.shape
    paths, bonus, near = [], [], [[] for _ in range(B)]
    for b in range(B):
        ok = np.zeros(N, bool)
        ok[0] = True
        depth = np.zeros(N, np.int64)
        for v in range(N):  # parents precede children
            kids = _children(first_child[b], next_sibling[b], v)
            if not kids or not ok[v]:
                for c in kids:
                    depth[c] = depth[v] + 1
                continue
            p, thr = typical_threshold(logits[b, v], eps, delta, T, dtype)
            for c in kids:
                depth[c] = depth[v] + 1
                pc = p[int(tok[b, c])]
                d = ("valid", c)
                if abs(float(pc) - float(thr)) <= NEAR_TYPICAL * float(thr):
                    near[b].append(d)
                ok[c] = bool(pc > thr) != ((b, d) in flip)
        reach = [i for i in range(N) if ok[i]]
        best = max(reach, key=lambda i: (depth[i], -i))
        path = []
        u = best
        while u != -1:
            path.append(u)
            u = int(parents[b, u]) if u else -1
        path.reverse()
        paths.append(path)
        bonus.append(int(np.argmax(np.asarray(logits[b, best], np.float64))))
    acc_len, acc_path, bon = _pack(paths, bonus, path_cap)
    return acc_len, acc_path, bon, near


def accept_reject(logits, tok, first_child, next_sibling, seed, step, T, path_cap,
                  dtype=np.float64, flip=()):
    """Rejection walk with point-mass sibling proposals and residual
    resampling.  Returns (acc_len, acc_path, bonus, near) with near[b] the
    list of near-tie decisions of sequence b; ``flip`` holds (b, decision)
    pairs to take the other way."""
    B, N, V = logits.shape
    paths, bonus, near = [], [], [[] for _ in range(B)]
    for b in range(B):
        v, path = 0, [0]
        while True:
            z = np.asarray(logits[b, v], dtype) / dtype(T)
            e = np.exp(z - z.max())
            S = e.sum(dtype=dtype)
            removed = dtype(0)
            excluded = []
            chosen = -1
            for c in _children(first_child[b], next_sibling[b], v):
                x = int(tok[b, c])
                # the residual's mass is at least x's own; the last token left
                # in the vocabulary holds all of it (r = 1)
                if x in excluded:
                    r = dtype(0)
                elif len(excluded) + 1 == V:
                    r = dtype(1)
                else:
                    r = e[x] / max(S - removed, e[x])
                u = rng.uniform_accept(seed, b, step, c)
                d = ("accept", c)
                if abs(float(u) - float(r)) <= NEAR_REJECT * max(float(r), 1e-30):
                    near[b].append(d)
                if bool(u < r) != ((b, d) in flip):
                    chosen = c
                    break
                if x not in excluded:
                    excluded.append(x)
                    removed = dtype(removed + e[x])
            if chosen == -1:
                u = rng.uniform_race(seed, b, step, v, np.arange(V))
                g = -np.log(-np.log(u.astype(dtype)))
                mask = np.zeros(V, bool)
                mask[excluded] = True
                d = ("race", v)
                x, is_near = _race(z, g, mask, (b, d) in flip)
                if is_near:
                    near[b].append(d)
                bonus.append(x)
                break
            v = chosen
            path.append(v)
        paths.append(path)
    acc_len, acc_path, bon = _pack(paths, bonus, path_cap)
    return acc_len, acc_path, bon, near


def reject_outcome_probs(probs, tok, first_child, next_sibling):
    """Exact distribution of (accepted path, bonus token) under the
    rejection walk for one sequence, by recursion over every accept/reject
    branch (no random numbers).  ``probs[v]`` is the target distribution at
    node v (float64 vector).  Returns {(path tuple, bonus): probability}."""
    out = {}

    def visit(v, path, mass):
        r = np.array(probs[v], np.float64)
        r = r / r.sum()
        for c in _children(first_child, next_sibling, v):
            x = int(tok[c])
            a = r[x]
            if a > 0:
                visit(c, path + (c,), mass * a)
            rest = 1.0 - a
            if rest <= 0:
                return
            mass *= rest
            r[x] = 0.0
            r /= r.sum()
        for x in np.nonzero(r)[0]:
            key = (path, int(x))
            out[key] = out.get(key, 0.0) + mass * r[x]

    visit(0, (0,), 1.0)
    return out


# ------------------------------------------------------------------------
# Rejection with stochastic siblings (the children of a node drawn
# independently from the drafter's distribution q at that node).
#
# "Drafters: ...", section "Why the answer does not change": keep a drafted
# token x with probability min(1, p(x)/q(x)); on rejection continue from
# the target with the drafter's probabilities subtracted, max(0, p - q)
# renormalised.  Applied to the siblings one after another, each test uses
# the residual left by the previous rejections: r <- norm(max(0, r - q)).
# With the siblings independent draws from q this keeps the output
# distribution the target's (pinned by exact enumeration in the tests).
# q_v = softmax(draft_logits[v] / T), the same temperature as the target.
# ------------------------------------------------------------------------


def _residual_after_rejection(r, q):
    """norm(max(0, r - q)); None when nothing is left (then the rejection
    had probability 0)."""
    res = np.maximum(r - q, 0.0)
    z = res.sum()
    return res / z if z > 0 else None


def reject_stochastic_outcome_probs(probs, qprobs, tok, first_child, next_sibling):
    """Exact distribution of (accepted path, bonus token) for one sequence
    whose child tokens are given, by recursion over every accept/reject
    branch (no random numbers).  ``probs[v]`` / ``qprobs[v]``: target and
    drafter distributions at node v (float64).  Returns {(path, bonus): p}."""
    out = {}

    def visit(v, path, mass):
        r = np.array(probs[v], np.float64)
        r = r / r.sum()
        q = np.array(qprobs[v], np.float64)
        q = q / q.sum()
        for c in _children(first_child, next_sibling, v):
            x = int(tok[c])
            a = 1.0 if q[x] <= 0 else min(1.0, r[x] / q[x])
            if a > 0:
                visit(c, path + (c,), mass * a)
            if a >= 1.0:
                return
            mass *= 1.0 - a
            r = _residual_after_rejection(r, q)
            if r is None:
                return
        for x in np.nonzero(r)[0]:
            key = (path, int(x))
            out[key] = out.get(key, 0.0) + mass * r[x]

    visit(0, (0,), 1.0)
    return out


def accept_reject_stochastic(logits, draft_logits, tok, first_child, next_sibling, seed, step, T, path_cap,
                             dtype=np.float64, flip=()):
    """The RNG-driven walk of the rule above: child c with token x is kept
    iff u_c < r(x) / q(x) (u_c the accept draw of the rejection rule; a
    token with q(x) = 0 is always kept); after a rejection
    r <- norm(max(0, r - q)); the bonus is the exponential race
    argmax_x (log r(x) + G_x) over the tokens with r(x) > 0,
    G_x = -log(-log u'_x).  Returns (acc_len, acc_path, bonus, near) as
    ``accept_reject``."""
    B, N, V = logits.shape
    paths, bonus, near = [], [], [[] for _ in range(B)]
    for b in range(B):
        v, path = 0, [0]
        while True:
            z = np.asarray(logits[b, v], dtype) / dtype(T)
            e = np.exp(z - z.max())
            r = e / e.sum(dtype=dtype)
            zq = np.asarray(draft_logits[b, v], dtype) / dtype(T)
            eq = np.exp(zq - zq.max())
            q = eq / eq.sum(dtype=dtype)
            chosen = -1
            for c in _children(first_child[b], next_sibling[b], v):
                x = int(tok[b, c])
                ratio = np.inf if q[x] <= 0 else float(r[x] / q[x])
                u = float(rng.uniform_accept(seed, b, step, c))
                d = ("accept", c)
                if np.isfinite(ratio) and abs(u - ratio) <= NEAR_REJECT * max(ratio, 1e-30):
                    near[b].append(d)
                if bool(u < ratio) != ((b, d) in flip):
                    chosen = c
                    break
                r = _residual_after_rejection(r.astype(np.float64), q.astype(np.float64))
                if r is None:       # a rejection of probability 0 (rounding): nothing to sample from
                    r = e / e.sum(dtype=dtype)
                    break
                r = r.astype(dtype)
            if chosen == -1:
                u = rng.uniform_race(seed, b, step, v, np.arange(V))
                g = -np.log(-np.log(u.astype(dtype)))
                with np.errstate(divide="ignore"):
                    logr = np.log(r).astype(dtype)
                d = ("race", v)
                x, is_near = _race(logr, g, r <= 0, (b, d) in flip)
                if is_near:
                    near[b].append(d)
                bonus.append(x)
                break
            v = chosen
            path.append(v)
        paths.append(path)
    acc_len, acc_path, bon = _pack(paths, bonus, path_cap)
    return acc_len, acc_path, bon, near
