"""Seeded synthetic inputs for the tree-verification step.

This module draws random numbers and random tree shapes and nothing else: it
performs none of the method's arithmetic (no masks, no depths-from-parents, no
attention, no softmax, no acceptance, no commit).  Both the CUDA path (tests,
``bench.py``) and the CPU oracle read their inputs from here, so that the two
sides see bit-identical data.

Conventions
-----------
* Random source: numpy PCG64, one generator per (workload seed, stream name).
* bf16 data is produced as float32 arrays whose values are exactly
  representable in bf16 (round-to-nearest-even applied here); the GPU side
  converts them to ``torch.bfloat16`` without further rounding and the oracle
  widens them to float64 without loss.
* "N(0, s)" in the workload descriptions is read as mean 0, standard
  deviation s (the same convention as the weight init "W ~ N(0, 0.02)").
* Tree shapes are emitted in breadth-first order (parents before children,
  siblings contiguous and ordered by candidate rank), the order used by the
  worked tree-mask example on the infra-guide page "5.3 Medusa、EAGLE 与 MTP",
  section 8.  A generator records the level at which it placed each node
  because it builds trees level by level; that is part of drawing the shape.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass, field

import numpy as np

# --------------------------------------------------------------------------
# random streams and number formats
# --------------------------------------------------------------------------


def stream(seed: int, name: str) -> np.random.Generator:
    """Independent PCG64 stream for (seed, name)."""
    return np.random.Generator(np.random.PCG64([seed, zlib.crc32(name.encode())]))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); float32 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def gaussian(g: np.random.Generator, shape, std: float, bf16: bool) -> np.ndarray:
    """float32 array ~ N(0, std); values rounded to bf16 when ``bf16``."""
    out = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return round_bf16(out) if bf16 else out


# --------------------------------------------------------------------------
# tree shapes
# --------------------------------------------------------------------------

#: parents array of the worked example on "5.3 Medusa、EAGLE 与 MTP", section 8
P4_PARENTS = (-1, 0, 0, 1, 2)


@dataclass
class TreeShape:
    """A drafted tree's shape: ``parents[i]`` (root = -1), the candidate
    rank of node i among its parent's children, and the level the generator
    placed it on.  Breadth-first order."""

    parents: np.ndarray  # int32 [N]
    rank: np.ndarray  # int32 [N]
    level: np.ndarray  # int32 [N]  (generator bookkeeping)

    @property
    def n(self) -> int:
        return int(self.parents.shape[0])

    @property
    def n_levels(self) -> int:
        return int(self.level.max()) + 1


def _bfs_shape(par, rank, level) -> TreeShape:
    """Re-emit an arbitrary-order shape in breadth-first order."""
    n = len(par)
    kids = [[] for _ in range(n)]
    for v in range(1, n):
        kids[par[v]].append(v)
    order = [0]
    head = 0
    while head < len(order):
        v = order[head]
        head += 1
        order.extend(sorted(kids[v], key=lambda c: rank[c]))
    new = {old: i for i, old in enumerate(order)}
    parents = np.array([-1] + [new[par[o]] for o in order[1:]], dtype=np.int32)
    return TreeShape(parents, np.array([rank[o] for o in order], np.int32),
                     np.array([level[o] for o in order], np.int32))


def p4_example() -> TreeShape:
    """The five-node example tree: root 0, siblings 1 and 2, 3 under 1, 4 under 2."""
    return TreeShape(np.array(P4_PARENTS, np.int32), np.array([0, 0, 1, 0, 0], np.int32),
                     np.array([0, 1, 1, 2, 2], np.int32))


def chain(n: int) -> TreeShape:
    """A single path root -> ... (the ordinary-sequence special case)."""
    par = np.arange(-1, n - 1, dtype=np.int32)
    return TreeShape(par, np.zeros(n, np.int32), np.arange(n, dtype=np.int32))


def random_tree(seed: int, n: int, caps) -> TreeShape:
    """Seeded sparse tree of ``n`` nodes with ``len(caps)+1`` levels.

    ``caps[l]`` bounds the children of a node on level l (the candidates per
    head).  The rank-0 chain down to the last level is always present (the
    top-1 guess of every head), then nodes are attached one at a time to a
    random open parent, favouring shallow levels and low ranks, the way a
    budgeted sparse tree spends its nodes on the likeliest branches.
    """
    g = stream(seed, "tree")
    depth_max = len(caps)
    assert n >= depth_max + 1
    par, rank, level, nkid = [-1], [0], [0], [0]
    for lv in range(1, depth_max + 1):  # rank-0 chain
        par.append(lv - 1); rank.append(0); level.append(lv); nkid.append(0)
        nkid[lv - 1] = 1
    while len(par) < n:
        open_ = [v for v in range(len(par)) if level[v] < depth_max and nkid[v] < caps[level[v]]]
        if not open_:
            raise ValueError("caps too small for the requested node count")
        w = np.array([0.45 ** level[v] * 0.7 ** nkid[v] for v in open_])
        v = open_[int(g.choice(len(open_), p=w / w.sum()))]
        par.append(v); rank.append(nkid[v]); level.append(level[v] + 1); nkid.append(0)
        nkid[v] += 1
    return _bfs_shape(par, rank, level)


def dense_tree(branching, n: int) -> TreeShape:
    """The Cartesian tree with ``branching[l]`` children per node on level l,
    breadth-first (children by rank), cut after its first ``n`` nodes: every
    node of level l + 1 before any of level l + 2 (the dense trees of the
    multi-candidate Medusa setting)."""
    par, rank, level = [-1], [0], [0]
    head = 0
    while len(par) < n and head < len(par):
        v = head
        head += 1
        if level[v] >= len(branching):
            continue
        for r in range(branching[level[v]]):
            if len(par) == n:
                break
            par.append(v); rank.append(r); level.append(level[v] + 1)
    return TreeShape(np.array(par, np.int32), np.array(rank, np.int32), np.array(level, np.int32))


def candidate_tokens(seed: int, batch: int, n_levels: int, s: int, vocab: int) -> np.ndarray:
    """cand_tok[b, l, r]: token proposed with rank r for level l+1 (distinct per row)."""
    g = stream(seed, "cand_tok")
    out = np.empty((batch, max(n_levels - 1, 0), s), np.int32)
    for b in range(batch):
        for l in range(n_levels - 1):
            out[b, l] = g.choice(vocab, size=s, replace=False)
    return out


def node_tokens_from_table(shape: TreeShape, cand_tok: np.ndarray, root_tok: np.ndarray) -> np.ndarray:
    """Tokens the generator assigned to each node when it filled ``cand_tok``
    (node at level l, rank r holds cand_tok[b, l-1, r]); used only to plant
    agreement into synthetic target logits."""
    B = cand_tok.shape[0]
    out = np.empty((B, shape.n), np.int32)
    out[:, 0] = root_tok
    for i in range(1, shape.n):
        out[:, i] = cand_tok[:, shape.level[i] - 1, shape.rank[i]]
    return out


# --------------------------------------------------------------------------
# synthetic target logits with planted agreement
# --------------------------------------------------------------------------

#: per-level planting rates: the head accuracies of the worked example on
#: "Medusa, explained" (0.8/0.65/0.5/0.35), extended with 0.25 and 0.2
PLANT_RATES = (0.8, 0.65, 0.5, 0.35, 0.25, 0.2)
PLANT_MARGIN = 8.0


def target_logits(seed: int, batch: int, n: int, vocab: int, std: float, bf16: bool) -> np.ndarray:
    """Unplanted target logits [B, N, V] ~ N(0, std)."""
    return gaussian(stream(seed, "target_logits"), (batch, n, vocab), std, bf16)


def plant_agreement(seed: int, logits: np.ndarray, parents: np.ndarray, level: np.ndarray,
                    tokens: np.ndarray, rates=PLANT_RATES, bf16: bool = True) -> np.ndarray:
    """In place: at each internal node v on level l, with probability
    rates[l] pick one of its children c and raise logits[b, v, tokens[b, c]]
    to (row max + PLANT_MARGIN), so that accepted paths have realistic
    lengths.  ``parents``/``level``/``tokens`` may be per-sequence [B, N] or
    shared [N] (tokens always [B, N])."""
    g = stream(seed, "plant")
    B, N, _ = logits.shape
    par2 = np.broadcast_to(parents, (B, N))
    lev2 = np.broadcast_to(level, (B, N))
    for b in range(B):
        kids = [[] for _ in range(N)]
        for c in range(1, N):
            if par2[b, c] >= 0:
                kids[par2[b, c]].append(c)
        for v in range(N):
            if not kids[v]:
                continue
            r = rates[min(int(lev2[b, v]), len(rates) - 1)]
            if g.random() < r:
                c = kids[v][int(g.integers(len(kids[v])))]
                row = logits[b, v]
                row[tokens[b, c]] = row.max() + np.float32(PLANT_MARGIN)
    if bf16:
        logits[...] = round_bf16(logits)
    return logits


# --------------------------------------------------------------------------
# EAGLE-2 style candidate pool (input of the confidence-product rerank)
# --------------------------------------------------------------------------


def candidate_pool(seed: int, batch: int, k: int, frontier: int, rounds: int, vocab: int):
    """A drafted candidate pool per sequence: pool[0] is the root; round 1
    gives the root ``k`` children; each later round gives ``k`` children to
    each of ``frontier`` earlier nodes of the previous round (drawn at
    random here: the pool is an input, the frontier choice by confidence is
    the method's job and is exercised by the expand step, not by this
    generator).  Confidences are draws from a seeded Dirichlet per parent, so
    siblings' confidences sum to at most 1 like softmax probabilities of
    distinct tokens.  Returns (pool_parent, pool_tok, pool_conf) [B, M]."""
    g = stream(seed, "pool")
    M = 1 + k + (rounds - 1) * frontier * k
    par = np.full((batch, M), -1, np.int32)
    tok = np.zeros((batch, M), np.int32)
    conf = np.zeros((batch, M), np.float32)
    for b in range(batch):
        tok[b, 0] = g.integers(vocab)
        conf[b, 0] = 1.0
        prev = [0]
        m = 1
        for rnd in range(rounds):
            parents_here = prev if rnd == 0 else sorted(g.choice(prev, size=min(frontier, len(prev)), replace=False).tolist())
            new = []
            for p in parents_here:
                toks = g.choice(vocab, size=k, replace=False)
                alpha = np.full(k + 1, 0.6)
                alpha[0] = 2.0
                pr = g.dirichlet(alpha)[:k].astype(np.float32)
                pr = np.sort(pr)[::-1]
                for j in range(k):
                    par[b, m] = p
                    tok[b, m] = toks[j]
                    conf[b, m] = pr[j]
                    new.append(m)
                    m += 1
            prev = new
        assert m == M
    return par, tok, conf


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------


@dataclass
class Workload:
    """One verify-step workload (sizes as in the workload descriptions)."""

    name: str
    seed: int
    batch: int
    hq: int
    hkv: int
    head_dim: int
    dtype: str  # "f32" or "bf16"
    prefix: tuple  # (lo, hi) inclusive; lo == hi for a fixed prefix
    n_nodes: int
    n_levels: int  # levels including the root
    vocab: int
    accept: str  # "greedy" | "reject" | "typical"
    tree: str  # "p4" | "random" | "dynamic"
    caps: tuple = ()
    medusa: dict = field(default_factory=dict)  # hidden, heads, topk
    eps: float = 0.3
    delta: float = 0.09
    temperature: float = 1.0
    logit_std: float = 2.0
    planted: bool = True
    dynamic: dict = field(default_factory=dict)  # k, frontier, rounds

    @property
    def group(self) -> int:
        return self.hq // self.hkv


WORKLOADS = {
    "tiny_exact": Workload(
        "tiny_exact", 1000, batch=1, hq=4, hkv=4, head_dim=64, dtype="f32", prefix=(128, 128),
        n_nodes=5, n_levels=3, vocab=1000, accept="greedy", tree="p4", planted=False),
    "vicuna7b_medusa": Workload(
        "vicuna7b_medusa", 1001, batch=1, hq=32, hkv=32, head_dim=128, dtype="bf16",
        prefix=(2048, 2048), n_nodes=64, n_levels=5, vocab=32000, accept="greedy", tree="random",
        caps=(10, 10, 10, 10), medusa=dict(hidden=4096, heads=4, topk=10, w_std=0.02),
        planted=False),
    "llama8b_eagle2": Workload(
        "llama8b_eagle2", 1002, batch=8, hq=32, hkv=8, head_dim=128, dtype="bf16",
        prefix=(512, 8192), n_nodes=60, n_levels=6, vocab=128256, accept="reject", tree="dynamic",
        dynamic=dict(k=10, frontier=10, rounds=5, draft=dict(ffn=14336, w_std=0.02))),
    "llama70b_serving": Workload(
        "llama70b_serving", 1003, batch=64, hq=64, hkv=8, head_dim=128, dtype="bf16",
        prefix=(4096, 4096), n_nodes=32, n_levels=4, vocab=128256, accept="greedy", tree="random",
        caps=(4, 3, 2)),
    "long_context": Workload(
        "long_context", 1004, batch=4, hq=32, hkv=8, head_dim=128, dtype="bf16",
        prefix=(32768, 32768), n_nodes=64, n_levels=6, vocab=128256, accept="typical",
        tree="random", caps=(8, 4, 3, 2, 2)),
}


def prefix_lengths(w: Workload) -> np.ndarray:
    lo, hi = w.prefix
    if lo == hi:
        return np.full(w.batch, lo, np.int32)
    return stream(w.seed, "prefix").integers(lo, hi + 1, size=w.batch).astype(np.int32)


def tree_shape(w: Workload) -> TreeShape:
    if w.tree == "p4":
        return p4_example()
    if w.tree == "random":
        return random_tree(w.seed, w.n_nodes, w.caps)
    raise ValueError("dynamic trees have no fixed shape")


def attention_inputs(w: Workload, prefix_len: np.ndarray, n: int | None = None,
                     s_max: int | None = None, q_scale: float = 1.0, batch: int | None = None):
    """Q [B,N,Hq,D], cache K/V [B,Hkv,S_max,D], tree K/V [B,Hkv,N,D] ~ N(0,1).

    The cache rows at and beyond each sequence's prefix length hold random
    values too (they are not part of the prefix and must be ignored)."""
    n = w.n_nodes if n is None else n
    B = w.batch if batch is None else batch
    bf16 = w.dtype == "bf16"
    if s_max is None:
        s_max = int(prefix_len.max()) + 64
    g = stream(w.seed, "attn")
    q = gaussian(g, (B, n, w.hq, w.head_dim), 1.0, False) * np.float32(q_scale)
    q = round_bf16(q) if bf16 else q
    kc = gaussian(g, (B, w.hkv, s_max, w.head_dim), 1.0, bf16)
    vc = gaussian(g, (B, w.hkv, s_max, w.head_dim), 1.0, bf16)
    kt = gaussian(g, (B, w.hkv, n, w.head_dim), 1.0, bf16)
    vt = gaussian(g, (B, w.hkv, n, w.head_dim), 1.0, bf16)
    return q, kc, vc, kt, vt


def medusa_inputs(w: Workload, batch: int | None = None, hidden: int | None = None,
                  vocab: int | None = None, heads: int | None = None):
    """h [B,d], W1 [K,d,d] ([out,in]), W2 [K,V,d], W_lm [V,d], all bf16 values."""
    m = w.medusa
    B = w.batch if batch is None else batch
    d = m["hidden"] if hidden is None else hidden
    V = w.vocab if vocab is None else vocab
    K = m["heads"] if heads is None else heads
    g = stream(w.seed, "medusa")
    h = gaussian(g, (B, d), 1.0, True)
    w1 = gaussian(g, (K, d, d), m["w_std"], True)
    w2 = gaussian(g, (K, V, d), m["w_std"], True)
    wlm = gaussian(g, (V, d), m["w_std"], True)
    return h, w1, w2, wlm


def root_tokens(w: Workload, batch: int | None = None) -> np.ndarray:
    B = w.batch if batch is None else batch
    return stream(w.seed, "root").integers(w.vocab, size=B).astype(np.int32)
