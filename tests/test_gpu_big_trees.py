"""GPU parity for trees of more than 64 nodes and for rejection with
stochastic siblings.

Trees of up to 256 nodes carry ceil(N / 64) ancestor-mask words per node.
The dense 256-node tree is the Cartesian product of per-level candidate
sets ("Medusa and EAGLE ... explained", section "Medusa: heads, losses and
trees"), cut breadth-first.  Stochastic siblings are independent draws from
the drafter's distribution at their parent (the multi-draft setting that
page attributes to SpecInfer); acceptance then follows "Drafters: ...",
section "Why the answer does not change": keep with min(1, r/q), otherwise
continue from norm(max(0, r - q)).
"""
import numpy as np
import pytest
import torch

from _util import dev, host, i32, within, zeros_i32
from oracle import accept as ACC
from oracle import attention as A
from oracle import commit as COM
from oracle import tree as T
from tree_speculative_decoding_attn_gb300 import specverify as sv
from tree_speculative_decoding_attn_gb300 import synth

pytestmark = pytest.mark.gpu

DENSE256 = synth.dense_tree((4, 4, 4, 4), 256)          # 1 + 4 + 16 + 64 + 171
BIG = [("dense256", DENSE256), ("sparse200", synth.random_tree(11, 200, (10, 8, 6, 4, 3))),
       ("dense65", synth.dense_tree((8, 8), 65)), ("chain130", synth.chain(130))]


def _build(shape, B, V, seed, prefix):
    cand = synth.candidate_tokens(seed, B, shape.n_levels, int(shape.rank.max()) + 1, V)
    root = synth.stream(seed, "root").integers(V, size=B).astype(np.int32)
    N, W = shape.n, sv.mask_words(shape.n)
    o = dict(tok=zeros_i32(B, N), depth=zeros_i32(B, N), pos=zeros_i32(B, N),
             anc=torch.zeros((B, N, W), dtype=torch.int64, device="cuda"), fc=zeros_i32(B, N),
             ns=zeros_i32(B, N))
    st = zeros_i32(1)
    sv.spec_build_tree(i32(shape.parents), i32(shape.rank), i32(cand), i32(root), i32(prefix), o["tok"], o["depth"],
                       o["pos"], o["anc"], o["fc"], o["ns"], st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = T.build_tree_static(shape.parents, shape.rank, cand, root, prefix)
    return o, ref, cand, root


@pytest.mark.parametrize("name,shape", BIG)
def test_static_build_multiword(name, shape):
    B = 3
    prefix = np.array([0, 17, 4096], np.int32)
    o, ref, _, _ = _build(shape, B, 32000, 5, prefix)
    np.testing.assert_array_equal(host(o["tok"]), ref["tok"])
    np.testing.assert_array_equal(host(o["depth"]), ref["depth"])
    np.testing.assert_array_equal(host(o["pos"]), ref["pos"])
    np.testing.assert_array_equal(host(o["fc"]), ref["first_child"])
    np.testing.assert_array_equal(host(o["ns"]), ref["next_sibling"])
    np.testing.assert_array_equal(host(o["anc"]).view(np.uint64), T.mask_words_multi(ref["mask"]))


@pytest.mark.parametrize("n", [65, 128, 200, 256])
def test_dynamic_rerank_multiword(n):
    """The EAGLE-2 pool of the 8B workload (411 drafted nodes) reranked to
    more than 64 nodes."""
    B, V = 3, 128256
    par, tok, conf = synth.candidate_pool(1002, B, 10, 10, 5, V)
    prefix = np.array([5, 600, 8000], np.int32)
    W = sv.mask_words(n)
    o = {k: zeros_i32(B, n) for k in ("tok", "par", "depth", "pos", "fc", "ns", "pidx")}
    anc = torch.zeros((B, n, W), dtype=torch.int64, device="cuda")
    val = torch.zeros((B, n), dtype=torch.float32, device="cuda")
    st = zeros_i32(1)
    sv.spec_build_tree_dynamic(i32(par), i32(tok), dev(conf), i32(prefix), o["tok"], o["par"], o["depth"], o["pos"],
                               anc, o["fc"], o["ns"], o["pidx"], val, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b in range(B):
        ref = T.rerank_dynamic(par[b], tok[b], conf[b], n, int(prefix[b]))
        np.testing.assert_array_equal(host(o["tok"])[b], ref["tok"])
        np.testing.assert_array_equal(host(o["par"])[b], ref["parent"])
        np.testing.assert_array_equal(host(o["pidx"])[b], ref["pool_index"])
        np.testing.assert_array_equal(host(o["pos"])[b], ref["pos"])
        np.testing.assert_array_equal(host(o["fc"])[b], ref["first_child"])
        np.testing.assert_array_equal(host(o["ns"])[b], ref["next_sibling"])
        np.testing.assert_array_equal(host(anc)[b].view(np.uint64), T.mask_words_multi(ref["mask"]))
        np.testing.assert_array_equal(host(val)[b], ref["val"])


ATTN = [
    # (dtype, B, hq, hkv, D, prefix per sequence, tree)
    ("bf16", 2, 8, 8, 128, [700, 0], DENSE256),            # MHA, 256 rows per KV head, one empty prefix
    ("bf16", 2, 16, 8, 128, [129, 2048], DENSE256),        # GQA 2: 512 rows
    ("f32", 1, 4, 4, 64, [300], synth.random_tree(11, 200, (10, 8, 6, 4, 3))),
    ("bf16", 1, 32, 8, 128, [1000], synth.dense_tree((8, 8), 65)),  # 260 rows, one node in the second word
    ("bf16", 1, 4, 4, 128, [333], synth.chain(130)),                 # 130 rows: the odd CTA mostly padding
    ("bf16", 2, 2, 2, 128, [5, 129], synth.random_tree(12, 100, (10, 8, 6, 4, 3))),  # 100 rows, one CTA's worth
    ("bf16", 3, 32, 4, 128, [6000, 1, 3000], DENSE256),             # 2048 rows per KV head: cut row groups
]


@pytest.mark.parametrize("case", range(len(ATTN)))
@pytest.mark.parametrize("tree_scale", [1.0, 4.0])
def test_attention_big_tree(case, tree_scale):
    """Every output against the oracle, Q scaled by 4 (peaked softmax);
    with the tree K scaled by 4 too, each node's ancestors carry most of its
    weight, so a wrong mask bit in any word fails the tolerance."""
    dtype, B, hq, hkv, D, prefix, shape = ATTN[case]
    w = synth.Workload("big", 40 + case, batch=B, hq=hq, hkv=hkv, head_dim=D, dtype=dtype, prefix=(0, 0),
                       n_nodes=shape.n, n_levels=shape.n_levels, vocab=10, accept="greedy", tree="random")
    prefix = np.asarray(prefix, np.int32)
    q, kc, vc, kt, vt = synth.attention_inputs(w, prefix, q_scale=4.0, s_max=int(prefix.max()) + 64)
    kt = kt * np.float32(tree_scale)   # a power of two: exact in bf16
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    mask = T.depth_and_mask(shape.parents)[1]
    anc = np.broadcast_to(T.mask_words_multi(mask), (B, shape.n, sv.mask_words(shape.n))).copy()
    N = shape.n
    ws_bytes = sv.tree_attn_workspace_bytes(tdt, B, N, hq, hkv, D, int(prefix.max()))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    out = torch.full(q.shape, float("nan"), dtype=tdt, device="cuda")
    st = zeros_i32(1)
    sv.tree_attn_verify(dev(q, tdt), dev(kc, tdt), dev(vc, tdt), dev(kt, tdt), dev(vt, tdt), i32(prefix),
                        dev(anc.view(np.int64)), out, int(prefix.max()), workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = A.tree_attention(q, kc, vc, kt, vt, prefix, mask)
    tol = (2e-2, 1e-2) if dtype == "bf16" else (1e-4, 1e-4)
    got = host(out)
    ok, excess = within(got, ref, *tol)
    err = np.abs(got - ref)
    print(f"{dtype} {hq}/{hkv} N={N} tree x{tree_scale}: max |err| {err.max():.3e}, "
          f"normalised RMS {np.sqrt((err ** 2).mean() / (ref ** 2).mean()):.3e}, ref std {ref.std():.3f}")
    assert ok, f"max excess over tolerance {excess}"
    assert ref.std() > 0.1


def _same(got, ref, b):
    return got[0][b] == ref[0][b] and (got[1][b] == ref[1][b]).all() and got[2][b] == ref[2][b]


def _decisions(got, ref, near, rerun, label, bound):
    excused = 0
    for b in range(len(ref[0])):
        if _same(got, ref, b):
            continue
        assert any(_same(got, rerun({(b, d)}), b) for d in near[b]), \
            f"{label}: sequence {b} differs from the oracle with no single flagged near tie explaining it"
        excused += 1
    print(f"{label}: {sum(len(x) for x in near)} near-tie decisions flagged, {excused} excused")
    assert excused <= bound


def _accept(mode, logits, o, par, cap, draft=None, **kw):
    B = logits.shape[0]
    tdt = torch.bfloat16 if kw.pop("bf16", False) else torch.float32
    acc_len, acc_path, bonus, st = zeros_i32(B), zeros_i32(B, cap), zeros_i32(B), zeros_i32(1)
    sv.spec_accept(mode, dev(logits, tdt), o["tok"], i32(par), o["fc"], o["ns"], acc_len, acc_path, bonus,
                   dev_status=st, draft_logits=None if draft is None else dev(draft, tdt), **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return host(acc_len), host(acc_path), host(bonus)


@pytest.mark.parametrize("mode", [sv.GREEDY, sv.TYPICAL, sv.REJECT])
def test_accept_on_256_nodes(mode):
    shape, B, V = DENSE256, 6, 5000
    o, ref, cand, root = _build(shape, B, V, 9, np.zeros(B, np.int32))
    lg = synth.target_logits(9, B, shape.n, V, 2.0, True)
    synth.plant_agreement(9, lg, shape.parents, shape.level, synth.node_tokens_from_table(shape, cand, root))
    par = np.broadcast_to(shape.parents, (B, shape.n)).copy()
    cap = shape.n_levels + 1
    got = _accept(mode, lg, o, par, cap, bf16=True, temperature=1.0, eps=0.3, delta=0.09, seed=3, step=1)
    t = ref
    if mode == sv.GREEDY:
        r = ACC.accept_greedy(lg, t["tok"], t["first_child"], t["next_sibling"], cap)
        for g_, r_ in zip(got, r):
            np.testing.assert_array_equal(g_, r_)
    elif mode == sv.TYPICAL:
        rerun = lambda flip: ACC.accept_typical(lg, t["tok"], par, t["first_child"], t["next_sibling"], 0.3, 0.09,
                                                1.0, cap, flip=flip)
        r = rerun(())
        _decisions(got, r[:3], r[3], rerun, "typical 256", 0)
    else:
        rerun = lambda flip: ACC.accept_reject(lg, t["tok"], t["first_child"], t["next_sibling"], 3, 1, 1.0, cap,
                                               flip=flip)
        r = rerun(())
        _decisions(got, r[:3], r[3], rerun, "reject 256", 0)
    assert got[0].mean() > 0.5
    # commit of the accepted paths out of a 256-node tree's K/V
    Hkv, D, S = 2, 64, 4 + cap + 2
    g = np.random.default_rng(4)
    kc = g.standard_normal((B, Hkv, S, D)).astype(np.float32)
    vc = g.standard_normal((B, Hkv, S, D)).astype(np.float32)
    kt = g.standard_normal((B, Hkv, shape.n, D)).astype(np.float32)
    vt = g.standard_normal((B, Hkv, shape.n, D)).astype(np.float32)
    prefix = np.full(B, 4, np.int32)
    dkc, dvc, plen, st = dev(kc), dev(vc), i32(prefix), zeros_i32(1)
    sv.kv_commit(dkc, dvc, dev(kt), dev(vt), i32(got[0]), i32(got[1]), plen, plen, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rk, rv, rlen = COM.kv_commit(kc, vc, kt, vt, prefix, got[0], got[1])
    np.testing.assert_array_equal(host(dkc), rk)
    np.testing.assert_array_equal(host(dvc), rv)
    np.testing.assert_array_equal(host(plen), rlen)


def _stochastic_case(shape, B, V, seed, bf16, similarity):
    """Target and drafter logits, and children drawn from the drafter's
    distribution at their parent (Gumbel-max draws, duplicates allowed).
    ``similarity`` mixes the target into the drafter so acceptances occur."""
    g = np.random.default_rng(seed)
    tgt = g.standard_normal((B, shape.n, V)) * 2.0
    drf = similarity * tgt + (1 - similarity) * g.standard_normal((B, shape.n, V)) * 2.0
    if bf16:
        tgt, drf = synth.round_bf16(tgt.astype(np.float32)), synth.round_bf16(drf.astype(np.float32))
    else:
        tgt, drf = tgt.astype(np.float32), drf.astype(np.float32)
    tok = np.zeros((B, shape.n), np.int32)
    for b in range(B):
        tok[b, 0] = g.integers(V)
        for c in range(1, shape.n):
            gum = -np.log(-np.log(g.random(V)))
            tok[b, c] = int(np.argmax(drf[b, shape.parents[c]].astype(np.float64) + gum))
    return tgt, drf, tok


SCASES = [("p4", synth.p4_example(), 6, 7), ("star8", synth.dense_tree((8,), 9), 5, 50),
          ("random32", synth.random_tree(1003, 32, (4, 3, 2)), 5, 3000),
          ("dense256", DENSE256, 3, 20011), ("chain7", synth.chain(7), 4, 1000)]


@pytest.mark.parametrize("si", range(len(SCASES)))
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("temperature", [1.0, 0.7])
def test_reject_stochastic_matches_oracle(si, bf16, temperature):
    name, shape, B, V = SCASES[si]
    tgt, drf, tok = _stochastic_case(shape, B, V, 100 + si, bf16, similarity=0.8)
    t = T.build_tree(shape.parents, 0)
    par = np.broadcast_to(shape.parents, (B, shape.n)).copy()
    fc = np.broadcast_to(t["first_child"], (B, shape.n)).copy()
    ns = np.broadcast_to(t["next_sibling"], (B, shape.n)).copy()
    o = dict(tok=i32(tok), fc=i32(fc), ns=i32(ns))
    cap = shape.n_levels + 1
    accepted = 0
    for step in range(3):
        got = _accept(sv.REJECT_STOCHASTIC, tgt, o, par, cap, draft=drf, bf16=bf16, temperature=temperature,
                      seed=0xABCDEF12345, step=step)
        rerun = lambda flip: ACC.accept_reject_stochastic(tgt, drf, tok, fc, ns, 0xABCDEF12345, step, temperature,
                                                          cap, flip=flip)
        r = rerun(())
        _decisions(got, r[:3], r[3], rerun, f"stochastic {name} step {step}", 1)
        accepted += int(got[0].sum())
    if shape.n > 1:
        assert accepted > 0            # the correlated drafter gets some drafts accepted


def test_reject_stochastic_point_mass_drafter_reduces_to_reject():
    """A drafter that is certain of each child's token (q a point mass, the
    deterministic-sibling case) makes the stochastic rule the point-mass
    rule: min(1, r/q) = r(x) and max(0, r - q) = r with x removed."""
    shape, B, V = synth.chain(6), 4, 700   # every node has one child: its proposal is that child's token
    o, ref, cand, root = _build(shape, B, V, 13, np.zeros(B, np.int32))
    lg = synth.target_logits(13, B, shape.n, V, 2.0, False)
    drf = np.full((B, shape.n, V), -1e4, np.float32)
    for b in range(B):
        for c in range(1, shape.n):
            drf[b, c - 1, ref["tok"][b, c]] = 0.0
    par = np.broadcast_to(shape.parents, (B, shape.n)).copy()
    cap = shape.n_levels + 1
    got_s = _accept(sv.REJECT_STOCHASTIC, lg, o, par, cap, draft=drf, temperature=1.0, seed=5, step=0)
    got_r = _accept(sv.REJECT, lg, o, par, cap, temperature=1.0, seed=5, step=0)
    # paths and lengths agree; the bonus of a rejection is drawn from the
    # same residual (r with the child removed) by the same race
    np.testing.assert_array_equal(got_s[0], got_r[0])
    np.testing.assert_array_equal(got_s[1], got_r[1])
    np.testing.assert_array_equal(got_s[2], got_r[2])
