"""GPU parity: paged prefix cache (block tables) and ragged per-request trees.

"5.3 Medusa、EAGLE 与 MTP", section 8, closing remarks: a serving engine keeps
the KV cache in blocks addressed by block tables and batches the trees of
different requests.  Here every request of a batch has its own tree (its own
node count and shape, padded to the batch's largest), its prefix lives in
blocks scattered over a shared pool, and the accepted path is appended to
its block list.

Reference: the oracle on the contiguous cache the block tables describe
(gathered here with plain indexing).  The paged kernels read the same values
in the same order as the contiguous ones, so paged and contiguous outputs
must also agree bit for bit.
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


def _ragged_trees(seed, B, n_max, caps_list):
    """Per-request trees of different sizes, parents padded with -1 past n_valid."""
    g = np.random.default_rng(seed)
    shapes, par = [], np.full((B, n_max), -1, np.int32)
    nv = np.zeros(B, np.int32)
    for b in range(B):
        caps = caps_list[b % len(caps_list)]
        cap_nodes, width = 1, 1
        for c in caps:                       # nodes the caps allow
            width *= c
            cap_nodes += width
        n = int(g.integers(len(caps) + 1, min(n_max, cap_nodes) + 1))
        sh = synth.random_tree(seed * 100 + b, n, caps)
        shapes.append(sh)
        par[b, :n] = sh.parents
        nv[b] = n
    return shapes, par, nv


def _pool(seed, B, Hkv, D, prefix, bs, dtype_bf16, extra_blocks=5):
    """A block pool with each sequence's blocks at shuffled positions, the
    block table, and the contiguous cache it describes."""
    g = np.random.default_rng(seed)
    need = [(int(p) + 64 + bs - 1) // bs for p in prefix]     # room for the commit
    max_blocks = max(need)
    nb = sum(need) + extra_blocks
    perm = g.permutation(nb)
    table = np.full((B, max_blocks), -1, np.int32)
    k = 0
    for b in range(B):
        for j in range(need[b]):
            table[b, j] = perm[k]
            k += 1
    kp = g.standard_normal((nb, Hkv, bs, D)).astype(np.float32)
    vp = g.standard_normal((nb, Hkv, bs, D)).astype(np.float32)
    if dtype_bf16:
        kp, vp = synth.round_bf16(kp), synth.round_bf16(vp)
    S = max_blocks * bs
    kc = np.zeros((B, Hkv, S, D), np.float32)
    vc = np.zeros((B, Hkv, S, D), np.float32)
    for b in range(B):
        for j in range(need[b]):
            kc[b, :, j * bs:(j + 1) * bs] = kp[table[b, j]]
            vc[b, :, j * bs:(j + 1) * bs] = vp[table[b, j]]
    return kp, vp, table, kc, vc


def _build_batch(par, nv, prefix, tok=None):
    B, N = par.shape
    W = sv.mask_words(N)
    o = dict(depth=zeros_i32(B, N), pos=zeros_i32(B, N), anc=torch.zeros((B, N, W), dtype=torch.int64, device="cuda"),
             fc=zeros_i32(B, N), ns=zeros_i32(B, N), tok=zeros_i32(B, N))
    st = zeros_i32(1)
    sv.spec_build_tree_batch(i32(par), i32(prefix), o["depth"], o["pos"], o["anc"], o["fc"], o["ns"],
                             n_valid=i32(nv), tok_in=None if tok is None else i32(tok),
                             tok=o["tok"] if tok is not None else None, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o


@pytest.mark.parametrize("n_max", [16, 64, 130])
def test_build_batch_per_request_trees(n_max):
    B = 6
    shapes, par, nv = _ragged_trees(n_max, B, n_max, [(4, 3, 2), (10, 2), (3, 3, 3, 3)])
    prefix = np.arange(B, dtype=np.int32) * 100
    tok = np.random.default_rng(1).integers(0, 32000, size=(B, n_max)).astype(np.int32)
    o = _build_batch(par, nv, prefix, tok)
    W = sv.mask_words(n_max)
    anc = host(o["anc"]).view(np.uint64).reshape(B, n_max, W)
    for b in range(B):
        n = int(nv[b])
        ref = T.build_tree(par[b, :n], int(prefix[b]))
        np.testing.assert_array_equal(host(o["depth"])[b, :n], ref["depth"])
        np.testing.assert_array_equal(host(o["pos"])[b, :n], ref["pos"])
        np.testing.assert_array_equal(host(o["fc"])[b, :n], ref["first_child"])
        np.testing.assert_array_equal(host(o["ns"])[b, :n], ref["next_sibling"])
        full = np.zeros((n_max, n_max), bool)
        full[:n, :n] = ref["mask"]
        for i in range(n, n_max):                 # absent nodes see only themselves
            full[i, i] = True
        np.testing.assert_array_equal(anc[b], T.mask_words_multi(full))
        assert (host(o["depth"])[b, n:] == 0).all() and (host(o["pos"])[b, n:] == prefix[b]).all()
        assert (host(o["fc"])[b, n:] == -1).all() and (host(o["ns"])[b, n:] == -1).all()
        np.testing.assert_array_equal(host(o["tok"])[b], tok[b])


CASES = [
    # (dtype, B, hq, hkv, D, block_size, prefix, n_max, caps)   kernel
    ("bf16", 4, 64, 8, 128, 128, [4096, 1000, 0, 2300], 32, [(4, 3, 2)]),       # SM pairs (256 rows)
    ("bf16", 3, 32, 32, 128, 256, [2048, 700, 129], 64, [(10, 10, 10, 10)]),   # single CTA, split KV
    ("f32", 2, 4, 4, 64, 128, [300, 129], 20, [(4, 3, 2)]),                     # CUDA cores
    ("bf16", 2, 8, 8, 128, 128, [700, 1500], 130, [(6, 5, 4, 3)]),              # three mask words, SM pairs
    ("bf16", 2, 32, 8, 128, 128, [3000, 129], 256, [(8, 6, 4, 3)]),             # two tree tiles, SM pairs
    ("f32", 2, 4, 4, 64, 128, [300, 129], 200, [(6, 5, 4, 3)]),                 # four mask words, CUDA cores
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_paged_attention_matches_contiguous_and_oracle(case):
    dtype, B, hq, hkv, D, bs, prefix, n_max, caps = CASES[case]
    bf = dtype == "bf16"
    tdt = torch.bfloat16 if bf else torch.float32
    prefix = np.asarray(prefix, np.int32)
    shapes, par, nv = _ragged_trees(50 + case, B, n_max, caps)
    kp, vp, table, kc, vc = _pool(60 + case, B, hkv, D, prefix, bs, bf)
    g = np.random.default_rng(70 + case)
    q = (g.standard_normal((B, n_max, hq, D)) * 4).astype(np.float32)
    kt = g.standard_normal((B, hkv, n_max, D)).astype(np.float32)
    vt = g.standard_normal((B, hkv, n_max, D)).astype(np.float32)
    if bf:
        q, kt, vt = synth.round_bf16(q), synth.round_bf16(kt), synth.round_bf16(vt)
    o = _build_batch(par, nv, prefix)
    mp = int(prefix.max())
    wsb = sv.tree_attn_workspace_bytes(tdt, B, n_max, hq, hkv, D, mp)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    st = zeros_i32(1)
    dq, dkt, dvt = dev(q, tdt), dev(kt, tdt), dev(vt, tdt)
    out_p = torch.full((B, n_max, hq, D), float("nan"), dtype=tdt, device="cuda")
    sv.tree_attn_verify_paged(dq, dev(kp, tdt), dev(vp, tdt), i32(table), dkt, dvt, i32(prefix), o["anc"], out_p, mp,
                              workspace=ws, dev_status=st)
    out_c = torch.full_like(out_p, float("nan"))
    sv.tree_attn_verify(dq, dev(kc, tdt), dev(vc, tdt), dkt, dvt, i32(prefix), o["anc"], out_c, mp, workspace=ws,
                        dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got_p, got_c = host(out_p), host(out_c)
    for b in range(B):
        n = int(nv[b])
        np.testing.assert_array_equal(got_p[b, :n], got_c[b, :n])         # same values, same order
        mask = T.depth_and_mask(par[b, :n])[1]
        ref = A.tree_attention(q[b:b + 1, :n], kc[b:b + 1], vc[b:b + 1], kt[b:b + 1, :, :n], vt[b:b + 1, :, :n],
                               prefix[b:b + 1], mask)
        ok, excess = within(got_p[b:b + 1, :n], ref, *((2e-2, 1e-2) if bf else (1e-4, 1e-4)))
        assert ok, f"sequence {b}: max excess {excess}"


def test_ragged_step_paged_greedy_commit():
    """One verify step over per-request trees and a paged cache: build ->
    paged attention -> greedy acceptance -> paged commit, against the oracle
    on the contiguous cache."""
    B, hq, hkv, D, bs, n_max, V = 5, 64, 8, 128, 128, 32, 5000
    prefix = np.array([1000, 4096, 130, 2047, 0], np.int32)
    shapes, par, nv = _ragged_trees(81, B, n_max, [(4, 3, 2), (6, 3), (2, 2, 2, 2)])
    kp, vp, table, kc, vc = _pool(82, B, hkv, D, prefix, bs, True)
    g = np.random.default_rng(83)
    tok = np.zeros((B, n_max), np.int32)
    for b in range(B):
        for v in range(int(nv[b])):
            kids = [c for c in range(1, int(nv[b])) if par[b, c] == v]
            tok[b, kids] = g.choice(V, size=len(kids), replace=False)
    lg = synth.round_bf16((g.standard_normal((B, n_max, V)) * 2).astype(np.float32))
    for b in range(B):                          # planted agreement along one branch
        v = 0
        while True:
            kids = [c for c in range(1, int(nv[b])) if par[b, c] == v]
            if not kids:
                break
            c = kids[int(g.integers(len(kids)))]
            lg[b, v, tok[b, c]] = lg[b, v].max() + 8
            v = c
    kt = synth.round_bf16(g.standard_normal((1, B, hkv, n_max, D)).astype(np.float32))
    vt = synth.round_bf16(g.standard_normal((1, B, hkv, n_max, D)).astype(np.float32))
    o = _build_batch(par, nv, prefix, tok)
    bf = torch.bfloat16
    dkp, dvp = dev(kp[None], bf), dev(vp[None], bf)
    st = zeros_i32(1)
    # greedy acceptance over the per-request trees
    cap = 8
    acc_len, acc_path, bonus = zeros_i32(B), zeros_i32(B, cap), zeros_i32(B)
    sv.spec_accept(sv.GREEDY, dev(lg, bf), o["tok"], i32(par), o["fc"], o["ns"], acc_len, acc_path, bonus,
                   dev_status=st)
    new_prefix = zeros_i32(B)
    sv.kv_commit_paged(dkp, dvp, i32(table), dev(kt, bf), dev(vt, bf), acc_len, acc_path, i32(prefix), new_prefix,
                       dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    fc = host(o["fc"]); ns = host(o["ns"])
    r_len, r_path, r_bonus = ACC.accept_greedy(lg, tok, fc, ns, cap)
    np.testing.assert_array_equal(host(acc_len), r_len)
    np.testing.assert_array_equal(host(acc_path), r_path)
    np.testing.assert_array_equal(host(bonus), r_bonus)
    assert r_len.mean() > 1
    # the pool after the commit, gathered back through the table, equals the
    # oracle's commit on the contiguous cache; blocks outside every table are untouched
    rk, rv, rnew = COM.kv_commit(kc, vc, kt[0], vt[0], prefix, r_len, r_path)
    kp2, vp2 = host(dkp)[0], host(dvp)[0]
    np.testing.assert_array_equal(host(new_prefix), rnew)
    for b in range(B):
        for j in range(table.shape[1]):
            blk = table[b, j]
            if blk < 0:
                continue
            np.testing.assert_array_equal(kp2[blk], rk[b, :, j * bs:(j + 1) * bs])
            np.testing.assert_array_equal(vp2[blk], rv[b, :, j * bs:(j + 1) * bs])
    unused = sorted(set(range(kp.shape[0])) - set(table[table >= 0].tolist()))
    np.testing.assert_array_equal(kp2[unused], kp[unused])


def test_paged_commit_bad_block_is_reported_and_skipped():
    B, hkv, D, bs = 2, 2, 64, 128
    prefix = np.array([126, 10], np.int32)
    kp, vp, table, kc, vc = _pool(91, B, hkv, D, prefix, bs, False)
    table[0, 1] = kp.shape[0] + 7                # sequence 0's second block does not exist
    kt = np.random.default_rng(92).standard_normal((1, B, hkv, 8, D)).astype(np.float32)
    acc_len = np.array([3, 2], np.int32)         # sequence 0 writes rows 126..129: blocks 0 and 1
    acc_path = np.array([[0, 1, 2, 3], [0, 4, 5, -1]], np.int32)
    dkp, dvp = dev(kp[None]), dev(vp[None])
    plen, st = i32(prefix), zeros_i32(1)
    sv.kv_commit_paged(dkp, dvp, i32(table), dev(kt), dev(kt), i32(acc_len), i32(acc_path), plen, plen,
                       dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == sv.DEV_BAD_BLOCK
    assert host(plen).tolist() == [126, 13]       # sequence 0 neither copied nor advanced
    kp2 = host(dkp)[0]
    np.testing.assert_array_equal(kp2[table[0, 0]], kp[table[0, 0]])
