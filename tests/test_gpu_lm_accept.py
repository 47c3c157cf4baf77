"""GPU parity: LM head fused with greedy / typical acceptance.

The fused call never writes the logits.  Its reference is the oracle's
acceptance applied to the logits the unfused LM head (spec_lm_head, the same
GEMM and summation order) writes: greedy must agree bit for bit; typical is
decided by the oracle in float64 and may differ only at a flagged near tie
(the fused path recomputes a child's logit as a float32 dot product).
Those logits themselves are checked against the float64 oracle LM head.
"""
import numpy as np
import pytest
import torch

from _util import dev, host, i32, within, zeros_i32
from oracle import accept as ACC
from oracle import heads as H
from oracle import tree as T
from tree_speculative_decoding_attn_gb300 import specverify as sv
from tree_speculative_decoding_attn_gb300 import synth

pytestmark = pytest.mark.gpu

CASES = [
    # (B, tree, hidden, V, temperature)
    (1, synth.random_tree(1001, 64, (10, 10, 10, 10)), 4096, 32000, 1.0),     # the Vicuna-7B step's shape
    (8, synth.random_tree(1002, 60, (10, 4, 3, 2, 2)), 1024, 128256, 1.0),   # 480 rows: two GEMM launches
    (2, synth.dense_tree((4, 4, 4, 4), 256), 512, 5000, 0.7),                # 256-node tree, four mask words
    (3, synth.p4_example(), 128, 1001, 1.0),                                 # vocabulary no multiple of 32
]


def _setup(case):
    B, shape, d, V, Tm = CASES[case]
    N = shape.n
    g = synth.stream(500 + case, "lm_accept")
    hid = synth.gaussian(g, (B, N, d), 1.0, True)
    w = synth.gaussian(g, (V, d), 0.02 if d >= 1024 else 0.05, True)
    dh, dw = dev(hid, torch.bfloat16), dev(w, torch.bfloat16)
    logits = torch.empty((B * N, V), dtype=torch.float32, device="cuda")
    sv.spec_lm_head(dh.view(B * N, d), dw, logits)
    torch.cuda.synchronize()
    lg = host(logits).reshape(B, N, V)
    # tokens: random distinct siblings, then planted agreement on the GPU's
    # own logits (a child takes its parent's argmax) so greedy paths are long
    tok = np.zeros((B, N), np.int32)
    t = T.build_tree(shape.parents, 0)
    for b in range(B):
        tok[b, 0] = g.integers(V)
        for v in range(N):
            kids = [c for c in range(1, N) if shape.parents[c] == v]
            if kids:
                tok[b, kids] = g.choice(V, size=len(kids), replace=False)
                if g.random() < 0.75:
                    c = kids[int(g.integers(len(kids)))]
                    a = int(np.argmax(lg[b, v]))
                    tok[b, [k for k in kids if tok[b, k] == a]] = tok[b, c]
                    tok[b, c] = a
    par = np.broadcast_to(shape.parents, (B, N)).copy()
    fc = np.broadcast_to(t["first_child"], (B, N)).copy()
    ns = np.broadcast_to(t["next_sibling"], (B, N)).copy()
    return B, shape, d, V, Tm, hid, w, dh, dw, lg, tok, par, fc, ns


def _fused(mode, dh, dw, tok, par, fc, ns, cap, **kw):
    B = tok.shape[0]
    acc_len, acc_path, bonus, st = zeros_i32(B), zeros_i32(B, cap), zeros_i32(B), zeros_i32(1)
    sv.spec_lm_head_accept(mode, dh, dw, i32(tok), i32(par), i32(fc), i32(ns), acc_len, acc_path, bonus,
                           dev_status=st, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, sv.spec_status_string(int(st.item()))
    return host(acc_len), host(acc_path), host(bonus)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fused_greedy_bit_exact(case):
    B, shape, d, V, Tm, hid, w, dh, dw, lg, tok, par, fc, ns = _setup(case)
    cap = shape.n_levels + 1
    got = _fused(sv.GREEDY, dh, dw, tok, par, fc, ns, cap)
    ref = ACC.accept_greedy(lg, tok, fc, ns, cap)
    for g_, r_ in zip(got, ref):
        np.testing.assert_array_equal(g_, r_)
    if shape.n > 5:
        assert got[0].mean() > 0.5
    # the unfused logits the reference used, against the float64 LM head
    rows = np.arange(0, B * shape.n, max(1, B * shape.n // 16))
    assert within(lg.reshape(-1, V)[rows], H.lm_head(hid.reshape(-1, d)[rows], w), 2e-2, 1e-2)[0]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("eps,delta", [(0.3, 0.09), (0.09, 0.3)])
def test_fused_typical_matches_oracle(case, eps, delta):
    B, shape, d, V, Tm, hid, w, dh, dw, lg, tok, par, fc, ns = _setup(case)
    cap = shape.n_levels + 1
    got = _fused(sv.TYPICAL, dh, dw, tok, par, fc, ns, cap, temperature=Tm, eps=eps, delta=delta)
    rerun = lambda flip: ACC.accept_typical(lg, tok, par, fc, ns, eps, delta, Tm, cap, flip=flip)
    ref = rerun(())
    excused = 0
    for b in range(B):
        same = got[0][b] == ref[0][b] and (got[1][b] == ref[1][b]).all() and got[2][b] == ref[2][b]
        if same:
            continue
        hit = [dd for dd in ref[3][b] if (lambda r: r[0][b] == got[0][b] and (r[1][b] == got[1][b]).all()
                                          and r[2][b] == got[2][b])(rerun({(b, dd)}))]
        assert hit, f"sequence {b} differs from the oracle with no single flagged near tie explaining it"
        excused += 1
    print(f"fused typical case {case}: {sum(len(x) for x in ref[3])} near ties flagged, {excused} excused")
    assert excused <= 1


def test_fused_refuses_rejection_and_small_workspace():
    B, shape, d, V, Tm, hid, w, dh, dw, lg, tok, par, fc, ns = _setup(3)
    cap = shape.n_levels + 1
    with pytest.raises(sv.SpecError) as e:
        _fused(sv.REJECT, dh, dw, tok, par, fc, ns, cap)
    assert e.value.code == sv.ERR_UNSUPPORTED
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        _fused(sv.GREEDY, dh, dw, tok, par, fc, ns, cap, workspace=small)
    assert e.value.code == sv.ERR_CAPACITY
