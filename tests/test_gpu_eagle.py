"""GPU parity: EAGLE drafting rounds (draft layer + confidence-product
expansion) against the oracle.

Three rounds grow a draft tree from the root ("Medusa and EAGLE ...
explained", section "EAGLE: autoregression over features"; "5.3 Medusa、EAGLE
与 MTP", section 5.2).  Each round is checked against the oracle fed with the
GPU's state before the round (pool, node features, node K/V), so errors do
not compound: new features, node K/V and draft logits within the bf16
tolerance of the float64 oracle; the expansion (children, tokens, pool
count) exactly, the next frontier except at flagged value near ties.
"""
import numpy as np
import pytest
import torch

from _util import dev, host, i32, within, zeros_i32
from oracle import eagle as E
from oracle import expand as X
from tree_speculative_decoding_attn_gb300 import specverify as sv
from tree_speculative_decoding_attn_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = (2e-2, 1e-2)


def _weights(g, d, hq, hkv, D, f, V, std):
    bf = lambda x: synth.round_bf16(x.astype(np.float32))
    n = lambda *s: bf(g.standard_normal(s) * std)
    return dict(fc=n(d, 2 * d), ln1=bf(1 + g.standard_normal(d) * 0.05), qkv=n((hq + 2 * hkv) * D, d),
                o=n(d, hq * D), ln2=bf(1 + g.standard_normal(d) * 0.05), gate_up=n(2, f, d), down=n(d, f),
                lnf=bf(1 + g.standard_normal(d) * 0.05), lm=n(V, d), emb=bf(g.standard_normal((V, d))))


@pytest.mark.parametrize("B,d,hq,hkv,D,f,V,k,fronts", [
    (2, 256, 4, 2, 64, 512, 1000, 4, (1, 4, 4)),          # CUDA-core attention (head_dim 64)
    (2, 512, 4, 1, 128, 1024, 3000, 6, (1, 6, 8)),        # tensor-core attention (4 x 64 rows per KV head)
])
def test_eagle_rounds_match_oracle(B, d, hq, hkv, D, f, V, k, fronts):
    g = np.random.default_rng(B * 1000 + d)
    wts = _weights(g, d, hq, hkv, D, f, V, 0.05)
    dw = {n: dev(x, torch.bfloat16) for n, x in wts.items()}
    prefix = np.array([37, 300], np.int32)[:B]
    S = int(prefix.max()) + 16
    kp = synth.round_bf16(g.standard_normal((B, hkv, S, D)).astype(np.float32))
    vp = synth.round_bf16(g.standard_normal((B, hkv, S, D)).astype(np.float32))
    M = 128                                   # pool capacity: 1 + k + k * F1 + k * F2 children
    feat0 = np.zeros((B, M + 1, d), np.float32)
    feat0[:, M] = synth.round_bf16(g.standard_normal((B, d)).astype(np.float32))
    par = np.full((B, M), -1, np.int32); tok = np.zeros((B, M), np.int32)
    conf = np.zeros((B, M), np.float32); val = np.zeros((B, M), np.float32)
    tok[:, 0] = g.integers(V, size=B); conf[:, 0] = 1; val[:, 0] = 1
    d_feat, d_kn, d_vn = dev(feat0, torch.bfloat16), torch.zeros((B, hkv, M, D), dtype=torch.bfloat16, device="cuda"), \
        torch.zeros((B, hkv, M, D), dtype=torch.bfloat16, device="cuda")
    d_par, d_tok, d_conf, d_val, d_cnt = i32(par), i32(tok), dev(conf), dev(val), i32(np.ones(B, np.int32))
    d_kp, d_vp, d_prefix = dev(kp, torch.bfloat16), dev(vp, torch.bfloat16), i32(prefix)
    front = np.zeros((B, 1), np.int32)
    st = zeros_i32(1)
    oracle_w = {n: x for n, x in wts.items() if n != "gate_up"}
    oracle_w["gate"], oracle_w["up"] = wts["gate_up"][0], wts["gate_up"][1]
    for depth in range(len(fronts)):
        F = front.shape[1]
        n_next = fronts[depth + 1] if depth + 1 < len(fronts) else 4
        state = dict(feat=host(d_feat), kn=host(d_kn), vn=host(d_vn), par=host(d_par), tok=host(d_tok),
                     conf=host(d_conf), val=host(d_val), cnt=host(d_cnt))
        nxt = zeros_i32(B, n_next)
        logits = torch.empty((B, F, V), dtype=torch.float32, device="cuda")
        sv.spec_eagle_round(dw, d_kp, d_vp, d_prefix, int(prefix.max()), d_kn, d_vn, d_feat, i32(front), depth, k,
                            1.0, d_par, d_tok, d_conf, d_val, d_cnt, nxt, draft_logits=logits, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"device status {int(st.item())}"
        rf, rk, rv, rl = E.draft_round(oracle_w, state["feat"], wts["emb"], state["par"], state["tok"], front, depth,
                                       prefix, kp, vp, state["kn"], state["vn"], hq, hkv)
        gf = host(d_feat)[np.arange(B)[:, None], front]
        ok, ex = within(gf, rf, *TOL)
        assert ok, f"round {depth}: features off by {ex}"
        gk = np.stack([host(d_kn)[b][:, front[b]] for b in range(B)])
        gv = np.stack([host(d_vn)[b][:, front[b]] for b in range(B)])
        assert within(gk, rk, *TOL)[0] and within(gv, rv, *TOL)[0], f"round {depth}: node K/V"
        gl = host(logits)
        ok, ex = within(gl, rl, *TOL)
        assert ok, f"round {depth}: draft logits off by {ex}"
        # the expansion from the GPU's own logits: exact
        rp, rt, rc, rvv, rcnt, rnxt, near = X.expand_round(gl, front, state["par"], state["tok"], state["conf"],
                                                           state["val"], state["cnt"], k, 1.0, n_next)
        np.testing.assert_array_equal(host(d_par), rp)
        np.testing.assert_array_equal(host(d_tok), rt)
        np.testing.assert_array_equal(host(d_cnt), rcnt)
        gnxt = host(nxt)
        flagged = set(near)
        for b in range(B):
            for j in range(n_next):
                if (b, j) not in flagged:
                    assert gnxt[b, j] == rnxt[b, j]
        print(f"round {depth}: features max |err| {np.abs(gf - rf).max():.2e}, logits max |err| "
              f"{np.abs(gl - rl).max():.2e}, {len(flagged)} frontier slots flagged")
        front = gnxt.astype(np.int32)
