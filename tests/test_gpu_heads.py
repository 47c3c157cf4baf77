"""GPU parity: Medusa heads, LM head and top-s selection."""
import numpy as np
import pytest
import torch

from _util import dev, host, within
from oracle import heads as H
from tree_speculative_decoding_attn_gb300 import specverify as sv
from tree_speculative_decoding_attn_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = (2e-2, 1e-2)   # bf16 weights/inputs, float32 accumulation vs float64


def _heads(h, w1, b1, w2, repeat=1):
    """z (bf16, as float) and the head logits; with ``repeat`` > 1 the call
    is repeated and every repeat must give identical bits."""
    B, d = h.shape
    K, V = w2.shape[:2]
    z = torch.empty((B, K, d), dtype=torch.bfloat16, device="cuda")
    logits = torch.empty((B, K, V), dtype=torch.float32, device="cuda")
    bf = torch.bfloat16
    args = (dev(h, bf), dev(w1, bf), None if b1 is None else dev(b1, bf), dev(w2, bf))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = None
    for _ in range(repeat):
        sv.spec_medusa_heads(*args, z, logits, dev_status=st)
        torch.cuda.synchronize()
        cur = (host(z), host(logits))
        if first is not None:
            np.testing.assert_array_equal(cur[0], first[0])
            np.testing.assert_array_equal(cur[1], first[1])
        first = cur
    assert int(st.item()) == 0
    return first


# batch 1 / 8 / 64 / 200 (activation tiles of 16, 16, 64 and 256 rows), 300
# (two launches of up to 256 rows); vocabularies that are no multiple of the
# 256-row weight tile; hidden sizes of 1 to 64 K chunks
@pytest.mark.parametrize("B,K,d,V,bias", [(1, 4, 256, 1000, False), (3, 2, 512, 777, True), (8, 1, 64, 50, True),
                                          (64, 3, 1024, 3000, False), (200, 2, 256, 513, True),
                                          (300, 1, 128, 700, False), (1, 1, 4096, 130, False)])
def test_medusa_heads_small(B, K, d, V, bias):
    """Weights ~ N(0, 0.02) as in the workloads.  z is bf16 (the W2
    operand), so the logits are checked twice: against the float64 oracle
    (within the bf16 tolerance; rounding z to bf16 moves them by at most
    ~0.01 at this weight scale) and, tightly, against W2 applied to the GPU's
    own z, which isolates the second product."""
    g = synth.stream(B * 100 + d, "h")
    h = synth.gaussian(g, (B, d), 1.0, True)
    w1 = synth.gaussian(g, (K, d, d), 0.02, True)
    b1 = synth.gaussian(g, (K, d), 0.1, True) if bias else None
    w2 = synth.gaussian(g, (K, V, d), 0.02, True)
    z, logits = _heads(h, w1, b1, w2, repeat=2)
    rz, rl = H.medusa_heads(h, w1, b1, w2)
    assert within(z, rz, *TOL)[0]                 # bf16 output of a float32 sum
    # the oracle's W2 product from the GPU's bf16 z isolates the second GEMM
    rl2 = np.einsum("bkd,kvd->bkv", z.astype(np.float64), w2.astype(np.float64))
    assert within(logits, rl2, 1e-4, 1e-4)[0]
    assert within(logits, rl, *TOL)[0]


def test_medusa_heads_zero_w1_reproduce_lm_head_topk():
    """W1 = 0 and W2 = copies of the LM head: every head's top-10 equals the
    LM head's (the heads' initialisation on the pages)."""
    g = synth.stream(3, "z")
    d, V = 256, 2000
    h = synth.gaussian(g, (2, d), 1.0, True)
    wlm = synth.gaussian(g, (V, d), 0.05, True)
    K = 3
    z, logits = _heads(h, np.zeros((K, d, d), np.float32), None, np.broadcast_to(wlm, (K, V, d)).copy())
    np.testing.assert_array_equal(z, np.broadcast_to(h[:, None, :], z.shape))   # h is bf16: exact
    lm = torch.empty((2, V), dtype=torch.float32, device="cuda")
    sv.spec_lm_head(dev(h, torch.bfloat16), dev(wlm, torch.bfloat16), lm)
    for k in range(K):
        np.testing.assert_array_equal(logits[:, k], logits[:, 0])
    idx = torch.empty((2, 10), dtype=torch.int32, device="cuda")
    sv.spec_topk(dev(logits[:, 0]), 10, idx)
    idx2 = torch.empty((2, 10), dtype=torch.int32, device="cuda")
    sv.spec_topk(lm, 10, idx2)
    torch.cuda.synchronize()
    assert (host(idx) == host(idx2)).all()


@pytest.mark.parametrize("B", [1, 8, 64])
def test_medusa_heads_full_size(B):
    """Hidden 4096, 4 heads, vocabulary 32000 (1.05 GB of head weights) at
    batch 1, 8 and 64: every z and every logit."""
    w = synth.WORKLOADS["vicuna7b_medusa"]
    h, w1, w2, _ = synth.medusa_inputs(w, batch=B)
    z, logits = _heads(h, w1, None, w2)
    rz, rl = H.medusa_heads(h, w1, None, w2)
    assert within(z, rz, *TOL)[0]
    assert within(logits, rl, *TOL)[0]


@pytest.mark.parametrize("R,d,V", [(5, 128, 300), (64, 4096, 32000), (130, 256, 1001), (600, 128, 900)])
def test_lm_head(R, d, V):
    g = synth.stream(R + d + V, "lm")
    hid = synth.gaussian(g, (R, d), 1.0, True)
    wlm = synth.gaussian(g, (V, d), 0.02, True)
    out = torch.empty((R, V), dtype=torch.float32, device="cuda")
    sv.spec_lm_head(dev(hid, torch.bfloat16), dev(wlm, torch.bfloat16), out)
    torch.cuda.synchronize()
    got = host(out)
    ref = H.lm_head(hid, wlm)
    assert within(got, ref, *TOL)[0]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
# (V, s): per-thread lists of 4, 8 and 16 keys; rows that fill one partial
# batch per thread and rows that fold many batches per thread
@pytest.mark.parametrize("V,s", [(1000, 10), (32000, 10), (128256, 16), (17, 1), (33, 16), (40000, 4), (9000, 7),
                                 (200000, 6), (3000, 12)])
def test_topk_bit_exact(dtype, V, s):
    g = synth.stream(V + s, "topk")
    rows = np.round(synth.gaussian(g, (6, V), 2.0, False) * 4) / 4   # plenty of exact ties
    rows = synth.round_bf16(rows) if dtype == torch.bfloat16 else rows.astype(np.float32)
    idx = torch.empty((6, s), dtype=torch.int32, device="cuda")
    val = torch.empty((6, s), dtype=torch.float32, device="cuda")
    sv.spec_topk(dev(rows, dtype), s, idx, val)
    torch.cuda.synchronize()
    ridx, rval = H.topk(rows, s)
    np.testing.assert_array_equal(host(idx), ridx)
    np.testing.assert_array_equal(host(val), rval)


def test_heads_then_topk_chain_matches_up_to_near_ties():
    """GPU heads -> GPU top-10 against oracle heads -> oracle top-10: equal,
    except where two candidates' oracle logits lie within the tolerance."""
    w = synth.WORKLOADS["vicuna7b_medusa"]
    h, w1, w2, _ = synth.medusa_inputs(w, hidden=512, vocab=4000)
    _, logits = _heads(h, w1, None, w2)
    idx = torch.empty((4, 10), dtype=torch.int32, device="cuda")
    sv.spec_topk(dev(logits.reshape(4, -1)), 10, idx)
    torch.cuda.synchronize()
    _, rl = H.medusa_heads(h, w1, None, w2)
    ridx, _ = H.topk(rl.reshape(4, -1), 10)
    got = host(idx)
    for r in range(4):
        for j in range(10):
            if got[r, j] != ridx[r, j]:
                a, b = rl.reshape(4, -1)[r, got[r, j]], rl.reshape(4, -1)[r, ridx[r, j]]
                assert abs(a - b) <= TOL[0] + TOL[1] * abs(b)
