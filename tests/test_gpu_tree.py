"""GPU parity: tree construction (static and confidence rerank) is bit-exact with the oracle."""
import numpy as np
import pytest
import torch

from _util import dev, host, i32, zeros_i32
from oracle import tree as T
from tree_speculative_decoding_attn_gb300 import specverify as sv
from tree_speculative_decoding_attn_gb300 import synth

pytestmark = pytest.mark.gpu


def _outs(B, N):
    return dict(tok=zeros_i32(B, N), depth=zeros_i32(B, N), pos_ids=zeros_i32(B, N),
                anc_mask=torch.zeros((B, N), dtype=torch.int64, device="cuda"),
                first_child=zeros_i32(B, N), next_sibling=zeros_i32(B, N))


def _static(shape, cand, root, prefix):
    B, N = len(root), shape.n
    o = _outs(B, N)
    st = zeros_i32(1)
    sv.spec_build_tree(i32(shape.parents), i32(shape.rank), i32(cand), i32(root), i32(prefix), o["tok"],
                       o["depth"], o["pos_ids"], o["anc_mask"], o["first_child"], o["next_sibling"], st)
    torch.cuda.synchronize()
    return {k: host(v) for k, v in o.items()}, int(host(st)[0])


SHAPES = [("p4", lambda: synth.p4_example()), ("single", lambda: synth.chain(1)),
          ("chain64", lambda: synth.chain(64)),
          ("medusa64", lambda: synth.random_tree(1001, 64, (10, 10, 10, 10))),
          ("static32", lambda: synth.random_tree(1003, 32, (4, 3, 2))),
          ("static64", lambda: synth.random_tree(1004, 64, (8, 4, 3, 2, 2)))]


@pytest.mark.parametrize("name,make", SHAPES)
def test_static_tree_bit_exact(name, make):
    shape = make()
    B = 5
    s = 10
    cand = synth.candidate_tokens(7, B, max(shape.n_levels, 2), s, 32000)
    root = synth.stream(7, "r").integers(32000, size=B).astype(np.int32)
    prefix = np.array([0, 1, 127, 2048, 32768], np.int32)
    got, status = _static(shape, cand, root, prefix)
    assert status == 0
    ref = T.build_tree_static(shape.parents, shape.rank, cand, root, prefix)
    np.testing.assert_array_equal(got["tok"], ref["tok"])
    np.testing.assert_array_equal(got["depth"], ref["depth"])
    np.testing.assert_array_equal(got["pos_ids"], ref["pos"])
    np.testing.assert_array_equal(got["anc_mask"].view(np.uint64), ref["anc"])
    np.testing.assert_array_equal(got["first_child"], ref["first_child"])
    np.testing.assert_array_equal(got["next_sibling"], ref["next_sibling"])


def test_worked_example_mask_on_gpu():
    got, status = _static(synth.p4_example(), np.zeros((1, 2, 2), np.int32), np.array([3], np.int32),
                          np.array([10], np.int32))
    words = got["anc_mask"][0].view(np.uint64)
    rows = [[int((int(w) >> j) & 1) for j in range(5)] for w in words]
    assert rows[4] == [1, 0, 1, 0, 1]
    assert got["depth"][0, 1] == got["depth"][0, 2] == 1
    assert got["pos_ids"][0].tolist() == [10, 11, 11, 12, 12]


@pytest.mark.parametrize("bad", [[0, 0, 1], [-1, 1, 0], [-1, 0, 3, 1]])
def test_bad_parents_reported_not_trapped(bad):
    shape = synth.TreeShape(np.array(bad, np.int32), np.zeros(len(bad), np.int32), np.zeros(len(bad), np.int32))
    _, status = _static(shape, np.zeros((1, 4, 2), np.int32), np.array([1], np.int32), np.array([0], np.int32))
    assert status == sv.DEV_BAD_PARENTS


def _dynamic(par, tok, conf, N, prefix):
    B, M = par.shape
    o = _outs(B, N)
    parents = zeros_i32(B, N)
    pidx = zeros_i32(B, N)
    val = torch.zeros((B, N), dtype=torch.float32, device="cuda")
    st = zeros_i32(1)
    sv.spec_build_tree_dynamic(i32(par), i32(tok), dev(conf), i32(prefix), o["tok"], parents, o["depth"],
                               o["pos_ids"], o["anc_mask"], o["first_child"], o["next_sibling"], pidx, val, st)
    torch.cuda.synchronize()
    got = {k: host(v) for k, v in o.items()}
    got.update(parent=host(parents), pool_index=host(pidx), val=host(val))
    return got, int(host(st)[0])


def _check_dynamic(par, tok, conf, N, prefix):
    got, status = _dynamic(par, tok, conf, N, prefix)
    assert status == 0
    for b in range(par.shape[0]):
        ref = T.rerank_dynamic(par[b], tok[b], conf[b], N, int(prefix[b]))
        np.testing.assert_array_equal(got["pool_index"][b], ref["pool_index"])
        np.testing.assert_array_equal(got["tok"][b], ref["tok"])
        np.testing.assert_array_equal(got["parent"][b], ref["parent"])
        np.testing.assert_array_equal(got["depth"][b], ref["depth"])
        np.testing.assert_array_equal(got["pos_ids"][b], ref["pos"])
        np.testing.assert_array_equal(got["anc_mask"][b].view(np.uint64), ref["anc"])
        np.testing.assert_array_equal(got["first_child"][b], ref["first_child"])
        np.testing.assert_array_equal(got["next_sibling"][b], ref["next_sibling"])
        np.testing.assert_array_equal(got["val"][b].view(np.uint32), ref["val"].view(np.uint32))


def test_dynamic_rerank_full_size_pool():
    """8 sequences, pool of 1 + 10 + 4 x 100 drafted nodes, 60 kept."""
    w = synth.WORKLOADS["llama8b_eagle2"]
    par, tok, conf = synth.candidate_pool(w.seed, w.batch, 10, 10, 5, w.vocab)
    _check_dynamic(par, tok, conf, 60, synth.prefix_lengths(w))


def test_dynamic_rerank_exact_value_ties():
    """Confidences on a 1/8 grid make many path values equal: ties must go
    to the shallower node, then the lower pool index."""
    par, tok, conf = synth.candidate_pool(5, 4, 4, 3, 4, 1000)
    conf = (np.round(conf * 8) / 8).astype(np.float32)
    conf[:, 0] = 1
    _check_dynamic(par, tok, conf, 17, np.array([3, 0, 9, 100], np.int32))


def test_dynamic_bad_confidence_reported():
    par = np.array([[-1, 0, 1]], np.int32)
    conf = np.array([[1.0, 0.5, 1.5]], np.float32)
    _, status = _dynamic(par, np.zeros((1, 3), np.int32), conf, 2, np.array([0], np.int32))
    assert status == sv.DEV_BAD_POOL
