"""GPU parity: tree attention against the oracle's explicit per-node attention.

Tolerances: bf16 inputs, float32 softmax/accumulation on the GPU, float64 in
the oracle: |gpu - ref| <= 2e-2 + 1e-2 |ref| (bf16 output rounding is 2^-9
relative, far inside); float32 inputs: 1e-4 + 1e-4 |ref|.
"""
import numpy as np
import pytest
import torch

from _util import dev, host, i32, within, zeros_i32
from oracle import attention as A
from oracle import tree as T
from tree_speculative_decoding_attn_gb300 import specverify as sv
from tree_speculative_decoding_attn_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 1e-2), "f32": (1e-4, 1e-4)}


def _run(w, shape, prefix, q, kc, vc, kt, vt, num_splits=0, max_prefix=None, repeats=1):
    """Runs tree_attn_verify ``repeats`` times (an L2 flush before each
    repeat after the first, so cold-cache timing is exercised too); returns
    the output and the device status of the last run."""
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    B, N = q.shape[0], q.shape[1]
    anc = np.broadcast_to(T.mask_words(T.depth_and_mask(shape.parents)[1]), (B, N)).copy()
    max_prefix = int(prefix.max()) if max_prefix is None else max_prefix
    ws_bytes = sv.tree_attn_workspace_bytes(tdt, B, N, w.hq, w.hkv, w.head_dim, max_prefix, num_splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    out = torch.full(q.shape, float("nan"), dtype=tdt, device="cuda")
    args = (dev(q, tdt), dev(kc, tdt), dev(vc, tdt), dev(kt, tdt), dev(vt, tdt), i32(prefix),
            dev(anc.view(np.int64)), out, max_prefix)
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda") if repeats > 1 else None
    for k in range(repeats):
        if k:
            flush.fill_(float(k))
        st = zeros_i32(1)
        sv.tree_attn_verify(*args, num_splits=num_splits, workspace=ws, dev_status=st)
        torch.cuda.synchronize()
        assert int(host(st)[0]) == 0 or k == repeats - 1, f"run {k}: status {int(host(st)[0])}"
    return host(out), int(host(st)[0]), anc


def _small(dtype, B, hq, hkv, D, prefix, shape, q_scale=1.0, seed=1):
    w = synth.Workload("t", seed, batch=B, hq=hq, hkv=hkv, head_dim=D, dtype=dtype, prefix=(0, 0),
                       n_nodes=shape.n, n_levels=shape.n_levels, vocab=10, accept="greedy", tree="random")
    prefix = np.asarray(prefix, np.int32)
    q, kc, vc, kt, vt = synth.attention_inputs(w, prefix, q_scale=q_scale, s_max=int(prefix.max()) + 70)
    return w, prefix, q, kc, vc, kt, vt


CASES = [
    # (dtype, B, hq, hkv, D, prefix per sequence, tree)
    ("f32", 1, 4, 4, 64, [128], synth.p4_example()),                       # the tiny exact workload
    ("bf16", 3, 16, 4, 128, [100, 37, 300], synth.random_tree(2, 24, (4, 3, 2))),
    ("bf16", 2, 8, 8, 64, [513, 1], synth.random_tree(3, 40, (6, 3, 2, 2))),
    ("f32", 2, 16, 2, 128, [257, 64], synth.random_tree(4, 32, (4, 3, 2))),  # 256 query rows / KV head
    ("bf16", 2, 16, 2, 128, [0, 5], synth.random_tree(5, 64, (8, 4, 3, 2, 2))),  # 512 rows, empty prefix
    ("bf16", 1, 4, 1, 128, [700], synth.chain(1)),                           # plain decode attention
    ("bf16", 2, 32, 8, 128, [1000, 4097], synth.chain(6)),
    ("bf16", 2, 64, 8, 128, [4096, 1111], synth.random_tree(7, 32, (4, 3, 2))),      # 256 rows per KV head
    ("bf16", 1, 32, 32, 128, [2048], synth.random_tree(8, 64, (10, 10, 10, 10))),    # MHA, 64 rows
    ("bf16", 3, 32, 8, 128, [513, 8192, 129], synth.random_tree(9, 60, (10, 4, 3, 2, 2))),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("q_scale", [1.0, 4.0])
def test_tree_attention_small(case, splits, q_scale):
    dtype, B, hq, hkv, D, prefix, shape = CASES[case]
    w, prefix, q, kc, vc, kt, vt = _small(dtype, B, hq, hkv, D, prefix, shape, q_scale, seed=case)
    got, status, anc = _run(w, shape, prefix, q, kc, vc, kt, vt, num_splits=splits)
    assert status == 0
    ref = A.tree_attention(q, kc, vc, kt, vt, prefix, T.depth_and_mask(shape.parents)[1])
    ok, excess = within(got, ref, *TOL[dtype])
    assert ok, f"max excess over tolerance {excess}"


def test_growing_scores_force_rescaling():
    """Keys whose norm grows along the prefix make each tile's row max
    exceed the running one, so the running output is rescaled many times."""
    w, prefix, q, kc, vc, kt, vt = _small("bf16", 2, 16, 4, 128, [1500, 700], synth.random_tree(3, 16, (4, 3)),
                                          q_scale=2.0, seed=21)
    grow = (1.0 + np.arange(kc.shape[2]) / 96.0).astype(np.float32)
    kc = synth.round_bf16(kc * grow[None, None, :, None])
    shape = synth.random_tree(3, 16, (4, 3))
    for splits in (1, 2):
        got, status, _ = _run(w, shape, prefix, q, kc, vc, kt, vt, num_splits=splits)
        assert status == 0
        ref = A.tree_attention(q, kc, vc, kt, vt, prefix, T.depth_and_mask(shape.parents)[1])
        ok, excess = within(got, ref, *TOL["bf16"])
        assert ok, f"max excess over tolerance {excess}"


def test_jumping_scores_force_the_exact_redo_and_rescale_on_sm_pairs():
    """Prefix keys scaled by 1.5 per 128-key tile on the SM-pair kernel (64
    nodes x 4 heads = 256 rows per KV head): from about the sixth tile on,
    each tile's scores exceed the running max by more than 2^16, so the
    one-pass tile fails its row-sum test, is redone with the exact max and O
    is rescaled, tile after tile."""
    shape = synth.random_tree(5, 64, (4, 4, 4))
    w, prefix, q, kc, vc, kt, vt = _small("bf16", 2, 16, 4, 128, [1200, 900], shape, q_scale=1.0, seed=23)
    f = (1.5 ** (np.arange(kc.shape[2]) // 128)).astype(np.float32)
    kc = synth.round_bf16(kc * f[None, None, :, None])
    for splits in (1, 0):
        got, status, _ = _run(w, shape, prefix, q, kc, vc, kt, vt, num_splits=splits)
        assert status == 0
        ref = A.tree_attention(q, kc, vc, kt, vt, prefix, T.depth_and_mask(shape.parents)[1])
        ok, excess = within(got, ref, *TOL["bf16"])
        assert ok, f"max excess over tolerance {excess}"
        assert np.abs(ref).max() > 0.1


def test_non_finite_stale_cache_rows_are_ignored():
    """Cache rows past the prefix hold NaN/Inf (never-written memory): the
    output must not see them."""
    shape = synth.random_tree(4, 24, (4, 3, 2))
    w, prefix, q, kc, vc, kt, vt = _small("bf16", 2, 32, 8, 128, [300, 77], shape, seed=22)
    for b, p in enumerate(prefix):
        kc[b, :, p:] = np.nan
        vc[b, :, p:] = np.inf
    got, status, _ = _run(w, shape, prefix, q, kc, vc, kt, vt)
    assert status == 0 and np.isfinite(got).all()
    kc2, vc2 = np.nan_to_num(kc, nan=0.0, posinf=0.0), np.nan_to_num(vc, nan=0.0, posinf=0.0)
    ref = A.tree_attention(q, kc2, vc2, kt, vt, prefix, T.depth_and_mask(shape.parents)[1])
    assert within(got, ref, *TOL["bf16"])[0]


def test_prefix_beyond_bound_is_reported():
    w, prefix, q, kc, vc, kt, vt = _small("bf16", 2, 8, 2, 128, [50, 60], synth.p4_example())
    got, status, _ = _run(w, synth.p4_example(), prefix, q, kc, vc, kt, vt, max_prefix=55)
    assert status == sv.DEV_CAPACITY
    ref = A.tree_attention(q[:1], kc[:1], vc[:1], kt[:1], vt[:1], prefix[:1], T.depth_and_mask(synth.P4_PARENTS)[1])
    assert within(got[:1], ref, *TOL["bf16"])[0]          # the in-bound sequence is still computed


def test_one_row_group_across_every_cluster():
    """One (sequence, KV head) of 256 query rows with a 20000-key prefix:
    its single row group is cut into one part per cluster of the persistent
    grid (more than 32), so the merge folds its contributors in rounds."""
    shape = synth.random_tree(31, 32, (4, 3, 2))
    w, prefix, q, kc, vc, kt, vt = _small("bf16", 1, 8, 1, 128, [20000], shape, seed=31)
    got, status, _ = _run(w, shape, prefix, q, kc, vc, kt, vt, repeats=2)
    assert status == 0
    ref = A.tree_attention(q, kc, vc, kt, vt, prefix, T.depth_and_mask(shape.parents)[1])
    assert within(got, ref, *TOL["bf16"])[0]


def test_pair_shape_prefix_beyond_bound_is_reported():
    """256 query rows per KV head (the SM-pair kernel): a sequence whose
    prefix exceeds max_prefix is reported, the others are still computed."""
    shape = synth.random_tree(32, 32, (4, 3, 2))
    w, prefix, q, kc, vc, kt, vt = _small("bf16", 3, 16, 2, 128, [300, 900, 2000], shape, seed=32)
    got, status, _ = _run(w, shape, prefix, q, kc, vc, kt, vt, max_prefix=1000)
    assert status == sv.DEV_CAPACITY
    ref = A.tree_attention(q[:2], kc[:2], vc[:2], kt[:2], vt[:2], prefix[:2], T.depth_and_mask(shape.parents)[1])
    assert within(got[:2], ref, *TOL["bf16"])[0]


FULL = ["vicuna7b_medusa", "llama8b_eagle2", "llama70b_serving", "long_context"]


@pytest.mark.parametrize("name", FULL)
def test_tree_attention_full_size_sampled(name):
    """The workload's full shapes in the default launch configuration;
    48 sampled (sequence, node, head) outputs against the oracle, plus
    properties of every output (finite, bounded by the value range)."""
    w = synth.WORKLOADS[name]
    shape = synth.random_tree(w.seed, w.n_nodes, w.caps if w.caps else (10, 4, 3, 2, 2))
    prefix = synth.prefix_lengths(w)
    q, kc, vc, kt, vt = synth.attention_inputs(w, prefix, q_scale=2.0)
    got, status, _ = _run(w, shape, prefix, q, kc, vc, kt, vt, repeats=3)
    assert status == 0
    assert np.isfinite(got).all()
    assert np.abs(got).max() <= max(np.abs(vc).max(), np.abs(vt).max()) * 1.01
    g = np.random.default_rng(0)
    mask = T.depth_and_mask(shape.parents)[1]
    for _ in range(48):
        b, i, h = int(g.integers(w.batch)), int(g.integers(w.n_nodes)), int(g.integers(w.hq))
        ref = A.tree_attention(q[b:b + 1], kc[b:b + 1], vc[b:b + 1], kt[b:b + 1], vt[b:b + 1], prefix[b:b + 1],
                               mask, nodes=[i], heads=[h])[0, i, h]
        ok, excess = within(got[b, i, h], ref, *TOL["bf16"])
        assert ok, (b, i, h, excess)
