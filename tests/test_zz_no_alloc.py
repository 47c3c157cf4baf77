"""tree_attn_verify_noalloc: the same tree attention for callers that cannot
allocate device memory (a plugin that is handed only its input and output
buffers by a host runtime owning all device memory, or a serving loop that
bans cudaMalloc/cudaFree after start-up because they synchronise the device).
Its split-KV partials live in the library's own fixed device array.

Called through the C ABI twice in a row, with different inputs, and compared
each time with tree_attn_verify given a caller-allocated workspace, within the
tolerance of the other attention tests.  Kept in a file of its own that
pytest collects last.
"""
import numpy as np
import pytest
import torch

from _util import dev, host, i32, within, zeros_i32
from oracle import tree as T
from tree_speculative_decoding_attn_gb300 import specverify as sv
from tree_speculative_decoding_attn_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = (2e-2, 1e-2)


def _inputs(seed, B=1, hq=32, hkv=32, D=128, P=2048, n=64, caps=(10, 10, 10, 10)):
    w = synth.Workload("noalloc", seed, batch=B, hq=hq, hkv=hkv, head_dim=D, dtype="bf16", prefix=(P, P),
                       n_nodes=n, n_levels=len(caps) + 1, vocab=10, accept="greedy", tree="random")
    shape = synth.random_tree(seed, n, caps)
    prefix = synth.prefix_lengths(w)
    q, kc, vc, kt, vt = synth.attention_inputs(w, prefix, q_scale=2.0)
    anc = np.broadcast_to(T.mask_words(T.depth_and_mask(shape.parents)[1]), (B, n)).copy()
    bf = torch.bfloat16
    return dict(q=dev(q, bf), kc=dev(kc, bf), vc=dev(vc, bf), kt=dev(kt, bf), vt=dev(vt, bf), prefix=i32(prefix),
                anc=dev(anc.view(np.int64)), max_prefix=int(prefix.max()))


def test_noalloc_matches_workspace_entry_point_twice():
    splits = 4                                      # forces split-KV partials (scratch in use)
    for call, seed in enumerate((11, 12)):
        x = _inputs(seed)
        need = sv.tree_attn_workspace_bytes(torch.bfloat16, 1, 64, 32, 32, 128, x["max_prefix"], splits)
        assert 0 < need <= sv.NOALLOC_SCRATCH_BYTES
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(x["q"])
        got = torch.full_like(x["q"], float("nan"))
        st = zeros_i32(1)
        sv.tree_attn_verify(x["q"], x["kc"], x["vc"], x["kt"], x["vt"], x["prefix"], x["anc"], ref, x["max_prefix"],
                            num_splits=splits, workspace=ws, dev_status=st)
        sv.tree_attn_verify_noalloc(x["q"], x["kc"], x["vc"], x["kt"], x["vt"], x["prefix"], x["anc"], got,
                                    x["max_prefix"], num_splits=splits, dev_status=st)
        torch.cuda.synchronize()
        assert int(host(st)[0]) == 0, f"call {call}"
        ok, excess = within(host(got), host(ref), *TOL)
        assert ok, f"call {call}: max excess {excess}"


def test_noalloc_sm_pair_path_matches_twice():
    """The 70B serving shape (64 query / 8 KV heads, 32 nodes: 256 query rows
    per KV head) runs on the SM-pair kernel, whose partial rows of cut row
    groups and cut descriptors also live in the fixed array."""
    B, hq, hkv, n = 16, 64, 8, 32
    for call, seed in enumerate((21, 22)):
        x = _inputs(seed, B=B, hq=hq, hkv=hkv, P=1000 + 300 * call, n=n, caps=(4, 3, 2))
        need = sv.tree_attn_workspace_bytes(torch.bfloat16, B, n, hq, hkv, 128, x["max_prefix"])
        assert 0 < need <= sv.NOALLOC_SCRATCH_BYTES
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(x["q"])
        got = torch.full_like(x["q"], float("nan"))
        st = zeros_i32(1)
        sv.tree_attn_verify(x["q"], x["kc"], x["vc"], x["kt"], x["vt"], x["prefix"], x["anc"], ref, x["max_prefix"],
                            workspace=ws, dev_status=st)
        sv.tree_attn_verify_noalloc(x["q"], x["kc"], x["vc"], x["kt"], x["vt"], x["prefix"], x["anc"], got,
                                    x["max_prefix"], dev_status=st)
        torch.cuda.synchronize()
        assert int(host(st)[0]) == 0, f"call {call}"
        ok, excess = within(host(got), host(ref), *TOL)
        assert ok, f"call {call}: max excess {excess}"


def test_noalloc_rejects_work_beyond_its_scratch():
    """64 KV splits of a 16384-token prefix need 68 MB of partials, more than
    the fixed array holds: refused before anything is launched.  The buffers
    are sized for these arguments all the same."""
    x = _inputs(13, P=16384)
    need = sv.tree_attn_workspace_bytes(torch.bfloat16, 1, 64, 32, 32, 128, x["max_prefix"], 64)
    assert need > sv.NOALLOC_SCRATCH_BYTES
    out = torch.empty_like(x["q"])
    with pytest.raises(sv.SpecError) as e:
        sv.tree_attn_verify_noalloc(x["q"], x["kc"], x["vc"], x["kt"], x["vt"], x["prefix"], x["anc"], out,
                                    x["max_prefix"], num_splits=64)
    assert e.value.code == sv.ERR_CAPACITY


def test_noalloc_256_node_tree_matches():
    """A dense 256-node tree (two tree tiles, four ancestor words per node)
    on the SM-pair kernel through the fixed array."""
    B, hq, hkv, n = 2, 16, 4, 256
    shape = synth.dense_tree((4, 4, 4, 4), n)
    w = synth.Workload("noalloc256", 31, batch=B, hq=hq, hkv=hkv, head_dim=128, dtype="bf16", prefix=(700, 1900),
                       n_nodes=n, n_levels=shape.n_levels, vocab=10, accept="greedy", tree="random")
    prefix = synth.prefix_lengths(w)
    q, kc, vc, kt, vt = synth.attention_inputs(w, prefix, q_scale=2.0)
    W = sv.mask_words(n)
    anc = np.broadcast_to(T.mask_words_multi(T.depth_and_mask(shape.parents)[1]), (B, n, W)).copy()
    bf = torch.bfloat16
    x = dict(q=dev(q, bf), kc=dev(kc, bf), vc=dev(vc, bf), kt=dev(kt, bf), vt=dev(vt, bf), prefix=i32(prefix),
             anc=dev(anc.view(np.int64)), max_prefix=int(prefix.max()))
    need = sv.tree_attn_workspace_bytes(bf, B, n, hq, hkv, 128, x["max_prefix"])
    assert 0 < need <= sv.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(x["q"])
    got = torch.full_like(x["q"], float("nan"))
    st = zeros_i32(1)
    sv.tree_attn_verify(x["q"], x["kc"], x["vc"], x["kt"], x["vt"], x["prefix"], x["anc"], ref, x["max_prefix"],
                        workspace=ws, dev_status=st)
    sv.tree_attn_verify_noalloc(x["q"], x["kc"], x["vc"], x["kt"], x["vt"], x["prefix"], x["anc"], got,
                                x["max_prefix"], dev_status=st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
    ok, excess = within(host(got), host(ref), *TOL)
    assert ok, f"max excess {excess}"
