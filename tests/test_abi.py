"""The C-ABI library builds, loads and exports every symbol its header declares (no GPU)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "specverify.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def built_lib():
    from tree_speculative_decoding_attn_gb300 import _build, specverify
    _build.build()
    return specverify.load()


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("spec_build_tree", "tree_attn_verify", "spec_accept", "kv_commit"):
        assert must in names


def test_library_exports_every_declared_symbol(built_lib):
    for name in _declared():
        assert hasattr(built_lib, name), name


def test_binding_covers_every_declared_symbol():
    from tree_speculative_decoding_attn_gb300 import specverify
    assert specverify.exported_symbols() == _declared()


def test_status_strings_without_gpu(built_lib):
    from tree_speculative_decoding_attn_gb300 import specverify as sv
    assert sv.spec_status_string(0) == "ok"
    assert "invalid" in sv.spec_status_string(1)
    assert sv.spec_abi_version() == 2


def test_split_planner_is_host_only_and_sane(built_lib):
    """tree_attn_plan_splits runs on the host.  Shapes with more than 128
    query rows per KV head go to the SM-pair kernel, which balances its own
    work (one "split"); for the single-CTA kernel a few long ragged
    sequences are split; bad arguments return an error."""
    import torch
    from tree_speculative_decoding_attn_gb300 import specverify as sv
    bf = torch.bfloat16
    ragged = [512, 8192, 1024, 3000, 700, 6000, 2048, 4000]
    assert sv.tree_attn_plan_splits(bf, 64, 32, 64, 8, 128, [4096] * 64) == 1
    assert sv.tree_attn_plan_splits(bf, 8, 60, 32, 8, 128, ragged) == 1
    assert sv.tree_attn_plan_splits(bf, 4, 64, 32, 8, 128, [32768] * 4) == 1
    assert sv.tree_attn_plan_splits(bf, 2, 64, 32, 32, 128, [8192, 600]) > 1       # MHA: 64 rows per KV head
    assert 1 <= sv.tree_attn_plan_splits(torch.float32, 1, 5, 4, 4, 64, [128]) <= 64
    with pytest.raises(sv.SpecError):
        sv.tree_attn_plan_splits(bf, 2, 257, 8, 8, 128, [10, 10])    # more than 256 tree nodes
