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
    assert sv.spec_abi_version() == 1
