"""Malformed arguments are refused at the C-ABI boundary with a status, before
any launch (host-side failure injection, no GPU).

Every case below breaks a rule that each entry point checks on the host
before its first CUDA call, so the placeholder device addresses are never
dereferenced.  The test is skipped where a GPU is visible: there a
validation order changed by mistake could hand a placeholder to a kernel.
"""
import pytest
import torch

from tree_speculative_decoding_attn_gb300 import _build
from tree_speculative_decoding_attn_gb300 import specverify as sv

pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="placeholder pointers only on a GPU-less host")

P = 0x100000          # 16-byte aligned placeholder address
MIS = 0x100004        # not 16-byte aligned
NULL = None
INV, UNS, CAP = sv.ERR_INVALID_ARG, sv.ERR_UNSUPPORTED, sv.ERR_CAPACITY
# one sequence, 32 heads of MHA, 64 nodes, prefix 2048: the single-CTA
# kernel with several KV splits, whose workspace size is a host computation
MHA = dict(B=1, N=64, hq=32, hkv=32, s_max=4096, max_prefix=2048)


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sv.load()


def _attn(lib, q=P, kc=P, dtype=sv.BF16, B=2, N=32, hq=16, hkv=2, D=128, s_max=1024, max_prefix=512,
          ws=NULL, ws_bytes=0, noalloc=False):
    if noalloc:
        return lib.tree_attn_verify_noalloc(q, kc, P, P, P, P, P, P, dtype, B, N, hq, hkv, D, s_max, max_prefix,
                                            0.0, 0, NULL, NULL)
    return lib.tree_attn_verify(q, kc, P, P, P, P, P, P, dtype, B, N, hq, hkv, D, s_max, max_prefix, 0.0, 0,
                                ws, ws_bytes, NULL, NULL)


@pytest.mark.parametrize("kw,code", [
    (dict(q=NULL), INV),
    (dict(kc=NULL), INV),
    (dict(dtype=7), UNS),
    (dict(hq=12, hkv=8), INV),                 # query heads not a multiple of KV heads
    (dict(D=96), UNS),
    (dict(N=257), UNS),                        # more nodes than the largest tree
    (dict(hq=128, hkv=8, N=64), UNS),          # 1024 query rows per KV head; 512 is the limit up to 64 nodes
    (dict(hq=16, hkv=1, N=200), UNS),          # 3200 rows per KV head; 2048 above 64 nodes
    (dict(B=0), INV),
    (dict(max_prefix=2048), CAP),              # prefix beyond the cache's capacity
    (dict(q=MIS), INV),
    (dict(MHA), CAP),                          # split KV needs a workspace; none given
    (dict(MHA, ws=P, ws_bytes=16), CAP),       # ... or one too small
    (dict(MHA, ws=MIS, ws_bytes=1 << 30), CAP),  # ... or one not 16-byte aligned
    (dict(hq=12, hkv=8, noalloc=True), INV),
    (dict(D=96, noalloc=True), UNS),
])
def test_tree_attn_verify_refuses(lib, kw, code):
    assert _attn(lib, **kw) == code


def test_workspace_query_is_zero_for_bad_shapes(lib):
    assert lib.tree_attn_workspace_bytes(sv.BF16, 2, 32, 12, 8, 128, 512, 0) == 0
    assert lib.tree_attn_workspace_bytes(sv.BF16, 2, 257, 16, 2, 128, 512, 0) == 0
    assert lib.tree_attn_workspace_bytes(sv.BF16, 1, 64, 32, 32, 128, 2048, 0) > 0


def _accept(lib, mode=sv.GREEDY, logits=P, draft=NULL, dtype=sv.BF16, B=2, N=16, V=1000, T=1.0, cap=8):
    return lib.spec_accept(mode, logits, draft, dtype, B, N, V, P, P, P, P, T, 0.3, 0.09, 1, 0, cap, P, P, P, NULL,
                           NULL)


@pytest.mark.parametrize("kw,code", [
    (dict(logits=NULL), INV),
    (dict(mode=4), INV),
    (dict(mode=sv.REJECT_STOCHASTIC), INV),            # stochastic siblings need the drafter's logits
    (dict(mode=sv.REJECT, draft=P), INV),              # ... and only that mode takes them
    (dict(mode=sv.REJECT_STOCHASTIC, draft=P, T=0.0), INV),
    (dict(dtype=5), UNS),
    (dict(N=257), UNS),
    (dict(V=0), INV),
    (dict(cap=0), INV),
    (dict(mode=sv.TYPICAL, T=0.0), INV),
    (dict(mode=sv.REJECT, T=-1.0), INV),
    (dict(mode=sv.REJECT, T=float("nan")), INV),
])
def test_spec_accept_refuses(lib, kw, code):
    assert _accept(lib, **kw) == code


def _commit(lib, kc=P, elem=2, layers=1, B=2, hkv=2, s_max=64, N=16, D=128, cap=8, prefix=P):
    return lib.kv_commit(kc, P, P, P, elem, layers, B, hkv, s_max, N, D, P, P, cap, prefix, NULL, NULL, NULL)


@pytest.mark.parametrize("kw,code", [
    (dict(kc=NULL), INV),
    (dict(prefix=NULL), INV),
    (dict(elem=3), UNS),
    (dict(layers=0), INV),
    (dict(N=257), UNS),
    (dict(cap=258), UNS),
    (dict(D=6), UNS),                          # a row of 12 bytes is not a whole number of 16-byte copies
    (dict(kc=MIS), INV),
])
def test_kv_commit_refuses(lib, kw, code):
    assert _commit(lib, **kw) == code


def test_build_tree_refuses(lib):
    # static: parents, rank, cand_tok, levels, s, root_tok, prefix_len, batch, n, tok, depth, pos, anc, fc, ns
    args = [P, P, P, 3, 4, P, P, 2, 16, P, P, P, P, P, P, NULL, NULL]
    assert lib.spec_build_tree(*args[:7], 2, 257, *args[9:]) == UNS
    assert lib.spec_build_tree(NULL, *args[1:]) == INV
    assert lib.spec_build_tree(P, NULL, *args[2:]) == INV          # candidate tokens without ranks
    assert lib.spec_build_tree(*args[:4], 0, *args[5:]) == INV     # zero candidates per level
    # dynamic: pool of fewer nodes than the tree, pool above the limit
    dyn = lambda M, N: lib.spec_build_tree_dynamic(P, P, P, M, P, 2, N, P, P, P, P, P, P, P, NULL, NULL, NULL,
                                                   NULL)
    assert dyn(10, 16) == INV
    assert dyn(4097, 16) == UNS
    assert dyn(300, 257) == UNS


def test_heads_topk_expand_lm_head_refuse(lib):
    heads = lambda h=P, B=1, d=4096, ws=P, nbytes=1 << 30: lib.spec_medusa_heads(h, P, NULL, P, B, 4, d, 32000, P, P,
                                                                                 ws, nbytes, NULL, NULL)
    assert heads(B=0) == INV                                                              # no rows
    assert heads(d=4100) == INV                                                           # hidden not a multiple of 64
    assert heads(h=MIS) == INV                                                            # misaligned input
    assert heads(ws=NULL) == INV                                                          # no workspace
    assert heads(nbytes=16) == CAP                                                        # workspace too small
    assert lib.spec_medusa_heads_workspace_bytes(64, 4, 4096, 32000) > 0
    assert lib.spec_medusa_heads_workspace_bytes(0, 4, 4096, 32000) == 0
    assert lib.spec_topk(P, sv.F32, 4, 1000, 1000, 17, P, P, NULL) == UNS                # s above 16
    assert lib.spec_topk(P, sv.F32, 4, 1000, 999, 10, P, P, NULL) == INV                 # stride below the row
    assert lib.spec_topk(P, sv.F32, 4, 8, 8, 9, P, P, NULL) == INV                       # s above the row
    assert lib.spec_tree_expand(P, sv.BF16, 2, 10, 1000, P, 17, 1.0, P, P, P, P, P, 512, P, 10, NULL,
                                NULL) == UNS
    assert lib.spec_tree_expand(P, sv.BF16, 2, 10, 1000, P, 10, 0.0, P, P, P, P, P, 512, P, 10, NULL,
                                NULL) == INV
    assert lib.spec_lm_head(P, P, 64, 100, 32000, P, P, 1 << 30, NULL, NULL) == INV       # hidden not a multiple of 64
    assert lib.spec_lm_head(P, P, 64, 4096, 32000, P, P, 16, NULL, NULL) == CAP          # workspace too small
    assert lib.spec_lm_head(P, P, 64, 4096, 32000, P, NULL, 1 << 30, NULL, NULL) == INV  # no workspace


def test_refusal_codes_have_their_texts(lib):
    assert _attn(lib, q=NULL) == INV and lib.spec_status_string(INV) == b"invalid argument"
    assert _attn(lib, D=96) == UNS and b"unsupported" in lib.spec_status_string(UNS)
    assert _attn(lib, max_prefix=2048) == CAP and b"capacity" in lib.spec_status_string(CAP)


def test_paged_batch_and_fused_entry_points_refuse(lib):
    # tree_attn_verify_paged(q, kp, vp, table, bs, nb, max_blocks, kt, vt, prefix, anc, out, dtype, B, N, hq, hkv,
    #                        D, max_prefix, scale, splits, ws, ws_bytes, status, stream)
    paged = lambda bs=128, nb=8, mb=4, table=P, mp=256, N=16: lib.tree_attn_verify_paged(
        P, P, P, table, bs, nb, mb, P, P, P, P, P, sv.BF16, 2, N, 16, 2, 128, mp, 0.0, 0, P, 1 << 30, NULL, NULL)
    assert paged(bs=64) == INV                   # blocks must hold whole 128-key tiles
    assert paged(table=NULL) == INV
    assert paged(nb=0) == INV
    assert paged(mp=600) == CAP                  # prefix beyond max_blocks * block_size
    assert paged(N=257) == UNS
    # kv_commit_paged(kp, vp, table, bs, nb, mb, kt, vt, esz, layers, B, hkv, N, D, len, path, cap, prefix, out, st, s)
    commit = lambda esz=2, table=P, D=128, cap=8: lib.kv_commit_paged(
        P, P, table, 128, 8, 4, P, P, esz, 1, 2, 2, 16, D, P, P, cap, P, NULL, NULL, NULL)
    assert commit(table=NULL) == INV
    assert commit(esz=3) == UNS
    assert commit(D=6) == UNS
    assert commit(cap=300) == UNS
    # spec_build_tree_batch(parents, n_valid, tok_in, prefix, B, N, tok, depth, pos, anc, fc, ns, status, stream)
    batch = lambda par=P, N=16, tok_in=NULL, tok=NULL: lib.spec_build_tree_batch(
        par, NULL, tok_in, P, 2, N, tok, P, P, P, P, P, NULL, NULL)
    assert batch(par=NULL) == INV
    assert batch(N=257) == UNS
    assert batch(tok_in=P) == INV                # tokens given but nowhere to copy them
    # spec_lm_head_accept(mode, hid, w, B, N, hidden, V, tok, par, fc, ns, T, eps, delta, cap, len, path, bonus,
    #                     ws, ws_bytes, status, stream)
    fused = lambda mode=sv.GREEDY, d=4096, ws_bytes=1 << 30, T=1.0: lib.spec_lm_head_accept(
        mode, P, P, 1, 64, d, 32000, P, P, P, P, T, 0.3, 0.09, 6, P, P, P, P, ws_bytes, NULL, NULL)
    assert fused(mode=sv.REJECT) == UNS          # rejection needs the whole residual row
    assert fused(mode=sv.REJECT_STOCHASTIC) == UNS
    assert fused(d=4100) == INV
    assert fused(mode=sv.TYPICAL, T=0.0) == INV
    assert fused(ws_bytes=16) == CAP
