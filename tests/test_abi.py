"""libmi.so loads on a GPU-less host and exports every entry point of include/mi.h."""
import ctypes
import os
import re

import pytest

from dynamic_sparse_attention_vertical_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "mi.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(mi_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return B.load()


def test_header_declares_the_five_calls():
    names = _declared()
    for n in ("mi_vs_estimate", "mi_vs_sparse_attn", "mi_block_sparse_attn", "mi_ashape_attn",
              "mi_dense_causal_attn"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) == set(B.SYMBOLS)
    raw = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_strerror_and_workspace_sizes_need_no_gpu(lib):
    assert B.mi_strerror(0) == "success"
    for code in range(-8, 0):
        assert B.mi_strerror(code) and "unknown" not in B.mi_strerror(code)
    assert B.mi_workspace_bytes(B.MI_OP_DENSE_CAUSAL_ATTN, 32, 8, 4096) == 256
    est = B.mi_workspace_bytes(B.MI_OP_VS_ESTIMATE, 32, 8, 131072)
    assert est >= 2 * 32 * 131072 * 4 and est % 256 == 0
    vs = B.mi_workspace_bytes(B.MI_OP_VS_SPARSE_ATTN, 24, 8, 131072)
    assert vs >= 2 * 24 * 131072 // 8
    assert B.mi_workspace_bytes(99, 1, 1, 64) == 0


def test_fault_injection_argument_checks(lib):
    assert B.mi_debug_inject(7, 1000) == B.MI_ERR_ARG
    assert B.mi_debug_inject(B.MI_FAULT_SKIP_Q_LOAD, 0) == B.MI_ERR_ARG
    assert B.mi_debug_inject(B.MI_FAULT_NONE, 0) == B.MI_OK


def test_layer_workspace_sizes_need_no_gpu(lib):
    H = B.HeadCfg
    cfg = [H.dense(), H.vs(64, 32), H.vs(128, 16), H.block(8), H.ashape(128, 512), H.skip(), H.skip(), H.skip()]
    n = B.mi_layer_workspace_bytes(8, 2, 4096, cfg)
    assert n > 0 and n % 256 == 0
    # more vertical-slash budget never needs less workspace
    cfg2 = list(cfg)
    cfg2[2] = H.vs(1000, 2000)
    assert B.mi_layer_workspace_bytes(8, 2, 4096, cfg2) >= n
    bad = list(cfg)
    bad[0] = B.HeadCfg(7, 0, 0, 0, 0, 0, 0)
    assert B.mi_layer_workspace_bytes(8, 2, 4096, bad) == 0
    assert B.mi_layer_workspace_bytes(8, 2, 4096, [H.skip()] * 8) == 0
    mixed_flags = list(cfg)
    mixed_flags[2] = H.vs(128, 16, expanded=True)
    assert B.mi_layer_workspace_bytes(8, 2, 4096, mixed_flags) == 0


def test_varlen_workspace_sizes_need_no_gpu(lib):
    H = B.HeadCfg
    cfg = [H.vs(64, 32), H.block(8), H.ashape(128, 512), H.dense()]
    n = B.mi_layer_workspace_bytes_varlen(4, 2, [0, 1000, 1081, 3581], cfg)
    assert n > 0 and n % 256 == 0
    # the workspace is that of the longest sequence
    assert n == B.mi_layer_workspace_bytes(4, 2, 2500, cfg)
    for bad in ([1, 1000], [0, 500, 400], [0]):
        assert B.mi_layer_workspace_bytes_varlen(4, 2, bad, cfg) == 0


def test_binding_constants_match_the_header():
    """Every MI_* integer constant the binding mirrors has the header's value."""
    with open(os.path.join(ROOT, "include", "mi.h")) as f:
        text = f.read()
    defined = {m.group(1): int(m.group(2))
               for m in re.finditer(r"^#define\s+(MI_\w+)\s+\(?(-?\d+)\)?", text, re.M)}
    mirrored = {n: getattr(B, n) for n in dir(B) if n.startswith("MI_") and isinstance(getattr(B, n), int)}
    common = sorted(set(defined) & set(mirrored))
    assert "MI_MAX_KV" in common and "MI_VS_BLOCK_EXPANDED" in common
    for n in common:
        assert mirrored[n] == defined[n], n
