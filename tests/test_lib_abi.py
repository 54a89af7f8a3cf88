"""The C-ABI library builds, loads and exports every declared symbol (no GPU
compute)."""

import os
import re

import pytest

from tree_verify_attention_gb300 import _lib
from tree_verify_attention_gb300 import build as B

HEADER = os.path.join(B.ROOT, "include", "dfv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dfv_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name


def test_binding_table_matches_header():
    assert set(_lib.SIGNATURES) == set(declared_functions())


def test_status_strings_and_version(lib):
    assert lib.dfv_status_string(0) == b"ok"
    assert lib.dfv_status_string(3) == b"workspace too small"
    assert lib.dfv_version() >= 100


def test_host_side_rejections(lib):
    # invalid shapes are rejected before any device call
    assert lib.dfv_tree_verify_attn_workspace_bytes(0, 24, 4, 256, 2048, 100) == 0
    assert lib.dfv_tree_verify_attn_workspace_bytes(66, 24, 4, 256, 2048, 100) == 0
    assert lib.dfv_tree_verify_attn_workspace_bytes(23, 24, 5, 256, 2048, 100) == 0
    assert lib.dfv_tree_verify_attn_workspace_bytes(23, 24, 4, 96, 2048, 100) == 0
    assert lib.dfv_greedy_accept_workspace_bytes(0, 10) == 0
    st = lib.dfv_greedy_accept(23, 100, 0, None, None, None, None, None, None, None, None, 0,
                               None, None)
    assert st == 1  # DFV_ERR_INVALID
    st = lib.dfv_kv_commit(23, 4, 256, 3, 100, None, None, None, None, None, None, None, None,
                           None)
    assert st == 2  # DFV_ERR_UNSUPPORTED (format)
    st = lib.dfv_kv_quantize_rows(4, 96, 2, 100, 0, 1, None, 0, 1, 1, None, None)
    assert st == 2


def test_header_constants_match_binding():
    """The binding's format codes, flags and status bits are the header's."""
    from tree_verify_attention_gb300 import api
    text = open(HEADER).read()
    defs = {m.group(1): int(m.group(2), 0)
            for m in re.finditer(r"#define\s+(DFV_\w+)\s+(0x[0-9a-fA-F]+|\d+)u?\b", text)}
    assert defs["DFV_KV_F16"] == api.KV_F16
    assert defs["DFV_KV_Q4_0"] == api.KV_Q4_0
    assert defs["DFV_KV_TREE_AS_CACHE"] == api.KV_TREE_AS_CACHE
    assert defs["DFV_STEP_PIPELINED"] == api.STEP_PIPELINED
    assert defs["DFV_DTYPE_F32"] == api.DTYPE_F32 and defs["DFV_DTYPE_BF16"] == api.DTYPE_BF16
    assert defs["DFV_MAX_NODES"] == api.MAX_NODES
    for name in ("BAD_TREE", "DEPTH", "CAPACITY", "CTX", "BAD_PATH", "TIMEOUT"):
        assert defs["DFV_DEV_" + name] == getattr(api, "DEV_" + name), name
    # flags sit above the format byte and do not overlap
    assert api.KV_TREE_AS_CACHE & 0xFF == 0 and api.STEP_PIPELINED & 0xFF == 0
    assert api.KV_TREE_AS_CACHE & api.STEP_PIPELINED == 0


def test_unknown_step_flag_rejected(lib):
    # a flag bit the library does not know is refused before any device call
    st = lib.dfv_verify_step(23, 16, 24, 4, 256, 2048, 2 | 0x400, 100, 1000, 1, None, None,
                             None, None, None, None, None, None, None, 0.0, None, None, None,
                             None, None, None, None, 0, None, None)
    assert st == 2  # DFV_ERR_UNSUPPORTED
    st = lib.dfv_tree_verify_attn(23, 16, 24, 4, 256, 2048, 2 | 0x800, 100, None, None, None,
                                  None, None, None, None, 0.0, None, None, None, 0, None, None)
    assert st == 2


def test_tree_mask_host_rejections(lib):
    # bad node counts and missing buffers are refused before any launch
    for n in (0, 66, -1):
        assert lib.dfv_build_tree_mask(n, None, None, None, None, None) == 1
    assert lib.dfv_build_tree_mask(5, None, None, None, None, None) == 1
