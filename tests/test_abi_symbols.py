"""The C-ABI library builds, loads without a GPU and exports every declared entry point."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(cpp_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib_path():
    from chunked_prefill_paged_slot_gb300 import build as b
    return b.build()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["cpp_kv_cache_write", "cpp_chunked_prefill_attn", "cpp_split_microbatch",
              "cpp_attn_workspace_bytes", "cpp_read_device_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_only_entry_points_without_gpu(lib_path):
    """Status strings, workspace sizing and the planner need no device."""
    import chunked_prefill_paged_slot_gb300 as cpsa
    lib = cpsa.load()
    assert lib.cpp_status_string(0) == b"ok"
    full = cpsa.cpp_attn_workspace_bytes(1537, 2048, 32, 8, 128, 8)
    small = cpsa.cpp_attn_workspace_min_bytes(1537, 2048, 32, 8, 128, 8)
    assert full > small > 0
    assert lib.cpp_attn_workspace_bytes(1, 16, 32, 8, 96, 8) == 0      # head_dim 96 unsupported
    assert lib.cpp_attn_workspace_bytes(1, 16, 30, 8, 128, 8) == 0     # 30 % 8 != 0
