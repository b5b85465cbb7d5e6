"""The C ABI library builds, loads without a GPU, and exports every entry point
that include/ula.h declares; the binding mirrors the declared structs."""
from __future__ import annotations

import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ula.h")


@pytest.fixture(scope="module")
def libpath():
    from serving_step_sparse_gb300.build import build
    return build()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(ula_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("ula_create", "ula_alloc", "ula_free", "ula_step_group", "ula_sync"):
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    lib = C.CDLL(libpath)
    names = declared_functions()
    assert len(names) >= 10
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_error_strings_without_gpu(libpath):
    lib = C.CDLL(libpath)
    lib.ula_error_string.restype = C.c_char_p
    for code in range(8):
        assert lib.ula_error_string(code)
    assert lib.ula_error_string(99) == b"unknown error"


def test_binding_struct_sizes_match_header(libpath):
    from serving_step_sparse_gb300 import ula
    # ula_config: 9 uint32 + 64 layer counts
    assert C.sizeof(ula.ula_config) == 4 * (8 + ula.MAX_GROUPS)
    assert C.sizeof(ula.ula_stats) == 8 * 13
    assert C.sizeof(ula.ula_debug_layout) == 4 * 8
    assert C.sizeof(ula.ula_debug_state) == 8 * 15 + 4 * 9 + 4  # padded to 8
    assert C.sizeof(ula.ula_span) == 4 * 2 + 8 * 2
    assert C.sizeof(ula.ula_profile) == (8 + 8 + 8) * len(ula.PHASES)
    src = open(HEADER).read()
    phases = re.search(r"ULA_PHASE_DEDUP = 0,(.*?)ULA_PHASE_COUNT", src, flags=re.S).group(1)
    names = re.findall(r"ULA_PHASE_(\w+)", re.sub(r"/\*.*?\*/", "", phases))
    assert ["dedup"] + [n.lower() for n in names] == ula.PHASES
    assert "#define ULA_MAX_GROUPS 64" in src and "#define ULA_MAX_BUCKETS 64" in src
    for name, val in (("ULA_ERR_INVALID_ARG", 1), ("ULA_ERR_CAPACITY", 2), ("ULA_ERR_UNMAPPED", 3),
                      ("ULA_ERR_CUDA", 4), ("ULA_ERR_TIMEOUT", 5), ("ULA_ERR_POISONED", 6),
                      ("ULA_ERR_INTERNAL", 7)):
        assert re.search(rf"{name}\s*=\s*{val}\b", src)
        assert getattr(ula, name[4:]) == val


def test_calls_reject_null_context_without_gpu(libpath):
    from serving_step_sparse_gb300 import ula
    base = C.c_uint32()
    assert ula.lib.ula_alloc(None, 1, None, C.byref(base)) == ula.ERR_INVALID_ARG
    assert ula.lib.ula_free(None, 0, 1) == ula.ERR_INVALID_ARG
    assert ula.lib.ula_sync(None, None) == ula.ERR_INVALID_ARG
    assert ula.lib.ula_create(None, None, None, None, None) == ula.ERR_INVALID_ARG
    ula.lib.ula_destroy(None)


def test_binding_flags_match_header(libpath):
    from serving_step_sparse_gb300 import ula
    src = open(HEADER).read()
    for name, val in (("ULA_FLAG_BYPASS_OVERFLOW", 1), ("ULA_FLAG_EXACT_LRU", 2),
                      ("ULA_FLAG_LAYER_SIGNAL", 4), ("ULA_FLAG_GATHER_BESIDE_MOVE", 8),
                      ("ULA_DEBUG_STALL_SCAN_BARRIER", 0x100),
                      ("ULA_NOALLOC_MAX_ENTRIES", 65536)):
        m = re.search(rf"#define {name} (0x[0-9a-fA-F]+|\d+)u?\b", src)
        assert m and int(m.group(1), 0) == val, name
        assert getattr(ula, name[4:]) == val, name


def test_tp_calls_reject_null_without_gpu(libpath):
    from serving_step_sparse_gb300 import ula
    base = C.c_uint32()
    assert ula.lib.ula_tp_alloc(None, 1, None, C.byref(base)) == ula.ERR_INVALID_ARG
    assert ula.lib.ula_tp_free(None, 0, 1) == ula.ERR_INVALID_ARG
    assert ula.lib.ula_tp_sync(None, None) == ula.ERR_INVALID_ARG
    assert ula.lib.ula_tp_destroy(None) == ula.ERR_INVALID_ARG
    assert not ula.lib.ula_tp_context(None, 0, 0)
    assert ula.lib.ula_tp_create(None, 2, 4, None, None, None, None, None) == ula.ERR_INVALID_ARG
    assert ula.lib.ula_layer_signal(None, 0, None, None) == ula.ERR_INVALID_ARG
