"""The C-ABI library loads and exports every function include/slotkv.h
declares; host-only argument checks work without a GPU."""
import ctypes
import os
import re

import sequence_slot_kv_gb300 as skv

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "slotkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if not n.startswith("SLOTKV")))


def test_header_declares_the_expected_calls():
    names = declared_functions()
    for n in ("slot_kv_alloc", "slot_kv_offset_bytes", "slot_kv_reset", "decode_batch_attn"):
        assert n in names


def test_library_exports_every_declared_function():
    lib = ctypes.CDLL(skv.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(skv.EXPORTS)


def test_host_only_checks_without_gpu():
    lib = skv._lib
    SIZE_MAX = ctypes.c_size_t(-1).value
    assert lib.slot_kv_offset_bytes(None, 0, 0) == SIZE_MAX
    h = ctypes.c_void_p()
    assert lib.slot_kv_alloc(ctypes.byref(h), 0, 16, 2, 64, None, None, 1, 2) == 1
    assert "n_slots" in skv.last_error()
    assert lib.slot_kv_alloc(ctypes.byref(h), 4, 16, 2, 96, None, None, 1, 2) == 3
    assert lib.slot_kv_alloc(ctypes.byref(h), 1 << 16, 1 << 15, 2, 64, None, None, 1, 2) == 1
    assert lib.slot_kv_alloc(ctypes.byref(h), 4, 16, 2, 64, ctypes.c_void_p(16), None, 1, 2) == 1
    assert lib.slot_kv_alloc(ctypes.byref(h), 4, 16, 2, 64, None, None, 1, 32) == 1
    assert not h.value
    assert lib.decode_batch_attn(None, 1, 2, *([None] * 10), 1e-6, 0.1, None) == 4
    assert lib.slot_kv_free(None) == 0
