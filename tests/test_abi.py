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


def test_more_host_checks_without_gpu():
    """Every size and pointer check that precedes a CUDA call, on the handle
    entry points and on the allocation-free one."""
    ARG, UNSUP, STATE = 1, 3, 4
    lib = skv._lib
    h = ctypes.c_void_p()
    byref = ctypes.byref
    # n_kv_head past 256, max_rows 0 and past 65535, max_n_head outside n_kv..8*n_kv
    assert lib.slot_kv_alloc(byref(h), 4, 16, 257, 64, None, None, 1, 257) == ARG
    assert "n_kv_head" in skv.last_error()
    assert lib.slot_kv_alloc(byref(h), 4, 16, 2, 64, None, None, 0, 2) == ARG
    assert lib.slot_kv_alloc(byref(h), 4, 16, 2, 64, None, None, 65536, 2) == ARG
    assert "max_rows" in skv.last_error()
    assert lib.slot_kv_alloc(byref(h), 4, 16, 2, 64, None, None, 1, 1) == ARG
    assert "max_n_head" in skv.last_error()
    # adopted buffers: both or neither, 16-byte aligned
    assert lib.slot_kv_alloc(byref(h), 4, 16, 2, 64, None, ctypes.c_void_p(256), 1, 2) == ARG
    assert lib.slot_kv_alloc(byref(h), 4, 16, 2, 64, ctypes.c_void_p(260), ctypes.c_void_p(256),
                             1, 2) == ARG
    assert "aligned" in skv.last_error()
    assert lib.slot_kv_alloc(None, 4, 16, 2, 64, None, None, 1, 2) == ARG
    assert not h.value
    # calls on no handle
    u = ctypes.c_uint32()
    assert lib.slot_kv_set_split(None, 64, 8) == STATE
    assert lib.slot_kv_set_options(None, 0) == STATE
    assert lib.slot_kv_call_shape(None, 1, 0, 0, byref(u), byref(u), byref(u)) == STATE
    assert lib.slot_kv_reset(None, 0, None) == STATE
    assert lib.slot_kv_get_status(None, None, byref(u)) == ARG
    # the allocation-free entry: checks before any device work
    p16 = ctypes.c_void_p(1 << 20)     # never dereferenced: every call below fails first
    p4 = ctypes.c_void_p((1 << 20) + 4)
    args = lambda **kw: [kw.get(k, d) for k, d in (
        ("K", p16), ("V", p16), ("n_slots", 4), ("slot_ctx", 16), ("n_kv", 2), ("hd", 64),
        ("B", 1), ("n_head", 4), ("q", p16), ("k", p16), ("v", p16), ("pos", p16),
        ("slots", p16), ("qw", p16), ("kw", p16), ("inv", p16), ("sinks", None),
        ("out", p16), ("flags", None), ("eps", 1e-6), ("scale", 0.125), ("stream", None))]
    na = lib.decode_batch_attn_noalloc
    assert na(*args(B=0, K=None)) == 0                      # nothing to do
    assert na(*args(K=None)) == ARG
    assert na(*args(q=p4)) == ARG and "16-byte" in skv.last_error()
    assert na(*args(pos=ctypes.c_void_p((1 << 20) + 2))) == ARG
    assert na(*args(hd=96)) == UNSUP
    assert na(*args(n_head=3)) == UNSUP
    assert na(*args(n_head=18)) == UNSUP                    # G = 9
    assert na(*args(n_kv=257, n_head=257)) == ARG
    assert na(*args(B=65536)) == ARG
    assert na(*args(n_slots=1 << 16, slot_ctx=1 << 15)) == ARG


def test_binding_refuses_mismatched_shapes():
    """The binding checks every step tensor's shape against (B, n_head) from
    q and the slot geometry before it passes an address on: a mismatched out
    or k_new would otherwise be read or written past its end."""
    import pytest
    import torch

    B, nh, nkv, hd = 3, 8, 2, 64
    K = torch.zeros((4, 16, nkv, hd))
    good = dict(q=torch.zeros((B, nh, hd)), k_new=torch.zeros((B, nkv, hd)),
                v_new=torch.zeros((B, nkv, hd)), positions=torch.zeros(B, dtype=torch.int32),
                slots=torch.zeros(B, dtype=torch.int32), q_norm_w=torch.ones(hd),
                k_norm_w=torch.ones(hd), inv_freq=torch.ones(hd // 2), sinks=None,
                out=torch.zeros((B, nh, hd)))
    bad = {"out": torch.zeros((B, nh - 1, hd)), "k_new": torch.zeros((B, nkv + 1, hd)),
           "v_new": torch.zeros((B + 1, nkv, hd)), "positions": torch.zeros(B + 1),
           "slots": torch.zeros(B - 1), "q_norm_w": torch.ones(hd + 1),
           "inv_freq": torch.ones(hd), "sinks": torch.zeros(nh + 1)}
    for name, t in bad.items():
        args = dict(good, **{name: t})
        with pytest.raises(ValueError, match=name):
            skv.decode_batch_attn_noalloc(K, K, eps=1e-6, scale=0.1, **args)

    class _Handle:          # the geometry a SlotKV carries, without a device
        n_kv_head, head_dim = nkv, hd

    with pytest.raises(ValueError, match="out"):
        skv.SlotKV.decode_batch_attn(_Handle(), **dict(good, out=bad["out"]), eps=1e-6,
                                     scale=0.1)
    with pytest.raises(ValueError, match="k_new"):
        skv.SlotKV.decode_batch_attn_host(_Handle(), **dict(good, k_new=bad["k_new"]),
                                          eps=1e-6, scale=0.1)
    # shapes that agree get as far as the placement check (CPU tensors here)
    with pytest.raises(ValueError, match="CUDA"):
        skv.decode_batch_attn_noalloc(K, K, eps=1e-6, scale=0.1, **good)


def test_host_call_checks_without_gpu():
    """The prepared host call refuses a missing handle or call pointer before
    any CUDA work; running or freeing a NULL call is refused or a no-op."""
    ARG, STATE = 1, 4
    lib = skv._lib
    c = ctypes.c_void_p()
    args = [1, 2] + [None] * 5 + [0] + [None] * 5 + [1e-6, 0.1]
    assert lib.slot_kv_host_call_create(None, ctypes.byref(c), *args) == STATE
    assert lib.slot_kv_host_call_create(None, None, *args) == ARG
    assert not c.value
    assert lib.slot_kv_host_call_run(None, None) == ARG
    assert lib.slot_kv_host_call_free(None) == 0
