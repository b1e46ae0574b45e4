"""CPU oracle for batched slot-KV decode attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline arm of
``bench.py`` may import this package.  The product path (the CUDA library
and its binding) never loads it.

``Oracle`` wraps ``liboracle.so`` (``oracle.c``): a plain f64 loop
statement of one batched decode step over slot KV.  See ``oracle.c`` for the
definition and the readings it takes where the pages are silent.
"""
import ctypes
import os

import numpy as np

from . import build as _build


VNORM = 1
NORM_PLUS_ONE = 2


class Oracle:
    def __init__(self, lib_path=None):
        if lib_path is None:
            lib_path = _build.build()
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        u32, f32, vp = ctypes.c_uint32, ctypes.c_float, ctypes.c_void_p
        lib.oracle_slot_kv_offset_bytes.argtypes = [u32, u32, u32, u32]
        lib.oracle_slot_kv_offset_bytes.restype = ctypes.c_uint64
        lib.oracle_norm_rope_head.argtypes = [vp, vp, u32, f32, u32, vp, vp]
        lib.oracle_norm_rope_head.restype = None
        lib.oracle_decode_batch.argtypes = [u32, u32, u32, u32, u32, u32,
                                            vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            f32, f32, vp, vp, vp, vp, ctypes.c_int]
        lib.oracle_decode_batch.restype = ctypes.c_int
        lib.oracle_decode_batch_opts.argtypes = [u32, u32, u32, u32, u32, u32,
                                                 vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                 f32, f32, u32, vp, vp, vp, vp, ctypes.c_int]
        lib.oracle_decode_batch_opts.restype = ctypes.c_int
        lib.oracle_decode_batch_paged.argtypes = [u32, u32, u32, u32, u32, u32,
                                                  vp, vp, vp, vp, vp, u32, vp, vp, vp, vp,
                                                  f32, f32, u32, vp, vp, vp, vp, ctypes.c_int]
        lib.oracle_decode_batch_paged.restype = ctypes.c_int
        self.lib = lib

    def offset_bytes(self, slot, pos, slot_ctx, kv_dim):
        return int(self.lib.oracle_slot_kv_offset_bytes(slot, pos, slot_ctx, kv_dim))

    def norm_rope_head(self, x, w, eps, pos, inv_freq):
        x = np.ascontiguousarray(x, dtype=np.float32)
        w = np.ascontiguousarray(w, dtype=np.float32)
        inv_freq = np.ascontiguousarray(inv_freq, dtype=np.float32)
        assert x.ndim == 1 and w.shape == x.shape and inv_freq.size == x.size // 2
        y = np.empty(x.size, dtype=np.float64)
        self.lib.oracle_norm_rope_head(x.ctypes.data, w.ctypes.data, x.size, eps, pos,
                                       inv_freq.ctypes.data, y.ctypes.data)
        return y

    def decode_batch(self, K, V, q, k_new, v_new, positions, slots, q_norm_w,
                     k_norm_w, inv_freq, sinks, eps, scale, n_threads=1, want64=False,
                     flags=0):
        """One decode step.  K, V: f32[n_slots][slot_ctx][n_kv_head][hd] (updated
        in place).  Returns (out f32[B][n_head][hd], out64 or None, skipped)."""
        assert K.dtype == np.float32 and V.dtype == np.float32
        assert K.flags.c_contiguous and V.flags.c_contiguous and K.shape == V.shape
        n_slots, slot_ctx, n_kv_head, hd = K.shape
        q = np.ascontiguousarray(q, dtype=np.float32)
        B, n_head = q.shape[0], q.shape[1]
        assert q.shape == (B, n_head, hd)
        k_new = np.ascontiguousarray(k_new, dtype=np.float32)
        v_new = np.ascontiguousarray(v_new, dtype=np.float32)
        assert k_new.shape == (B, n_kv_head, hd) and v_new.shape == k_new.shape
        positions = np.ascontiguousarray(positions, dtype=np.uint32)
        slots = np.ascontiguousarray(slots, dtype=np.uint32)
        assert positions.shape == (B,) and slots.shape == (B,)
        qw = np.ascontiguousarray(q_norm_w, dtype=np.float32)
        kw = np.ascontiguousarray(k_norm_w, dtype=np.float32)
        fr = np.ascontiguousarray(inv_freq, dtype=np.float32)
        sk = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float32)
        out = np.zeros((B, n_head, hd), dtype=np.float32)
        out64 = np.zeros((B, n_head, hd), dtype=np.float64) if want64 else None
        rc = self.lib.oracle_decode_batch_opts(
            n_slots, slot_ctx, n_head, n_kv_head, hd, B,
            q.ctypes.data, k_new.ctypes.data, v_new.ctypes.data,
            positions.ctypes.data, slots.ctypes.data, qw.ctypes.data, kw.ctypes.data,
            fr.ctypes.data, None if sk is None else sk.ctypes.data, eps, scale, int(flags),
            K.ctypes.data, V.ctypes.data, out.ctypes.data,
            None if out64 is None else out64.ctypes.data, int(n_threads))
        if rc < 0:
            raise ValueError("oracle_decode_batch rejected its arguments")
        return out, out64, rc

    def decode_batch_paged(self, K, V, q, k_new, v_new, positions, block_tables, q_norm_w,
                           k_norm_w, inv_freq, sinks, eps, scale, n_threads=1, want64=False,
                           flags=0):
        """One decode step over a paged pool.  K, V:
        f32[n_blocks][block_size][n_kv_head][hd] (updated in place);
        block_tables: u32[B][max_blocks] (row b's key t lives in block
        block_tables[b][t // block_size] at offset t % block_size).
        Returns (out, out64 or None, skipped)."""
        assert K.dtype == np.float32 and V.dtype == np.float32
        assert K.flags.c_contiguous and V.flags.c_contiguous and K.shape == V.shape
        n_blocks, block_size, n_kv_head, hd = K.shape
        q = np.ascontiguousarray(q, dtype=np.float32)
        B, n_head = q.shape[0], q.shape[1]
        assert q.shape == (B, n_head, hd)
        k_new = np.ascontiguousarray(k_new, dtype=np.float32)
        v_new = np.ascontiguousarray(v_new, dtype=np.float32)
        assert k_new.shape == (B, n_kv_head, hd) and v_new.shape == k_new.shape
        positions = np.ascontiguousarray(positions, dtype=np.uint32)
        bt = np.ascontiguousarray(block_tables, dtype=np.uint32)
        assert positions.shape == (B,) and bt.ndim == 2 and bt.shape[0] == B
        qw = np.ascontiguousarray(q_norm_w, dtype=np.float32)
        kw = np.ascontiguousarray(k_norm_w, dtype=np.float32)
        fr = np.ascontiguousarray(inv_freq, dtype=np.float32)
        sk = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float32)
        out = np.zeros((B, n_head, hd), dtype=np.float32)
        out64 = np.zeros((B, n_head, hd), dtype=np.float64) if want64 else None
        rc = self.lib.oracle_decode_batch_paged(
            n_blocks, block_size, n_head, n_kv_head, hd, B,
            q.ctypes.data, k_new.ctypes.data, v_new.ctypes.data,
            positions.ctypes.data, bt.ctypes.data, bt.shape[1], qw.ctypes.data,
            kw.ctypes.data, fr.ctypes.data, None if sk is None else sk.ctypes.data, eps, scale,
            int(flags), K.ctypes.data, V.ctypes.data, out.ctypes.data,
            None if out64 is None else out64.ctypes.data, int(n_threads))
        if rc < 0:
            raise ValueError("oracle_decode_batch_paged rejected its arguments")
        return out, out64, rc


_default = None


def default():
    global _default
    if _default is None:
        _default = Oracle()
    return _default
