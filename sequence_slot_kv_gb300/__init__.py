"""Python binding of libslotkv: batched decode attention over slot KV on GB300.

Argument marshalling only.  Every step of the decode attention runs in the
library's CUDA kernels; PyTorch supplies device memory and streams.  There is
no CPU fallback: importing this package raises if ``libslotkv.so`` has not
been built (``__graft_entry__.build()`` or ``python -m
sequence_slot_kv_gb300.build``).

The functions mirror the C ABI in ``include/slotkv.h`` name for name
(``EXPORTS`` lists every symbol): the handle (``slot_kv_alloc``,
``slot_kv_free``, ``slot_kv_offset_bytes``, ``slot_kv_reset``), the step
(``decode_batch_attn``, its host-buffer form ``decode_batch_attn_host``,
``prefill_batch_attn`` and its host-buffer form ``prefill_batch_attn_host``
(with ``slot_kv_prefill_host_parts``), ``decode_batch_attn_paged`` and its
host-buffer form ``decode_batch_attn_paged_host``, the allocation-free
``decode_batch_attn_noalloc``), multi-step support
(``slot_kv_advance_positions``), and control (``slot_kv_get_status``,
``slot_kv_set_split``, ``slot_kv_set_options``, ``slot_kv_call_shape``).
``SlotKV`` wraps a handle.
"""
import ctypes
import os

__all__ = [
    "SlotKV", "SlotKVError", "slot_kv_alloc", "slot_kv_free", "slot_kv_offset_bytes",
    "slot_kv_reset", "decode_batch_attn", "decode_batch_attn_host", "prefill_batch_attn",
    "prefill_batch_attn_host", "slot_kv_prefill_host_parts", "PREFILL_HOST_MAX_PARTS",
    "decode_batch_attn_paged", "decode_batch_attn_paged_host", "decode_batch_attn_noalloc",
    "slot_kv_advance_positions",
    "slot_kv_get_status", "slot_kv_set_split", "HostCall", "LIB_PATH", "EXPORTS", "DEV_RANGE",
    "DEV_TIMEOUT", "OPT_VNORM", "OPT_NORM_PLUS_ONE", "OPT_TEST_STALL",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libslotkv.so")
DEV_RANGE = 1
DEV_TIMEOUT = 2
OPT_VNORM = 1
OPT_NORM_PLUS_ONE = 2
OPT_TEST_STALL = 0x80000000
PREFILL_HOST_MAX_PARTS = 8  # SLOTKV_PREFILL_HOST_MAX_PARTS
SIZE_MAX = ctypes.c_size_t(-1).value

_u32, _f32, _vp, _int = ctypes.c_uint32, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
_DECODE_ARGS = [_vp, _u32, _u32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                _f32, _f32, _vp]
EXPORTS = {
    "slot_kv_alloc": ([ctypes.POINTER(_vp), _u32, _u32, _u32, _u32, _vp, _vp, _u32, _u32],
                      _int),
    "slot_kv_free": ([_vp], _int),
    "slot_kv_offset_bytes": ([_vp, _u32, _u32], ctypes.c_size_t),
    "slot_kv_reset": ([_vp, _u32, _vp], _int),
    "slot_kv_k_ptr": ([_vp, ctypes.POINTER(_vp)], _int),
    "slot_kv_v_ptr": ([_vp, ctypes.POINTER(_vp)], _int),
    "slot_kv_geometry": ([_vp] + [ctypes.POINTER(_u32)] * 6, _int),
    "decode_batch_attn": (_DECODE_ARGS, _int),
    "decode_batch_attn_host": (_DECODE_ARGS, _int),
    "prefill_batch_attn": (_DECODE_ARGS, _int),
    "prefill_batch_attn_host": (_DECODE_ARGS, _int),
    "slot_kv_prefill_host_parts": ([_u32, _vp, ctypes.POINTER(_u32), _u32,
                                    ctypes.POINTER(_u32)], _int),
    "decode_batch_attn_paged": ([_vp, _u32, _u32, _vp, _vp, _vp, _vp, _vp, _u32, _vp, _vp, _vp,
                                 _vp, _vp, _f32, _f32, _vp], _int),
    "decode_batch_attn_paged_host": ([_vp, _u32, _u32, _vp, _vp, _vp, _vp, _vp, _u32, _vp, _vp,
                                      _vp, _vp, _vp, _f32, _f32, _vp], _int),
    "slot_kv_get_status": ([_vp, _vp, ctypes.POINTER(_u32)], _int),
    "slot_kv_set_split": ([_vp, _u32, _u32], _int),
    "slot_kv_call_shape": ([_vp, _u32, _u32, _u32, ctypes.POINTER(_u32), ctypes.POINTER(_u32),
                            ctypes.POINTER(_u32)], _int),
    "slot_kv_advance_positions": ([_vp, _u32, _u32, _vp], _int),
    "slot_kv_set_options": ([_vp, _u32], _int),
    "decode_batch_attn_noalloc": ([_vp, _vp, _u32, _u32, _u32, _u32, _u32, _u32, _vp, _vp, _vp,
                                   _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _f32, _vp],
                                  _int),
    "slot_kv_shard_range": ([_u32, _u32, _u32, ctypes.POINTER(_u32), ctypes.POINTER(_u32)],
                            _int),
    "slot_kv_shard_route": ([_u32, _u32, _u32, _vp, _vp, _vp, _vp], _int),
    "slot_kv_host_call_create": ([_vp, ctypes.POINTER(_vp), _u32, _u32, _vp, _vp, _vp, _vp, _vp,
                                  _u32, _vp, _vp, _vp, _vp, _vp, _f32, _f32], _int),
    "slot_kv_host_call_run": ([_vp, _vp], _int),
    "slot_kv_host_call_enqueue": ([_vp, _vp], _int),
    "slot_kv_host_call_free": ([_vp], _int),
    "slot_kv_last_error": ([], ctypes.c_char_p),
}


class SlotKVError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what} failed with status {code}: {last_error()}")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run __graft_entry__.build() (no CPU fallback exists)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def last_error():
    msg = _lib.slot_kv_last_error()
    return msg.decode() if msg else ""


def _check(code, what):
    if code != 0:
        raise SlotKVError(code, what)


def _ptr(t, dtype=None, what="tensor", cuda=True):
    """Address of a contiguous tensor that lives on the GPU (cuda=True) or in
    host memory (cuda=False); None stays NULL.  The library reads these
    addresses from its kernels or copies, so a tensor in the wrong place is
    refused here."""
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if cuda is not None and t.is_cuda != cuda:
        raise ValueError(f"{what} must be a {'CUDA' if cuda else 'CPU'} tensor")
    return t.data_ptr()


def _shape(t):
    return None if t is None else tuple(int(x) for x in t.shape)


def _check_step(q, k_new, v_new, positions, rows_idx, out, q_norm_w, k_norm_w, inv_freq,
                sinks, n_kv_head, head_dim, idx_name="slots"):
    """Shapes of one step's tensors against (B, n_head) taken from q and the
    slot geometry (n_kv_head, head_dim).  The library reads and writes these
    buffers by those sizes, so a mismatch is refused before any call."""
    if q is None or q.dim() != 3:
        raise ValueError("q must be [B][n_head][head_dim]")
    B, n_head, hd = _shape(q)
    if hd != head_dim:
        raise ValueError(f"q's head_dim {hd} != the slot buffers' {head_dim}")
    want = {
        "q": (q, (B, n_head, hd)), "k_new": (k_new, (B, n_kv_head, hd)),
        "v_new": (v_new, (B, n_kv_head, hd)), "positions": (positions, (B,)),
        "out": (out, (B, n_head, hd)), "q_norm_w": (q_norm_w, (hd,)),
        "k_norm_w": (k_norm_w, (hd,)), "inv_freq": (inv_freq, (hd // 2,)),
    }
    if idx_name == "slots":
        want["slots"] = (rows_idx, (B,))
    for name, (t, shape) in want.items():
        if t is None:
            raise ValueError(f"{name} is required")
        if _shape(t) != shape:
            raise ValueError(f"{name} has shape {_shape(t)}, expected {shape}")
    if sinks is not None and _shape(sinks) != (n_head,):
        raise ValueError(f"sinks has shape {_shape(sinks)}, expected ({n_head},)")
    return B, n_head


def _stream_ptr(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class SlotKV:
    """One attention layer's slot KV: ``[n_slots][slot_ctx][n_kv_head][head_dim]``
    f32 K and V, plus the split-K workspace for up to ``max_rows`` rows and
    ``max_n_head`` query heads.  ``k_buf``/``v_buf`` (torch CUDA tensors) are
    adopted in place when given; otherwise the library allocates them."""

    def __init__(self, n_slots, slot_ctx, n_kv_head, head_dim, max_rows, max_n_head,
                 k_buf=None, v_buf=None):
        import torch
        self._h = _vp()
        self.n_slots, self.slot_ctx = int(n_slots), int(slot_ctx)
        self.n_kv_head, self.head_dim = int(n_kv_head), int(head_dim)
        self.kv_dim = self.n_kv_head * self.head_dim
        self.max_rows, self.max_n_head = int(max_rows), int(max_n_head)
        self._keep = (k_buf, v_buf)
        kp = _ptr(k_buf, torch.float32, "k_buf")
        vp = _ptr(v_buf, torch.float32, "v_buf")
        _check(_lib.slot_kv_alloc(ctypes.byref(self._h), n_slots, slot_ctx, n_kv_head,
                                  head_dim, kp, vp, max_rows, max_n_head), "slot_kv_alloc")

    @property
    def handle(self):
        return self._h.value

    def free(self):
        if self._h.value:
            _check(_lib.slot_kv_free(self._h), "slot_kv_free")
            self._h = _vp()
        self._keep = (None, None)

    def __del__(self):
        try:
            self.free()
        except Exception:  # noqa: BLE001 -- interpreter shutdown
            pass

    def offset_bytes(self, slot, pos):
        v = _lib.slot_kv_offset_bytes(self._h, slot, pos)
        return None if v == SIZE_MAX else int(v)

    def reset(self, slot, stream=None):
        _check(_lib.slot_kv_reset(self._h, slot, _stream_ptr(stream)), "slot_kv_reset")

    def k_ptr(self):
        p = _vp()
        _check(_lib.slot_kv_k_ptr(self._h, ctypes.byref(p)), "slot_kv_k_ptr")
        return p.value

    def v_ptr(self):
        p = _vp()
        _check(_lib.slot_kv_v_ptr(self._h, ctypes.byref(p)), "slot_kv_v_ptr")
        return p.value

    def kv_tensors(self):
        """(K, V) as torch views of the slot buffers (adopted or owned)."""
        if self._keep[0] is not None:
            return self._keep
        # owned buffers: wrap the device addresses without copying
        n = self.n_slots * self.slot_ctx * self.kv_dim
        shape = (self.n_slots, self.slot_ctx, self.n_kv_head, self.head_dim)
        return tuple(_wrap_device(ptr, n).view(shape) for ptr in (self.k_ptr(), self.v_ptr()))

    def decode_batch_attn(self, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                          inv_freq, sinks, out, eps, scale, stream=None):
        import torch
        B, n_head = _check_step(q, k_new, v_new, positions, slots, out, q_norm_w, k_norm_w,
                                inv_freq, sinks, self.n_kv_head, self.head_dim)
        f, u = torch.float32, torch.int32
        _check(_lib.decode_batch_attn(
            self._h, B, n_head, _ptr(q, f, "q"), _ptr(k_new, f, "k_new"),
            _ptr(v_new, f, "v_new"), _ptr(positions, u, "positions"), _ptr(slots, u, "slots"),
            _ptr(q_norm_w, f, "q_norm_w"), _ptr(k_norm_w, f, "k_norm_w"),
            _ptr(inv_freq, f, "inv_freq"), _ptr(sinks, f, "sinks"), _ptr(out, f, "out"),
            eps, scale, _stream_ptr(stream)), "decode_batch_attn")
        return out

    def prefill_batch_attn(self, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                           inv_freq, sinks, out, eps, scale, stream=None):
        """Batched causal prefill: tokens (rows of q, k_new, v_new, positions,
        slots, out) are written into their slots and each attends keys
        0..pos of its slot, the call's other new rows included."""
        import torch
        n, n_head = _check_step(q, k_new, v_new, positions, slots, out, q_norm_w, k_norm_w,
                                inv_freq, sinks, self.n_kv_head, self.head_dim)
        f, u = torch.float32, torch.int32
        _check(_lib.prefill_batch_attn(
            self._h, n, n_head, _ptr(q, f, "q"), _ptr(k_new, f, "k_new"),
            _ptr(v_new, f, "v_new"), _ptr(positions, u, "positions"), _ptr(slots, u, "slots"),
            _ptr(q_norm_w, f, "q_norm_w"), _ptr(k_norm_w, f, "k_norm_w"),
            _ptr(inv_freq, f, "inv_freq"), _ptr(sinks, f, "sinks"), _ptr(out, f, "out"),
            eps, scale, _stream_ptr(stream)), "prefill_batch_attn")
        return out

    def prefill_batch_attn_host(self, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                                inv_freq, sinks, out, eps, scale, stream=None):
        """As prefill_batch_attn, with q/k_new/v_new/positions/slots/out in host
        memory (CPU tensors, ideally pinned); synchronous."""
        import torch
        n, n_head = _check_step(q, k_new, v_new, positions, slots, out, q_norm_w, k_norm_w,
                                inv_freq, sinks, self.n_kv_head, self.head_dim)
        f, u = torch.float32, torch.int32
        _check(_lib.prefill_batch_attn_host(
            self._h, n, n_head, _ptr(q, f, "q", cuda=False), _ptr(k_new, f, "k_new", cuda=False),
            _ptr(v_new, f, "v_new", cuda=False), _ptr(positions, u, "positions", cuda=False),
            _ptr(slots, u, "slots", cuda=False), _ptr(q_norm_w, f, "q_norm_w"),
            _ptr(k_norm_w, f, "k_norm_w"), _ptr(inv_freq, f, "inv_freq"), _ptr(sinks, f, "sinks"),
            _ptr(out, f, "out", cuda=False), eps, scale, _stream_ptr(stream)),
            "prefill_batch_attn_host")
        return out

    def decode_batch_attn_paged(self, q, k_new, v_new, positions, block_tables, q_norm_w,
                                k_norm_w, inv_freq, sinks, out, eps, scale, stream=None):
        """Decode over a paged pool (this handle's buffers as blocks of
        slot_ctx positions): block_tables is int32 [B][max_blocks], row b's
        key t in block block_tables[b][t // slot_ctx]."""
        import torch
        B, n_head = _check_step(q, k_new, v_new, positions, block_tables, out, q_norm_w,
                                k_norm_w, inv_freq, sinks, self.n_kv_head, self.head_dim,
                                idx_name="block_tables")
        f, u = torch.float32, torch.int32
        if block_tables.dim() != 2 or int(block_tables.shape[0]) != B:
            raise ValueError("block_tables must be [B][max_blocks]")
        _check(_lib.decode_batch_attn_paged(
            self._h, B, n_head, _ptr(q, f, "q"), _ptr(k_new, f, "k_new"),
            _ptr(v_new, f, "v_new"), _ptr(positions, u, "positions"),
            _ptr(block_tables, u, "block_tables"), int(block_tables.shape[1]),
            _ptr(q_norm_w, f, "q_norm_w"), _ptr(k_norm_w, f, "k_norm_w"),
            _ptr(inv_freq, f, "inv_freq"), _ptr(sinks, f, "sinks"), _ptr(out, f, "out"),
            eps, scale, _stream_ptr(stream)), "decode_batch_attn_paged")
        return out

    def decode_batch_attn_paged_host(self, q, k_new, v_new, positions, block_tables, q_norm_w,
                                     k_norm_w, inv_freq, sinks, out, eps, scale, stream=None):
        """As decode_batch_attn_paged, with q/k_new/v_new/positions/block_tables/out
        in host memory (CPU tensors, ideally pinned); synchronous."""
        import torch
        B, n_head = _check_step(q, k_new, v_new, positions, block_tables, out, q_norm_w,
                                k_norm_w, inv_freq, sinks, self.n_kv_head, self.head_dim,
                                idx_name="block_tables")
        f, u = torch.float32, torch.int32
        if block_tables.dim() != 2 or int(block_tables.shape[0]) != B:
            raise ValueError("block_tables must be [B][max_blocks]")
        _check(_lib.decode_batch_attn_paged_host(
            self._h, B, n_head, _ptr(q, f, "q", cuda=False),
            _ptr(k_new, f, "k_new", cuda=False), _ptr(v_new, f, "v_new", cuda=False),
            _ptr(positions, u, "positions", cuda=False),
            _ptr(block_tables, u, "block_tables", cuda=False), int(block_tables.shape[1]),
            _ptr(q_norm_w, f, "q_norm_w"), _ptr(k_norm_w, f, "k_norm_w"),
            _ptr(inv_freq, f, "inv_freq"), _ptr(sinks, f, "sinks"),
            _ptr(out, f, "out", cuda=False), eps, scale, _stream_ptr(stream)),
            "decode_batch_attn_paged_host")
        return out

    def prepare_host_call(self, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                          inv_freq, sinks, out, eps, scale, block_tables=None):
        """A prepared host step (slot_kv_host_call_create): the arguments of
        decode_batch_attn_host -- or, with ``block_tables`` given in place of
        ``slots`` (pass slots=None), of decode_batch_attn_paged_host --
        checked once.  Calling the returned HostCall runs one step on the
        buffers' current contents, synchronously."""
        return HostCall(self, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w, inv_freq,
                        sinks, out, eps, scale, block_tables)

    def decode_batch_attn_host(self, q, k_new, v_new, positions, slots, q_norm_w,
                               k_norm_w, inv_freq, sinks, out, eps, scale, stream=None):
        """As decode_batch_attn, with q/k_new/v_new/positions/slots/out in host
        memory (CPU tensors, ideally pinned); synchronous."""
        import torch
        B, n_head = _check_step(q, k_new, v_new, positions, slots, out, q_norm_w, k_norm_w,
                                inv_freq, sinks, self.n_kv_head, self.head_dim)
        f, u = torch.float32, torch.int32
        _check(_lib.decode_batch_attn_host(
            self._h, B, n_head, _ptr(q, f, "q", cuda=False),
            _ptr(k_new, f, "k_new", cuda=False), _ptr(v_new, f, "v_new", cuda=False),
            _ptr(positions, u, "positions", cuda=False), _ptr(slots, u, "slots", cuda=False),
            _ptr(q_norm_w, f, "q_norm_w"), _ptr(k_norm_w, f, "k_norm_w"),
            _ptr(inv_freq, f, "inv_freq"), _ptr(sinks, f, "sinks"),
            _ptr(out, f, "out", cuda=False), eps, scale, _stream_ptr(stream)),
            "decode_batch_attn_host")
        return out

    def get_status(self, stream=None):
        v = _u32()
        _check(_lib.slot_kv_get_status(self._h, _stream_ptr(stream), ctypes.byref(v)),
               "slot_kv_get_status")
        return int(v.value)

    def set_options(self, flags):
        """OPT_VNORM and/or OPT_NORM_PLUS_ONE (see slot_kv_set_options)."""
        _check(_lib.slot_kv_set_options(self._h, flags), "slot_kv_set_options")

    def call_shape(self, B, bt_stride=0, prefill=False):
        """(chunk_keys, ctas, kernels) of a call of B rows (slot_kv_call_shape)."""
        c, n, k = _u32(), _u32(), _u32()
        _check(_lib.slot_kv_call_shape(self._h, B, bt_stride, 1 if prefill else 0,
                                       ctypes.byref(c), ctypes.byref(n), ctypes.byref(k)),
               "slot_kv_call_shape")
        return c.value, n.value, k.value

    def set_split(self, min_chunk_keys, max_splits):
        _check(_lib.slot_kv_set_split(self._h, min_chunk_keys, max_splits), "slot_kv_set_split")


def _wrap_device(ptr, numel):
    """A float32 CUDA tensor aliasing ``numel`` floats at device address ``ptr``."""
    import torch

    class _Holder:
        pass

    h = _Holder()
    h.__cuda_array_interface__ = {
        "shape": (numel,), "typestr": "<f4", "data": (ptr, False), "version": 3,
        "strides": None,
    }
    return torch.as_tensor(h, device="cuda")


# ---- C-ABI names ---------------------------------------------------------
def slot_kv_alloc(n_slots, slot_ctx, n_kv_head, head_dim, max_rows, max_n_head,
                  k_buf=None, v_buf=None):
    return SlotKV(n_slots, slot_ctx, n_kv_head, head_dim, max_rows, max_n_head, k_buf, v_buf)


def slot_kv_free(h):
    h.free()


def slot_kv_offset_bytes(h, slot, pos):
    return h.offset_bytes(slot, pos)


def slot_kv_reset(h, slot, stream=None):
    h.reset(slot, stream)


def decode_batch_attn(h, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w, inv_freq,
                      sinks, out, eps, scale, stream=None):
    return h.decode_batch_attn(q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                               inv_freq, sinks, out, eps, scale, stream)


def prefill_batch_attn(h, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w, inv_freq,
                       sinks, out, eps, scale, stream=None):
    return h.prefill_batch_attn(q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                                inv_freq, sinks, out, eps, scale, stream)


def prefill_batch_attn_host(h, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                            inv_freq, sinks, out, eps, scale, stream=None):
    return h.prefill_batch_attn_host(q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                                     inv_freq, sinks, out, eps, scale, stream)


def slot_kv_prefill_host_parts(slots):
    """Where prefill_batch_attn_host cuts a call with these slots (one per
    token, a host sequence of ints): the part boundaries [0, ..., n_tok].
    Host only."""
    import numpy as np
    sl = np.ascontiguousarray(np.asarray(slots).astype(np.uint32, copy=False))
    cuts = (_u32 * (PREFILL_HOST_MAX_PARTS + 1))()
    n = _u32()
    _check(_lib.slot_kv_prefill_host_parts(len(sl), sl.ctypes.data if len(sl) else None, cuts,
                                           len(cuts), ctypes.byref(n)),
           "slot_kv_prefill_host_parts")
    return [int(cuts[i]) for i in range(n.value + 1)]


def decode_batch_attn_paged(h, q, k_new, v_new, positions, block_tables, q_norm_w, k_norm_w,
                            inv_freq, sinks, out, eps, scale, stream=None):
    return h.decode_batch_attn_paged(q, k_new, v_new, positions, block_tables, q_norm_w,
                                     k_norm_w, inv_freq, sinks, out, eps, scale, stream)


class HostCall:
    """A prepared host step on a SlotKV handle (slot_kv_host_call_create):
    the host tensors (q, k_new, v_new, positions, slots or block_tables, out;
    ideally pinned) and the device parameters are checked once and kept
    referenced; ``call(stream=None)`` runs one synchronous step on their
    current contents (slot_kv_host_call_run), the same step the host entry
    runs; ``call(stream, sync=False)`` only enqueues it
    (slot_kv_host_call_enqueue).  ``free()`` releases it (also on garbage
    collection)."""

    def __init__(self, kv, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w, inv_freq,
                 sinks, out, eps, scale, block_tables=None):
        import torch
        paged = block_tables is not None
        idx = block_tables if paged else slots
        B, n_head = _check_step(q, k_new, v_new, positions, idx, out, q_norm_w, k_norm_w,
                                inv_freq, sinks, kv.n_kv_head, kv.head_dim,
                                idx_name="block_tables" if paged else "slots")
        if paged and (block_tables.dim() != 2 or int(block_tables.shape[0]) != B):
            raise ValueError("block_tables must be [B][max_blocks]")
        f, u = torch.float32, torch.int32
        self._c = _vp()
        self._kv = kv
        self._keep = (q, k_new, v_new, positions, idx, q_norm_w, k_norm_w, inv_freq, sinks, out)
        _check(_lib.slot_kv_host_call_create(
            kv._h, ctypes.byref(self._c), B, n_head, _ptr(q, f, "q", cuda=False),
            _ptr(k_new, f, "k_new", cuda=False), _ptr(v_new, f, "v_new", cuda=False),
            _ptr(positions, u, "positions", cuda=False),
            _ptr(idx, u, "block_tables" if paged else "slots", cuda=False),
            int(block_tables.shape[1]) if paged else 0,
            _ptr(q_norm_w, f, "q_norm_w"), _ptr(k_norm_w, f, "k_norm_w"),
            _ptr(inv_freq, f, "inv_freq"), _ptr(sinks, f, "sinks"),
            _ptr(out, f, "out", cuda=False), eps, scale), "slot_kv_host_call_create")
        self.out = out

    def __call__(self, stream=None, sync=True):
        """One step.  sync=False only enqueues it (slot_kv_host_call_enqueue):
        out is complete, and the host inputs may be refilled, once the stream
        has been synchronised."""
        if sync:
            _check(_lib.slot_kv_host_call_run(self._c, _stream_ptr(stream)),
                   "slot_kv_host_call_run")
        else:
            _check(_lib.slot_kv_host_call_enqueue(self._c, _stream_ptr(stream)),
                   "slot_kv_host_call_enqueue")
        return self.out

    def free(self):
        if self._c.value:
            _check(_lib.slot_kv_host_call_free(self._c), "slot_kv_host_call_free")
            self._c = _vp()
        self._keep = None

    def __del__(self):
        try:
            self.free()
        except Exception:  # noqa: BLE001 -- interpreter shutdown
            pass


def decode_batch_attn_host(h, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                           inv_freq, sinks, out, eps, scale, stream=None):
    return h.decode_batch_attn_host(q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                                    inv_freq, sinks, out, eps, scale, stream)


def decode_batch_attn_paged_host(h, q, k_new, v_new, positions, block_tables, q_norm_w,
                                 k_norm_w, inv_freq, sinks, out, eps, scale, stream=None):
    return h.decode_batch_attn_paged_host(q, k_new, v_new, positions, block_tables, q_norm_w,
                                          k_norm_w, inv_freq, sinks, out, eps, scale, stream)


def slot_kv_get_status(h, stream=None):
    return h.get_status(stream)


def slot_kv_set_split(h, min_chunk_keys, max_splits):
    h.set_split(min_chunk_keys, max_splits)


def slot_kv_advance_positions(positions, delta=1, stream=None):
    """positions += delta on the device (int32 CUDA tensor), on ``stream``."""
    import torch
    _check(_lib.slot_kv_advance_positions(_ptr(positions, torch.int32, "positions"),
                                          int(positions.numel()), int(delta),
                                          _stream_ptr(stream)), "slot_kv_advance_positions")


def decode_batch_attn_noalloc(K, V, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                              inv_freq, sinks, out, eps, scale, dev_flags=None, stream=None):
    """The decode step for callers that cannot allocate device memory: no
    handle; the slot buffers K, V ([n_slots][slot_ctx][n_kv_head][head_dim]
    torch CUDA tensors) and every input and output come from the caller, and
    the library's split-K scratch is a fixed array inside it.  ``dev_flags``
    is an optional int32 CUDA tensor of one element that receives the device
    flags.  The first call on a device should come before any stream capture;
    calls that overlap on the GPU race on the shared scratch."""
    import torch
    if K.dim() != 4 or _shape(V) != _shape(K):
        raise ValueError("K and V must both be [n_slots][slot_ctx][n_kv_head][head_dim]")
    n_slots, slot_ctx, n_kv_head, head_dim = _shape(K)
    B, n_head = _check_step(q, k_new, v_new, positions, slots, out, q_norm_w, k_norm_w,
                            inv_freq, sinks, n_kv_head, head_dim)
    if dev_flags is not None and int(dev_flags.numel()) < 1:
        raise ValueError("dev_flags must hold one element")
    f, u = torch.float32, torch.int32
    _check(_lib.decode_batch_attn_noalloc(
        _ptr(K, f, "K"), _ptr(V, f, "V"), n_slots, slot_ctx, n_kv_head, head_dim, B, n_head,
        _ptr(q, f, "q"), _ptr(k_new, f, "k_new"), _ptr(v_new, f, "v_new"),
        _ptr(positions, u, "positions"), _ptr(slots, u, "slots"), _ptr(q_norm_w, f, "q_norm_w"),
        _ptr(k_norm_w, f, "k_norm_w"), _ptr(inv_freq, f, "inv_freq"), _ptr(sinks, f, "sinks"),
        _ptr(out, f, "out"), _ptr(dev_flags, u, "dev_flags"), eps, scale, _stream_ptr(stream)),
        "decode_batch_attn_noalloc")
    return out
