"""Seeded synthetic inputs for batched slot-KV decode attention.

Shared by the CPU oracle side and the CUDA side as *inputs only*: nothing in
this package computes any step of the attention method.  Every value is a
pure function of (seed, stream, index) (see ``synth.h``), so a tensor of any
size can be regenerated piecewise on the host, and the history K/V can be
filled on the device with bit-identical values.

The five workloads below follow the batched-decode configurations this
library is measured on; where a recipe leaves a detail open the choice is
stated next to it.
"""
import ctypes
import dataclasses
import os

import numpy as np

from . import build as _build

S_HIST_K, S_HIST_V, S_Q, S_KNEW, S_VNEW = 1, 2, 3, 4, 5
S_QNORM_W, S_KNORM_W, S_SINKS, S_POS, S_SLOTS = 6, 7, 8, 9, 10
S_BLOCKS = 11
STEP_STRIDE = 16

_host = None
_dev = None


def host_lib():
    global _host
    if _host is None:
        path = _build.HOST_LIB
        if not os.path.exists(path):
            _build.build_host()
        lib = ctypes.CDLL(path)
        u64, i32, f32 = ctypes.c_uint64, ctypes.c_int, ctypes.c_float
        vp = ctypes.c_void_p
        lib.synth_fill_normal.argtypes = [vp, u64, u64, u64, u64, i32]
        lib.synth_fill_normal.restype = i32
        lib.synth_fill_normal_affine.argtypes = [vp, u64, u64, u64, u64, f32, f32, i32]
        lib.synth_fill_normal_affine.restype = i32
        lib.synth_fill_below.argtypes = [vp, u64, u64, u64, ctypes.c_uint32]
        lib.synth_fill_below.restype = i32
        lib.synth_subset.argtypes = [vp, ctypes.c_uint32, ctypes.c_uint32, u64, u64, vp]
        lib.synth_subset.restype = i32
        lib.synth_key_of.argtypes = [u64, u64]
        lib.synth_key_of.restype = u64
        _host = lib
    return _host


def dev_lib():
    global _dev
    if _dev is None:
        path = _build.DEV_LIB
        if not os.path.exists(path):
            raise ImportError(f"{path} is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        u64 = ctypes.c_uint64
        lib.synth_dev_fill_normal.argtypes = [ctypes.c_void_p, u64, u64, u64, u64,
                                              ctypes.c_void_p]
        lib.synth_dev_fill_normal.restype = ctypes.c_int
        _dev = lib
    return _dev


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


def normal(count, seed, stream, index0=0):
    out = np.empty(int(count), dtype=np.float32)
    rc = host_lib().synth_fill_normal(out.ctypes.data, out.size, seed, stream, index0,
                                      _threads())
    assert rc == 0
    return out


def normal_affine(count, seed, stream, mean, sd, index0=0):
    out = np.empty(int(count), dtype=np.float32)
    rc = host_lib().synth_fill_normal_affine(out.ctypes.data, out.size, seed, stream,
                                             index0, mean, sd, _threads())
    assert rc == 0
    return out


def below(count, seed, stream, n):
    out = np.empty(int(count), dtype=np.uint32)
    rc = host_lib().synth_fill_below(out.ctypes.data, out.size, seed, stream, n)
    assert rc == 0
    return out


def subset(n, k, seed, stream):
    out = np.empty(int(k), dtype=np.uint32)
    scratch = np.empty(int(n), dtype=np.uint32)
    rc = host_lib().synth_subset(out.ctypes.data, n, k, seed, stream, scratch.ctypes.data)
    assert rc == 0
    return out


def dev_fill_normal(ptr, count, seed, stream, index0=0, cuda_stream=0):
    """Fill ``count`` f32 at device address ``ptr`` with N01(seed, stream, index0+i)."""
    rc = dev_lib().synth_dev_fill_normal(ctypes.c_void_p(ptr), count, seed, stream,
                                         index0, ctypes.c_void_p(cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill_normal failed: cuda error {rc}")


@dataclasses.dataclass(frozen=True)
class Workload:
    """One batched-decode configuration and its input recipe."""
    name: str
    index: int
    B: int
    n_slots: int
    slot_ctx: int
    n_head: int
    n_kv_head: int
    head_dim: int
    theta: float
    sinks: bool
    steps: int = 1
    eps: float = 1e-6
    pos_rule: str = "uniform"      # uniform | fixed | skew | uniform_start
    slot_rule: str = "perm"        # perm | subset
    fixed_positions: tuple = ()
    start_hi: int = 0              # uniform_start: start positions in [0, start_hi]

    @property
    def seed(self):
        return 0x510751070000 + self.index

    @property
    def kv_dim(self):
        return self.n_kv_head * self.head_dim

    @property
    def scale(self):
        return float(np.float32(1.0 / np.sqrt(self.head_dim)))

    def replace(self, **kw):
        return dataclasses.replace(self, **kw)

    # --- integer inputs -------------------------------------------------
    def positions0(self):
        """Positions of the first step (u32[B])."""
        if self.pos_rule == "fixed":
            return np.asarray(self.fixed_positions, dtype=np.uint32)
        if self.pos_rule == "skew":
            # "interleaved": even rows at 16, odd rows at slot_ctx - 1
            p = np.empty(self.B, dtype=np.uint32)
            p[0::2] = 16
            p[1::2] = self.slot_ctx - 1
            return p
        if self.pos_rule == "uniform_start":
            return below(self.B, self.seed, S_POS, self.start_hi + 1)
        return below(self.B, self.seed, S_POS, self.slot_ctx)

    def positions(self, step=0):
        return (self.positions0() + np.uint32(step)).astype(np.uint32)

    def slots(self):
        if self.slot_rule == "subset":
            return subset(self.n_slots, self.B, self.seed, S_SLOTS)
        return subset(self.n_slots, self.n_slots, self.seed, S_SLOTS)[: self.B].copy()

    # --- float inputs ---------------------------------------------------
    def q(self, step=0):
        n = self.B * self.n_head * self.head_dim
        return normal(n, self.seed, S_Q + STEP_STRIDE * step).reshape(
            self.B, self.n_head, self.head_dim)

    def k_new(self, step=0):
        n = self.B * self.kv_dim
        return normal(n, self.seed, S_KNEW + STEP_STRIDE * step).reshape(
            self.B, self.n_kv_head, self.head_dim)

    def v_new(self, step=0):
        n = self.B * self.kv_dim
        return normal(n, self.seed, S_VNEW + STEP_STRIDE * step).reshape(
            self.B, self.n_kv_head, self.head_dim)

    def q_norm_w(self):
        return normal_affine(self.head_dim, self.seed, S_QNORM_W, 1.0, 0.1)

    def k_norm_w(self):
        return normal_affine(self.head_dim, self.seed, S_KNORM_W, 1.0, 0.1)

    def sink_logits(self):
        return normal(self.n_head, self.seed, S_SINKS) if self.sinks else None

    def inv_freq(self):
        """RoPE inverse frequencies theta^(-2i/hd), formed in f64, stored f32."""
        i = np.arange(self.head_dim // 2, dtype=np.float64)
        return (self.theta ** (-2.0 * i / self.head_dim)).astype(np.float32)

    # --- history K/V ------------------------------------------------------
    def hist_index0(self, slot, pos=0):
        return (int(slot) * self.slot_ctx + int(pos)) * self.kv_dim

    def hist_rows(self, which, slot, pos_begin, pos_end):
        """Host copy of history rows [pos_begin, pos_end) of ``slot``:
        f32[pos_end - pos_begin][n_kv_head][head_dim]."""
        stream = S_HIST_K if which == "k" else S_HIST_V
        n = (pos_end - pos_begin) * self.kv_dim
        return normal(n, self.seed, stream, self.hist_index0(slot, pos_begin)).reshape(
            pos_end - pos_begin, self.n_kv_head, self.head_dim)

    def kv_elems(self):
        return self.n_slots * self.slot_ctx * self.kv_dim

    def dev_fill_history(self, k_ptr, v_ptr, cuda_stream=0):
        """Fill the whole device K and V slot buffers with the history values."""
        chunk = 1 << 30
        total = self.kv_elems()
        for which, ptr in ((S_HIST_K, k_ptr), (S_HIST_V, v_ptr)):
            off = 0
            while off < total:
                n = min(chunk, total - off)
                dev_fill_normal(ptr + 4 * off, n, self.seed, which, off, cuda_stream)
                off += n

    # --- paged layout ------------------------------------------------------
    # The paged pool of a workload is its slot buffers cut into blocks of
    # ``block_size`` positions and shuffled: slot s's i-th block goes to pool
    # block perm[s * per + i] (per = slot_ctx / block_size), and a row's table
    # lists the pool blocks of its slot in order.
    def block_perm(self, block_size):
        assert self.slot_ctx % block_size == 0
        n_blocks = self.n_slots * (self.slot_ctx // block_size)
        return subset(n_blocks, n_blocks, self.seed, S_BLOCKS)

    def block_tables(self, block_size):
        """u32[B][slot_ctx / block_size]: row b's pool blocks, in key order."""
        per = self.slot_ctx // block_size
        perm = self.block_perm(block_size).reshape(self.n_slots, per)
        return perm[self.slots()].copy()

    def alg_bytes(self, positions):
        """Algorithmic HBM bytes of one decode step at ``positions``: history
        K+V read once per kv head, plus q/out/k_new/v_new and the K/V write."""
        p = np.asarray(positions, dtype=np.int64)
        hist = int(p.sum()) * 2 * self.kv_dim * 4
        io = self.B * (2 * self.n_head * self.head_dim + 2 * self.kv_dim) * 4
        wr = self.B * 2 * self.kv_dim * 4
        return hist + io + wr


WORKLOADS = {
    "tiny": Workload("tiny", 0, B=4, n_slots=4, slot_ctx=64, n_head=8, n_kv_head=2,
                     head_dim=64, theta=10000.0, sinks=False, pos_rule="fixed",
                     fixed_positions=(0, 5, 17, 63), slot_rule="perm"),
    "mid": Workload("mid", 1, B=32, n_slots=64, slot_ctx=4096, n_head=32, n_kv_head=8,
                    head_dim=128, theta=1e6, sinks=False, slot_rule="subset"),
    "skewed": Workload("skewed", 2, B=64, n_slots=64, slot_ctx=32768, n_head=16,
                       n_kv_head=8, head_dim=256, theta=10000.0, sinks=False,
                       pos_rule="skew", slot_rule="perm"),
    "sinks": Workload("sinks", 3, B=128, n_slots=128, slot_ctx=8192, n_head=64,
                      n_kv_head=8, head_dim=64, theta=150000.0, sinks=True,
                      slot_rule="perm"),
    "large": Workload("large", 4, B=256, n_slots=512, slot_ctx=2048, n_head=40,
                      n_kv_head=8, head_dim=128, theta=10000.0, sinks=False, steps=64,
                      pos_rule="uniform_start", start_hi=1983, slot_rule="subset"),
}

# Shapes the library accepts beyond the five workloads: eight query heads per
# kv head (the most the kernels take), where the per-key arithmetic is
# highest.  Same slots, positions and KV bytes per key as the batch-32
# workload.
EXTRA_WORKLOADS = {
    "gqa8_hd128": WORKLOADS["mid"].replace(name="gqa8_hd128", index=40, n_head=64),
    "gqa8_hd256": WORKLOADS["mid"].replace(name="gqa8_hd256", index=41, n_head=32, n_kv_head=4,
                                           head_dim=256),
}

# Scaled-down cases of two workloads, for profiler captures that must hold a
# few GB at most: the same head geometry, split chunk and persistent grid as
# the full workload, fewer rows and slots.
#   skewed_8:  8 rows (4 at position 16, 4 at 32767) on 8 slots of 32768;
#   large_32:  32 rows of the batch-256 workload's first step on 64 slots
#              (run with the full workload's 2048-key chunk: --split 2048 64).
PROFILE_WORKLOADS = {
    "skewed_8": WORKLOADS["skewed"].replace(name="skewed_8", index=30, B=8, n_slots=8),
    "large_32": WORKLOADS["large"].replace(name="large_32", index=31, B=32, n_slots=64, steps=1),
}
