"""Slot-ownership sharding of the decode step over several GPUs.

The rows of a step are independent sequences in disjoint slots ("Forward
Cuda Gemma", decodeBatch: B sequences each advance by one token over their
own slot; allocSlotKv: one slot per concurrent sequence).  So each rank --
one process, one GPU -- holds the slot KV of a contiguous range of the
global slots and runs only the rows whose slots it owns, reading only its
own HBM.  The step needs no collective.  ``all_gather_out`` is the optional
gather for a consumer that wants every row's output on every rank: one
all-gather over the process group (NCCL between GPUs, gloo on CPU).

The partition and the routing are the library's ``slot_kv_shard_range`` and
``slot_kv_shard_route``; this module marshals their arguments and moves rows
(an index gather of a step's inputs for this rank, the all-gather of
outputs).  The attention itself runs in the library's kernels through a
``SlotKV`` handle over this rank's slots.
"""
import ctypes

import numpy as np

from . import SlotKV, _check, _lib

__all__ = ["Route", "shard_range", "shard_route", "assemble", "all_gather_out",
           "ShardedSlotKV"]


def shard_range(n_ranks, n_slots, rank):
    """(first, count): rank ``rank`` owns global slots [first, first + count)."""
    first, count = ctypes.c_uint32(), ctypes.c_uint32()
    _check(_lib.slot_kv_shard_range(n_ranks, n_slots, rank, ctypes.byref(first),
                                    ctypes.byref(count)), "slot_kv_shard_range")
    return int(first.value), int(count.value)


class Route:
    """One step's rows grouped by the rank that owns their slot: rank r runs
    rows ``order[offsets[r]:offsets[r + 1]]`` with local slots
    ``local_slots[offsets[r]:offsets[r + 1]]``."""

    def __init__(self, n_ranks, order, offsets, local_slots):
        self.n_ranks = n_ranks
        self.order, self.offsets, self.local_slots = order, offsets, local_slots

    def rows(self, rank):
        return self.order[self.offsets[rank]:self.offsets[rank + 1]]

    def local(self, rank):
        return self.local_slots[self.offsets[rank]:self.offsets[rank + 1]]

    def count(self, rank):
        return int(self.offsets[rank + 1] - self.offsets[rank])

    def max_count(self):
        return int(np.max(np.diff(self.offsets.astype(np.int64)))) if self.n_ranks else 0


def shard_route(n_ranks, n_slots, slots):
    """Route a step's rows by the global slot ids ``slots`` (host array-like
    of B u32) to their owners (``slot_kv_shard_route``)."""
    s = np.ascontiguousarray(np.asarray(slots).astype(np.uint32))
    B = int(s.size)
    order = np.empty(B, dtype=np.uint32)
    local = np.empty(B, dtype=np.uint32)
    offsets = np.empty(n_ranks + 1, dtype=np.uint32)
    _check(_lib.slot_kv_shard_route(n_ranks, n_slots, B, s.ctypes.data if B else None,
                                    order.ctypes.data if B else None, offsets.ctypes.data,
                                    local.ctypes.data if B else None), "slot_kv_shard_route")
    return Route(n_ranks, order, offsets, local)


def assemble(route, outs, out=None):
    """Put the ranks' outputs (``outs[r]``: rank r's rows in route order)
    back at the rows' original indices of the step: out[order[i]] =
    cat(outs)[i]."""
    import torch
    cat = torch.cat([o[:route.count(r)] for r, o in enumerate(outs)], dim=0)
    if out is None:
        out = torch.empty_like(cat)
    idx = torch.from_numpy(route.order.astype(np.int64)).to(cat.device)
    out.index_copy_(0, idx, cat)
    return out


def all_gather_out(route, local_out, group=None):
    """Every rank's rows of the step on every rank, at their original
    indices: one all-gather over ``group`` (the ranks' outputs padded to the
    largest share), then ``assemble``."""
    import torch
    import torch.distributed as dist
    width = route.max_count()
    pad = torch.zeros((width,) + tuple(local_out.shape[1:]), dtype=local_out.dtype,
                      device=local_out.device)
    pad[:local_out.shape[0]] = local_out
    parts = [torch.empty_like(pad) for _ in range(route.n_ranks)]
    dist.all_gather(parts, pad, group=group)
    return assemble(route, parts)


class ShardedSlotKV:
    """Rank ``rank`` of ``n_ranks``: a ``SlotKV`` over the global slots this
    rank owns (``shard_range``), on the current device.  ``k_buf``/``v_buf``,
    if given, hold only those slots: [count][slot_ctx][n_kv_head][head_dim]."""

    def __init__(self, n_ranks, rank, n_slots, slot_ctx, n_kv_head, head_dim, max_rows,
                 max_n_head, k_buf=None, v_buf=None):
        self.n_ranks, self.rank, self.n_slots = int(n_ranks), int(rank), int(n_slots)
        self.first, self.count = shard_range(n_ranks, n_slots, rank)
        self.kv = SlotKV(self.count, slot_ctx, n_kv_head, head_dim, max_rows, max_n_head,
                         k_buf=k_buf, v_buf=v_buf)

    def route(self, slots):
        return shard_route(self.n_ranks, self.n_slots, slots)

    def decode_batch_attn(self, route, q, k_new, v_new, positions, q_norm_w, k_norm_w,
                          inv_freq, sinks, eps, scale, out=None, stream=None):
        """This rank's rows of one step.  q, k_new, v_new, positions are the
        whole step's tensors ([B] rows) on this rank's device; ``route`` is
        ``shard_route`` of the step's global slots.  Returns the rows'
        outputs [count][n_head][head_dim], in route order."""
        import torch
        n = route.count(self.rank)
        shape = (n, int(q.shape[1]), int(q.shape[2]))
        if out is None:
            out = torch.empty(shape, dtype=torch.float32, device=q.device)
        if n == 0:
            return out
        rows = torch.from_numpy(route.rows(self.rank).astype(np.int64)).to(q.device)
        local = torch.from_numpy(route.local(self.rank).astype(np.int32)).to(q.device)
        sel = lambda t: t.index_select(0, rows).contiguous()  # noqa: E731
        self.kv.decode_batch_attn(sel(q), sel(k_new), sel(v_new), sel(positions), local,
                                  q_norm_w, k_norm_w, inv_freq, sinks, out, eps, scale,
                                  stream=stream)
        return out

    def free(self):
        self.kv.free()
