"""Benchmark: batched slot-KV decode attention on GB300.

A step is one decode_batch_attn call over the workload's B rows (for the
multi-step workload, its 64 consecutive calls).  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload large]
                    [--impl gpu|reference]

The default workload is the largest single-GPU configuration: 256 rows on
512 slots of 2048 positions, 40 query / 8 kv heads, head dim 128, 64
consecutive decode steps per bench step.

value       rows/s with every input resident in HBM, CUDA events on the
            launching stream around exactly K steps (max over ranks); the
            W warm-up steps run directly before the timed region;
e2e         the same metric through decode_batch_attn_host: per step the
            inputs are copied from pinned host memory and the output back;
roofline    one decode call's algorithmic HBM bytes over its mean (and
            median) CUDA-event time, against the measured copy bandwidth;
per_config  the same figures for each of the four bandwidth-target
            workloads (mid, skewed, sinks, large), each timed on its own in
            the same run;
cpu_baseline  the CPU oracle on the host's cores over a bounded sample, and
            the same rows on one thread.
Under torchrun each rank runs its own copy of the workload on its own GPU
(rows are independent; no collective on the data path): weak scaling.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

HBM_FALLBACK_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024     # GB300 L2
FLUSH_BYTES = 256 * 1024 * 1024  # written between calls of a step that fits in L2

# DRAM bytes (read + write) per decode call (plan + decode kernels) from ncu
# captures of dram__bytes_read.sum and dram__bytes_write.sum, valid only for
# the kernel code they were taken on (code_hash of decode_attn.cuh).
MEASURED_TRAFFIC = {
    # all at full size; large's is its first step's ratio to the algorithmic
    # bytes times the mean algorithmic bytes of its 64 steps
    # (plan + decode kernel bytes, the mean of two calls; of 18 calls for the
    # eight-heads-per-kv-head workloads)
    "26542fcb3b784732": {"mid": 551_830_912, "sinks": 2_336_513_024,
                         "skewed": 17_227_054_208, "large": 2_238_835_960,
                         "gqa8_hd128": 509_073_606, "gqa8_hd256": 627_442_587},
}


def code_hash(name):
    """sha256 prefix of a kernel source with its comments and whitespace
    removed: the measured counters below stay tied to the code, not to the
    wording of its comments."""
    import hashlib
    import re
    with open(os.path.join(ROOT, "sequence_slot_kv_gb300", "csrc", name)) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = " ".join(text.split())
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def kernel_source_hash():
    return code_hash("decode_attn.cuh")


def measured_traffic(workload):
    return MEASURED_TRAFFIC.get(kernel_source_hash(), {}).get(workload)


# DRAM read + write bytes of one tensor-core prefill kernel launch on the
# prefill workload of a geometry (ncu one-pass counters, the mean over the
# full-size calls' launches), keyed by code_hash of prefill_tc.cuh; reported
# only while the kernel is the one measured.
MEASURED_PREFILL_TRAFFIC = {"56858cc248ba86b3": {"mid": 247_501_909, "sinks": 170_577_280}}


def prefill_source_hash():
    return code_hash("prefill_tc.cuh")


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return HBM_FALLBACK_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if self.t0 - 0.06 <= r[0] <= self.t1 + 0.06]
        used = inside if inside else sorted(rows, key=lambda r: abs(r[0] - self.t0))[:2]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in used:
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                pass
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(used),
                "samples_in_region": len(inside)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, device=None):
    """The largest value of ``x`` over all ranks (identity when not
    distributed).  Timing only; rows never cross ranks."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rows_per_s(rows_per_rank_step, steps, world, max_seconds):
    """Weak scaling: every rank runs its own copy of the workload."""
    return world * rows_per_rank_step * steps / max_seconds


def oracle_sample(w, rows, n_threads):
    """Compact host slot buffers for the oracle over ``rows`` (untimed set-up)."""
    slots = w.slots()
    p = w.positions(0)
    ctx = int(max(p[r] for r in rows)) + w.steps
    K = np.empty((len(rows), ctx, w.n_kv_head, w.head_dim), dtype=np.float32)
    V = np.empty_like(K)
    for i, r in enumerate(rows):
        K[i] = w.hist_rows("k", slots[r], 0, ctx)
        V[i] = w.hist_rows("v", slots[r], 0, ctx)
    return K, V


class OracleSample:
    """The CPU oracle, as it stands, over a fixed sample of the workload's
    rows (min(B, cores) rows of its first step, at evenly spaced quantiles of
    position).  The sample's slot
    history is regenerated on the host once, outside any timing; the oracle
    rewrites the same K/V rows on every call, so calls repeat exactly."""

    def __init__(self, w, n_threads, flags=0, paged_bs=0, n_rows=None):
        import oracle
        self.o = oracle.default()
        self.w = w
        self.n_threads = n_threads
        self.flags = flags
        self.paged_bs = paged_bs
        # rows at evenly spaced quantiles of position, so the sample has the
        # workload's mix of history lengths
        k = min(w.B, n_rows or n_threads)
        order = np.argsort(w.positions(0), kind="stable")
        self.rows = sorted(int(order[int(i)]) for i in
                           np.linspace(0, w.B - 1, k).round().astype(int))
        r = self.rows
        if paged_bs:
            # the sampled rows' blocks only, in a compact pool, with tables into it
            self.K, self.V, addr = paged_oracle_sample(w, r, paged_bs)
        else:
            self.K, self.V = oracle_sample(w, r, n_threads)
            addr = np.arange(len(r), dtype=np.uint32)
        self.args = (w.q(0)[r], w.k_new(0)[r], w.v_new(0)[r], w.positions(0)[r],
                     addr, w.q_norm_w(), w.k_norm_w(),
                     w.inv_freq(), w.sink_logits(), w.eps, w.scale)

    @property
    def threads(self):
        """Threads the oracle actually runs (one row per thread at most)."""
        return min(self.n_threads, len(self.rows))

    def step(self):
        t0 = time.perf_counter()
        if self.paged_bs:
            self.o.decode_batch_paged(self.K, self.V, *self.args, n_threads=self.n_threads,
                                      flags=self.flags)
        else:
            self.o.decode_batch(self.K, self.V, *self.args, n_threads=self.n_threads,
                                flags=self.flags)
        return time.perf_counter() - t0

    def describe(self, steps, seconds):
        pos = self.w.positions(0)[self.rows]
        how = (f" over {self.paged_bs}-key blocks" if self.paged_bs else "") + \
              (f", norm options {self.flags}" if self.flags else "")
        return (f"{len(self.rows)} rows (positions {pos.min()}..{pos.max()}, mean "
                f"{pos.mean():.0f}) of the {self.w.name} workload's "
                f"first step per oracle call{how}, {steps} calls, {seconds:.1f} s, "
                + ("on one thread" if self.n_threads == 1 else
                   f"rows split over {self.n_threads} threads"))


def paged_oracle_sample(w, rows, bs):
    """Compact host block pool holding only the blocks of ``rows``, and their
    tables into it (untimed set-up)."""
    slots = w.slots()
    p = w.positions(0)
    used = [int(p[r]) // bs + 1 for r in rows]
    K = np.empty((sum(used), bs, w.n_kv_head, w.head_dim), dtype=np.float32)
    V = np.empty_like(K)
    tab = np.zeros((len(rows), max(used)), dtype=np.uint32)
    base = 0
    for i, r in enumerate(rows):
        n = used[i]
        K[base:base + n] = w.hist_rows("k", slots[r], 0, n * bs).reshape(n, bs, w.n_kv_head,
                                                                        w.head_dim)
        V[base:base + n] = w.hist_rows("v", slots[r], 0, n * bs).reshape(n, bs, w.n_kv_head,
                                                                        w.head_dim)
        tab[i, :n] = np.arange(base, base + n, dtype=np.uint32)
        base += n
    return K, V, tab


def time_oracle(w, budget_s, n_threads, flags=0, paged_bs=0, n_rows=None):
    """rows/s of the oracle over calls on its sample until ``budget_s``."""
    smp = OracleSample(w, n_threads, flags, paged_bs, n_rows)
    smp.step()                                       # warm caches and pages
    calls, spent = 0, 0.0
    while spent < budget_s:
        spent += smp.step()
        calls += 1
    return len(smp.rows) * calls / spent, smp.describe(calls, spent), smp.threads


def run_reference(args, w):
    """The CPU oracle, as it stands, on this arm's workload (prefill, paged
    layout and norm options included), each step a bounded sample of it."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    if args.prefill:
        w, slots, pos = prefill_workload(args.prefill_geometry)
        smp = PrefillOracleSample(w, slots, pos, cores)
        per_step, unit = smp.n_seq, "tokens/s"
        metric, config = "slot-attn prefill tokens/s", prefill_config(w)
    else:
        smp = OracleSample(w, cores, flags=args.options, paged_bs=args.paged)
        per_step, unit = len(smp.rows), "rows/s"
        metric, config = "slot-attn decode rows/s", config_of(w, args)
    for _ in range(args.warmup):
        smp.step()
    spent = sum(smp.step() for _ in range(args.steps))
    value = per_step * args.steps / spent
    line = {
        "impl": "reference", "metric": metric, "value": value,
        "unit": unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * spent / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": value, "unit": unit, "cores": smp.threads, "kind": "oracle",
                         "sample": smp.describe(args.steps, spent)},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# the library's and the oracle's option bits agree: 1 weightless V norm,
# 2 (1 + w) norm weights
OPTION_NAMES = {1: "weightless V norm", 2: "(1 + w) Q/K norm weights",
                3: "weightless V norm and (1 + w) Q/K norm weights"}


def config_of(w, args=None):
    """The workload's config; with ``args``, its layout and norm options."""
    cfg = {"workload": w.name, "B": w.B, "n_slots": w.n_slots, "slot_ctx": w.slot_ctx,
           "n_head": w.n_head, "n_kv_head": w.n_kv_head, "head_dim": w.head_dim,
           "steps_per_call_sequence": w.steps, "sinks": w.sinks,
           "l2": ("inputs larger than L2 (history K/V read per step >> 129 MB)"
                  if w.alg_bytes(w.positions(0)) >= 2 * L2_BYTES else
                  f"L2 flushed between calls ({FLUSH_BYTES >> 20} MiB written outside "
                  f"the timed calls)")}
    if args is not None and args.paged:
        cfg.update({"kv_layout": "paged", "block_size": args.paged,
                    "block_order": "seeded shuffle over the pool"})
    if args is not None and args.options:
        cfg["norm_options"] = OPTION_NAMES[args.options]
    return cfg


# The four workloads the bandwidth target covers; each is timed in every run
# and reported under per_config.
TARGET_WORKLOADS = ("mid", "skewed", "sinks", "large")
# A per-config entry's timed region runs at least this long (more steps than
# --steps where one step is short), so its clock record has several samples.
MIN_REGION_S = 0.25


class DeviceWorkload:
    """A workload resident on one device: slot (or paged) K/V filled with the
    history recipe, a handle adopting it, every step's inputs uploaded."""

    def __init__(self, w, dev, stream, paged=0, split=None, options=0):
        import torch
        import sequence_slot_kv_gb300 as skv
        self.w, self.dev, self.stream, self.bs = w, dev, stream, paged
        sp = self.sp = stream.cuda_stream
        shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
        with torch.cuda.stream(stream):
            K = torch.empty(shape, dtype=torch.float32, device=dev)
            V = torch.empty(shape, dtype=torch.float32, device=dev)
        w.dev_fill_history(K.data_ptr(), V.data_ptr(), sp)
        bs = paged
        self.tables_np = None
        if bs:
            # paged layout: the same history cut into blocks of bs positions,
            # shuffled over a pool; each row reads its blocks through its table
            pshape = (w.n_slots * (w.slot_ctx // bs), bs, w.n_kv_head, w.head_dim)
            perm = self.dev_t(w.block_perm(bs).astype(np.int64))
            torch.cuda.synchronize(dev)
            pools = []
            for src in (K, V):
                dst = torch.empty(pshape, dtype=torch.float32, device=dev)
                dst[perm] = src.view(pshape)
                pools.append(dst)
            torch.cuda.synchronize(dev)
            del K, V
            K, V = pools
            self.tables_np = w.block_tables(bs).astype(np.int32)
            self.tables = self.dev_t(self.tables_np)
            self.kv = skv.SlotKV(pshape[0], bs, w.n_kv_head, w.head_dim, w.B, w.n_head,
                                 k_buf=K, v_buf=V)
        else:
            self.kv = skv.SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head,
                                 k_buf=K, v_buf=V)
        self.K, self.V = K, V
        if split:
            self.kv.set_split(*split)
        if options:
            self.kv.set_options(options)
        self.qw, self.kw, self.inv = (self.dev_t(w.q_norm_w()), self.dev_t(w.k_norm_w()),
                                      self.dev_t(w.inv_freq()))
        self.sinks = None if not w.sinks else self.dev_t(w.sink_logits())
        self.slots_np = w.slots().astype(np.int32)
        self.slots = self.dev_t(self.slots_np)
        self.nsub = w.steps
        self.q = [self.dev_t(w.q(t)) for t in range(self.nsub)]
        self.kn = [self.dev_t(w.k_new(t)) for t in range(self.nsub)]
        self.vn = [self.dev_t(w.v_new(t)) for t in range(self.nsub)]
        self.pos = [self.dev_t(w.positions(t).astype(np.int32)) for t in range(self.nsub)]
        self.out = torch.empty((w.B, w.n_head, w.head_dim), dtype=torch.float32, device=dev)
        # paged mode also reads each used table entry once
        self.bytes_per_launch = [
            w.alg_bytes(w.positions(t)) +
            (int((w.positions(t).astype(np.int64) // bs + 1).sum()) * 4 if bs else 0)
            for t in range(self.nsub)]
        torch.cuda.synchronize(dev)

    def dev_t(self, a):
        import torch
        return torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def decode(self, t):
        w = self.w
        if self.bs:
            self.kv.decode_batch_attn_paged(self.q[t], self.kn[t], self.vn[t], self.pos[t],
                                            self.tables, self.qw, self.kw, self.inv, self.sinks,
                                            self.out, w.eps, w.scale, stream=self.sp)
        else:
            self.kv.decode_batch_attn(self.q[t], self.kn[t], self.vn[t], self.pos[t],
                                      self.slots, self.qw, self.kw, self.inv, self.sinks,
                                      self.out, w.eps, w.scale, stream=self.sp)

    def one_step(self):
        for t in range(self.nsub):
            self.decode(t)

    def launches_per_call(self):
        w = self.w
        return self.kv.call_shape(w.B, bt_stride=(w.slot_ctx // self.bs if self.bs else 0))[2]

    def free(self):
        import torch
        self.kv.free()
        for name in ("K", "V", "q", "kn", "vn", "pos", "out", "slots", "tables"):
            if hasattr(self, name):
                delattr(self, name)
        torch.cuda.synchronize(self.dev)
        torch.cuda.empty_cache()


GROUP_CALLS = 64   # calls between two events of the timed region


def time_device(dw, steps, warmup, local, world, graph=False):
    """Time ``steps`` steps of ``dw`` on its stream with CUDA events.  The
    warm-up runs directly before the timed region (no idle gap in which
    clocks could drop), with the clock sampler already running.

    Calls run back to back, as a decode loop runs them: events are recorded
    only at the boundaries of groups of about GROUP_CALLS calls (whole
    steps).  An event between two calls would serialise the stream there
    (about 4 us a call on GB300) and keep the next call's plan kernel from
    launching during the previous call's tail.  The per-call samples are the
    groups' mean call times.

    A workload whose bytes fit in L2 twice over would be timed warm: a buffer
    larger than L2 is written before every call, outside a pair of events
    around the call, and the step time is the sum of the calls' times.

    Returns (total_ms, calls, per-call ms samples, clocks)."""
    import torch
    dev, stream = dw.dev, dw.stream
    nsub = dw.nsub

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    g = None
    if graph:
        # one step (all its decode calls) captured once and replayed per step
        dw.one_step()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                dw.one_step()
    flush = None
    if statistics.mean(dw.bytes_per_launch) < 2 * L2_BYTES:
        flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(warmup):
        g.replay() if g is not None else dw.one_step()
    torch.cuda.synchronize(dev)
    assert dw.kv.get_status(dw.sp) == 0
    for _ in range(2):       # warm again after the status read, right before timing
        g.replay() if g is not None else dw.one_step()
    calls = steps * nsub
    event = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    if flush is not None:
        # one (flush, timed unit) per call, or per replay of a captured step
        units = steps if g is not None else calls
        ev = [(event(), event()) for _ in range(units)]
        barrier()
        clocks.mark("begin")
        with torch.cuda.stream(stream):
            for i in range(units):
                flush.fill_(float(i))
                ev[i][0].record(stream)
                g.replay() if g is not None else dw.decode(i % nsub)
                ev[i][1].record(stream)
        barrier()
        clocks.mark("end")
        unit_ms = [a.elapsed_time(b) for a, b in ev]
        total_ms = sum(unit_ms)  # the flushes are not the step's
        samples = [x / nsub for x in unit_ms] if g is not None else unit_ms
        del flush
    else:
        group = max(1, -(-GROUP_CALLS // nsub))  # steps per group
        marks = [event() for _ in range(-(-steps // group) + 1)]
        barrier()
        clocks.mark("begin")
        with torch.cuda.stream(stream):
            for s in range(steps):
                if s % group == 0:
                    marks[s // group].record(stream)
                g.replay() if g is not None else dw.one_step()
            marks[-1].record(stream)
        barrier()
        clocks.mark("end")
        total_ms = marks[0].elapsed_time(marks[-1])
        samples = []
        for k in range(len(marks) - 1):
            n = (min(steps, (k + 1) * group) - k * group) * nsub
            samples.append(marks[k].elapsed_time(marks[k + 1]) / n)
    clk = clocks.stop()
    assert dw.kv.get_status(dw.sp) == 0
    return total_ms, calls, samples, clk


def roofline_of(dw, total_ms, calls, samples, traffic=None):
    """The decode call's roofline entry: algorithmic bytes over the mean call
    time (the timed region over its calls), against the measured copy
    bandwidth; the median over the per-call samples beside it."""
    peak, peak_kind = peak_hbm()
    mean_s = total_ms / calls / 1e3
    med_s = statistics.median(samples) / 1e3
    alg = statistics.mean(dw.bytes_per_launch)
    achieved = alg / mean_s / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
            "traffic_per_alg_byte": (traffic / alg if traffic else None),
            "alg_bytes_per_launch": alg, "avg_launch_us": mean_s * 1e6,
            "median_launch_us": med_s * 1e6,
            "median_frac": alg / med_s / 1e9 / peak,
            "kernel": "slotkv_plan_kernel + slotkv_decode_attn_kernel (one decode call)"}


def time_e2e(dw, steps, warmup, world):
    """The same metric end to end: every step copies its inputs from pinned
    host memory and reads the output back, through prepared host calls
    (SlotKV.prepare_host_call: the host entry decode_batch_attn_host, or
    decode_batch_attn_paged_host, with its arguments checked once, as a
    serving loop that reuses its pinned buffers would call it).  The calls
    are prepared before the timed region; a step enqueues its calls and
    synchronises its stream once at its end."""
    import torch
    w, dev, stream, nsub, bs = dw.w, dw.dev, dw.stream, dw.nsub, dw.bs
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    hq = [pin(w.q(t)) for t in range(nsub)]
    hk = [pin(w.k_new(t)) for t in range(nsub)]
    hv = [pin(w.v_new(t)) for t in range(nsub)]
    hp = [pin(w.positions(t).astype(np.int32)) for t in range(nsub)]
    hs = pin(dw.tables_np if bs else dw.slots_np)
    hout = torch.empty((w.B, w.n_head, w.head_dim), dtype=torch.float32).pin_memory()
    calls = [dw.kv.prepare_host_call(hq[t], hk[t], hv[t], hp[t], None if bs else hs, dw.qw,
                                     dw.kw, dw.inv, dw.sinks, hout, w.eps, w.scale,
                                     block_tables=hs if bs else None)
             for t in range(nsub)]

    def e2e_step():
        # the step's calls are enqueued back to back; the step ends when its
        # stream is synchronised (its outputs are then in host memory)
        for c in calls:
            c(stream=dw.sp, sync=False)
        dw.stream.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(1, warmup)):
        e2e_step()
    barrier()
    if statistics.mean(dw.bytes_per_launch) < 2 * L2_BYTES:
        # as for the device time: L2 written over between steps, outside them
        flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        e2e_s = 0.0
        for k in range(steps):
            with torch.cuda.stream(stream):
                flush.fill_(float(k))
            stream.synchronize()
            t0 = time.perf_counter()
            e2e_step()
            e2e_s += time.perf_counter() - t0
        del flush
        barrier()
    else:
        t0 = time.perf_counter()
        for _ in range(steps):
            e2e_step()
        barrier()
        e2e_s = time.perf_counter() - t0
    for c in calls:
        c.free()
    h2d = nsub * (hq[0].numel() + hk[0].numel() + hv[0].numel() + hp[0].numel()
                  + hs.numel()) * 4
    d2h = nsub * hout.numel() * 4
    return e2e_s, h2d, d2h


def per_config_entry(name, args, dev, stream, local):
    """One target workload timed on its own (same --warmup; at least --steps
    steps, more where a step is short, so the region lasts MIN_REGION_S)."""
    w = synth.WORKLOADS[name]
    dw = DeviceWorkload(w, dev, stream, split=args.split)
    try:
        est_ms, _, _, _ = time_device(dw, 3, 1, local, 1)
        steps = max(args.steps, int(np.ceil(MIN_REGION_S * 1e3 / max(est_ms / 3, 1e-3))))
        total_ms, calls, samples, clk = time_device(dw, steps, args.warmup, local, 1)
        rl = roofline_of(dw, total_ms, calls, samples, traffic=measured_traffic(name))
        return {"value": w.B * dw.nsub * steps / (total_ms / 1e3), "unit": "rows/s",
                "steps": steps, "calls": calls, "ms_per_step": total_ms / steps,
                "avg_launch_us": rl["avg_launch_us"],
                "median_launch_us": rl["median_launch_us"],
                "alg_bytes_per_launch": rl["alg_bytes_per_launch"],
                "achieved_GBps": rl["achieved"], "frac": rl["frac"],
                "median_frac": rl["median_frac"], "traffic": rl["traffic"],
                "traffic_per_alg_byte": rl["traffic_per_alg_byte"], "clocks": clk}
    finally:
        dw.free()


def run_ncu_target(args, w):
    """For profiler captures: set the workload up, make one warm-up call and
    one more call of its first step, nothing else.  Prints no bench line."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    dw = DeviceWorkload(w, dev, stream, paged=args.paged, split=args.split, options=args.options)
    for _ in range(2):
        dw.decode(0)
    torch.cuda.synchronize(dev)
    assert dw.kv.get_status(dw.sp) == 0
    print(json.dumps({"ncu_target": w.name, "calls": 2,
                      "alg_bytes_per_launch": dw.bytes_per_launch[0],
                      "chunk_ctas_kernels": dw.kv.call_shape(w.B)}), flush=True)
    dw.free()


def run_gpu(args, w):
    import torch
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)

    dw = DeviceWorkload(w, dev, stream, paged=args.paged, split=args.split,
                        options=args.options)
    total_ms, calls, samples, clk = time_device(dw, args.steps, args.warmup, local, world,
                                                graph=args.graph)
    total_ms = max_over_ranks(total_ms, dev)
    rows_per_step = w.B * dw.nsub
    value = whole_job_rows_per_s(rows_per_step, args.steps, world, total_ms / 1e3)
    e2e_s, h2d, d2h = time_e2e(dw, args.steps, args.warmup, world)
    e2e_s = max_over_ranks(e2e_s, dev)
    e2e_value = whole_job_rows_per_s(rows_per_step, args.steps, world, e2e_s)
    traffic = (args.traffic if args.traffic is not None
               else (None if args.paged or args.options else measured_traffic(w.name)))
    line = {
        "metric": "slot-attn decode rows/s", "value": value, "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_of(w, args),
        "roofline": roofline_of(dw, total_ms, calls, samples, traffic),
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        # the library's kernels per decode call (plan + decode, or decode alone)
        "gpu_launches": args.steps * dw.nsub * dw.launches_per_call(),
        "graph": bool(args.graph),
        "clocks": clk,
    }
    headline_entry = None
    if w.name in TARGET_WORKLOADS and not (args.paged or args.options or args.graph):
        rl = line["roofline"]
        headline_entry = {
            "value": value, "unit": "rows/s", "steps": args.steps,
            "calls": calls, "ms_per_step": total_ms / args.steps,
            "avg_launch_us": rl["avg_launch_us"], "median_launch_us": rl["median_launch_us"],
            "alg_bytes_per_launch": rl["alg_bytes_per_launch"], "achieved_GBps": rl["achieved"],
            "frac": rl["frac"], "median_frac": rl["median_frac"], "traffic": rl["traffic"],
            "traffic_per_alg_byte": rl["traffic_per_alg_byte"], "clocks": clk}
    dw.free()
    if rank == 0 and world == 1 and not args.no_per_config:
        per = {}
        for name in TARGET_WORKLOADS:
            if headline_entry is not None and name == w.name:
                per[name] = headline_entry
            else:
                per[name] = per_config_entry(name, args, dev, stream, local)
        line["per_config"] = per
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        v, desc, used = time_oracle(w, args.cpu_budget, cores, flags=args.options,
                                    paged_bs=args.paged)
        # the same rows on one thread
        v1, desc1, _ = time_oracle(w, args.cpu_budget / 3, 1, flags=args.options,
                                   paged_bs=args.paged, n_rows=cores)
        line["cpu_baseline"] = {"value": v, "unit": "rows/s", "cores": used, "kind": "oracle",
                                "sample": desc,
                                "single_thread": {"value": v1, "sample": desc1}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


PREFILL_SEQ, PREFILL_HIST, PREFILL_CHUNK = 8, 1536, 512


def prefill_workload(geometry="mid"):
    """The prefill workload at a decode workload's head geometry (mid: 32 / 8
    heads at hd 128; sinks: 64 / 8 heads at hd 64): 8 sequences in slots 0,
    2, .., 14, each adding a 512-token prompt chunk after 1536 positions of
    history.  Returns the workload (one row per token) and the tokens' slots
    and positions."""
    n_seq, hist, chunk = PREFILL_SEQ, PREFILL_HIST, PREFILL_CHUNK
    n_tok = n_seq * chunk
    w = synth.WORKLOADS[geometry].replace(
        name="prefill" if geometry == "mid" else f"prefill_{geometry}", index=20, B=n_tok,
        n_slots=16, slot_ctx=hist + chunk, pos_rule="fixed",
        fixed_positions=tuple([0] * n_tok))
    slots = np.repeat(np.arange(n_seq, dtype=np.int32) * 2, chunk)
    pos = np.tile(np.arange(hist, hist + chunk, dtype=np.int32), n_seq)
    return w, slots, pos


def prefill_config(w):
    return {"workload": w.name, "sequences": PREFILL_SEQ, "history": PREFILL_HIST,
            "prompt_chunk": PREFILL_CHUNK, "n_head": w.n_head, "n_kv_head": w.n_kv_head,
            "head_dim": w.head_dim}


def run_prefill(args):
    """Batched causal prefill (prefill_workload).  A step is one
    prefill_batch_attn call over all 4096 tokens."""
    import torch
    import sequence_slot_kv_gb300 as skv
    w, slots, pos = prefill_workload(args.prefill_geometry)
    n_tok = w.B
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    K = torch.empty(shape, device=dev)
    V = torch.empty(shape, device=dev)
    w.dev_fill_history(K.data_ptr(), V.data_ptr(), sp)
    kv = skv.SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, n_tok, w.n_head,
                    k_buf=K, v_buf=V)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    q, kn, vn = d(w.q()), d(w.k_new()), d(w.v_new())
    ps, ss = d(pos), d(slots)
    qw, kw, inv = d(w.q_norm_w()), d(w.k_norm_w()), d(w.inv_freq())
    out = torch.empty((n_tok, w.n_head, w.head_dim), device=dev)

    def step():
        kv.prefill_batch_attn(q, kn, vn, ps, ss, qw, kw, inv, None, out, w.eps, w.scale,
                              stream=sp)

    step()
    torch.cuda.synchronize(dev)
    assert kv.get_status(sp) == 0
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):      # directly before the timed region
        step()
    b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark("begin")
    b.record(stream)
    for _ in range(args.steps):
        step()
    e.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark("end")
    clk = clocks.stop()
    ms = b.elapsed_time(e) / args.steps
    assert kv.get_status(sp) == 0

    # End to end: every step moves its inputs from page-locked host memory
    # and its output back through the host entry (prefill_batch_attn_host,
    # synchronous).
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    hq, hkn, hvn, hps, hss = pin(w.q()), pin(w.k_new()), pin(w.v_new()), pin(pos), pin(slots)
    hout = torch.empty(tuple(out.shape), dtype=torch.float32).pin_memory()

    def e2e_step():  # the same call as the device step (no sinks)
        kv.prefill_batch_attn_host(hq, hkn, hvn, hps, hss, qw, kw, inv, None, hout, w.eps,
                                   w.scale, stream=sp)

    e2e_step()
    e2e_steps = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in (hq, hkn, hvn, hps, hss))
    d2h = hout.numel() * hout.element_size()
    # distinct K/V bytes the call reads (each sequence's keys once per kv
    # head) and its per-token inputs and outputs
    seq_keys = int(sum(int(pos[slots == s].max()) + 1 for s in np.unique(slots)))
    key_bytes = seq_keys * 2 * w.kv_dim * 4
    io = n_tok * (2 * w.n_head * w.head_dim + 4 * w.kv_dim) * 4
    # Useful f32 flops: per token and query head, 2 hd per key for the score
    # and 2 hd per key for the value sum, over keys 0..pos.
    flops = 4 * w.head_dim * w.n_head * int((pos.astype(np.int64) + 1).sum())
    tflops = flops / (ms / 1e3) / 1e12
    if kv.call_shape(n_tok, prefill=True)[2] == 3:
        # tensor cores: every f32 product is three TF32 products (hi*hi,
        # hi*lo, lo*hi), against the dense TF32 peak
        peak, peak_kind = tf32_peak()
        roof = {"bound": "tensor", "achieved": 3 * tflops, "peak": peak, "unit": "TFLOP/s",
                "frac": 3 * tflops / peak, "peak_kind": peak_kind,
                "achieved_is": "3 TF32 products per useful f32 product, useful (causal) keys only",
                "kernel": "slotkv_prefill_tc_kernel (with its prep and plan kernels)",
                "traffic": MEASURED_PREFILL_TRAFFIC.get(prefill_source_hash(), {}).get(
                    args.prefill_geometry),
                "traffic_unit": "DRAM bytes per tensor-core kernel launch (read + write)"}
    else:
        peak, peak_kind = alu_peak_f32(dev)
        roof = {"bound": "alu", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                "frac": tflops / peak, "peak_kind": peak_kind,
                "kernel": "slotkv_decode_attn_kernel (prefill mode)"}
    roof.setdefault("traffic", None)
    roof.update({"alg_flops_per_launch": flops, "avg_launch_us": ms * 1e3,
                 "effective_f32_TFLOPs": tflops})
    line = {"metric": "slot-attn prefill tokens/s", "value": n_tok / (ms / 1e3),
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": prefill_config(w),
            "roofline": roof,
            "key_bytes_per_step": key_bytes, "io_bytes_per_step": io,
            "e2e": {"value": n_tok / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * kv.call_shape(n_tok, prefill=True)[2],
            "clocks": clk}
    if not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        v, desc, used = time_oracle_prefill(w, slots, pos, args.cpu_budget, cores)
        v1, desc1, _ = time_oracle_prefill(w, slots, pos, args.cpu_budget / 3, 1)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": used,
                                "kind": "oracle", "sample": desc,
                                "single_thread": {"value": v1, "sample": desc1}}
    print(json.dumps(line), flush=True)
    kv.free()


def tf32_peak():
    """Dense TF32 tensor peak: the measured bf16 GEMM peak (burst) times the
    nominal TF32/bf16 ratio 1.1/2.25, in TFLOP/s."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
        kind = "measured bf16 burst x 1.1/2.25"
    except (OSError, KeyError, ValueError):
        bf16, kind = 1900.0, "fallback bf16 1.9 PFLOP/s x 1.1/2.25"
    return bf16 * 1.1 / 2.25, kind


def alu_peak_f32(dev):
    """f32 FMA peak: SMs x 128 FP32 lanes x 2 flops x the maximum SM clock
    (MEASURED_PEAKS.json's sm_max_mhz, else 2070 MHz), in TFLOP/s."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except (OSError, ValueError):
        pass
    return sms * 128 * 2 * mhz * 1e6 / 1e12, f"derived: {sms} SMs x 128 FP32 lanes x 2 x {mhz:.0f} MHz"


class PrefillOracleSample:
    """The CPU oracle on the prefill workload, as it stands: each call takes
    the next prompt token of every sequence (one decode step per token, in
    position order, the sequences' tokens in parallel) on host copies of the
    sequences' slots (regenerated once, outside any timing).  After the last
    token of the chunk it starts again from the first; the rows a call
    rewrites are the ones it wrote the first time, so calls repeat exactly."""

    def __init__(self, w, slots, pos, n_threads):
        import oracle
        self.o = oracle.default()
        self.w, self.pos = w, pos
        n_seq, chunk = PREFILL_SEQ, PREFILL_CHUNK
        self.n_seq, self.chunk = n_seq, chunk
        self.n_threads = min(n_threads, n_seq)
        seq_slots = slots[::chunk].astype(np.int64)
        self.first = pos[::chunk].astype(np.int64)
        ctx = int(self.first.max()) + chunk
        self.K = np.empty((n_seq, ctx, w.n_kv_head, w.head_dim), dtype=np.float32)
        self.V = np.empty_like(self.K)
        for i, s_ in enumerate(seq_slots):
            self.K[i] = w.hist_rows("k", s_, 0, ctx)
            self.V[i] = w.hist_rows("v", s_, 0, ctx)
        self.q, self.kn, self.vn = w.q(), w.k_new(), w.v_new()
        self.compact = np.arange(n_seq, dtype=np.uint32)
        self.calls = 0
        self.threads = self.n_threads  # one sequence per thread at most

    def step(self):
        w = self.w
        rows = np.arange(self.n_seq) * self.chunk + self.calls % self.chunk
        t0 = time.perf_counter()
        self.o.decode_batch(self.K, self.V, self.q[rows], self.kn[rows], self.vn[rows],
                            self.pos[rows].astype(np.uint32), self.compact, w.q_norm_w(),
                            w.k_norm_w(), w.inv_freq(), w.sink_logits(), w.eps, w.scale,
                            n_threads=self.n_threads)
        self.calls += 1
        return time.perf_counter() - t0

    def describe(self, calls, seconds):
        last = int(self.first.max()) + min(calls, self.chunk) - 1
        return (f"{calls} calls of one prompt token of each of the {self.n_seq} sequences "
                f"(one decode step per token, positions {int(self.first.min())}..{last}), "
                f"{seconds:.1f} s, " + ("on one thread" if self.n_threads == 1 else
                                         f"the sequences split over {self.n_threads} threads"))


def time_oracle_prefill(w, slots, pos, budget_s, n_threads):
    """tokens/s of the oracle on the prefill workload over calls until
    ``budget_s`` (at most one pass over the chunk)."""
    smp = PrefillOracleSample(w, slots, pos, n_threads)
    calls, spent = 0, 0.0
    while spent < budget_s and calls < PREFILL_CHUNK:
        spent += smp.step()
        calls += 1
    return smp.n_seq * calls / spent, smp.describe(calls, spent), smp.threads


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="large",
                    choices=sorted(synth.WORKLOADS) + sorted(synth.EXTRA_WORKLOADS) +
                    sorted(synth.PROFILE_WORKLOADS))
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--split", type=int, nargs=2, default=None,
                    metavar=("MIN_CHUNK_KEYS", "MAX_SPLITS"))
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill", action="store_true",
                    help="time batched causal prefill instead of the decode step")
    ap.add_argument("--prefill-geometry", default="mid", choices=["mid", "sinks"],
                    help="head geometry of the prefill workload (mid: hd 128; sinks: hd 64)")
    ap.add_argument("--options", default="", choices=["", "vnorm", "plus_one", "both"],
                    help="Gemma norm forms: weightless V norm, (1 + w) Q/K weights, or both")
    ap.add_argument("--paged", type=int, default=0, metavar="BLOCK_SIZE",
                    help="run the workload over a shuffled paged pool of this block size")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step in a CUDA graph and time its replays")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the decode kernel, if measured")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the four target workloads beside the headline")
    ap.add_argument("--ncu", action="store_true",
                    help="profiler target: two calls of the workload's first step, no line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    args.options = {"": 0, "vnorm": 1, "plus_one": 2, "both": 3}[args.options]
    w = {**synth.WORKLOADS, **synth.EXTRA_WORKLOADS, **synth.PROFILE_WORKLOADS}[args.workload]
    if args.ncu:
        run_ncu_target(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    elif args.prefill:
        run_prefill(args)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
