"""Benchmark of one paged decode step: KV write + decode attention (+ reduce).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config opt13b]
                    [--impl ours|reference] [--partition P]

A step is one pass of the hot path over one batch: the slot-mapped KV write
of the step's new keys and values, then paged decode attention (partition
pass and, when a sequence spans several partitions, the split-K merge); on
the parallel-sampling workload the copy-on-write block copies run first.
The default workload is the OPT-13B-shaped decode (40 heads MHA, head_dim
128, fp16, block 16, batch 64, lengths uniform over 200..2000, shuffled pool
= need + 10%), one layer.  The default line also carries, under the key
"gqa", the same measurement of the GQA Llama-3-8B-shaped decode (32 query /
8 KV heads, bf16, batch 256).  Inputs are seeded synthetic data resident in
HBM; the pools (about 1.6 and 1.3 GB) are larger than L2, so no flush is
needed between steps.

The timed region runs K steps back to back (device time between one event
before the first and one after the last) and then K decode launches alone,
whose mean duration is the roofline's per-launch time.  Pools smaller than
twice L2 (the parallel-sampling workload) are flushed before every step and
every decode launch, and each is bracketed by its own events.

Under torchrun (N > 1) every rank runs its own batch on its own GPU with no
collective on the data path (sequences are independent: weak scaling); the
timed region is bracketed by barriers and the slowest rank's time is used.

``--impl reference`` times the float64 CPU oracle on the same workload (one
bounded sample of sequences per step) on rank 0; other ranks exit at once.
"""

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_cache_145_gb300 import synth  # noqa: E402

METRIC = "paged decode attention KV GB/s and tokens/s on 1 GB300, % of HBM roofline"

# DRAM bytes (read + write) per launch of the decode partition kernel (for
# the shared-prefix decode: of its kernels together, per call), from
# ncu (dram__bytes_read.sum + dram__bytes_write.sum), keyed by workload, KV
# dtype or decode form, and partition length, with the hash of the sources
# of that kernel family they were taken on.  A stale hash reports null.
TRAFFIC = {
    "opt13b/native/512": (1277931520, "c5e6dfe8a34e9dc5"),
    "gqa/native/512": (1127068928, "c5e6dfe8a34e9dc5"),
    "long/native/512": (875515520, "c5e6dfe8a34e9dc5"),
    "fork/native/512": (77181440, "c5e6dfe8a34e9dc5"),
    "fork/shared/512": (79970304, "c5e6dfe8a34e9dc5"),
    "opt13b/fp8/2048": (641383936, "13cf79d9ff22aa7b"),
    "gqa/fp8/2048": (563038336, "13cf79d9ff22aa7b"),
    "long/fp8/1536": (437340288, "13cf79d9ff22aa7b"),
}

KERNEL_SOURCES = {
    "native": ("common.cuh", "decode.cuh", "decode_mma.cuh", "decode_launch.cuh",
               "decode_shared.cuh", "tcgen05.cuh"),
    "fp8": ("common.cuh", "decode.cuh", "decode_mma_fp8.cuh", "decode_launch.cuh"),
}


def kernel_source_hash(family="native"):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, "paged_kv_cache_145_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def pack_pinned(tensors, dev, align=256):
    """One pinned host buffer holding every tensor's bytes (each at an
    ``align``-byte offset), its device twin, and device views of the twin
    with the tensors' dtypes and shapes: a step's inputs then cross the host
    link in one copy."""
    import torch

    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // align) * align
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        host[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
    devbuf = torch.empty(total, dtype=torch.uint8, device=dev)
    views = [devbuf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for t, o in zip(tensors, offs)]
    return host, devbuf, views


def e2e_pipelined(host_tensors, dev, step, out_like, steps):
    """End-to-end steps through the public API from pinned host memory.

    Every step's inputs cross the host link in one copy (into one of two
    device staging buffers, on a host-to-device stream) and its output comes
    back in one copy (from one of two device outputs, on a device-to-host
    stream), so step i's copies overlap the kernels of steps i - 1 and
    i + 1, as a serving loop would stage them.  ``step(views, out)`` runs
    one step on the current stream.  Returns (seconds per step, h2d bytes
    per step, d2h bytes per step, the last output copied to the host, the
    device output it came from)."""
    import torch

    compute = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    staged = [pack_pinned(host_tensors, dev) for _ in range(2)]
    outs = [torch.empty_like(out_like) for _ in range(2)]
    outs_h = [torch.empty(out_like.shape, dtype=out_like.dtype).pin_memory() for _ in range(2)]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ev_in, ev_done, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(compute)
    h2d.wait_stream(compute)
    d2h.wait_stream(compute)
    for i in range(steps):
        k = i % 2
        host_in, dev_in, views = staged[k]
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(ev_done[k])  # step i - 2 has read this staging buffer
            dev_in.copy_(host_in, non_blocking=True)
            ev_in[k].record(h2d)
        compute.wait_event(ev_in[k])
        if i >= 2:
            compute.wait_event(ev_out[k])  # step i - 2's output has left this buffer
        step(views, outs[k])
        ev_done[k].record(compute)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_done[k])
            outs_h[k].copy_(outs[k], non_blocking=True)
            ev_out[k].record(d2h)
    compute.wait_stream(h2d)
    compute.wait_stream(d2h)
    end.record(compute)
    torch.cuda.synchronize()
    last = (steps - 1) % 2
    return (start.elapsed_time(end) / 1e3 / steps, staged[0][0].numel(),
            outs_h[0].numel() * outs_h[0].element_size(), outs_h[last], outs[last])


def e2e_graphed(host_tensors, dev, step, out_like, steps, per_graph=8):
    """``e2e_pipelined`` with the per-step host work taken out of the loop:
    ``per_graph`` consecutive steps (the same copies, stream hand-offs and
    API calls, buffers alternating) are captured once in a CUDA graph and
    the graph is replayed, as a serving loop replays its decode step.  Every
    replayed step still copies its inputs from pinned host memory and its
    output back.  Returns the same tuple as ``e2e_pipelined`` and the number
    of steps run (a multiple of ``per_graph``)."""
    import torch

    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    staged = [pack_pinned(host_tensors, dev) for _ in range(2)]
    outs = [torch.empty_like(out_like) for _ in range(2)]
    outs_h = [torch.empty(out_like.shape, dtype=out_like.dtype).pin_memory() for _ in range(2)]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        cap = torch.cuda.current_stream()
        h2d.wait_stream(cap)
        d2h.wait_stream(cap)
        ev_done, ev_out = [None, None], [None, None]
        for i in range(per_graph):
            k = i % 2
            host_in, dev_in, views = staged[k]
            ev_in = ev()
            with torch.cuda.stream(h2d):
                if ev_done[k] is not None:
                    h2d.wait_event(ev_done[k])  # step i - 2 has read this staging buffer
                dev_in.copy_(host_in, non_blocking=True)
                ev_in.record(h2d)
            cap.wait_event(ev_in)
            if ev_out[k] is not None:
                cap.wait_event(ev_out[k])  # step i - 2's output has left this buffer
            step(views, outs[k])
            ev_done[k] = ev()
            ev_done[k].record(cap)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_done[k])
                outs_h[k].copy_(outs[k], non_blocking=True)
                ev_out[k] = ev()
                ev_out[k].record(d2h)
        cap.wait_stream(h2d)
        cap.wait_stream(d2h)
    reps = max(1, steps // per_graph)
    g.replay()  # one untimed replay
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    start.record(stream)
    for _ in range(reps):
        g.replay()
    end.record(stream)
    torch.cuda.synchronize()
    n = reps * per_graph
    last = (per_graph - 1) % 2
    return (start.elapsed_time(end) / 1e3 / n, staged[0][0].numel(),
            outs_h[0].numel() * outs_h[0].element_size(), outs_h[last], outs[last]), n


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def read_stream_gbs(dev, nbytes=4 << 30, reps=10):
    """A measured read-only streaming rate: the library's read-stream
    self-test kernel over a buffer far larger than L2, best of ``reps``
    CUDA-event timed passes.  Context for the roofline, next to the
    copy-rate peak."""
    import torch

    import paged_kv_cache_145_gb300 as pkv

    x = torch.ones(nbytes, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(3):
        pkv.paged_selftest_read_stream(x, sink)
    best = None
    stream = torch.cuda.current_stream()
    for _ in range(reps):
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pkv.paged_selftest_read_stream(x, sink)
        z.record(stream)
        z.synchronize()
        t = a.elapsed_time(z) / 1e3
        best = t if best is None else min(best, t)
    del x
    return {"gbs": round(nbytes / best / 1e9, 1),
            "how": "paged_selftest_read_stream (16-byte non-caching loads, whole GPU) over "
                   "%d MiB, best of %d" % (nbytes >> 20, reps)}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# workload (product side: the native block manager plans the step)
# ---------------------------------------------------------------------------
class Workload:
    """One decode step of a named workload, planned by the native block manager.

    ``block_size`` overrides the workload's block size; ``table="identity"``
    hands out physical blocks in order (each sequence's blocks contiguous and
    sequences back to back) instead of from a shuffled free list, which
    isolates the cost of scattered pages from the rest of the paging.
    """

    def __init__(self, name, rank=0, block_size=None, table="shuffled", kv_dtype=None):
        import paged_kv_cache_145_gb300 as pkv

        cfg = synth.CONFIGS[name]
        self.name, self.cfg = name, cfg
        self.b = b = block_size or cfg["block_size"]
        self.table_kind = table
        self.H, self.Hk, self.D, self.dtype = cfg["heads"], cfg["kv_heads"], cfg["head_dim"], cfg["dtype"]
        self.elt = synth.ELEM_BYTES[self.dtype]                # q, out, new k/v
        self.kv_dtype = kv_dtype or self.dtype
        self.kv_elt = synth.ELEM_BYTES[self.kv_dtype]          # cache elements
        ceil_div = lambda a, c: -(-a // c)  # noqa: E731
        if name == "fork":
            g, f, prompt = cfg["groups"], cfg["forks"], cfg["prompt"]
            self.ids = [i * f + j for i in range(g) for j in range(f)]
            need = g * (ceil_div(prompt, b) + f - 1)
        else:
            lengths = synth.lengths(name)
            self.ids = list(range(len(lengths)))
            need = sum(ceil_div(int(t) + 1, b) for t in lengths)
        self.N = cfg.get("pool_blocks") or synth.pool_with_slack(need, cfg["slack"])
        order = (np.arange(self.N, dtype=np.int64) if table == "identity"
                 else synth.free_order(synth.seed_of(name, 2) + rank, self.N))
        bm = pkv.BlockManager(self.N, b, order)
        if name == "fork":
            for i in range(g):
                bm.admit(i * f, prompt)
                for j in range(1, f):
                    bm.fork(i * f, i * f + j)
        else:
            for i, t in enumerate(lengths):
                bm.admit(i, int(t))
        self.slots, self.pairs = bm.append(self.ids)
        self.max_blocks = max(bm.num_seq_blocks(i) for i in self.ids)
        self.tables, self.seq_lens = bm.tables(self.ids, self.max_blocks)
        self.S = len(self.ids)
        self.max_len = int(self.seq_lens.max())
        # Stored positions over allocated slots (tail waste of the last blocks).
        self.utilization = float(self.seq_lens.sum()) / float(b * sum(
            bm.num_seq_blocks(i) for i in self.ids))

    # Algorithmic bytes, counted without reuse across sequences.
    def decode_bytes(self, part):
        L = self.seq_lens.astype(np.int64)
        kv = 2 * L * self.Hk * self.D * self.kv_elt
        qo = 2 * self.H * self.D * self.elt
        table = 4 * (-(-L // self.b)) + 4
        nparts = -(-L // part)
        ws = np.where(nparts > 1, 2 * self.H * nparts * (self.D + 2) * 4, 0)
        return int((kv + qo + table + ws).sum()), int(kv.sum())

    def unique_kv_bytes(self):
        """K+V bytes of the distinct positions read (a page shared by several
        tables counted once): what a step must fetch from DRAM at least."""
        held = {}
        for row, L in zip(self.tables, self.seq_lens):
            for j in range(-(-int(L) // self.b)):
                pb = int(row[j])
                held[pb] = max(held.get(pb, 0), min(self.b, int(L) - j * self.b))
        return 2 * sum(held.values()) * self.Hk * self.D * self.kv_elt

    def pool_bytes(self):
        return 2 * self.N * self.Hk * self.b * self.D * self.kv_elt

    def write_bytes(self):
        n = self.S
        return 2 * n * self.Hk * self.D * (self.elt + self.kv_elt) + 8 * n

    def copy_bytes(self):
        return 2 * 2 * len(self.pairs) * self.Hk * self.b * self.D * self.kv_elt + 16 * len(self.pairs)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def smi_gpu_id(local_index):
    """nvidia-smi's name for a CUDA device: its UUID (robust to remapping)."""
    import torch

    try:
        u = str(torch.cuda.get_device_properties(local_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x for x in vis.split(",") if x.strip()]
        return ids[local_index] if local_index < len(ids) else str(local_index)


class ClockSampler:
    def __init__(self, gpu_index):
        self.proc = None
        self.path = None
        self.gpu = smi_gpu_id(gpu_index)

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + CLOCK_FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed helpers (replicas; no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def combine_ranks(local_bytes, local_seconds):
    """Whole-job throughput: bytes of all ranks over the slowest rank's time."""
    import torch
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
        b = torch.tensor([float(local_bytes)], dtype=torch.float64, device=dev)
        s = torch.tensor([float(local_seconds)], dtype=torch.float64, device=dev)
        dist.all_reduce(b, op=dist.ReduceOp.SUM)
        dist.all_reduce(s, op=dist.ReduceOp.MAX)
        return float(b.item()), float(s.item())
    return float(local_bytes), float(local_seconds)


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle leg (spawned child, single BLAS thread)
# ---------------------------------------------------------------------------
def _oracle_prepare(name, i, t, seed):
    """Inputs of one oracle decode step for a sequence of t cached tokens:
    its pool after the append (slot and table planned by the oracle's block
    pool), the new key/value and the query.  Not timed."""
    from oracle import blocks as B
    from oracle import paging as P

    cfg = synth.CONFIGS[name]
    b, H, Hk, D, dt = cfg["block_size"], cfg["heads"], cfg["kv_heads"], cfg["head_dim"], cfg["dtype"]
    nblk = P.blocks_needed(t + 1, b)
    pool = B.BlockPool(nblk, b, free_order=synth.free_order(seed + i, nblk), auto_verify=False)
    pool.admit(0, list(range(t)))
    slot = pool.append(0, -1).slot
    return dict(
        kp=synth.storage_numpy(synth.normal(seed + 3 * i, (nblk, Hk, b, D), dt), dt),
        vp=synth.storage_numpy(synth.normal(seed + 3 * i + 1, (nblk, Hk, b, D), dt), dt),
        kn=synth.storage_numpy(synth.normal(seed + 3 * i + 2, (1, Hk, D), dt), dt),
        q=synth.storage_numpy(synth.normal(seed + 7 * i, (1, H, D), dt), dt),
        slot=slot, table=pool.table(0), length=t + 1, b=b, D=D, dt=dt,
        kv_bytes=2 * (t + 1) * Hk * D * synth.ELEM_BYTES[dt])


def _oracle_step(x):
    """The oracle's KV write + attention for one prepared sequence; seconds."""
    from oracle import attention as A

    t0 = time.perf_counter()
    kp2, vp2, _ = A.write_tokens(x["kp"], x["vp"], x["kn"], x["kn"], [x["slot"]], x["b"])
    A.attention(x["q"], kp2, vp2, [x["table"]], [x["length"]], 1.0 / math.sqrt(x["D"]), x["b"],
                x["dt"])
    return time.perf_counter() - t0


def _lengths(name):
    cfg = synth.CONFIGS[name]
    if name == "fork":
        return np.full(cfg["groups"] * cfg["forks"], cfg["prompt"])
    return synth.lengths(name)


def _oracle_sample(name, budget_s, seed):
    """Times the oracle's KV write + attention over sequences of the workload
    until ``budget_s`` seconds of oracle work have passed; returns
    (kv_bytes, seconds, seqs)."""
    kv_bytes, done, spent = 0, 0, 0.0
    for i, t in enumerate(_lengths(name)):
        x = _oracle_prepare(name, i, int(t), seed)
        spent += _oracle_step(x)
        kv_bytes += x["kv_bytes"]
        done += 1
        if spent >= budget_s:
            break
    return kv_bytes, spent, done


def _reference_steps(name, steps, warmup, seed, distinct=8, target_s=120.0):
    """The reference arm: warm-up and timed steps of the oracle, each one
    sequence of the workload (cycling over ``distinct`` prepared ones).
    So that K + W steps take about ``target_s`` seconds of oracle work,
    a step covers the first h KV heads of its sequence (with their query
    heads), h chosen from one timed full step.  Returns (kv_bytes, seconds,
    steps, h, kv_heads)."""
    cfg = synth.CONFIGS[name]
    Hk, G = cfg["kv_heads"], cfg["heads"] // cfg["kv_heads"]
    lengths = _lengths(name)
    xs = [_oracle_prepare(name, i, int(lengths[i % len(lengths)]), seed) for i in range(distinct)]
    full = sum(_oracle_step(x) for x in xs) / distinct
    h = int(max(1, min(Hk, Hk * target_s / max(steps + warmup, 1) / max(full, 1e-9))))
    for x in xs:
        x["kp"], x["vp"] = x["kp"][:, :h].copy(), x["vp"][:, :h].copy()
        x["kn"], x["q"] = x["kn"][:, :h].copy(), x["q"][:, :h * G].copy()
        x["kv_bytes"] = x["kv_bytes"] * h // Hk
    for k in range(warmup):
        _oracle_step(xs[k % distinct])
    kv_bytes, spent = 0, 0.0
    for k in range(steps):
        spent += _oracle_step(xs[k % distinct])
        kv_bytes += xs[k % distinct]["kv_bytes"]
    return kv_bytes, spent, steps, h, Hk


def _oracle_child(conn, fn, args):
    conn.send(fn(*args))
    conn.close()


def oracle_child(fn, *args):
    """Runs fn(*args) in a spawned child limited to one BLAS thread."""
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    ctx = mp.get_context("spawn")
    parent, child = ctx.Pipe()
    p = ctx.Process(target=_oracle_child, args=(child, fn, args))
    p.start()
    result = parent.recv()
    p.join()
    return result


def oracle_timed(name, budget_s, seed=4242):
    return oracle_child(_oracle_sample, name, budget_s, seed)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _oracle_worker(name, budget_s, seed, w, workers, start, results):
    """One of ``workers`` oracle processes: sequences w, w + workers, ... of
    the workload (cycling), prepared before the common start, then timed
    until ``budget_s`` seconds of oracle work have passed."""
    lengths = _lengths(name)
    mine = list(range(w, len(lengths), workers)) or [w % len(lengths)]
    prepared = {}

    def get(i):
        if i not in prepared:
            prepared[i] = _oracle_prepare(name, i, int(lengths[i]), seed)
        return prepared[i]

    get(mine[0])
    start.wait()
    kv_bytes, done, spent, k = 0, 0, 0.0, 0
    while spent < budget_s:
        x = get(mine[k % len(mine)])
        spent += _oracle_step(x)
        kv_bytes += x["kv_bytes"]
        done += 1
        k += 1
    results.put((kv_bytes, spent, done))


def oracle_all_cores(name, budget_s, seed=4242):
    """The oracle spread over every host core the process may use: one
    spawned process per core (one BLAS thread each), each on its own share
    of the workload's sequences, started together.  Returns (kv_bytes,
    seconds, seqs, workers); throughput = all bytes over the longest
    worker's time."""
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    workers = host_cores()
    ctx = mp.get_context("spawn")
    start, results = ctx.Barrier(workers), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker,
                         args=(name, budget_s, seed, w, workers, start, results))
             for w in range(workers)]
    for p in procs:
        p.start()
    got = [results.get() for _ in procs]
    for p in procs:
        p.join()
    return (sum(g[0] for g in got), max(g[1] for g in got), sum(g[2] for g in got), workers)


def cpu_baseline_record(name, single, pool, num_seqs, what):
    """cpu_baseline: the one-process oracle figure, with the all-cores one
    beside it."""
    cb, cs, cn = single
    rec = {"value": round(cb / cs / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": "%d of %d sequences (all heads), %s, float64 NumPy oracle, 1 process, "
                     "1 BLAS thread, %.1f s" % (cn, num_seqs, what, cs),
           "host_cores": host_cores(), "blas_threads": 1}
    if pool is not None:
        pb, ps, pn, pw = pool
        rec["all_cores"] = {
            "value": round(pb / ps / 1e9, 6), "unit": "GB/s", "cores": pw, "kind": "oracle",
            "sample": "%d processes (one per host core, 1 BLAS thread each) over strided "
                      "shares of the %d sequences, cycling, %d sequence steps in %.1f s; "
                      "all bytes over the longest process's time" % (pw, num_seqs, pn, ps)}
    return rec


def _oracle_prefill_sample(name, budget_s, seed, fp8):
    """Times the oracle's chunk write + causal prefill attention over the
    workload's sequences, one (sequence, KV head) pair at a time with that
    head's query heads, until ``budget_s`` seconds of oracle work have
    passed.  Each pair gets a private pool of its sequence's blocks, handed
    out in shuffled order.  Returns (flops, seconds, pairs, queries)."""
    from oracle import attention as A

    cfg = synth.CONFIGS[name]
    b, H, Hk, D, dt = cfg["block_size"], cfg["heads"], cfg["kv_heads"], cfg["head_dim"], cfg["dtype"]
    prefix, chunk, G = cfg["prefix"], cfg["chunk"], H // Hk
    L = prefix + chunk
    nblk = -(-L // b)
    kdt = "e4m3" if fp8 else dt
    sc = [1.0 / 64]
    flops_pair = 4 * D * G * sum(prefix + i + 1 for i in range(chunk))
    flops, spent, pairs = 0, 0.0, 0
    for s in range(cfg["batch"]):
        table = synth.free_order(seed + s, nblk)
        pos = np.arange(prefix, L)
        slots = table[pos // b] * b + pos % b
        for kvh in range(Hk):
            r = seed + 1000 * s + 10 * kvh
            if fp8:
                kp = synth.storage_numpy(synth.random_codes(r, (nblk, 1, b, D)), "e4m3")
                vp = synth.storage_numpy(synth.random_codes(r + 1, (nblk, 1, b, D)), "e4m3")
            else:
                kp = synth.storage_numpy(synth.normal(r, (nblk, 1, b, D), dt), dt)
                vp = synth.storage_numpy(synth.normal(r + 1, (nblk, 1, b, D), dt), dt)
            kn = synth.storage_numpy(synth.normal(r + 2, (chunk, 1, D), dt), dt)
            vn = synth.storage_numpy(synth.normal(r + 3, (chunk, 1, D), dt), dt)
            q = synth.storage_numpy(synth.normal(r + 4, (chunk, G, D), dt), dt)
            t0 = time.perf_counter()
            if fp8:
                kp, vp, _ = A.write_tokens_fp8(kp, vp, kn, vn, slots, b, sc, sc, dt)
            else:
                kp, vp, _ = A.write_tokens(kp, vp, kn, vn, slots, b)
            A.prefill_attention(q, kp, vp, [table], [L], [0, chunk], 1.0 / math.sqrt(D), b, kdt,
                                q_dtype=dt, k_scale=sc if fp8 else None,
                                v_scale=sc if fp8 else None)
            spent += time.perf_counter() - t0
            flops += flops_pair
            pairs += 1
            if spent >= budget_s:
                return flops, spent, pairs, chunk
    return flops, spent, pairs, chunk


def _oracle_op_sample(name, op, budget_s, seed, block_size=None):
    """Times the oracle's KV write, block copy or block swap on samples of
    the workload until ``budget_s`` seconds of oracle work have passed.
    write: every position of one sequence after another, each into a private
    pool of its blocks; copy: 256 shuffled disjoint pairs over a 512-block
    pool per call; swap: 256 blocks out to a host pool and back per call.
    Returns (algorithmic bytes, seconds, units) with the bytes counted as the
    GPU line counts them."""
    from oracle import attention as A

    cfg = synth.CONFIGS[name]
    b = block_size or cfg["block_size"]
    Hk, D, dt = cfg["kv_heads"], cfg["head_dim"], cfg["dtype"]
    elt = synth.ELEM_BYTES[dt]
    block_bytes = Hk * b * D * elt
    nbytes, spent, units = 0, 0.0, 0
    if op == "write":
        for i, L in enumerate(_lengths(name)):
            L = int(L)
            nblk = -(-L // b)
            table = synth.free_order(seed + i, nblk)
            t = np.arange(L)
            slots = table[t // b] * b + t % b
            kp = synth.storage_numpy(synth.normal(seed + 4 * i, (nblk, Hk, b, D), dt), dt)
            vp = synth.storage_numpy(synth.normal(seed + 4 * i + 1, (nblk, Hk, b, D), dt), dt)
            kn = synth.storage_numpy(synth.normal(seed + 4 * i + 2, (L, Hk, D), dt), dt)
            vn = synth.storage_numpy(synth.normal(seed + 4 * i + 3, (L, Hk, D), dt), dt)
            t0 = time.perf_counter()
            A.write_tokens(kp, vp, kn, vn, slots, b)
            spent += time.perf_counter() - t0
            nbytes += 2 * 2 * L * Hk * D * elt + 8 * L
            units += L
            if spent >= budget_s:
                break
        return nbytes, spent, units
    half = 256
    kp = synth.storage_numpy(synth.normal(seed, (2 * half, Hk, b, D), dt), dt)
    vp = synth.storage_numpy(synth.normal(seed + 1, (2 * half, Hk, b, D), dt), dt)
    perm = synth.free_order(seed + 2, 2 * half)
    while spent < budget_s:
        if op == "copy":
            pairs = np.stack([perm[:half], perm[half:]], 1)
            t0 = time.perf_counter()
            A.copy_blocks(kp, vp, pairs)
            spent += time.perf_counter() - t0
            nbytes += 2 * 2 * half * block_bytes + 16 * half
        else:
            hk = np.zeros((half, Hk, b, D), dtype=kp.dtype)
            hv = np.zeros_like(hk)
            out_pairs = np.stack([perm[:half], np.arange(half)], 1)
            in_pairs = np.stack([np.arange(half), perm[:half]], 1)
            t0 = time.perf_counter()
            _, _, hk2, hv2, _ = A.swap_blocks(kp, vp, hk, hv, out_pairs, "out")
            A.swap_blocks(kp, vp, hk2, hv2, in_pairs, "in")
            spent += time.perf_counter() - t0
            # one swap out and one swap in, each moving 2 * half blocks
            nbytes += 2 * (2 * half * block_bytes + 16 * half)
        units += half
    return nbytes, spent, units


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    total_b, total_s, seqs, h, hk = oracle_child(_reference_steps, args.config, args.steps,
                                                 args.warmup, 4242)
    gbs = total_b / total_s / 1e9
    cfg = synth.CONFIGS[args.config]
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total_s / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.config, "about": cfg["about"],
                   "sample": "one sequence of the workload per step (8 distinct sequences "
                             "cycled), its first %d of %d KV heads" % (h, hk)},
        # a step over h of the KV heads counts as h / kv_heads of a sequence
        "decode_tokens_per_s": round(seqs * h / hk / total_s, 3),
        "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "host_cores": host_cores(), "blas_threads": 1,
                         "sample": "%d steps of one sequence each (8 distinct, cycled; "
                                   "%d of %d KV heads), float64 NumPy oracle (write + "
                                   "attention), 1 BLAS thread" % (seqs, h, hk)},
        "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import paged_kv_cache_145_gb300 as pkv

    rank, local_rank, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pkv._lib.lib()

    # The default line also measures the GQA workload (32 query / 8 KV heads,
    # bf16, batch 256), under the key "gqa", with its own roofline, clocks,
    # end-to-end figure and CPU baseline; the headline stays the
    # OPT-13B-shaped workload.
    names = [args.config]
    if (args.config == "opt13b" and args.kv_dtype == "native" and args.partition == 0
            and args.block_size == 0 and args.table == "shuffled" and not args.no_gqa):
        names.append("gqa")

    # The CPU baselines run before any GPU work, so the oracle processes do
    # not compete with the timed region for host cores.
    cpu = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        for name in names:
            single = oracle_timed(name, args.cpu_budget)
            pool = oracle_all_cores(name, args.cpu_budget / 2) if not args.no_all_cores else None
            cpu[name] = (single, pool)

    line = decode_line(args, args.config, cpu.get(args.config), rank, local_rank, world, dev)
    for name in names[1:]:
        torch.cuda.empty_cache()
        sub = decode_line(args, name, cpu.get(name), rank, local_rank, world, dev)
        if rank == 0:
            line[name] = {k: sub[k] for k in SUB_RECORD_KEYS if k in sub}
    if rank == 0:
        print(json.dumps(line), flush=True)


SUB_RECORD_KEYS = ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "dtype", "config",
                   "decode_tokens_per_s", "kv_gbs", "layer_stack_extrapolation", "roofline",
                   "clocks", "gpu_launches", "e2e", "e2e_eager", "cpu_baseline")


def decode_line(args, name, cpu, rank, local_rank, world, dev):
    """Times the decode step of workload ``name`` and returns its JSON line
    (rank 0) or None (other ranks)."""
    import torch

    import paged_kv_cache_145_gb300 as pkv

    kv_dtype = "e4m3" if args.kv_dtype == "fp8" else None
    w = Workload(name, rank=rank, block_size=args.block_size or None, table=args.table,
                 kv_dtype=kv_dtype)
    dt = synth.TORCH_DTYPE[w.dtype]
    seed = synth.seed_of(name, 3) + 10 * rank
    shape = (w.N, w.Hk, w.b, w.D)
    if kv_dtype:
        # FP8 E4M3 pool with one scale per KV head (1/64: N(0, 1) values
        # within +-4 land inside the format's +-448 range).
        scale = torch.full((w.Hk,), 1.0 / 64, dtype=torch.float32, device=dev)
        cache = pkv.PagedKVCache(synth.random_codes(seed, shape, device="cuda"),
                                 synth.random_codes(seed + 1, shape, device="cuda"),
                                 scale, scale.clone(), dt)
    else:
        cache = pkv.PagedKVCache(synth.normal(seed, shape, w.dtype, device="cuda"),
                                 synth.normal(seed + 1, shape, w.dtype, device="cuda"))
    q_h = synth.normal(seed + 2, (w.S, w.H, w.D), w.dtype).pin_memory()
    k_h = synth.normal(seed + 3, (w.S, w.Hk, w.D), w.dtype).pin_memory()
    v_h = synth.normal(seed + 4, (w.S, w.Hk, w.D), w.dtype).pin_memory()
    slots_h = torch.from_numpy(w.slots).pin_memory()
    tables_h = torch.from_numpy(w.tables).pin_memory()
    lens_h = torch.from_numpy(w.seq_lens).pin_memory()
    pairs_h = torch.from_numpy(np.asarray(w.pairs, dtype=np.int64).reshape(-1, 2)).pin_memory()
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    slots, tables, lens, pairs = slots_h.to(dev), tables_h.to(dev), lens_h.to(dev), pairs_h.to(dev)
    out = torch.empty_like(q)
    out_h = torch.empty_like(q_h).pin_memory()
    part = pkv.paged_attention_partition_size(cache, w.S, w.H, w.max_len, args.partition)
    ws_bytes = pkv.paged_attention_workspace_bytes(cache, w.S, w.H, w.max_len, part)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(w.D)
    has_pairs = len(w.pairs) > 0
    nparts_max = -(-w.max_len // part)
    shared = name == "fork" and args.decode == "shared"
    # Forked batches (the parallel-sampling workload) decode their shared
    # prompt once per group with the shared-prefix entry point; --decode
    # plain times the plain decode instead.
    tail_parts = 0
    if shared:
        groups, forks = w.cfg["groups"], w.cfg["forks"]
        g_starts = torch.arange(0, groups * forks + 1, forks, dtype=torch.int32, device=dev)
        g_prefix = torch.full((groups,), (w.cfg["prompt"] // w.b) * w.b, dtype=torch.int32,
                              device=dev)
        # Partitions the partition pass covers per fork after its group's
        # shared ones: the host knows every length and prefix.
        tail_parts = max(-(-int(L) // part) for L in w.seq_lens) - \
            ((w.cfg["prompt"] // w.b) * w.b) // part
    # Kernels per decode call: partition pass (+ merge when any sequence has
    # several partitions); shared-prefix decode: its kernel, then either the
    # tail-and-merge pass (every tail within one partition) or the partition
    # pass and merge.
    if shared and 0 < tail_parts < nparts_max and tail_parts == 1:
        decode_launches = 2
    else:
        decode_launches = 1 + (1 if nparts_max > 1 else 0) + (1 if shared else 0)
    launches_per_step = 1 + decode_launches + (1 if has_pairs else 0)

    stream = torch.cuda.current_stream()

    resident = (q, k, v, slots, tables, lens, pairs)


    def decode(x=resident, o=out):
        if shared:
            pkv.paged_attention_decode_shared(cache, x[0], x[4], x[5], scale, g_starts, g_prefix,
                                              forks, out=o, max_seq_len=w.max_len, workspace=ws,
                                              partition_size=part, tail_parts=tail_parts)
        else:
            pkv.paged_attention_decode(cache, x[0], x[4], x[5], scale, out=o,
                                       max_seq_len=w.max_len, workspace=ws, partition_size=part)

    def step(x=resident, o=out):
        if has_pairs:
            pkv.paged_block_copy(cache, x[6])
        pkv.paged_kv_write(cache, x[1], x[2], x[3])
        decode(x, o)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pkv.paged_get_device_error() == 0

    # A pool smaller than twice L2 would be served from L2 across steps: L2
    # is then flushed (a write of 2 x L2 bytes) before every timed step and
    # only the steps themselves are timed; the warm figures are reported
    # beside the flushed ones.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_l2 = w.pool_bytes() < 2 * l2_bytes
    flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if flush_l2 else None

    def span(fn, n, flush):
        """Device time of n calls of fn.  Without a flush only the first
        and last call are bracketed by events (an event record between two
        kernels costs about 2 us of device time); with a flush every call is
        bracketed and the flushes are left out."""
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(n if flush else 1)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(n if flush else 1)]
        for i in range(n):
            if flush:
                flush_buf.fill_(i & 0xFF)
            if flush or i == 0:
                e0[i if flush else 0].record(stream)
            fn()
            if flush or i == n - 1:
                e1[i if flush else 0].record(stream)
        return e0, e1

    def elapsed(e0, e1):
        return sum(a.elapsed_time(b) for a, b in zip(e0, e1))

    def timed(n, flush, sampler=None):
        """The timed region: n steps, then n decode launches alone (the
        roofline's per-launch duration), between barriers and syncs."""
        barrier()
        torch.cuda.synchronize()
        if sampler is not None:
            sampler.start()
            time.sleep(0.3)  # let the sampler start before the timed region
        steps = span(step, n, flush)
        decodes = span(decode, n, flush)
        torch.cuda.synchronize()
        barrier()
        clk = sampler.stop() if sampler is not None else None
        assert pkv.paged_get_device_error() == 0
        return elapsed(*steps), elapsed(*decodes) / n, clk

    total_ms, decode_ms, clocks = timed(args.steps, flush_l2, ClockSampler(local_rank))
    warm = timed(args.steps, False) if flush_l2 else None

    # End to end through the public API with host buffers: the step's inputs
    # (q, new k/v, slots, tables, lengths and copy pairs) staged in one
    # pinned host buffer cross to HBM in one copy, the step runs on views of
    # its device twin, and the output is copied back to the host.  Without
    # an L2 flush the copies run on their own streams, overlapping the
    # neighbouring steps' kernels; with one (a pool that fits in L2) each
    # step is copied in, run and copied out in turn, timed without the
    # flushes.
    e2e_steps = args.steps
    e2e_inputs = [q_h, k_h, v_h, slots_h, tables_h, lens_h, pairs_h]
    eager_s = None  # seconds per step of the eager loop, when graph replay is reported
    barrier()
    if flush_l2:
        host_in, dev_in, views = pack_pinned(e2e_inputs, dev)
        h2d = host_in.numel()
        d2h = out_h.numel() * out_h.element_size()
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
        torch.cuda.synchronize()
        for i in range(e2e_steps):
            flush_buf.fill_(i & 0xFF)
            e0[i].record(stream)
            dev_in.copy_(host_in, non_blocking=True)
            step(views)
            out_h.copy_(out, non_blocking=True)
            e1[i].record(stream)
        torch.cuda.synchronize()
        e2e_ms = sum(e0[i].elapsed_time(e1[i]) for i in range(e2e_steps))
        e2e_host, e2e_dev = out_h, out
        e2e_mode = "serial (L2 flushed between steps)"
    else:
        per_step, h2d, d2h, e2e_host, e2e_dev = e2e_pipelined(e2e_inputs, dev, step, out, e2e_steps)
        assert torch.equal(e2e_host, e2e_dev.cpu()), "end-to-end output differs from the device output"
        eager_s = per_step
        e2e_ms = per_step * 1e3 * e2e_steps
        e2e_mode = "copies on their own streams, overlapping the neighbouring steps"
        try:
            (g_step, h2d, d2h, g_host, g_dev), g_n = e2e_graphed(e2e_inputs, dev, step, out,
                                                                 e2e_steps)
            if not torch.equal(g_host, g_dev.cpu()) or not torch.equal(g_dev, e2e_dev):
                raise RuntimeError("graph-replayed output differs")
            e2e_steps, e2e_ms, e2e_host, e2e_dev = g_n, g_step * 1e3 * g_n, g_host, g_dev
            e2e_mode = ("copies on their own streams, overlapping the neighbouring steps; "
                        "8 steps' copies and API calls captured in a CUDA graph and replayed")
        except Exception as exc:  # the eager figure stands
            eager_s = None
            e2e_mode += " (graph replay unavailable: %s)" % str(exc).splitlines()[0][:120]
    barrier()
    assert pkv.paged_get_device_error() == 0
    assert torch.equal(e2e_host, e2e_dev.cpu()), "end-to-end output differs from the device output"

    dec_bytes, kv_bytes = w.decode_bytes(part)
    step_bytes = dec_bytes + w.write_bytes() + (w.copy_bytes() if has_pairs else 0)
    all_bytes, max_s = combine_ranks(step_bytes * args.steps, total_ms / 1e3)
    all_e2e_bytes, max_e2e_s = combine_ranks(step_bytes * e2e_steps, e2e_ms / 1e3)
    eager_bytes, eager_max_s = combine_ranks(step_bytes, eager_s or 0.0)  # every rank calls it
    all_seqs, _ = combine_ranks(w.S * args.steps, total_ms / 1e3)
    if rank != 0:
        return None
    peak, peak_kind = hbm_peak()
    read_peak = read_stream_gbs(dev)
    unique_bytes = w.unique_kv_bytes()
    # Pages shared by several tables (forks) are fetched from DRAM once and
    # then served from L2: the roofline counts them once.
    roof_bytes = dec_bytes - kv_bytes + unique_bytes
    achieved = roof_bytes / (decode_ms / 1e3) / 1e9
    layers = w.cfg.get("layers", 1)
    src_hash = kernel_source_hash("fp8" if kv_dtype else "native")
    default_shape = args.partition == 0 and args.block_size == 0 and args.table == "shuffled"
    key = "%s/%s/%d" % (name, "fp8" if kv_dtype else ("shared" if shared else "native"), part)
    tr = TRAFFIC.get(key) if default_shape else None
    traffic = tr[0] if tr and tr[1] == src_hash else None
    line = {
        "metric": METRIC,
        "value": round(all_bytes / max_s / 1e9, 3),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_s * 1e3 / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype if not kv_dtype else "%s (KV cache e4m3)" % w.dtype,
        "data": "synthetic",
        "config": {"workload": name, "about": w.cfg["about"], "num_seqs": w.S,
                   "kv_dtype": w.kv_dtype,
                   "kv_heads": w.Hk, "heads": w.H, "head_dim": w.D, "block_size": w.b,
                   "pool_blocks": w.N, "partition_size": part, "table": w.table_kind,
                   "decode": ("shared prefix: %d groups of %d forks, %d positions shared, "
                              "tail grid of %d partition(s)"
                              % (w.cfg["groups"], w.cfg["forks"], (w.cfg["prompt"] // w.b) * w.b,
                                 tail_parts) if shared else "plain"),
                   "slot_utilization": round(w.utilization, 5),
                   "l2": ("flushed before every timed step (pool %.1f MB < 2 x L2 %.0f MB)"
                          % (w.pool_bytes() / 1e6, l2_bytes / 1e6) if flush_l2 else
                          "no flush: the %.2f GB pool read per step exceeds the %.0f MB L2"
                          % (kv_bytes / 1e9, l2_bytes / 1e6)),
                   "parallelism": "replicas" if world > 1 else "single"},
        "decode_tokens_per_s": round(all_seqs / max_s, 1),
        "kv_gbs": round(kv_bytes / (decode_ms / 1e3) / 1e9, 3),
        "kv_unique_bytes": unique_bytes,
        "kv_unique_gbs": round(unique_bytes / (decode_ms / 1e3) / 1e9, 3),
        "layer_stack_extrapolation": {
            "layers": layers,
            "decode_tokens_per_s": round(all_seqs / max_s / layers, 1),
            "note": "attention-only, extrapolated: one layer's step timed, times %d layers "
                    "(no projections, MLP or sampling)" % layers},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": (("paged_attention_decode_shared (shared-prefix pass + tail and "
                                 "merge)" if decode_launches == 2 else
                                 "paged_attention_decode_shared (shared-prefix pass + partition "
                                 "pass + split-K merge)") if shared else
                                "paged_attention_decode (partition pass + split-K merge)"),
                     "peak_source": peak_kind,
                     "peak_note": ("the measured device-to-device copy rate (half reads, half "
                                   "writes); decode only reads, so it can exceed 1.0"),
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "read_stream": read_peak,
                     "decode_us": round(decode_ms * 1e3, 2),
                     "decode_bytes": roof_bytes, "source_hash": src_hash,
                     "basis": ("distinct positions (shared pages counted once)"
                               if unique_bytes < kv_bytes else "every position read")},
        "clocks": clocks,
        "gpu_launches": (launches_per_step + decode_launches) * args.steps,
        "e2e": {"value": round(all_e2e_bytes / max_e2e_s / 1e9, 3), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(max_e2e_s * 1e3 / e2e_steps, 5), "copies": e2e_mode,
                "mode": "graph replay" if eager_s is not None else "eager (one API call per step)"},
    }
    if eager_s is not None:
        line["e2e_eager"] = {
            "value": round(eager_bytes / eager_max_s / 1e9, 3), "unit": "GB/s",
            "ms_per_step": round(eager_max_s * 1e3, 5),
            "mode": "eager (one API call per step)",
            "note": "the per-call API figure: the same pipelined steps issued one at a time "
                    "from Python through the binding and the C ABI; bound by the host's "
                    "per-step launch work when that exceeds the step's device time"}
    if warm is not None:
        line["warm_l2"] = {
            "ms_per_step": round(warm[0] / args.steps, 5),
            "decode_us": round(warm[1] * 1e3, 2),
            "kv_gbs": round(kv_bytes / (warm[1] / 1e3) / 1e9, 3),
            "kv_unique_gbs": round(unique_bytes / (warm[1] / 1e3) / 1e9, 3),
            "note": "same steps back to back with no flush: shared and small pools hit L2"}
    if cpu is not None:
        line["cpu_baseline"] = cpu_baseline_record(name, cpu[0], cpu[1], w.S,
                                                   "KV write + attention")
    return line


# ---------------------------------------------------------------------------
# data-movement kernels at bandwidth-sized launches (--op write|copy|swap)
# ---------------------------------------------------------------------------
def _timed(fn, steps, warmup, stream):
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, z in evs:
        a.record(stream)
        fn()
        z.record(stream)
    torch.cuda.synchronize()
    return statistics.fmean(a.elapsed_time(z) for a, z in evs) / 1e3


PREFILL_CONFIGS = ("prefill", "chunked")
DECODE_CONFIGS = ("opt13b", "gqa", "fork", "long")


def run_prefill(args):
    """Prefill step: write each sequence's chunk of new keys/values, then
    causal attention of the chunk's queries over prefix + chunk."""
    import torch

    import paged_kv_cache_145_gb300 as pkv

    rank, local_rank, world = dist_env()
    if rank != 0:
        return
    fp8 = args.kv_dtype == "fp8"
    # The CPU baseline child is spawned before any GPU work.
    cpu = None
    if not args.no_cpu_baseline:
        cpu = oracle_child(_oracle_prefill_sample, args.config, args.cpu_budget, 4242, fp8)
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = synth.CONFIGS[args.config]
    b, H, Hk, D, dt = cfg["block_size"], cfg["heads"], cfg["kv_heads"], cfg["head_dim"], cfg["dtype"]
    S, prefix, chunk = cfg["batch"], cfg["prefix"], cfg["chunk"]
    need = S * (-(-(prefix + chunk) // b))
    n = synth.pool_with_slack(need, cfg["slack"])
    bm = pkv.BlockManager(n, b, synth.free_order(synth.seed_of(args.config, 2), n))
    slots = []
    for i in range(S):
        bm.admit(i, prefix + chunk)
        slots.append(bm.slots(i, prefix, chunk))
    slots = np.concatenate(slots)
    width = max(bm.num_seq_blocks(i) for i in range(S))
    tables, lens = bm.tables(range(S), width)
    seed = synth.seed_of(args.config, 3)
    if fp8:
        # FP8 E4M3 pool with one scale per KV head (1/64, as for decode): the
        # step's KV write quantizes the chunk, the prefill reads codes.
        sc = torch.full((Hk,), 1.0 / 64, dtype=torch.float32, device=dev)
        cache = pkv.PagedKVCache(synth.random_codes(seed, (n, Hk, b, D), device="cuda"),
                                 synth.random_codes(seed + 1, (n, Hk, b, D), device="cuda"),
                                 sc, sc.clone(), synth.TORCH_DTYPE[dt])
    else:
        cache = pkv.PagedKVCache(synth.normal(seed, (n, Hk, b, D), dt, device="cuda"),
                                 synth.normal(seed + 1, (n, Hk, b, D), dt, device="cuda"))
    T = S * chunk
    q_h = synth.normal(seed + 2, (T, H, D), dt).pin_memory()
    k_h = synth.normal(seed + 3, (T, Hk, D), dt).pin_memory()
    v_h = synth.normal(seed + 4, (T, Hk, D), dt).pin_memory()
    sl_h = torch.from_numpy(slots).pin_memory()
    starts_h = torch.arange(0, T + 1, chunk, dtype=torch.int32).pin_memory()
    tab_h = torch.from_numpy(tables).pin_memory()
    ln_h = torch.from_numpy(lens).pin_memory()
    host = [q_h, k_h, v_h, sl_h, starts_h, tab_h, ln_h]
    resident = tuple(t.to(dev) for t in host)
    out = torch.empty_like(resident[0])
    scale = 1.0 / math.sqrt(D)
    stream = torch.cuda.current_stream()

    def attend(x=resident, o=out):
        pkv.paged_attention_prefill(cache, x[0], x[4], x[5], x[6], scale, chunk, out=o)

    def step(x=resident, o=out):
        pkv.paged_kv_write(cache, x[1], x[2], x[3])
        attend(x, o)

    def span(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        return e0, e1

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pkv.paged_get_device_error() == 0
    # Timed region: K steps back to back, then K attention launches alone
    # (the roofline's per-launch time), one event pair each.
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    steps_ev = span(step)
    attn_ev = span(attend)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    assert pkv.paged_get_device_error() == 0
    step_s = steps_ev[0].elapsed_time(steps_ev[1]) / 1e3 / args.steps
    attn_s = attn_ev[0].elapsed_time(attn_ev[1]) / 1e3 / args.steps

    # End to end through the public API with host buffers: the step's inputs
    # (queries, new keys/values, slots, chunk starts, tables, lengths) staged
    # in one pinned host buffer cross to HBM in one copy, the step runs on
    # views of its device twin, and the output is copied back to the host,
    # the copies on their own streams overlapping the neighbouring steps.
    e2e_s, h2d, d2h, e2e_host, e2e_dev = e2e_pipelined(host, dev, step, out, args.steps)
    assert pkv.paged_get_device_error() == 0
    assert torch.equal(e2e_host, e2e_dev.cpu()), "end-to-end output differs from the device output"
    # Algorithmic FLOPs: QK^T and PV, 2 * D each, per (query, head, visible key).
    visible = S * sum(prefix + i + 1 for i in range(chunk))
    flops = 4 * D * H * visible
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            peak, kind = float(json.load(fh)["bf16_tflops"]), "measured cuBLAS bf16 burst"
    except (OSError, KeyError, ValueError):
        peak, kind = 1900.0, "fallback"
    line = {
        "metric": "paged prefill attention TFLOP/s (causal, GQA)", "value": round(flops / step_s / 1e12, 3),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dt if not fp8 else "%s (KV cache e4m3, fp16 MMAs)" % dt,
        "data": "synthetic",
        "config": {"workload": args.config, "about": cfg["about"], "sequences": S, "prefix": prefix,
                   "chunk": chunk, "pool_blocks": n, "kv_dtype": "e4m3" if fp8 else dt},
        "prefill_tokens_per_s": round(T / step_s, 1),
        "roofline": {"bound": "tensor", "achieved": round(flops / attn_s / 1e12, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(flops / attn_s / 1e12 / peak, 4), "traffic": None,
                     "kernel": ("prefill_mma_kernel (mma.sync m16n8k16)"
                                if os.environ.get("PKV_PREFILL_KERNEL") == "mma" else
                                "prefill_tc_kernel (tcgen05.mma, TMEM accumulators)"),
                     "peak_source": kind,
                     "attention_us": round(attn_s * 1e6, 2)},
        "clocks": clocks, "gpu_launches": 3 * args.steps,
        "e2e": {"value": round(flops / e2e_s / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_s * 1e3, 4),
                "copies": "copies on their own streams, overlapping the neighbouring steps"},
    }
    if cpu is not None:
        cf, cs, cpairs, cq = cpu
        line["cpu_baseline"] = {
            "value": round(cf / cs / 1e12, 9), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": "%d (sequence, KV head) pairs of %d x %d, each its %d-token chunk write + "
                      "causal prefill of %d queries x %d query heads, float64 NumPy oracle, "
                      "1 BLAS thread, %.1f s" % (cpairs, S, Hk, cq, cq, H // Hk, cs)}
    print(json.dumps(line), flush=True)


def run_op(args):
    """Bandwidth of the KV write, block copy or block swap at sizes of our
    choosing (a decode step's write and copies are too small to time for
    bandwidth): every cached position written once; half the pool copied to
    the other half by shuffled disjoint pairs; half the pool swapped out to
    pinned host memory and back."""
    import torch

    import paged_kv_cache_145_gb300 as pkv

    rank, local_rank, world = dist_env()
    if rank != 0:
        return
    # The CPU baseline child is spawned before any GPU work.
    cpu = None
    if not args.no_cpu_baseline:
        cpu = oracle_child(_oracle_op_sample, args.config, args.op, args.cpu_budget, 4242,
                           args.block_size or None)
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = Workload(args.config, block_size=args.block_size or None, table=args.table)
    seed = synth.seed_of(args.config, 3)
    shape = (w.N, w.Hk, w.b, w.D)
    cache = pkv.PagedKVCache(synth.normal(seed, shape, w.dtype, device="cuda"),
                             synth.normal(seed + 1, shape, w.dtype, device="cuda"))
    stream = torch.cuda.current_stream()
    block_bytes = w.Hk * w.b * w.D * w.elt
    peak, peak_kind = hbm_peak()
    extra = {}
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    if args.op == "write":
        # Slots of every cached position of every sequence, through its table.
        t = [np.arange(L) for L in w.seq_lens]
        slots = np.concatenate([w.tables[i][ti // w.b].astype(np.int64) * w.b + ti % w.b
                                for i, ti in enumerate(t)])
        n = len(slots)
        host = [synth.normal(seed + 2, (n, w.Hk, w.D), w.dtype).pin_memory(),
                synth.normal(seed + 3, (n, w.Hk, w.D), w.dtype).pin_memory(),
                torch.from_numpy(slots).pin_memory()]
        k, v, sl = (t.to(dev) for t in host)
        secs = _timed(lambda: pkv.paged_kv_write(cache, k, v, sl), args.steps, args.warmup, stream)
        # End to end: the new keys, values and slots cross from pinned host
        # memory in one copy before every write (the result stays in the pool).
        host_in, dev_in, views = pack_pinned(host, dev)

        def e2e_step():
            dev_in.copy_(host_in, non_blocking=True)
            pkv.paged_kv_write(cache, *views)
        e2e = (_timed(e2e_step, args.steps, args.warmup, stream), host_in.numel(), 0)
        nbytes = 2 * 2 * n * w.Hk * w.D * w.elt + 8 * n
        metric, unit_count, kernel = "paged KV write GB/s (prefill-sized)", n, "kv_write_kernel"
        extra["tokens"] = n
    elif args.op == "copy":
        perm = synth.free_order(seed + 4, w.N)
        half = w.N // 2
        pairs_h = torch.from_numpy(np.stack([perm[:half], perm[half:2 * half]], 1)).pin_memory()
        pairs = pairs_h.to(dev)
        secs = _timed(lambda: pkv.paged_block_copy(cache, pairs), args.steps, args.warmup, stream)
        # End to end: the pair list crosses from pinned host memory first.
        pairs_d = torch.empty_like(pairs)

        def e2e_step():
            pairs_d.copy_(pairs_h, non_blocking=True)
            pkv.paged_block_copy(cache, pairs_d)
        e2e = (_timed(e2e_step, args.steps, args.warmup, stream), pairs_h.numel() * 8, 0)
        nbytes = 2 * 2 * half * block_bytes + 16 * half
        metric, unit_count, kernel = "paged block copy GB/s (half the pool)", half, "block_move_kernel"
        extra["pairs"] = half
    else:
        half = w.N // 2
        hk = torch.empty((half, w.Hk, w.b, w.D), dtype=synth.TORCH_DTYPE[w.dtype]).pin_memory()
        hv = torch.empty_like(hk).pin_memory()
        perm = synth.free_order(seed + 4, w.N)
        out_pairs = torch.from_numpy(np.stack([perm[:half], np.arange(half)], 1)).to(dev)
        in_pairs = torch.from_numpy(np.stack([np.arange(half), perm[:half]], 1)).to(dev)
        t_out = _timed(lambda: pkv.paged_block_swap(cache, hk, hv, out_pairs, pkv.PKV_SWAP_OUT),
                       args.steps, args.warmup, stream)
        t_in = _timed(lambda: pkv.paged_block_swap(cache, hk, hv, in_pairs, pkv.PKV_SWAP_IN),
                      args.steps, args.warmup, stream)
        moved = 2 * half * block_bytes
        # Denominator: the copy engines moving the same bytes as one plain
        # contiguous cudaMemcpyAsync each way.
        dbuf = torch.empty(moved, dtype=torch.uint8, device=dev)
        hbuf = torch.empty(moved, dtype=torch.uint8).pin_memory()
        c_out = _timed(lambda: hbuf.copy_(dbuf, non_blocking=True), args.steps, args.warmup, stream)
        c_in = _timed(lambda: dbuf.copy_(hbuf, non_blocking=True), args.steps, args.warmup, stream)
        secs = (t_out + t_in) / 2
        # The swap's own launches already move host memory: the pair lists
        # are the only extra inputs that cross the link end to end.
        e2e = (secs, 16 * half, 0)
        nbytes = moved + 16 * half
        peak = moved / ((c_out + c_in) / 2) / 1e9
        peak_kind = "measured in this run: contiguous cudaMemcpyAsync of the same bytes"
        metric, unit_count, kernel = "block swap GB/s (HBM <-> pinned host, half the pool)", half, "block_move_kernel"
        extra.update(swap_out_gbs=round(moved / t_out / 1e9, 2), swap_in_gbs=round(moved / t_in / 1e9, 2),
                     memcpy_d2h_gbs=round(moved / c_out / 1e9, 2), memcpy_h2d_gbs=round(moved / c_in / 1e9, 2),
                     pairs=half)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    assert pkv.paged_get_device_error() == 0
    achieved = nbytes / secs / 1e9
    line = {
        "metric": metric, "value": round(achieved, 3), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": dict(workload=args.config, op=args.op, block_size=w.b, pool_blocks=w.N,
                       block_bytes=block_bytes, **extra),
        "roofline": {"bound": "hbm" if args.op != "swap" else "host-link", "achieved": round(achieved, 2),
                     "peak": round(peak, 2), "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None, "kernel": kernel, "peak_source": peak_kind},
        "clocks": clocks,
        "gpu_launches": args.steps * (2 if args.op == "swap" else 1),
        "e2e": {"value": round(nbytes / e2e[0] / 1e9, 3), "unit": "GB/s",
                "h2d_bytes_per_step": e2e[1], "d2h_bytes_per_step": e2e[2],
                "ms_per_step": round(e2e[0] * 1e3, 5)},
    }
    if cpu is not None:
        cb, cs, cu = cpu
        what = {"write": "%d tokens of whole sequences, each into a private pool of its blocks",
                "copy": "%d pairs, 256 per call over a 512-block pool",
                "swap": "%d blocks, 256 out to a host pool and back per call"}[args.op] % cu
        line["cpu_baseline"] = {
            "value": round(cb / cs / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%s, NumPy oracle, 1 thread, %.1f s" % (what, cs)}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="opt13b", choices=sorted(k for k in synth.CONFIGS if k != "tiny"))
    ap.add_argument("--partition", type=int, default=0, help="positions per partition (0 = default)")
    ap.add_argument("--block-size", type=int, default=0, help="override the workload's block size")
    ap.add_argument("--kv-dtype", choices=("native", "fp8"), default="native",
                    help="cache element type: the workload's own (default) or FP8 E4M3 with "
                         "per-head scales")
    ap.add_argument("--table", choices=("shuffled", "identity"), default="shuffled",
                    help="physical block order: shuffled pool (default) or consecutive blocks")
    ap.add_argument("--op", choices=("step", "write", "copy", "swap", "prefill"), default="step",
                    help="step: the decode step (default); write/copy/swap: bandwidth of the KV "
                         "write, block copy or host swap at sizes of our choosing; prefill: "
                         "chunk write + causal prefill attention (--config prefill|chunked)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-all-cores", action="store_true",
                    help="skip the all-cores oracle figure beside the one-process one")
    ap.add_argument("--decode", choices=("shared", "plain"), default="shared",
                    help="forked workload: shared-prefix decode (default) or the plain decode")
    ap.add_argument("--no-gqa", action="store_true",
                    help="default line: skip the GQA workload's sub-record")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "prefill" or args.config in PREFILL_CONFIGS:
        if args.config not in PREFILL_CONFIGS:
            ap.error("--op prefill needs --config prefill or chunked")
        run_prefill(args)
    elif args.op != "step":
        run_op(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
