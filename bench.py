"""Benchmark of the GB300 Leyline AMORTIZE splice.

Workload (default): the largest synthetic configuration, a concurrency sweep of
C = 16 requests sharing one 61-layer paged MLA pool (block size 16, latent 512 +
rope 64 bf16, lengths lognormal with median 24000 clipped to [2048, 131072]) and
1-3 directives per request: 36 directives, about 153k rewritten slots in every
layer, 21.5 GB of algorithmic bytes per call.  A step is one leyline_splice call
over all 16 requests (plan, move+rotate, commit kernels).

The requests stay resident: a rewrite splice only reads its source pages, so
between steps the caller's tables and lengths are put back from a saved copy and
the pool's page accounting is rolled back (leyline_pool_checkpoint /
leyline_pool_rollback); the next step splices the same 29.6 GB of rows again.
Those restores are a few device copies of tables and the free-page ring, and
they lie inside the timed region.  Smaller workloads keep as many copies as the
memory budget holds and restore only when all have been used.

Metric: downstream slots spliced per second (each slot covers all layers), plus
HBM GB/s of the move+rotate kernel against the measured copy bandwidth and the
8 TB/s nominal.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl reference] [--workload cfg5-C16-B16]
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
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

METRIC = "downstream slots spliced/sec (all layers) and HBM GB/s vs 8 TB/s on 1 GB300"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # the GB300 HBM3e figure the metric names
# Resident copies of a workload's requests are kept within this many bytes of pool.
DEFAULT_MEM_GB = 96.0
# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of a kernel on a
# workload, from one ncu capture of that kernel, valid only for the kernel code it was
# taken on (kernel_sha).  "scale": the capture ran on fewer layers and its traffic is
# multiplied by the ratio of the units (tile x layer) the full launch processes.
NCU_TRAFFIC = {
    # the move kernel on the largest workload, captured on 4 of its 61 layers (DRAM read
    # 704.28 MB = the algorithmic read; write 654.73 MB, the rest still in L2 at kernel end)
    ("sweep-C16-61L-B16", "move_rotate_vector"): {
        "kernel_sha256": "2ef00ccd9feaf4b162dd17472d88bf800b50479db73ede0fe9b44c6d14c453a3",
        "bytes": 704278016 + 654730752, "captured_layers": 4, "scale": 61 / 4},
    # the move kernel on the DeepSeek-V2-Lite shape (one call, 27 layers)
    ("dsv2lite-27L-32k-B16", "move_rotate_vector"): {
        "kernel_sha256": "2ef00ccd9feaf4b162dd17472d88bf800b50479db73ede0fe9b44c6d14c453a3",
        "bytes": 210919424 + 161249024},
    # the whole-line rotate kernel of a re-index call, block-1 sweep of 4 requests on 16 layers
    ("sweep-C4-61L-B1-as-16L", "rotate_in_place"): {
        "kernel_sha256": "e18d01e54a2418d387cdd03ae681b8d1df59b8c6e2830fe101411272b97dfcbb",
        "bytes": 130887680 + 71868672},
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="cfg5-C16-B16")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--reindex", action="store_true",
                    help="block size 1 pools: keep survivors in their pages (LEYLINE_POOL_REINDEX)")
    ap.add_argument("--lazy", action="store_true",
                    help="lazy pools: splices count pending turns instead of rotating (LEYLINE_POOL_LAZY)")
    ap.add_argument("--read", action="store_true",
                    help="lazy pools: also time leyline_materialize of the timed steps' requests")
    ap.add_argument("--split", action="store_true",
                    help="latents and rope bands in two arrays (LEYLINE_POOL_SPLIT_ROPE)")
    ap.add_argument("--e2e-copy", action="store_true",
                    help="e2e leg: copy rows of R to device buffers first, instead of passing pinned host rows")
    ap.add_argument("--single-leg", action="store_true",
                    help="time the move kernel inside the value leg and skip the other legs (large workloads)")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the workload's layer count (small cases for profiler captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="wall-time budget of each CPU-baseline sample (single core, then all cores)")
    ap.add_argument("--mem-gb", type=float, default=DEFAULT_MEM_GB,
                    help="device memory for resident copies of the workload's requests (at least one copy)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(seed: int, rank: int) -> int:
    """Each rank splices its own synthetic requests: the units are sharded, nothing is exchanged."""
    return seed + 1000 * rank


def reduce_max_over_ranks(values, world: int, device):
    """Element-wise max of per-rank timings (the job ends when its slowest rank does)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_value(slots_per_rank_step: int, steps: int, world: int, elapsed_ms_max: float) -> float:
    """Whole-job throughput: slots spliced by all ranks / the slowest rank's time."""
    return slots_per_rank_step * steps * world / (elapsed_ms_max / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources each timed kernel is compiled from: the shared headers and its own file.
KERNEL_COMMON = ("leyline_device.cuh", "leyline_plan.h", "leyline_internal.h")
KERNEL_FILES = {"move_rotate": "leyline_move.cu", "rotate_in_place": "leyline_reindex.cu",
                "materialize": "leyline_read.cu"}


def kernel_sha(kernel: str = "move_rotate"):
    """sha256 of one kernel's sources with comments and whitespace runs removed: a change to
    its code invalidates its stored ncu counters, a change to a comment or to another
    kernel's file does not."""
    text = ""
    for name in KERNEL_COMMON + (KERNEL_FILES[kernel],):
        with open(os.path.join(ROOT, "rope_rotation_gb300", "csrc", name)) as f:
            text += f.read() + "\n"
    text = re.sub(r"//[^\n]*", "", text)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"leyline_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.05)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workload --

def workload(name: str, layers: int = 0, chain_ok: bool = False):
    from synth import configs
    w = configs.by_name(name)
    w.key, w.layers_override = name, layers  # how a spawned worker rebuilds the same workload
    if len(w.steps) != 1 and not chain_ok:
        raise SystemExit(f"workload {name} is a multi-step chain; bench runs single-call workloads")
    if layers > 0:
        w.num_layers = layers
        w.name = f"{w.name}-as-{layers}L"
    return w


def _dry_directives(w, step):
    """The workload's directives for a host-only dry run: a 16-byte aligned stand-in for each
    directive's rows of R (the planner never reads them)."""
    from rope_rotation_gb300 import leyline
    fake = 1 << 40
    return [leyline.Directive(d.req, d.mode, d.s_start, d.s_end, d.n_repl, 0, fake if d.n_repl else None)
            for d in step]


def plan_stats(w, flags: int = 0):
    """The work accounting of one call of the workload (leyline_splice_plan: host planner, no
    device): downstream and replacement slots, algorithmic bytes, fresh pages taken."""
    from rope_rotation_gb300 import leyline
    desc = leyline.pool_desc(w.num_layers, w.block_size, 1, w.latent_dim, w.rope_dim, w.theta, flags=flags,
                             rope_heads=w.rope_heads)
    nb = max(-(-(L + 64 * 3) // w.block_size) for L in w.lengths)
    st, _ = leyline.leyline_splice_plan(desc, np.array(w.lengths, dtype=np.int64), nb, _dry_directives(w, w.steps[0]))
    return st


def host_plan_us(w, flags: int, reps: int = 50) -> float:
    """Median time of the host planner alone (leyline_splice_plan, C, no device) for one call."""
    from rope_rotation_gb300 import leyline
    desc = leyline.pool_desc(w.num_layers, w.block_size, 1, w.latent_dim, w.rope_dim, w.theta, flags=flags)
    dirs = _dry_directives(w, w.steps[0])
    nb = max(-(-(L + 64 * 3) // w.block_size) for L in w.lengths)
    lens = np.array(w.lengths, dtype=np.int64)
    times = []
    for _ in range(reps):
        t = time.perf_counter()
        leyline.leyline_splice_plan(desc, lens, nb, dirs)
        times.append((time.perf_counter() - t) * 1e6)
    return float(statistics.median(times))


def resident_copies(copy_bytes: int, wanted: int, mem_gb: float) -> int:
    """How many copies of the workload's requests stay resident: at most `wanted` (one per
    step of a leg), at least one, within mem_gb of pool."""
    fit = int(mem_gb * 1e9 // max(copy_bytes, 1))
    return max(1, min(wanted, fit))


# ---------------------------------------------------------------- our arm ---

# The value leg times the device (the metric runs from the first kernel of the first
# timed step to the last kernel of the last): before its first event the stream is held
# by a short spin, so that the host has queued steps when the timed region starts and
# the region holds the K steps' GPU work alone.  The e2e leg has no head start.
HEAD_START_CYCLES = 2_000_000  # about 1 ms at 2 GHz
L2_BYTES = 128 << 20  # GB300's L2 (129 MB), rounded down: the flush before a lazy read reads 4x this
READ_REPS = 4  # lazy reads: one after the splices, then three after a read pass that cleans L2


def hold_stream(torch, cycles: int = HEAD_START_CYCLES):
    torch.cuda._sleep(cycles)


def copy_gbps_now(torch, gib: float = 2.0, reps: int = 5) -> float:
    """A plain device copy (torch) of gib GiB on this GPU now, read + write bytes over the best of
    reps CUDA-event timings: context for the kernel fractions, beside the stored peak."""
    n = int(gib * (1 << 30)) // 2
    a = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    a.fill_(1.0)
    best = float("inf")
    for _ in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del a, b
    torch.cuda.empty_cache()
    return 2 * n * 2 / (best / 1e3) / 1e9


class Resident:
    """`copies` copies of the workload's requests in one pool, and the state to put them back.

    Copy g holds requests g*C .. g*C + C - 1.  After filling, the caller's table and lengths
    are saved and the pool's page accounting is checkpointed.  next_group() hands out the
    copies in turn; once all have been spliced it first restores the table, the lengths and
    the accounting (device copies on the stream, so they order after the last splice and
    before the next one), which makes every copy splice-able again: a rewrite splice only
    reads its source pages, and the rollback is refused if any of them was taken again."""

    def __init__(self, torch, cache, copies: int, C: int, flags: int, stream):
        from rope_rotation_gb300 import leyline
        self.torch, self.cache, self.copies, self.C = torch, cache, copies, C
        self.leyline = leyline
        self.stream = stream
        # bands turned in place (eager re-index) stay turned across a rollback: the work of
        # the repeated call is the same, its values are not compared
        self.flags = (leyline.LEYLINE_ROLLBACK_ACCEPT_TURNED
                      if (flags & leyline.LEYLINE_POOL_REINDEX) and not (flags & leyline.LEYLINE_POOL_LAZY)
                      else 0)
        self.table = cache.table.clone()
        self.lens_dev = cache.seq_lens_dev.clone()
        self.lens_host = cache.seq_lens_host.copy()
        leyline.leyline_pool_checkpoint(cache.pool, stream)
        self.used = 0
        self.restores = 0

    def restore(self, flags=None):
        c = self.cache
        c.table.copy_(self.table, non_blocking=True)
        c.seq_lens_dev.copy_(self.lens_dev, non_blocking=True)
        c.seq_lens_host[:] = self.lens_host
        self.leyline.leyline_pool_rollback(c.pool, self.flags if flags is None else flags, self.stream)
        self.used = 0
        self.restores += 1

    def next_group(self) -> int:
        if self.used == self.copies:
            self.restore()
        g = self.used
        self.used += 1
        return g


def run_ours(args, rank, world, local):
    import torch
    import __graft_entry__
    from rope_rotation_gb300 import leyline
    from rope_rotation_gb300.runtime import PagedCache
    from synth import fill

    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = workload(args.workload, args.layers)
    K, W = args.steps, args.warmup
    C = w.num_reqs
    B = w.block_size
    flags = ((leyline.LEYLINE_POOL_REINDEX if args.reindex else 0) | (leyline.LEYLINE_POOL_LAZY if args.lazy else 0)
             | (leyline.LEYLINE_POOL_SPLIT_ROPE if args.split else 0))
    if args.single_leg:
        args.no_e2e = True
    plan = plan_stats(w, flags)
    max_blocks = max(-(-(L + 64 * 3) // B) for L in w.lengths)
    # pages of one copy: its requests, plus the fresh pages one call takes
    copy_pages = sum(-(-L // B) for L in w.lengths) + plan.pages_popped + C
    page_bytes = w.num_layers * B * w.row_elems * 2
    copies = resident_copies(copy_pages * page_bytes, W + K, args.mem_gb)
    cache = PagedCache(w.num_layers, B, copies * copy_pages, copies * C, max_blocks, w.latent_dim, w.rope_dim,
                       w.theta, flags=flags)
    seed = rank_seed(w.seed, rank)
    for g in range(copies):
        for r, L in enumerate(w.lengths):
            cache.add_request(g * C + r, L)
            fill.fill_request(cache, seed, g * C + r, L)
    # replacement rows: device copies (value and kernel legs) and pinned host copies (e2e leg)
    repl_dev, repl_host = {}, {}
    for d in w.steps[0]:
        if d.n_repl:
            t = fill.repl_tensor(seed, d.req, d.key, w.num_layers, d.n_repl, cache.row, dev)
            repl_dev[d.key] = t
            repl_host[d.key] = t.cpu().pin_memory()

    # each step's directives: one checked template per source of R (directive_batch), of
    # which a step changes only the request ids
    templates = {}

    def dirs_for(g, repl_map):
        key = id(repl_map)
        if key not in templates:
            templates[key] = leyline.directive_batch([d.req for d in w.steps[0]], [d.s_start for d in w.steps[0]],
                                                     [d.s_end for d in w.steps[0]],
                                                     [repl_map.get(d.key) for d in w.steps[0]],
                                                     n_repl=[d.n_repl for d in w.steps[0]])
        b = templates[key].copy()
        b["req"] += g * C
        return b

    stream = torch.cuda.current_stream()
    stream_ptr = stream.cuda_stream
    torch.cuda.synchronize()
    res = Resident(torch, cache, copies, C, flags, stream_ptr)

    def step(repl_map):
        g = res.next_group()
        cache.splice(dirs_for(g, repl_map), stream_ptr)
        return g

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # warm-up
    for _ in range(W):
        step(repl_dev)
    torch.cuda.synchronize()
    cache.check_status()
    st = cache.last_stats()
    assert st["downstream_slots"] == plan.downstream_slots and st["algorithmic_bytes"] == plan.algorithmic_bytes

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.single_leg:
        leyline.leyline_kernel_timing_enable(cache.pool, True)
    restores0 = res.restores
    barrier()
    torch.cuda.synchronize()
    hold_stream(torch)
    ev0.record(stream)
    t_host = time.perf_counter()
    for _ in range(K):
        step(repl_dev)
    enqueue_us = (time.perf_counter() - t_host) * 1e6 / K
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    value_restores = res.restores - restores0
    cache.check_status()
    last = cache.last_stats()

    kernel_leg_ms = elapsed_ms  # --single-leg: the value leg carries the kernel events
    kl0, kl1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if not args.single_leg:
        # kernel leg: the same steps with events around each move (or rotate) kernel
        for _ in range(W):
            step(repl_dev)
        torch.cuda.synchronize()
        leyline.leyline_kernel_timing_enable(cache.pool, True)
        barrier()
        torch.cuda.synchronize()
        hold_stream(torch)
        kl0.record(stream)
        for _ in range(K):
            step(repl_dev)
        kl1.record(stream)
        torch.cuda.synchronize()
        barrier()
        kernel_leg_ms = kl0.elapsed_time(kl1)
    k2_ms, k2_n = leyline.leyline_kernel_timing_read(cache.pool)
    leyline.leyline_kernel_timing_enable(cache.pool, False)
    cache.check_status()

    e2e = None
    if not args.no_e2e:
        # End to end through the public API: each step's rows of R come from pinned host
        # memory, and the step's new lengths and table rows are read back to the host.
        rbuf = {k: torch.empty_like(v) for k, v in repl_dev.items()}
        out_tab = torch.empty((K, C, max_blocks), dtype=torch.int32).pin_memory()
        out_len = torch.empty((K, C), dtype=torch.int32).pin_memory()
        exp_len = np.zeros((K, C), dtype=np.int64)
        # rows of R: by default the splice is given the pinned host rows and its move kernel
        # reads them in place over the host link; --e2e-copy stages them on the device first
        src = rbuf if args.e2e_copy else repl_host
        for _ in range(W):  # warm the copy path
            if args.e2e_copy:
                for k2, v in repl_host.items():
                    rbuf[k2].copy_(v, non_blocking=True)
            step(src)
        torch.cuda.synchronize()
        h2d = sum(v.numel() * v.element_size() for v in repl_host.values())
        d2h = C * max_blocks * 4 + C * 4
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for k in range(K):
            if args.e2e_copy:
                for k2, v in repl_host.items():
                    rbuf[k2].copy_(v, non_blocking=True)
            g = step(src)
            out_tab[k].copy_(cache.table[g * C:(g + 1) * C], non_blocking=True)
            out_len[k].copy_(cache.seq_lens_dev[g * C:(g + 1) * C], non_blocking=True)
            exp_len[k] = cache.seq_lens_host[g * C:(g + 1) * C]
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = e0.elapsed_time(e1)
        cache.check_status()
        assert np.array_equal(out_len.numpy(), exp_len), "e2e read-back lengths differ"
        e2e = {"ms": e2e_ms, "h2d": h2d, "d2h": d2h,
               "inputs": "rows of R copied to device buffers, then spliced" if args.e2e_copy
               else "rows of R read in place from pinned host memory by the move kernel"}
    lazy_read = None
    if args.lazy and args.read:
        # the cost a lazy pool defers to its reads: splice every resident copy once, then
        # materialize all their requests (every pending band turned in place once, counts
        # cleared).  Repeated READ_REPS times: each repeat rolls the accounting and the
        # pending counts back (the bands stay turned: the same work on other values) and
        # splices the copies again.  The first read runs right after the splices, whose
        # writes still sit dirty in L2 and are written back during it; before each later one
        # a read-only pass over a buffer 4x the L2 writes them back, so that the read moves
        # its own bytes.  The reported figure is the median of the later reads.
        reqs = list(range(copies * C))
        turned = 0
        flush = torch.empty(4 * L2_BYTES // 4, dtype=torch.float32, device=dev).fill_(1.0)
        read_ms = []
        for rep in range(READ_REPS):
            res.restore(leyline.LEYLINE_ROLLBACK_ACCEPT_TURNED if rep else None)
            for _ in range(copies):
                step(repl_dev)
            if rep == 0:
                pend = cache.pending().view(-1)
                for q in reqs:
                    t = torch.arange(int(cache.seq_lens_host[q]), device=dev)
                    slots = cache.table[q][t // B].long() * B + t % B
                    turned += int((pend[slots] != 0).sum())
            r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            if rep:
                flush.sum()
                torch.cuda.synchronize()
            hold_stream(torch)
            r0.record(stream)
            cache.materialize_requests(reqs, stream_ptr)
            r1.record(stream)
            torch.cuda.synchronize()
            cache.check_status()
            read_ms.append(r0.elapsed_time(r1))
        del flush
        clean_ms = statistics.median(read_ms[1:])
        band_bytes = 2 * w.num_layers * w.rope_heads * w.rope_dim * 2  # read + write per turned slot
        lazy_read = {"op": "leyline_materialize_requests", "requests": len(reqs), "turned_slots": turned,
                     "ms": clean_ms, "slots_per_s": turned / (clean_ms / 1e3),
                     "algorithmic_gbps": turned * band_bytes / (clean_ms / 1e3) / 1e9,
                     "ms_each": read_ms, "l2": "written back before each read after the first (median of those); "
                     "the first read follows the splices with their writes dirty in L2",
                     "algorithmic_gbps_l2_dirty": turned * band_bytes / (read_ms[0] / 1e3) / 1e9}
    copy_now = copy_gbps_now(torch)
    clocks = sampler.stop()

    # max over ranks
    elapsed_ms, e2e_ms_max = reduce_max_over_ranks([elapsed_ms, e2e["ms"] if e2e else 0.0], world, dev)
    if e2e:
        e2e["ms"] = e2e_ms_max
    slots = st["downstream_slots"] * K * world
    reindexed = st["reindexed"] == 1
    value = job_value(st["downstream_slots"], K, world, elapsed_ms)
    peak, peak_kind = measured_peaks()
    k2_avg_s = (k2_ms / max(k2_n, 1)) / 1e3
    achieved = st["timed_kernel_bytes"] / k2_avg_s / 1e9
    kernel_name = (("prep_repl_reindex" if args.lazy else "rotate_in_place") if reindexed
                   else "move_rotate_" + os.environ.get("LEYLINE_MOVE_KERNEL", "vector"))
    traffic = stored_traffic(w, kernel_name, "rotate_in_place" if reindexed else "move_rotate",
                             eligible=not args.lazy and not args.split)
    step_achieved = st["algorithmic_bytes"] / (elapsed_ms / K / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "slots/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": elapsed_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "layers": w.num_layers, "requests": C,
                   "tokens": w.lengths if C > 1 else w.lengths[0],
                   "block_size": B, "latent_dim": w.latent_dim, "rope_dim": w.rope_dim, "storage": "bf16",
                   "directives": [[d.req, d.s_start, d.s_end, d.n_repl] for d in w.steps[0]],
                   "downstream_slots_per_step": st["downstream_slots"], "repl_slots_per_step": st["repl_slots"],
                   "algorithmic_bytes_per_step": st["algorithmic_bytes"],
                   "resident_copies": copies,
                   "restores_in_value_leg": value_restores,
                   "l2": "inputs larger than L2: each step splices "
                         + (f"{st['algorithmic_bytes'] / 2e9:.2f} GB of source rows" if copies == 1
                            else f"one of {copies} resident copies of the requests in turn"),
                   "repeat": "between steps the caller's table and lengths are copied back and the pool's page "
                             "accounting is rolled back (leyline_pool_rollback), once all resident copies have "
                             "been spliced; these restores run inside the timed region",
                   "timing": "value: CUDA events around K steps queued behind a ~1 ms spin on the stream "
                             "(device time of the steps); e2e: events around the steps with no head start",
                   "pool": ("lazy (pending turns, rotation on read)" if args.lazy else "eager")
                   + (", re-index" if reindexed else "") + (", split rope" if args.split else ""),
                   "move_kernel": ("rotate_in_place" if reindexed
                                   else os.environ.get("LEYLINE_MOVE_KERNEL", "vector")),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gbps_step": st["algorithmic_bytes"] * K * world / (elapsed_ms / 1e3) / 1e9,
        "slot_layers_per_s": value * w.num_layers,
        "host_plan_us": host_plan_us(w, flags & (leyline.LEYLINE_POOL_REINDEX | leyline.LEYLINE_POOL_LAZY)),
        # host side of the timed steps: the Python loop per step, and the library's own
        # account of its last call (leyline_stats_t host_ns, resolve_ns, plan_ns)
        "host": {"enqueue_us_per_step": enqueue_us, "splice_call_us": last["host_ns"] / 1e3,
                 "resolve_us": last["resolve_ns"] / 1e3, "plan_us": last["plan_ns"] / 1e3},
        "clocks": clocks,
        "gpu_launches": K * st["kernels_launched"],
        "roofline": {"kernel": kernel_name, "bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "frac_nominal": achieved / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS,
                     # a plain torch copy timed in this run, on this GPU: boxes differ by a few
                     # per cent, and this puts the fraction above in the run's own terms
                     "copy_gbps_this_run": copy_now, "frac_of_copy_this_run": achieved / copy_now,
                     "launch_ms": k2_avg_s * 1e3, "launches_timed": k2_n,
                     "algorithmic_bytes_per_launch": st["timed_kernel_bytes"],
                     # the value leg's steps (with their restores), against the same peaks
                     "step_achieved": step_achieved,
                     "step_frac": step_achieved / peak,
                     "step_frac_nominal": step_achieved / NOMINAL_HBM_GBS,
                     # the kernel's share of the kernel leg's own steps (serialised like an ncu
                     # launch list, so the two shares compare)
                     "launch_share": k2_ms / kernel_leg_ms if kernel_leg_ms > 0 else None},
    }
    if lazy_read:
        line["lazy_read"] = lazy_read
    if e2e:
        line["e2e"] = {"value": slots / (e2e["ms"] / 1e3), "unit": "slots/s", "h2d_bytes_per_step": e2e["h2d"],
                       "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": e2e["ms"] / K,
                       "inputs": e2e["inputs"]}
    cache.close()
    return line, w


def stored_traffic(w, kernel_name: str, kernel_src: str, eligible: bool = True):
    """Per-launch DRAM bytes of the timed kernel on this workload from the stored ncu capture,
    or None when there is none or the kernel's code changed since it was taken."""
    stored = NCU_TRAFFIC.get((w.name, kernel_name))
    if not eligible or not stored or stored["kernel_sha256"] != kernel_sha(kernel_src):
        return None
    return stored["bytes"] * stored.get("scale", 1.0)


def run_chain(args, rank, world, local):
    """A workload of successive splices of one request (the 64-splice chain): a step is the
    whole chain on a fresh copy of the request, its splices enqueued back to back (each one
    planned on the lengths the one before left).  Value: downstream slots of all splices per
    second; the roofline kernel is timed around every splice's move (or rotate) kernel."""
    import torch
    import __graft_entry__
    from rope_rotation_gb300 import leyline
    from rope_rotation_gb300.runtime import PagedCache
    from synth import fill

    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = workload(args.workload, args.layers, chain_ok=True)
    K, W = args.steps, args.warmup
    assert w.num_reqs == 1 and all(len(step) == 1 for step in w.steps), "one request, one directive per splice"
    L0, B = w.lengths[0], w.block_size
    nb = -(-max(L0, max(d.s_start + d.n_repl for step in w.steps for d in step)) // B) + 1
    flags = ((leyline.LEYLINE_POOL_REINDEX if args.reindex else 0) | (leyline.LEYLINE_POOL_LAZY if args.lazy else 0)
             | (leyline.LEYLINE_POOL_SPLIT_ROPE if args.split else 0))
    # As many copies of the request as the memory budget holds.  A chain's splices recycle the
    # pages they return, so a spent copy cannot be rolled back: between chains (outside the
    # timed events) its pages are returned and the request is written afresh.
    copies = resident_copies(nb * w.num_layers * B * w.row_elems * 2, W + K, args.mem_gb)
    # every chain copy's pages, plus one request's worth for the fresh pages a rewrite takes
    cache = PagedCache(w.num_layers, B, (copies + 1) * nb, copies, nb, w.latent_dim, w.rope_dim, w.theta, flags=flags)
    seed = rank_seed(w.seed, rank)
    for g in range(copies):
        cache.add_request(g, L0)
        fill.fill_request(cache, seed, g, L0)
    spent = [False] * copies

    def fresh_copy(k):
        """The copy chain k runs on, written afresh first if an earlier chain spent it."""
        g = k % copies
        if spent[g]:
            n_old = -(-int(cache.seq_lens_host[g]) // B)
            leyline.leyline_free_pages(cache.pool, cache.table[g, :n_old].cpu().numpy())
            cache.table[g].fill_(-1)
            cache.add_request(g, L0)
            fill.fill_request(cache, seed, g, L0)
            torch.cuda.synchronize()
        spent[g] = True
        return g
    tmpl = []
    for step in w.steps:
        d = step[0]
        r = fill.repl_tensor(seed, 0, d.key, w.num_layers, d.n_repl, cache.row, dev) if d.n_repl else None
        tmpl.append((leyline.directive_batch([0], [d.s_start], [d.s_end], [r], n_repl=[d.n_repl],
                                             mode=[d.mode]), r))
    stream = torch.cuda.current_stream()
    stream_ptr = stream.cuda_stream

    def chain(g, stats=None):
        for t, _ in tmpl:
            b = t.copy()
            b["req"] = g
            cache.splice(b, stream_ptr)
            if stats is not None:
                for k, v in cache.last_stats().items():
                    stats[k] = stats.get(k, 0) + v

    per_chain = {}
    for k in range(W):
        chain(fresh_copy(k), per_chain if k == 0 else None)
        torch.cuda.synchronize()
    if W == 0:
        raise SystemExit("a chain needs at least one warm-up chain (its work counts come from it)")
    cache.check_status()
    n_splices = len(tmpl)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    leyline.leyline_kernel_timing_enable(cache.pool, True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    # each chain has its own events, behind a spin long enough for the host to queue the
    # whole chain; a copy written afresh between chains lies outside them
    elapsed_ms, enqueue_s = 0.0, 0.0
    for k in range(W, W + K):
        g = fresh_copy(k)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_stream(torch, 4 * HEAD_START_CYCLES)
        ev0.record(stream)
        t_host = time.perf_counter()
        chain(g)
        enqueue_s += time.perf_counter() - t_host
        ev1.record(stream)
        torch.cuda.synchronize()
        elapsed_ms += ev0.elapsed_time(ev1)
    enqueue_us = enqueue_s * 1e6 / K
    if world > 1:
        dist.barrier()
    cache.check_status()
    k2_ms, k2_n = leyline.leyline_kernel_timing_read(cache.pool)
    leyline.leyline_kernel_timing_enable(cache.pool, False)
    clocks = sampler.stop()
    (elapsed_ms,) = reduce_max_over_ranks([elapsed_ms], world, dev)
    value = job_value(per_chain["downstream_slots"], K, world, elapsed_ms)
    peak, peak_kind = measured_peaks()
    # per launch: the timed kernels' algorithmic bytes over their summed time
    achieved = per_chain["timed_kernel_bytes"] * K / (k2_ms / 1e3) / 1e9 if k2_ms > 0 else 0.0
    reindexed = per_chain["reindexed"] > 0
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "slots/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": elapsed_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "layers": w.num_layers, "tokens": L0, "block_size": B,
                   "latent_dim": w.latent_dim, "rope_dim": w.rope_dim, "storage": "bf16",
                   "splices_per_step": n_splices,
                   "step": "the whole chain of successive splices on a fresh copy of the request",
                   "downstream_slots_per_step": per_chain["downstream_slots"],
                   "repl_slots_per_step": per_chain["repl_slots"],
                   "algorithmic_bytes_per_step": per_chain["algorithmic_bytes"],
                   "reindexed_splices": per_chain["reindexed"],
                   "l2": "inputs larger than L2: each chain splices its own pre-filled request",
                   "resident_copies": copies,
                   "timing": "CUDA events around each of the K chains, each queued behind a ~4 ms spin on the "
                             "stream; a copy spent by an earlier chain is written afresh outside the events",
                   "pool": ("lazy (pending turns, rotation on read)" if args.lazy else "eager")
                   + (", re-index" if args.reindex else "") + (", split rope" if args.split else ""),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gbps_step": per_chain["algorithmic_bytes"] * K * world / (elapsed_ms / 1e3) / 1e9,
        "slot_layers_per_s": value * w.num_layers,
        "host": {"enqueue_us_per_step": enqueue_us, "enqueue_us_per_splice": enqueue_us / n_splices},
        "clocks": clocks,
        "gpu_launches": K * per_chain["kernels_launched"],
        "roofline": {"kernel": (("prep_repl_reindex" if args.lazy else "rotate_in_place") if reindexed
                                else "move_rotate_vector"), "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "launch_ms": k2_ms / max(k2_n, 1), "launches_timed": k2_n,
                     "algorithmic_bytes_per_launch": per_chain["timed_kernel_bytes"] / n_splices,
                     "step_achieved": per_chain["algorithmic_bytes"] / (elapsed_ms / K / 1e3) / 1e9,
                     "step_frac": per_chain["algorithmic_bytes"] / (elapsed_ms / K / 1e3) / 1e9 / peak,
                     "launch_share": k2_ms / elapsed_ms if elapsed_ms > 0 else None},
    }
    cache.close()
    return line, w


# -------------------------------------------------------------- CPU oracle --
#
# The oracle (fp64 C, as it stands) timed on the host cores.  A call's work is cut into
# units of one request's splice in one layer (layers are independent: the same plan turns
# every layer).  A unit's rows are generated first and only the oracle call is timed.  The
# single-core figure runs units one after another in this process; the all-core figure
# runs them in a pool of spawned processes (spawned, not forked: this process may hold a
# CUDA context), one per core, and divides their slots by the longest summed oracle time
# of any process.  Slots are counted as the metric counts them: a unit of request r in one
# layer is worth downstream(r) / layers slots.

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_units(w):
    """[(request, layer, slot worth)] of one call, layer-major, and the call's downstream slots."""
    import oracle
    per_req = {}
    for r in range(w.num_reqs):
        ds = [d for d in w.steps[0] if d.req == r]
        if not ds:
            continue
        _, kind, idx, _ = oracle.splice_map(w.lengths[r], [(d.s_start, d.s_end, d.n_repl) for d in ds])
        first_end = min(d.s_end for d in ds)
        per_req[r] = int(np.count_nonzero((kind == 0) & (idx >= first_end)))
    units = [(r, layer, per_req[r] / w.num_layers) for layer in range(w.num_layers) for r in sorted(per_req)]
    return units, sum(per_req.values())


def _oracle_unit(job):
    """One unit in a worker: generate the request's rows of one layer, time the oracle's splice."""
    import oracle
    import synth
    seed, key, layers, r, layer = job
    w = workload(key, layers)
    ds = [d for d in w.steps[0] if d.req == r]
    cache = synth.cache_rows(seed, r, layer, np.arange(w.lengths[r]), w.row_elems)[None]
    reps = [synth.repl_rows(seed, r, d.key, w.num_layers, d.n_repl, w.row_elems)[layer:layer + 1] for d in ds]
    t0 = time.perf_counter()
    oracle.splice_request(cache, [(d.s_start, d.s_end, d.n_repl) for d in ds], reps, w.latent_dim, w.theta)
    return time.perf_counter() - t0, os.getpid()


class OraclePool:
    """Spawned worker processes, one per host core, that run oracle units."""

    def __init__(self, procs: int):
        import multiprocessing as mp
        import oracle
        oracle.build()  # once, here; the workers load the built library
        self.procs = procs
        self.pool = mp.get_context("spawn").Pool(procs)

    def run(self, seed: int, w, units) -> tuple[float, float]:
        """(longest summed oracle seconds of any worker, wall seconds) over the units."""
        per_pid = {}
        t0 = time.perf_counter()
        jobs = [(seed, w.key, w.layers_override, r, l) for r, l, _ in units]
        for dt, pid in self.pool.imap_unordered(_oracle_unit, jobs):
            per_pid[pid] = per_pid.get(pid, 0.0) + dt
        return max(per_pid.values()), time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def single_core_sample(w, units, budget_s: float, seed: int):
    """Units one after another in this process until budget_s of oracle time: (slots, seconds, units)."""
    slots, spent, n = 0.0, 0.0, 0
    for r, layer, worth in units:
        dt, _ = _oracle_unit((seed, w.key, w.layers_override, r, layer))
        slots += worth
        spent += dt
        n += 1
        if spent >= budget_s:
            break
    return slots, spent, n


def parallel_units(units, rate_1: float, budget_core_s: float, procs: int = 1):
    """The first units (layer-major, so every request is in the sample) whose single-core
    estimate fits budget_core_s core-seconds; at least one layer of every request.  When the
    sample holds at least `procs` units it is cut to a multiple of procs, so that no process
    runs one unit more than the others."""
    per_layer = len({r for r, _, _ in units})
    out, est = [], 0.0
    for i, u in enumerate(units):
        est += u[2] / rate_1
        if est > budget_core_s and i >= per_layer:
            break
        out.append(u)
    if procs > 1 and len(out) >= procs:
        out = out[:len(out) // procs * procs]
    return out


def cpu_oracle_sample(w, budget_s: float, seed: int = 0):
    """The oracle on the host cores: a single-core sample, then a sample on all cores."""
    units, _ = oracle_units(w)
    s1, t1, n1 = single_core_sample(w, units, budget_s / 2, seed)
    rate_1 = s1 / t1
    procs = host_cores()
    pool = OraclePool(procs)
    try:
        pu = parallel_units(units, rate_1, budget_s * procs, procs)
        busy, wall = pool.run(seed, w, pu)
    finally:
        pool.close()
    slots_n = sum(u[2] for u in pu)
    whole = len(pu) == len(units)
    return {"value": slots_n / busy, "unit": "slots/s", "cores": procs, "kind": "oracle",
            "single_core_value": rate_1,
            "sample": f"{'one whole call' if whole else f'{len(pu)} of {len(units)} (request, layer) units of a call'}"
                      f" of {w.name} ({w.num_layers} layers) through the fp64 C oracle in {procs} spawned "
                      f"processes: {slots_n:.0f} slots over the longest per-process oracle time {busy:.2f} s "
                      f"({wall:.2f} s wall with row generation); single core: {n1} units, {s1:.0f} slots in "
                      f"{t1:.2f} s"}


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle, as it stands, on all host cores.  A step is a
    bounded sample of one call of the same workload: (request, layer) units, layer-major,
    every request in it, sized from a single-core calibration to about cpu_seconds of wall
    time on the host's cores."""
    if rank != 0:
        return None
    w = workload(args.workload, args.layers)
    seed = w.seed
    units, _ = oracle_units(w)
    s1, t1, _ = single_core_sample(w, units, 1.0, seed)
    procs = host_cores()
    pu = parallel_units(units, s1 / t1, args.cpu_seconds * procs / 4, procs)
    slots = sum(u[2] for u in pu)
    pool = OraclePool(procs)
    try:
        for _ in range(args.warmup):
            pool.run(seed, w, pu)
        busy = [pool.run(seed, w, pu)[0] for _ in range(args.steps)]
    finally:
        pool.close()
    dt = sum(busy)
    value = slots * args.steps / dt
    sample = (f"{len(pu)} of {len(units)} (request, layer) units of one call of {w.name} per step "
              f"({slots:.0f} slots), fp64 C oracle in {procs} spawned processes; a step's time is the longest "
              f"per-process oracle time")
    return {"metric": METRIC, "value": value, "unit": "slots/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "layers": w.num_layers, "block_size": w.block_size, "storage": "bf16"},
            "cpu_baseline": {"value": value, "unit": "slots/s", "cores": procs, "kind": "oracle",
                             "single_core_value": s1 / t1, "sample": sample},
            "e2e": {"value": value, "unit": "slots/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    from synth import configs
    is_chain = len(configs.by_name(args.workload).steps) > 1
    line, w = (run_chain if is_chain else run_ours)(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1 and not is_chain:
            cb = cpu_oracle_sample(w, args.cpu_seconds)
            line["cpu_baseline"] = cb
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
