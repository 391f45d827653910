"""Benchmark of the GB300 Leyline AMORTIZE splice.

Workload (default): the DeepSeek-V2-Lite-shaped paged MLA cache -- 27 layers,
32768 tokens, block size 16, latent 512 + rope 64 bf16 -- and one directive that
replaces [20000, 26000) by 12 rows (Delta = -5988): 6768 downstream slots, each
moved and rotated in all 27 layers.  A step is one leyline_splice call (plan,
move+rotate, commit kernels) on one request.  Each timed step splices a
different, pre-filled request, so every step reads 0.42 GB that no earlier step
touched (inputs larger than L2; no reset inside the timed region).

Metric: downstream slots spliced per second (each slot covers all layers), plus
HBM GB/s of the move+rotate kernel against the measured copy bandwidth.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl reference] [--workload cfg2]
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
# Per-launch DRAM traffic (read + write bytes) of a kernel on a workload, from an ncu
# capture, valid only for the kernel code it was taken on (kernel_sha)
# (profiles/move_rotate_dsv2lite_27L_32k_B16_full.md: read 210.9 MB + write 160.8 MB; the
# rest of the 210.9 MB written was still in L2 when the single captured launch ended).
NCU_TRAFFIC = {
    ("dsv2lite-27L-32k-B16", "move_rotate_vector"): {
        "kernel_sha256": "cb5ffd94aae258a0a13a19b61dad06767e0bff66acc83ae01ddca7f255930f65",
        "bytes": 210919168 + 160825344},
    # profiles/rotate_in_place_sweep_C4_B1_16L_full.md (the rotate kernel alone)
    ("sweep-C4-61L-B1-as-16L", "rotate_in_place"): {
        "kernel_sha256": "2d7517d189d93b0a50478fd95ba3c605c4f05540a7e8e380a390b1ef1cf6ff2b",
        "bytes": 130889984 + 75299584},
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="cfg2")
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
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the CPU-baseline sample")
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
    if len(w.steps) != 1 and not chain_ok:
        raise SystemExit(f"workload {name} is a multi-step chain; bench runs single-call workloads")
    if layers > 0:
        w.num_layers = layers
        w.name = f"{w.name}-as-{layers}L"
    return w


def per_request_counts(w):
    """Downstream and replacement slots of one call of the workload (oracle-free: planner dry run)."""
    from rope_rotation_gb300 import leyline
    desc = leyline.pool_desc(w.num_layers, w.block_size, 1, w.latent_dim, w.rope_dim, w.theta)
    dirs = [leyline.directive(d.req, d.s_start, d.s_end, None, n_repl=0) for d in w.steps[0]]
    nb = max(-(-(L + 64 * 3) // w.block_size) for L in w.lengths)
    st, _ = leyline.leyline_splice_plan(desc, np.array(w.lengths, dtype=np.int64), nb, dirs)
    return st


def host_plan_us(w, flags: int, reps: int = 50) -> float:
    """Median time of the host planner alone (leyline_splice_plan, C, no device) for one call."""
    from rope_rotation_gb300 import leyline
    desc = leyline.pool_desc(w.num_layers, w.block_size, 1, w.latent_dim, w.rope_dim, w.theta, flags=flags)
    fake = 1 << 40  # a 16-byte aligned stand-in for the rows of R: the dry run never reads them
    dirs = [leyline.Directive(d.req, d.mode, d.s_start, d.s_end, d.n_repl, 0, fake if d.n_repl else None)
            for d in w.steps[0]]
    nb = max(-(-(L + 64 * 3) // w.block_size) for L in w.lengths)
    lens = np.array(w.lengths, dtype=np.int64)
    times = []
    for _ in range(reps):
        t = time.perf_counter()
        leyline.leyline_splice_plan(desc, lens, nb, dirs)
        times.append((time.perf_counter() - t) * 1e6)
    return float(statistics.median(times))


# ---------------------------------------------------------------- our arm ---

# The value leg times the device (the metric runs from the first kernel of the first
# timed step to the last kernel of the last): before its first event the stream is held
# by a short spin, so that the host has queued steps when the timed region starts and
# the region holds the K steps' GPU work alone.  The e2e leg has no head start.
HEAD_START_CYCLES = 2_000_000  # about 1 ms at 2 GHz


def hold_stream(torch):
    torch.cuda._sleep(HEAD_START_CYCLES)


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
    # legs: value (plain steps), kernel (the same steps with CUDA events around the
    # move+rotate kernel, for the roofline), e2e (host buffers); each step and warm-up
    # of each leg splices its own copy of the workload's requests
    if args.single_leg:
        args.no_e2e = True
    legs = 1 if args.single_leg else (2 if args.no_e2e else 3)
    groups = (W + K) * legs
    B = w.block_size
    max_blocks = max(-(-(L + 64 * 3) // B) for L in w.lengths)
    pages = groups * sum(-(-L // B) for L in w.lengths) + sum(-(-L // B) + 1 for L in w.lengths)
    cache = PagedCache(w.num_layers, B, pages, groups * C, max_blocks, w.latent_dim, w.rope_dim, w.theta,
                       flags=(leyline.LEYLINE_POOL_REINDEX if args.reindex else 0)
                       | (leyline.LEYLINE_POOL_LAZY if args.lazy else 0)
                       | (leyline.LEYLINE_POOL_SPLIT_ROPE if args.split else 0))
    seed = rank_seed(w.seed, rank)
    for g in range(groups):
        for r, L in enumerate(w.lengths):
            cache.add_request(g * C + r, L)
            fill.fill_request(cache, seed, g * C + r, L)
    # replacement rows: device copies (value leg) and pinned host copies (e2e leg)
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
    # warm-up
    for g in range(W):
        cache.splice(dirs_for(g, repl_dev))
    torch.cuda.synchronize()
    cache.check_status()
    st = cache.last_stats()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.single_leg:
        leyline.leyline_kernel_timing_enable(cache.pool, True)
    barrier()
    torch.cuda.synchronize()
    hold_stream(torch)
    ev0.record(stream)
    t_host = time.perf_counter()
    for k in range(K):
        cache.splice(dirs_for(W + k, repl_dev), stream_ptr)
    enqueue_us = (time.perf_counter() - t_host) * 1e6 / K
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    cache.check_status()
    last = cache.last_stats()

    kernel_leg_ms = elapsed_ms  # --single-leg: the value leg carries the kernel events
    kl0, kl1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if not args.single_leg:
        # kernel leg: the same steps on fresh requests, with events around move+rotate
        base = W + K
        for g in range(W):
            cache.splice(dirs_for(base + g, repl_dev))
        torch.cuda.synchronize()
        leyline.leyline_kernel_timing_enable(cache.pool, True)
        barrier()
        torch.cuda.synchronize()
        hold_stream(torch)
        kl0.record(stream)
        for k in range(K):
            cache.splice(dirs_for(base + W + k, repl_dev))
        kl1.record(stream)
        torch.cuda.synchronize()
        barrier()
        kernel_leg_ms = kl0.elapsed_time(kl1)
    k2_ms, k2_n = leyline.leyline_kernel_timing_read(cache.pool)
    leyline.leyline_kernel_timing_enable(cache.pool, False)
    cache.check_status()

    e2e = None
    if not args.no_e2e:
        # End to end through the public API: each step copies its replacement rows from
        # pinned host memory, splices, and reads back the request's new lengths and table row.
        base = 2 * (W + K)
        rbuf = {k: torch.empty_like(v) for k, v in repl_dev.items()}
        out_tab = torch.empty((K, C, max_blocks), dtype=torch.int32).pin_memory()
        out_len = torch.empty((K, C), dtype=torch.int32).pin_memory()
        # rows of R: by default the splice is given the pinned host rows and its move kernel
        # reads them in place over the host link; --e2e-copy stages them on the device first
        src = rbuf if args.e2e_copy else repl_host
        for g in range(W):  # warm the copy path
            if args.e2e_copy:
                for k2, v in repl_host.items():
                    rbuf[k2].copy_(v, non_blocking=True)
            cache.splice(dirs_for(base + g, src))
        torch.cuda.synchronize()
        h2d = sum(v.numel() * v.element_size() for v in repl_host.values())
        d2h = C * max_blocks * 4 + C * 4
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for k in range(K):
            g = base + W + k
            if args.e2e_copy:
                for k2, v in repl_host.items():
                    rbuf[k2].copy_(v, non_blocking=True)
            cache.splice(dirs_for(g, src), stream_ptr)
            out_tab[k].copy_(cache.table[g * C:(g + 1) * C], non_blocking=True)
            out_len[k].copy_(cache.seq_lens_dev[g * C:(g + 1) * C], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = e0.elapsed_time(e1)
        cache.check_status()
        exp_len = cache.seq_lens_host[(base + W) * C:(base + W + K) * C].reshape(K, C)
        assert np.array_equal(out_len.numpy(), exp_len), "e2e read-back lengths differ"
        e2e = {"ms": e2e_ms, "h2d": h2d, "d2h": d2h,
               "inputs": "rows of R copied to device buffers, then spliced" if args.e2e_copy
               else "rows of R read in place from pinned host memory by the move kernel"}
    lazy_read = None
    if args.lazy and args.read:
        # the cost a lazy pool defers to its reads: materialize each request of the value
        # leg's timed steps (every pending band turned in place once, counts cleared)
        reqs = [g * C + r for g in range(W, W + K) for r in range(C)]
        pend = cache.pending().view(-1)
        turned = 0
        for q in reqs:
            t = torch.arange(int(cache.seq_lens_host[q]), device=dev)
            slots = cache.table[q][t // B].long() * B + t % B
            turned += int((pend[slots] != 0).sum())
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        hold_stream(torch)
        r0.record(stream)
        cache.materialize_requests(reqs, stream_ptr)
        r1.record(stream)
        torch.cuda.synchronize()
        cache.check_status()
        read_ms = r0.elapsed_time(r1)
        band_bytes = 2 * w.num_layers * w.rope_heads * w.rope_dim * 2  # read + write per turned slot
        lazy_read = {"op": "leyline_materialize_requests", "requests": len(reqs), "turned_slots": turned,
                     "ms": read_ms, "slots_per_s": turned / (read_ms / 1e3),
                     "algorithmic_gbps": turned * band_bytes / (read_ms / 1e3) / 1e9}
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
    achieved = st["algorithmic_bytes"] / k2_avg_s / 1e9
    kernel_name = "rotate_in_place" if reindexed else "move_rotate_" + os.environ.get("LEYLINE_MOVE_KERNEL", "vector")
    traffic = None
    stored = NCU_TRAFFIC.get((w.name, kernel_name))
    if stored and not args.lazy and not args.split and stored["kernel_sha256"] == kernel_sha(
            "rotate_in_place" if reindexed else "move_rotate"):
        traffic = stored["bytes"]
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
        "config": {"workload": w.name, "layers": w.num_layers, "tokens": w.lengths if C > 1 else w.lengths[0],
                   "block_size": B, "latent_dim": w.latent_dim, "rope_dim": w.rope_dim, "storage": "bf16",
                   "directives": [[d.s_start, d.s_end, d.n_repl] for d in w.steps[0]],
                   "downstream_slots_per_step": st["downstream_slots"], "repl_slots_per_step": st["repl_slots"],
                   "algorithmic_bytes_per_step": st["algorithmic_bytes"],
                   "l2": "inputs larger than L2: each step splices its own pre-filled request",
                   "timing": "value: CUDA events around K steps queued behind a ~1 ms spin on the stream "
                             "(device time of the steps); e2e: events around the steps with no head start",
                   "pool": ("lazy (pending turns, rotation on read)" if args.lazy else "eager")
                   + (", re-index" if reindexed else "") + (", split rope" if args.split else ""),
                   "move_kernel": ("rotate_in_place" if reindexed
                                   else os.environ.get("LEYLINE_MOVE_KERNEL", "vector")),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gbps_step": st["algorithmic_bytes"] * K * world / (elapsed_ms / 1e3) / 1e9,
        "slot_layers_per_s": value * w.num_layers,
        "host_plan_us": host_plan_us(w, (leyline.LEYLINE_POOL_REINDEX if args.reindex else 0)
                                     | (leyline.LEYLINE_POOL_LAZY if args.lazy else 0)),
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
                     "launch_ms": k2_avg_s * 1e3, "launches_timed": k2_n,
                     "algorithmic_bytes_per_launch": st["algorithmic_bytes"],
                     # the value leg's steps: consecutive calls overlap there, which the
                     # per-launch events of the kernel leg rule out
                     "step_achieved": st["algorithmic_bytes"] / (elapsed_ms / K / 1e3) / 1e9,
                     "step_frac": st["algorithmic_bytes"] / (elapsed_ms / K / 1e3) / 1e9 / peak,
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


# -------------------------------------------------------------- CPU oracle --

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
    groups = W + K
    flags = ((leyline.LEYLINE_POOL_REINDEX if args.reindex else 0) | (leyline.LEYLINE_POOL_LAZY if args.lazy else 0)
             | (leyline.LEYLINE_POOL_SPLIT_ROPE if args.split else 0))
    # every chain copy's pages, plus one request's worth for the fresh pages a rewrite takes
    cache = PagedCache(w.num_layers, B, (groups + 1) * nb, groups, nb, w.latent_dim, w.rope_dim, w.theta, flags=flags)
    seed = rank_seed(w.seed, rank)
    for g in range(groups):
        cache.add_request(g, L0)
        fill.fill_request(cache, seed, g, L0)
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
    for g in range(W):
        chain(g, per_chain if g == 0 else None)
    if W == 0:
        raise SystemExit("a chain needs at least one warm-up chain (its work counts come from it)")
    torch.cuda.synchronize()
    cache.check_status()
    n_splices = len(tmpl)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    leyline.leyline_kernel_timing_enable(cache.pool, True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    hold_stream(torch)
    ev0.record(stream)
    t_host = time.perf_counter()
    for g in range(W, W + K):
        chain(g)
    enqueue_us = (time.perf_counter() - t_host) * 1e6 / K
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    cache.check_status()
    k2_ms, k2_n = leyline.leyline_kernel_timing_read(cache.pool)
    leyline.leyline_kernel_timing_enable(cache.pool, False)
    clocks = sampler.stop()
    (elapsed_ms,) = reduce_max_over_ranks([elapsed_ms], world, dev)
    value = job_value(per_chain["downstream_slots"], K, world, elapsed_ms)
    peak, peak_kind = measured_peaks()
    # per launch: the chain's algorithmic bytes spread over its timed launches
    achieved = per_chain["algorithmic_bytes"] * K / (k2_ms / 1e3) / 1e9 if k2_ms > 0 else 0.0
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
                   "timing": "CUDA events around K chains queued behind a ~1 ms spin on the stream",
                   "pool": ("lazy (pending turns, rotation on read)" if args.lazy else "eager")
                   + (", re-index" if args.reindex else "") + (", split rope" if args.split else ""),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gbps_step": per_chain["algorithmic_bytes"] * K * world / (elapsed_ms / 1e3) / 1e9,
        "slot_layers_per_s": value * w.num_layers,
        "host": {"enqueue_us_per_step": enqueue_us, "enqueue_us_per_splice": enqueue_us / n_splices},
        "clocks": clocks,
        "gpu_launches": K * per_chain["kernels_launched"],
        "roofline": {"kernel": "rotate_in_place" if reindexed else "move_rotate_vector", "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "launch_ms": k2_ms / max(k2_n, 1), "launches_timed": k2_n,
                     "algorithmic_bytes_per_launch": per_chain["algorithmic_bytes"] / n_splices,
                     "step_achieved": per_chain["algorithmic_bytes"] / (elapsed_ms / K / 1e3) / 1e9,
                     "step_frac": per_chain["algorithmic_bytes"] / (elapsed_ms / K / 1e3) / 1e9 / peak,
                     "launch_share": k2_ms / elapsed_ms if elapsed_ms > 0 else None},
    }
    cache.close()
    return line, w


def cpu_oracle_sample(w, budget_s: float, seed: int = 0):
    """Time the fp64 oracle (single thread, as it stands) on whole calls of the workload,
    repeated until about budget_s seconds of CPU work."""
    import oracle
    import synth
    st = per_request_counts(w)
    caches = [synth.cache_request(seed, r, w.num_layers, L, w.row_elems) for r, L in enumerate(w.lengths)]
    reps = {d.key: synth.repl_rows(seed, d.req, d.key, w.num_layers, d.n_repl, w.row_elems) for d in w.steps[0]}
    calls, t_total = 0, 0.0
    while t_total < budget_s or calls == 0:
        t0 = time.perf_counter()
        for r in range(w.num_reqs):
            ds = [d for d in w.steps[0] if d.req == r]
            if ds:
                oracle.splice_request(caches[r], [(d.s_start, d.s_end, d.n_repl) for d in ds],
                                      [reps[d.key] for d in ds], w.latent_dim, w.theta)
        t_total += time.perf_counter() - t0
        calls += 1
    value = st.downstream_slots * calls / t_total
    return {"value": value, "unit": "slots/s", "cores": 1, "kind": "oracle",
            "sample": f"{calls} whole call(s) of {w.name} ({w.num_layers} layers) through the fp64 C oracle, "
                      f"single thread, {t_total:.1f} s"}, t_total / calls


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle timed as it stands on the same workload."""
    if rank != 0:
        return None
    w = workload(args.workload, args.layers)
    import oracle
    import synth
    st = per_request_counts(w)
    seed = w.seed
    caches = [synth.cache_request(seed, r, w.num_layers, L, w.row_elems) for r, L in enumerate(w.lengths)]
    reps = {d.key: synth.repl_rows(seed, d.req, d.key, w.num_layers, d.n_repl, w.row_elems) for d in w.steps[0]}

    def one_call():
        for r in range(w.num_reqs):
            ds = [d for d in w.steps[0] if d.req == r]
            if ds:
                oracle.splice_request(caches[r], [(d.s_start, d.s_end, d.n_repl) for d in ds],
                                      [reps[d.key] for d in ds], w.latent_dim, w.theta)
    for _ in range(args.warmup):
        one_call()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_call()
    dt = time.perf_counter() - t0
    value = st.downstream_slots * args.steps / dt
    return {"metric": METRIC, "value": value, "unit": "slots/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "layers": w.num_layers, "block_size": w.block_size, "storage": "bf16"},
            "cpu_baseline": {"value": value, "unit": "slots/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} timed whole call(s) of {w.name} through the fp64 C oracle, "
                                       "single thread"},
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
            cb, _ = cpu_oracle_sample(w, args.cpu_seconds)
            line["cpu_baseline"] = cb
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
