"""The five synthetic splice workloads: context lengths and directive spans.

Shapes follow the workloads the splice is specified on: a 1-layer contiguous
cache, a DeepSeek-V2-Lite-shaped 27-layer paged cache, a batch of 8 requests, a
61-layer 64-splice chain, and a concurrency sweep over a shared pool.  Only
integers are produced here (lengths, spans, replacement counts, seeds); the rows
themselves come from ``synth.cache_rows`` / ``synth.repl_rows``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

from . import Draw


@dataclass(frozen=True)
class Dir:
    """One AMORTIZE directive: replace tokens [s_start, s_end) of request ``req`` by ``n_repl`` rows.

    ``key`` selects the replacement rows in ``synth.repl_rows`` (unique per directive).
    """
    req: int
    s_start: int
    s_end: int
    n_repl: int
    key: int
    mode: int = 0  # 0 AMORTIZE (re-encode survivors), 2 EVICT (keep their positions)


@dataclass
class Workload:
    name: str
    num_layers: int
    block_size: int
    lengths: list[int]
    steps: list[list[Dir]]  # one list of directives per splice call, applied in order
    seed: int = 0
    identity_table: bool = False
    latent_dim: int = 512
    rope_dim: int = 64
    theta: float = 10000.0
    rope_heads: int = 1  # RoPE bands per row (GQA/MHA keys); 1 for MLA
    notes: dict = field(default_factory=dict)

    @property
    def num_reqs(self) -> int:
        return len(self.lengths)

    @property
    def row_elems(self) -> int:
        return self.latent_dim + self.rope_heads * self.rope_dim


def contiguous_4k(seed: int = 0) -> Workload:
    """1 request, 1 layer, 4096 tokens, block size 1, identity table; s=1024, e=2048, |R|=16."""
    return Workload("contiguous-1L-4k-B1", 1, 1, [4096], [[Dir(0, 1024, 2048, 16, 0)]],
                    seed=seed, identity_table=True)


def dsv2_lite_32k(seed: int = 0) -> Workload:
    """DeepSeek-V2-Lite shape: 27 layers, 32768 tokens, block 16; drop [20000, 26000), |R|=12."""
    return Workload("dsv2lite-27L-32k-B16", 27, 16, [32768], [[Dir(0, 20000, 26000, 12, 0)]], seed=seed)


def batched_c8(seed: int = 0) -> Workload:
    """8 requests, 27 layers, block 16, L~U[16384,65536]; one directive each, request 7 has Delta=+48."""
    d = Draw(seed, 3)
    lengths, dirs = [], []
    for r in range(8):
        L = d.integer(16384, 65536)
        s = d.integer(0, L // 2 - 1)
        span = d.integer(256, 8192)
        n_repl = d.integer(4, 64)
        if r == 7:
            span, n_repl = 16, 64
        lengths.append(L)
        dirs.append(Dir(r, s, s + span, n_repl, r))
    return Workload("batched-C8-27L-B16", 27, 16, lengths, [dirs], seed=seed)


def chain_64(seed: int = 0, num_layers: int = 61, length: int = 131072, n_steps: int = 64) -> Workload:
    """1 request, 61 layers, 131072 tokens, block 1; 64 successive splices, span~U[512,2048], |R|=12."""
    d = Draw(seed, 4)
    L = length
    steps = []
    for k in range(n_steps):
        span = d.integer(512, 2048)
        s = d.integer(0, L - span)
        steps.append([Dir(0, s, s + span, 12, k)])
        L = L - span + 12
    return Workload("chain64-61L-128k-B1", num_layers, 1, [length], steps, seed=seed)


def sweep(C: int, block_size: int, seed: int = 0, num_layers: int = 61) -> Workload:
    """C requests sharing one pool; L ~ lognormal(ln 24000, 0.75) clipped to [2048, 131072];
    1-3 non-overlapping directives per request, span~U[128,16384] (clipped to fit), |R|~U[4,64].

    Non-overlap is drawn by splitting [0, L) into k equal zones and placing one span in each.
    """
    d = Draw(seed, 500 + C)
    lengths, dirs = [], []
    for r in range(C):
        L = int(round(math.exp(math.log(24000.0) + 0.75 * d.normal())))
        L = max(2048, min(131072, L))
        k = d.integer(1, 3)
        zone = L // k
        for z in range(k):
            span = min(d.integer(128, 16384), zone)
            s = z * zone + d.integer(0, zone - span)
            dirs.append(Dir(r, s, s + span, d.integer(4, 64), r * 8 + z))
        lengths.append(L)
    return Workload(f"sweep-C{C}-61L-B{block_size}", num_layers, block_size, lengths, [dirs], seed=seed)


def sweep_aligned(C: int, block_size: int, seed: int = 0, num_layers: int = 61) -> Workload:
    """The sweep with every directive moved onto the block grid: s_start and s_end rounded
    down to multiples of the block size, |R| rounded up to one (page-granular compaction)."""
    w = sweep(C, block_size, seed, num_layers)
    B = block_size
    dirs = []
    for d in w.steps[0]:
        s, e = (d.s_start // B) * B, (d.s_end // B) * B
        dirs.append(Dir(d.req, s, max(s, e), -(-d.n_repl // B) * B, d.key))
    return Workload(f"sweep-aligned-C{C}-61L-B{B}", num_layers, B, w.lengths, [dirs], seed=seed)


def sweep_shift_aligned(C: int, block_size: int, seed: int = 0, num_layers: int = 61) -> Workload:
    """The sweep with spans as drawn and |R| raised to the next value that makes Delta a
    multiple of the block size: survivors shift by whole blocks, boundary blocks do not."""
    w = sweep(C, block_size, seed, num_layers)
    B = block_size
    dirs = []
    for d in w.steps[0]:
        span = d.s_end - d.s_start
        n = d.n_repl + (span - d.n_repl) % B  # n - span is a multiple of B
        dirs.append(Dir(d.req, d.s_start, d.s_end, n, d.key))
    return Workload(f"sweep-shift-aligned-C{C}-61L-B{B}", num_layers, B, w.lengths, [dirs], seed=seed)


def by_name(name: str, seed: int = 0) -> Workload:
    table = {
        "cfg1": contiguous_4k,
        "cfg2": dsv2_lite_32k,
        "cfg3": batched_c8,
        "cfg4": chain_64,
    }
    if name in table:
        return table[name](seed)
    if name.startswith("cfg5-"):  # cfg5-C16-B16
        _, c, b = name.split("-")
        return sweep(int(c[1:]), int(b[1:]), seed)
    if name.startswith("cfg5a-"):  # cfg5a-C16-B16: the same sweep on the block grid
        _, c, b = name.split("-")
        return sweep_aligned(int(c[1:]), int(b[1:]), seed)
    if name.startswith("cfg5s-"):  # cfg5s-C16-B16: the same sweep with Delta a multiple of B
        _, c, b = name.split("-")
        return sweep_shift_aligned(int(c[1:]), int(b[1:]), seed)
    raise KeyError(name)
