"""Test harness: run splices on the GPU through the C ABI and compare with the oracle.

Tolerance for the rope band of moved rows ("Leyline: KV Cache Directives for
Agentic Inference", section 2.2: R(Delta) applied to R(i) equals R(i + Delta);
section 4.3: fp32 rotation, bf16 storage):
  an element passes if |gpu - oracle| <= 1 bf16 step at the oracle's value, or
  |gpu - oracle| <= 2^-16 * |pair|  (|pair| = norm of the element's RoPE pair).
The second clause covers cancellations: an output much smaller than its pair
norm carries an fp32 error of order 2^-23 |pair|, which can exceed one bf16 step
of the small output.  Per splice, the relative L2 error of the moved rope bands
must also stay <= 1e-3.  Latents, prefix rows, rows of R, lengths and block-table
structure must be bit-exact.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth
from synth import fill as sfill
from synth.configs import Dir, Workload

FLOOR = 2.0 ** -16
REL_L2_MAX = 1e-3


def bf16_step(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def pair_norms(vals: np.ndarray, layout: int) -> np.ndarray:
    """Norm of each element's RoPE pair, same shape as vals [..., d]."""
    d = vals.shape[-1]
    out = np.empty_like(vals)
    if layout == 0:
        n = np.hypot(vals[..., : d // 2], vals[..., d // 2:])
        out[..., : d // 2] = n
        out[..., d // 2:] = n
    else:
        n = np.hypot(vals[..., 0::2], vals[..., 1::2])
        out[..., 0::2] = n
        out[..., 1::2] = n
    return out


def compare_kpe(got_bits: np.ndarray, want_bits: np.ndarray, layout: int, exact: bool = False) -> dict:
    """Check moved rope bands [n][d]; returns counters.  exact=True demands equal bits."""
    if got_bits.size == 0:
        return {"n": 0, "floor_used": 0, "max_steps": 0.0, "rel_l2": 0.0}
    g = oracle.bf16_value(got_bits)
    w = oracle.bf16_value(want_bits)
    diff = np.abs(g - w)
    step = bf16_step(w)
    pn = pair_norms(w, layout)
    ok_step = diff <= step
    ok_floor = diff <= FLOOR * pn
    bad = ~(ok_step | ok_floor)
    if exact:
        bad = got_bits != want_bits
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(f"rope band mismatch at {tuple(i)}: gpu {g[tuple(i)]!r} oracle {w[tuple(i)]!r} "
                             f"({int(bad.sum())} bad of {bad.size})")
    rel = float(np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-300))
    assert rel <= REL_L2_MAX, f"relative L2 {rel} > {REL_L2_MAX}"
    return {"n": int(diff.size), "floor_used": int((~ok_step & ok_floor).sum()),
            "max_steps": float(np.max(diff / step)), "rel_l2": rel}


def pages_for(w: Workload, slack_pages: int = 0) -> int:
    """Pool size: at every step, the live pages before it plus a full rewrite after it."""
    B = w.block_size
    lens = list(w.lengths)
    need = 0
    for step in w.steps or [[]]:
        before = sum(-(-L // B) for L in lens)
        for r in range(w.num_reqs):
            lens[r] += sum(d.n_repl - (d.s_end - d.s_start) for d in step if d.req == r)
        need = max(need, before + sum(-(-L // B) + 1 for L in lens))
    return need + slack_pages


def make_cache(w: Workload, pair_layout: int = 0, precision: int = 0, slack_pages: int = 0,
               max_blocks: int | None = None):
    from rope_rotation_gb300.runtime import PagedCache
    B = w.block_size
    lens = list(w.lengths)
    mx = max(lens)
    for step in w.steps:
        for r in range(w.num_reqs):
            lens[r] += sum(d.n_repl - (d.s_end - d.s_start) for d in step if d.req == r)
            mx = max(mx, lens[r])
    if max_blocks is None:
        max_blocks = -(-mx // B) + 1
    cache = PagedCache(w.num_layers, B, pages_for(w, slack_pages), w.num_reqs, max_blocks, w.latent_dim,
                       w.rope_dim, w.theta, pair_layout, precision)
    for r, L in enumerate(w.lengths):
        cache.add_request(r, L)
        sfill.fill_request(cache, w.seed, r, L)
    return cache


def repl_for(w: Workload, d: Dir, device="cuda"):
    if d.n_repl == 0:
        return None
    return sfill.repl_tensor(w.seed, d.req, d.key, w.num_layers, d.n_repl, w.row_elems, device)


def gpu_directives(w: Workload, step: list[Dir]):
    from rope_rotation_gb300 import leyline
    repl = [repl_for(w, d) for d in step]
    dirs = [leyline.directive(d.req, d.s_start, d.s_end, r, n_repl=d.n_repl) for d, r in zip(step, repl)]
    return dirs, repl


def logical_rows(cache, req: int, length: int) -> np.ndarray:
    """All layers of one request gathered through the C ABI, as uint16 [layers][L][row]."""
    import torch
    out = np.empty((cache.num_layers, length, cache.row), dtype=np.uint16)
    buf = torch.empty((max(length, 1), cache.row), dtype=torch.bfloat16, device=cache.device)
    for layer in range(cache.num_layers):
        cache.gather(req, layer, 0, length, buf[:length])
        out[layer] = buf[:length].view(torch.int16).cpu().numpy().view(np.uint16)
    return out


def check_tables(cache, before_table: np.ndarray, after_table: np.ndarray, before_lens, after_lens,
                 touched: dict) -> None:
    """Block-table structure after a splice.  touched[r] = b0 (first rewritten block)."""
    B = cache.block_size
    live = set()
    for r in range(after_table.shape[0]):
        nb = -(-int(after_lens[r]) // B)
        row = after_table[r]
        assert np.all(row[nb:] == -1), f"request {r}: entries past the length are not -1"
        ids = row[:nb]
        assert np.all((ids >= 0) & (ids < cache.num_pages)), f"request {r}: page id out of range"
        assert len(set(ids.tolist())) == nb, f"request {r}: repeated page id"
        assert not (live & set(ids.tolist())), f"request {r}: page shared with another request"
        live |= set(ids.tolist())
        if r in touched:
            b0 = touched[r]
            assert np.array_equal(row[:b0], before_table[r][:b0]), f"request {r}: prefix entries changed"
            old_live = set(before_table[r][: -(-int(before_lens[r]) // B)].tolist())
            assert not (set(row[b0:nb].tolist()) & old_live), f"request {r}: rewritten block reuses a source page"
        else:
            assert np.array_equal(row, before_table[r]), f"request {r}: untouched request changed"


def splice_step_and_check(w: Workload, cache, state: list[np.ndarray], step: list[Dir], layout: int = 0,
                          precision: int = 0, guard: bool = True) -> dict:
    """Run one splice step on the GPU and check it against the oracle applied to `state`
    (the oracle's own logical caches, uint16 [layers][L][row] per request; updated in place)."""
    import torch
    B = w.block_size
    before_table = cache.table.cpu().numpy().copy()
    before_lens = cache.seq_lens_host.copy()
    snap = cache.kv.clone() if guard else None
    free_before = cache.free_pages()
    dirs, repl_t = gpu_directives(w, step)
    cache.splice(dirs)
    torch.cuda.synchronize()
    cache.check_status()
    stats = cache.last_stats()
    after_table = cache.table.cpu().numpy()
    after_lens_dev = cache.seq_lens_dev.cpu().numpy()
    touched = {}
    counters = {"moved": 0, "floor_used": 0, "rel_l2_max": 0.0}
    for r in range(w.num_reqs):
        ds = [d for d in step if d.req == r]
        eff = [d for d in ds if not (d.s_start == d.s_end and d.n_repl == 0)]
        if not eff:
            assert after_lens_dev[r] == before_lens[r]
            continue
        touched[r] = min(d.s_start for d in eff) // B
        tup = [(d.s_start, d.s_end, d.n_repl) for d in ds]
        newlen, kind, idx, which = oracle.splice_map(int(before_lens[r]), tup)
        reps = [synth.repl_rows(w.seed, r, d.key, w.num_layers, d.n_repl, w.row_elems) for d in ds]
        assert int(cache.seq_lens_host[r]) == newlen and int(after_lens_dev[r]) == newlen
        got = logical_rows(cache, r, newlen)
        lat = w.latent_dim
        if precision == 0:
            want = oracle.splice_request(state[r], tup, reps, lat, w.theta, layout)
        else:
            want = np.empty_like(got)
            for p in range(newlen):
                if kind[p] == 1:
                    want[:, p] = reps[which[p]][:, idx[p]]
                else:
                    t = int(idx[p])
                    want[:, p, :lat] = state[r][:, t, :lat]
                    want[:, p, lat:] = oracle.rotate_bf16only(state[r][:, t, lat:], p - t, w.theta, layout)
        assert np.array_equal(got[:, :, :lat], want[:, :, :lat]), f"request {r}: latent bits differ"
        moved = (kind == 0) & (idx != np.arange(newlen))
        assert np.array_equal(got[:, ~moved], want[:, ~moved]), f"request {r}: prefix / R rows differ"
        c = compare_kpe(got[:, moved, lat:].reshape(-1, w.rope_dim), want[:, moved, lat:].reshape(-1, w.rope_dim),
                        layout, exact=(precision != 0))
        counters["moved"] += c["n"]
        counters["floor_used"] += c["floor_used"]
        counters["rel_l2_max"] = max(counters["rel_l2_max"], c["rel_l2"])
        state[r] = want
    check_tables(cache, before_table, after_table, before_lens, cache.seq_lens_host, touched)
    assert cache.free_pages() == free_before - stats["pages_popped"] + stats["pages_pushed"]
    if guard:
        new_pages = set()
        for r in touched:
            nb = -(-int(cache.seq_lens_host[r]) // B)
            new_pages |= set(after_table[r][touched[r]:nb].tolist())
        keep = np.ones(cache.num_pages, dtype=bool)
        keep[list(new_pages)] = False
        kv_b = snap.view(cache.num_layers, cache.num_pages, -1)
        kv_a = cache.kv.view(cache.num_layers, cache.num_pages, -1)
        keep_t = torch.from_numpy(keep).to(cache.device)
        assert torch.equal(kv_a[:, keep_t].view(torch.int16), kv_b[:, keep_t].view(torch.int16)), \
            "a page outside the rewritten blocks changed"
    del repl_t
    counters["stats"] = stats
    return counters


def oracle_state(w: Workload) -> list[np.ndarray]:
    return [synth.cache_request(w.seed, r, w.num_layers, L, w.row_elems) for r, L in enumerate(w.lengths)]
