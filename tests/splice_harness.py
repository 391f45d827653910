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
    """Check rope bands [n][d] at the per-splice tolerance; returns counters.  exact=True
    demands equal bits.  want_bits is the oracle applied to the same stored input the GPU
    turned (for chained calls: the GPU's own state before the call)."""
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
               max_blocks: int | None = None, flags: int = 0):
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
                       w.rope_dim, w.theta, pair_layout, precision, flags, w.rope_heads)
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
    dirs = [leyline.directive(d.req, d.s_start, d.s_end, r, n_repl=d.n_repl, mode=d.mode) for d, r in zip(step, repl)]
    return dirs, repl


def work_stats(cache) -> dict:
    """The last call's work accounting, without its host timings (which differ call to call)."""
    return {k: v for k, v in cache.last_stats().items() if not k.endswith("_ns")}


def logical_rows(cache, req: int, length: int) -> np.ndarray:
    """All layers of one request gathered through the C ABI, as uint16 [layers][L][row]."""
    import torch
    out = np.empty((cache.num_layers, length, cache.row), dtype=np.uint16)
    buf = torch.empty((max(length, 1), cache.row), dtype=torch.bfloat16, device=cache.device)
    for layer in range(cache.num_layers):
        cache.gather(req, layer, 0, length, buf[:length])
        out[layer] = buf[:length].view(torch.int16).cpu().numpy().view(np.uint16)
    return out


def turn_of(t: int, dirs) -> int:
    """Rotation of a survivor at old position t: the summed Delta of the AMORTIZE directives
    left of it (EVICT directives shift it without re-encoding)."""
    return sum(n - (e - s) for (s, e, n, m) in dirs if e <= t and m == 0)


def check_tables(cache, before_table: np.ndarray, after_table: np.ndarray, before_lens, after_lens,
                 touched: dict, reindex: bool = False) -> None:
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
            if not reindex:
                old_live = set(before_table[r][: -(-int(before_lens[r]) // B)].tolist())
                assert not (set(row[b0:nb].tolist()) & old_live), f"request {r}: rewritten block reuses a source page"
        else:
            assert np.array_equal(row, before_table[r]), f"request {r}: untouched request changed"


def splice_step_and_check(w: Workload, cache, state: list[np.ndarray], step: list[Dir], layout: int = 0,
                          precision: int = 0, guard: bool = True) -> dict:
    """Run one splice step on the GPU and check it against the oracle applied to `state`, the
    logical caches (uint16 [layers][L][row] per request) the GPU held before the call.  On
    return `state` holds the GPU's caches after the call, checked: the generator's rows
    before the first call, the GPU's own output before every later one."""
    import torch
    B = w.block_size
    before_table = cache.table.cpu().numpy().copy()
    before_lens = cache.seq_lens_host.copy()
    snap = [v.clone() for v in cache.page_views()] if guard else None
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
        modes = [d.mode for d in ds]
        newlen, kind, idx, which = oracle.splice_map(int(before_lens[r]), tup)
        reps = [synth.repl_rows(w.seed, r, d.key, w.num_layers, d.n_repl, w.row_elems) for d in ds]
        assert int(cache.seq_lens_host[r]) == newlen and int(after_lens_dev[r]) == newlen
        got = logical_rows(cache, r, newlen)
        lat = w.latent_dim
        dm = [(d.s_start, d.s_end, d.n_repl, d.mode) for d in ds]
        turn = np.array([turn_of(int(idx[p]), dm) if kind[p] == 0 else 0 for p in range(newlen)], dtype=np.int64)
        H_ = w.rope_heads
        if precision == 0:
            want = oracle.splice_request(state[r], tup, reps, lat, w.theta, layout,
                                         None if (all(m == 0 for m in modes) and H_ == 1) else modes,
                                         rope_heads=H_)
        else:
            want = np.empty_like(got)
            for p in range(newlen):
                if kind[p] == 1:
                    want[:, p] = reps[which[p]][:, idx[p]]
                else:
                    t = int(idx[p])
                    want[:, p, :lat] = state[r][:, t, :lat]
                    bands = state[r][:, t, lat:].reshape(w.num_layers, H_, w.rope_dim)
                    want[:, p, lat:] = oracle.rotate_bf16only(bands, int(turn[p]), w.theta,
                                                              layout).reshape(w.num_layers, -1)
        assert np.array_equal(got[:, :, :lat], want[:, :, :lat]), f"request {r}: latent bits differ"
        moved = turn != 0  # rows this call turned
        assert np.array_equal(got[:, ~moved], want[:, ~moved]), f"request {r}: prefix / R / unturned rows differ"
        c = compare_kpe(got[:, moved, lat:].reshape(-1, w.rope_dim), want[:, moved, lat:].reshape(-1, w.rope_dim),
                        layout, exact=(precision != 0))
        counters["moved"] += c["n"]
        counters["floor_used"] += c["floor_used"]
        counters["rel_l2_max"] = max(counters["rel_l2_max"], c["rel_l2"])
        # the next call is checked against the oracle applied to what the GPU holds now, so
        # every call of a chain meets the per-splice tolerance on its own input
        state[r] = got
    check_tables(cache, before_table, after_table, before_lens, cache.seq_lens_host, touched,
                 reindex=stats["reindexed"] == 1)  # re-indexed calls keep pages
    assert cache.free_pages() == free_before - stats["pages_popped"] + stats["pages_pushed"]
    if guard:
        new_pages = set()
        for r in touched:
            nb = -(-int(cache.seq_lens_host[r]) // B)
            new_pages |= set(after_table[r][touched[r]:nb].tolist())
        keep = np.ones(cache.num_pages, dtype=bool)
        keep[list(new_pages)] = False
        keep_t = torch.from_numpy(keep).to(cache.device)
        for kv_b, kv_a in zip(snap, cache.page_views()):
            assert torch.equal(kv_a[:, keep_t].view(torch.int16), kv_b[:, keep_t].view(torch.int16)), \
                "a page outside the rewritten blocks changed"
    del repl_t
    counters["stats"] = stats
    return counters


def oracle_state(w: Workload) -> list:
    """The logical caches before the first call: the generator's rows, per request."""
    return [synth.cache_request(w.seed, r, w.num_layers, L, w.row_elems) for r, L in enumerate(w.lengths)]


def checked_sequential_run(w: Workload, flags: int = 0, slack_pages: int = 0, layout: int = 0) -> list:
    """Every call of w, one at a time on a pool of its own, each checked at the per-splice
    tolerance against the oracle applied to the GPU's caches before it.  Returns the final
    caches (uint16 [layers][L][row] per request).  Calls that ran without synchronisation
    (in flight, overlapping) run the same kernels on the same inputs, so their final caches
    must equal these bit for bit."""
    cache = make_cache(w, pair_layout=layout, slack_pages=slack_pages, flags=flags)
    state = oracle_state(w)
    for step in w.steps:
        splice_step_and_check(w, cache, state, step, layout=layout, guard=False)
    cache.close()
    return state


def aligned_steps(seed, B, lengths, n_steps, evict_every=0) -> list[list[Dir]]:
    """Chained calls whose directives all lie on block boundaries (s_start a multiple of B;
    s_end and |R| multiples of B unless s_end is the request's end), one per request."""
    rng = np.random.default_rng(seed)
    lens = list(lengths)
    steps, key = [], 0
    for k in range(n_steps):
        step = []
        for r, L in enumerate(lens):
            nb = -(-L // B)
            b0 = int(rng.integers(0, nb + 1))
            if rng.random() < 0.25 and L % B:  # to the end, with a partial last block
                s, e, n = b0 * B if b0 * B <= L else (nb - 1) * B, L, int(rng.integers(0, 2 * B + 3))
            else:
                b1 = int(rng.integers(b0, min(nb, b0 + 6) + 1))
                s, e = b0 * B, min(b1 * B, L)
                if e % B and e != L:
                    e = (e // B) * B
                s = min(s, e)
                n = B * int(rng.integers(0, 3)) if e != L else int(rng.integers(0, 2 * B + 3))
                if s % B:  # past a partial last block: nothing to do here
                    s, e, n = 0, 0, 0
            mode = 2 if (evict_every and k % evict_every == evict_every - 1) else 0
            step.append(Dir(r, s, e, n, key, mode))
            key += 1
            lens[r] = L - (e - s) + n
        steps.append(step)
    return steps


# ------------------------------------------------------------ full-size checks --

def sample_positions(newlen: int, kind: np.ndarray, idx: np.ndarray, n: int, rng) -> np.ndarray:
    """Every segment boundary (and its neighbours), both ends, and n random positions."""
    if newlen == 0:
        return np.zeros(0, dtype=np.int64)
    jump = np.flatnonzero((np.diff(kind) != 0) | (np.diff(idx) != 1)) + 1
    cand = np.concatenate([[0, newlen - 1], jump - 1, jump, jump + 1, rng.integers(0, newlen, size=n)])
    return np.unique(np.clip(cand, 0, newlen - 1))


def fetch_rows(cache, req: int, layers: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """GPU rows (uint16 [n][row]) of (layer, position) pairs, read through the block table."""
    import torch
    B = cache.block_size
    row = cache.table[req].cpu().numpy().astype(np.int64)
    page = torch.from_numpy(row[pos // B]).to(cache.device)
    slot = torch.from_numpy(pos % B).to(cache.device)
    lay = torch.from_numpy(layers.astype(np.int64)).to(cache.device)
    got = cache.read_rows(lay, page, slot)
    return got.view(torch.int16).cpu().numpy().view(np.uint16)


def check_sampled_single_call(w: Workload, cache, step, before_lens, rng, n_samples: int = 1500) -> dict:
    """One call from the generator's initial state: sampled rows against the oracle, element by element."""
    lat = w.latent_dim
    tot = {"rows": 0, "moved": 0, "floor_used": 0, "rel_l2_max": 0.0}
    for r in range(w.num_reqs):
        ds = [d for d in step if d.req == r]
        if not ds:
            continue
        tup = [(d.s_start, d.s_end, d.n_repl) for d in ds]
        newlen, kind, idx, which = oracle.splice_map(int(before_lens[r]), tup)
        assert int(cache.seq_lens_host[r]) == newlen
        pos = sample_positions(newlen, kind, idx, n_samples, rng)
        if pos.size == 0:
            continue
        layers = rng.integers(0, w.num_layers, size=pos.size)
        got = fetch_rows(cache, r, layers, pos)
        want = np.empty_like(got)
        moved = np.zeros(pos.size, dtype=bool)
        reps = {k: synth.repl_rows(w.seed, r, ds[k].key, w.num_layers, ds[k].n_repl, w.row_elems)
                for k in set(which[pos][kind[pos] == 1].tolist())}
        for i, (p, layer) in enumerate(zip(pos, layers)):
            if kind[p] == 1:
                want[i] = reps[which[p]][layer, idx[p]]
            else:
                t = int(idx[p])
                orig = synth.cache_rows(w.seed, r, int(layer), [t], w.row_elems)[0]
                want[i, :lat] = orig[:lat]
                want[i, lat:] = oracle.rerotate(orig[lat:], t, int(p), w.theta) if t != p else orig[lat:]
                moved[i] = t != p
        assert np.array_equal(got[:, :lat], want[:, :lat]), f"request {r}: latent bits differ"
        assert np.array_equal(got[~moved], want[~moved]), f"request {r}: prefix / R rows differ"
        c = compare_kpe(got[moved, lat:], want[moved, lat:], 0)
        tot["rows"] += int(pos.size)
        tot["moved"] += c["n"]
        tot["floor_used"] += c["floor_used"]
        tot["rel_l2_max"] = max(tot["rel_l2_max"], c["rel_l2"])
    return tot


def check_full_layers(w: Workload, cache, step, before_lens, layers) -> dict:
    """Every row of the given layers of every request the call touched, element by element
    against the oracle's splice of the generator's rows: latents, prefix rows and rows of R
    bit-exact, turned rope bands at the per-splice tolerance."""
    import torch
    lat = w.latent_dim
    tot = {"rows": 0, "moved": 0, "floor_used": 0, "rel_l2_max": 0.0, "layers": [int(x) for x in layers]}
    for r in range(w.num_reqs):
        ds = [d for d in step if d.req == r]
        if not ds:
            continue
        L0 = int(before_lens[r])
        tup = [(d.s_start, d.s_end, d.n_repl) for d in ds]
        newlen, kind, idx, _ = oracle.splice_map(L0, tup)
        assert int(cache.seq_lens_host[r]) == newlen
        turned = (kind == 0) & (idx != np.arange(newlen))
        reps_all = [synth.repl_rows(w.seed, r, d.key, w.num_layers, d.n_repl, w.row_elems) for d in ds]
        buf = torch.empty((max(newlen, 1), w.row_elems), dtype=torch.bfloat16, device=cache.device)
        for layer in layers:
            layer = int(layer)
            src = synth.cache_rows(w.seed, r, layer, np.arange(L0), w.row_elems)[None]
            want = oracle.splice_request(src, tup, [x[layer:layer + 1] for x in reps_all], lat, w.theta)[0]
            cache.gather(r, layer, 0, newlen, buf[:newlen])
            got = buf[:newlen].view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got[:, :lat], want[:, :lat]), f"request {r} layer {layer}: latent bits differ"
            assert np.array_equal(got[~turned], want[~turned]), f"request {r} layer {layer}: unturned rows differ"
            c = compare_kpe(got[turned, lat:], want[turned, lat:], 0)
            tot["rows"] += newlen
            tot["moved"] += c["n"]
            tot["floor_used"] += c["floor_used"]
            tot["rel_l2_max"] = max(tot["rel_l2_max"], c["rel_l2"])
    return tot


def check_layers(num_layers: int, rng, n: int = 4) -> list:
    """The first and last layer and n - 2 others drawn from rng."""
    mid = [l for l in range(1, num_layers - 1)]
    pick = rng.choice(mid, size=min(n - 2, len(mid)), replace=False).tolist() if mid else []
    return sorted({0, num_layers - 1, *[int(x) for x in pick]})


def check_properties_all_rows(w: Workload, cache, step, before_lens) -> int:
    """Every row of every touched request and layer, on the device: latents and unmoved rows
    bit-exact against the generator's rows through the oracle's slot map, R rows bit-exact,
    and each moved RoPE pair's norm preserved within bf16 rounding (2^-7 relative)."""
    import torch
    base = sfill._base_on_device(w.seed, w.row_elems, str(cache.device))
    lat = w.latent_dim
    h = w.rope_dim // 2
    checked = 0
    for r in range(w.num_reqs):
        ds = [d for d in step if d.req == r]
        if not ds:
            continue
        tup = [(d.s_start, d.s_end, d.n_repl) for d in ds]
        newlen, kind, idx, which = oracle.splice_map(int(before_lens[r]), tup)
        if newlen == 0:
            continue
        kept = np.flatnonzero(kind == 0)
        moved_np = idx[kept] != kept
        kept_t = torch.from_numpy(kept).to(cache.device)
        moved_t = torch.from_numpy(moved_np).to(cache.device)
        reps = [sfill.repl_tensor(w.seed, r, d.key, w.num_layers, d.n_repl, w.row_elems, str(cache.device))
                if d.n_repl else None for d in ds]
        buf = torch.empty((newlen, w.row_elems), dtype=torch.bfloat16, device=cache.device)
        for layer in range(w.num_layers):
            cache.gather(r, layer, 0, newlen, buf)
            ids = torch.from_numpy(synth.row_ids(w.seed, synth.STREAM_CACHE, r, layer, idx[kept])).to(cache.device)
            src = base.index_select(0, ids)
            got = buf.index_select(0, kept_t)
            gi, si = got.view(torch.int16), src.view(torch.int16)
            assert torch.equal(gi[:, :lat], si[:, :lat]), f"request {r} layer {layer}: latent bits differ"
            assert torch.equal(gi[~moved_t], si[~moved_t]), f"request {r} layer {layer}: unmoved rows differ"
            a = got[moved_t, lat:].float()
            b = src[moved_t, lat:].float()
            na = torch.hypot(a[:, :h], a[:, h:])
            nb = torch.hypot(b[:, :h], b[:, h:])
            assert bool(torch.all((na - nb).abs() <= 2.0 ** -7 * nb + 1e-30)), \
                f"request {r} layer {layer}: a rope pair's norm changed"
            for k, d in enumerate(ds):
                if not d.n_repl:
                    continue
                pk = np.flatnonzero((kind == 1) & (which == k))
                rows = buf.index_select(0, torch.from_numpy(pk).to(cache.device))
                assert torch.equal(rows.view(torch.int16), reps[k][layer].view(torch.int16)), \
                    f"request {r} layer {layer}: replacement rows differ"
            checked += newlen
    return checked
