"""Lazy pools (LEYLINE_POOL_LAZY): a splice moves stored bits and counts pending turns.

The page's AMORTIZE definition ("Leyline: KV Cache Directives for Agentic
Inference", section 2.1) re-encodes a survivor at its new position; section 2.2
gives R(a) R(b) = R(a + b), so the turns of successive splices may be summed and
applied once when the row is read.  A lazy pool does exactly that, which makes
every read of a row a single rounding of R(pending) x (section 4.3's drift,
one bf16 rounding per splice, no longer accumulates).

Checks, per splice, against state tracked here from ``oracle.splice_map``:
* the stored bits of every row are the written bits, moved exactly (latent and band);
* each slot's pending count is the sum of the AMORTIZE deltas it went through
  (0 for rows of R), and every page outside a block table has count 0;
* a gather equals ``oracle.rerotate(stored band, 0, pending)`` within one rounding;
* for AMORTIZE-only chains, pending = final position - original position.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from synth.configs import Dir, Workload
import splice_harness as H

pytestmark = pytest.mark.gpu

LAZY = 2
REINDEX = 1


def _raw_rows(cache, req: int, length: int) -> np.ndarray:
    """Stored bits of a request's rows, uint16 [layers][L][row], read through the table (no gather)."""
    import torch
    B = cache.block_size
    nb = -(-length // B)
    pages = cache.table[req, :nb].long()
    rows = torch.cat((cache.latent_view()[:, pages], cache.rope_view()[:, pages]), -1)
    rows = rows.reshape(cache.num_layers, nb * B, cache.row)[:, :length]
    return rows.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _pending_of(cache, req: int, length: int) -> np.ndarray:
    """Counts of a request's slots [0, length); the unused slots of its last page must be 0
    (a row appended there later is written at its own position)."""
    B = cache.block_size
    nb = -(-length // B)
    pages = cache.table[req, :nb].long()
    every = cache.pending()[pages].reshape(-1).cpu().numpy().astype(np.int64)
    assert not every[length:].any(), f"request {req}: an unused slot of its last page has a pending turn"
    return every[:length]


def _check_free_pages_clear(cache) -> None:
    table = cache.table.cpu().numpy()
    live = set()
    for r in range(table.shape[0]):
        nb = -(-int(cache.seq_lens_host[r]) // cache.block_size)
        live |= set(table[r, :nb].tolist())
    pend = cache.pending().cpu().numpy()
    free = np.ones(cache.num_pages, dtype=bool)
    free[list(live)] = False
    assert not pend[free].any(), "a page outside every block table carries a pending turn"


class LazyState:
    """Per request: the bits that should be stored (uint16 [layers][L][row]), the pending
    count of each row, and the original position of each row (-1 - p for a row of R written
    at position p)."""

    def __init__(self, w: Workload):
        self.base = [synth.cache_request(w.seed, r, w.num_layers, L, w.row_elems) for r, L in enumerate(w.lengths)]
        self.pend = [np.zeros(L, dtype=np.int64) for L in w.lengths]
        self.origin = [np.arange(L, dtype=np.int64) for L in w.lengths]

    def apply(self, w: Workload, step: list[Dir], before_lens) -> dict:
        touched = {}
        for r in range(w.num_reqs):
            ds = [d for d in step if d.req == r]
            if not [d for d in ds if not (d.s_start == d.s_end and d.n_repl == 0)]:
                continue
            tup = [(d.s_start, d.s_end, d.n_repl) for d in ds]
            dm = [(d.s_start, d.s_end, d.n_repl, d.mode) for d in ds]
            newlen, kind, idx, which = oracle.splice_map(int(before_lens[r]), tup)
            reps = [synth.repl_rows(w.seed, r, d.key, w.num_layers, d.n_repl, w.row_elems) for d in ds]
            base = np.empty((w.num_layers, newlen, w.row_elems), dtype=np.uint16)
            pend = np.zeros(newlen, dtype=np.int64)
            origin = np.full(newlen, -1, dtype=np.int64)
            for p in range(newlen):
                if kind[p] == 1:
                    base[:, p] = reps[which[p]][:, idx[p]]
                    origin[p] = -1 - p  # written at p
                else:
                    t = int(idx[p])
                    base[:, p] = self.base[r][:, t]
                    pend[p] = self.pend[r][t] + H.turn_of(t, dm)
                    origin[p] = self.origin[r][t]
            self.base[r], self.pend[r], self.origin[r] = base, pend, origin
            touched[r] = min(d.s_start for d in ds if not (d.s_start == d.s_end and d.n_repl == 0)) // w.block_size
        return touched

    def rebase(self, r: int, stored: np.ndarray) -> None:
        """After a materialize checked against the oracle: the stored bits are the GPU's, with
        nothing pending, and later reads are checked against one rounding of those bits."""
        self.base[r] = stored.copy()
        self.pend[r][:] = 0


def _want_read(w: Workload, st: LazyState, r: int, precision: int, layout: int) -> np.ndarray:
    lat = w.latent_dim
    base = st.base[r]
    want = base.copy()
    moved = st.pend[r] != 0
    if moved.any():
        bands = base[:, moved, lat:].reshape(w.num_layers, -1, w.rope_heads, w.rope_dim)
        pend = np.broadcast_to(st.pend[r][moved][None, :, None], bands.shape[:3]).reshape(-1)
        if precision == 0:
            turned = oracle.rerotate(bands, 0, pend, w.theta, layout)
        else:
            turned = oracle.rotate_bf16only(bands, pend, w.theta, layout)
        want[:, moved, lat:] = turned.reshape(w.num_layers, -1, w.rope_heads * w.rope_dim)
    return want


def _check_read(w: Workload, cache, st: LazyState, r: int, precision: int, layout: int) -> dict:
    lat = w.latent_dim
    L = int(cache.seq_lens_host[r])
    got = H.logical_rows(cache, r, L)
    want = _want_read(w, st, r, precision, layout)
    assert np.array_equal(got[:, :, :lat], want[:, :, :lat]), f"request {r}: latent bits differ"
    moved = st.pend[r] != 0
    assert np.array_equal(got[:, ~moved], want[:, ~moved]), f"request {r}: rows with nothing pending differ"
    # one rounding per read, of the stored bits
    return H.compare_kpe(got[:, moved, lat:].reshape(-1, w.rope_dim), want[:, moved, lat:].reshape(-1, w.rope_dim),
                         layout, exact=(precision != 0))


def _step(w: Workload, cache, st: LazyState, step: list[Dir], precision: int = 0, layout: int = 0) -> dict:
    import torch
    before_table = cache.table.cpu().numpy().copy()
    before_lens = cache.seq_lens_host.copy()
    free_before = cache.free_pages()
    dirs, repl_t = H.gpu_directives(w, step)
    cache.splice(dirs)
    torch.cuda.synchronize()
    cache.check_status()
    stats = cache.last_stats()
    touched = st.apply(w, step, before_lens)
    out = {"rel_l2_max": 0.0, "moved": 0}
    for r in touched:
        L = int(cache.seq_lens_host[r])
        assert L == st.base[r].shape[1]
        assert np.array_equal(_raw_rows(cache, r, L), st.base[r]), f"request {r}: stored bits differ"
        assert np.array_equal(_pending_of(cache, r, L), st.pend[r]), f"request {r}: pending counts differ"
        c = _check_read(w, cache, st, r, precision, layout)
        out["rel_l2_max"] = max(out["rel_l2_max"], c["rel_l2"])
        out["moved"] += c["n"]
    H.check_tables(cache, before_table, cache.table.cpu().numpy(), before_lens, cache.seq_lens_host, touched,
                   reindex=stats["reindexed"] == 1)
    assert cache.free_pages() == free_before - stats["pages_popped"] + stats["pages_pushed"]
    _check_free_pages_clear(cache)
    del repl_t
    out["stats"] = stats
    return out


def _chain(seed: int, n_steps: int, L0: int, n_reqs: int = 1, evict_every: int = 0) -> list[list[Dir]]:
    rng = np.random.default_rng(seed)
    lens = [L0] * n_reqs
    steps = []
    for k in range(n_steps):
        step = []
        for r in range(n_reqs):
            L = lens[r]
            span = int(rng.integers(0, max(L // 6, 2)))
            s = int(rng.integers(0, L - span + 1))
            n = int(rng.integers(0, 40))
            mode = 2 if (evict_every and k % evict_every == evict_every - 1) else 0
            step.append(Dir(r, s, s + span, n, 100 * k + r, mode))
            lens[r] = L - span + n
        steps.append(step)
    return steps


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("B", [16, 1])
def test_lazy_single_splice(layout, B):
    w = Workload(f"lazy-B{B}", 3, B, [3001, 1777], [[Dir(0, 500, 1800, 12, 0), Dir(0, 2000, 2100, 0, 1),
                                                     Dir(1, 64, 65, 40, 2)]], seed=11)
    cache = H.make_cache(w, pair_layout=layout, flags=LAZY)
    st = LazyState(w)
    st.layout = layout
    c = _step(w, cache, st, w.steps[0], layout=layout)
    assert c["moved"] > 0
    cache.close()


@pytest.mark.parametrize("flags,B", [(LAZY, 16), (LAZY, 1), (LAZY | REINDEX, 1)])
def test_lazy_chain_pending_is_position_shift(flags, B):
    """AMORTIZE only: a surviving row's pending count is its final position minus its original one."""
    steps = _chain(5, 10, 4000, n_reqs=2)
    w = Workload("lazy-chain", 2, B, [4000, 4000], steps, seed=21)
    cache = H.make_cache(w, flags=flags, slack_pages=64)
    st = LazyState(w)
    for step in steps:
        _step(w, cache, st, step)
    for r in range(w.num_reqs):
        L = int(cache.seq_lens_host[r])
        orig = st.origin[r]
        pos = np.arange(L)
        old = orig >= 0
        assert np.array_equal(st.pend[r][old], pos[old] - orig[old])
        wr = ~old  # rows of R: pending = final position - position written
        assert np.array_equal(st.pend[r][wr], pos[wr] - (-1 - orig[wr]))
        assert np.array_equal(_pending_of(cache, r, L), st.pend[r])
    cache.close()


@pytest.mark.parametrize("flags,B", [(LAZY, 16), (LAZY | REINDEX, 1)])
def test_lazy_modes_and_heads(flags, B):
    """EVICT directives shift without adding to the count; GQA rows (4 bands) turn band by band."""
    steps = _chain(9, 6, 2500, n_reqs=1, evict_every=2)
    w = Workload("lazy-modes-gqa", 2, B, [2500], steps, seed=31, latent_dim=128, rope_dim=64, rope_heads=4)
    cache = H.make_cache(w, flags=flags, slack_pages=64)
    st = LazyState(w)
    for step in steps:
        _step(w, cache, st, step)
    cache.close()


def test_lazy_block_reindex():
    """Pages of 16 slots on a lazy re-index pool: calls on block boundaries move whole
    pages and only their counts change."""
    lengths = [16 * 40 + 9, 16 * 12]
    steps = H.aligned_steps(91, 16, lengths, 8, evict_every=3)
    w = Workload("lazy-block-reindex", 2, 16, lengths, steps, seed=91)
    cache = H.make_cache(w, flags=LAZY | REINDEX, slack_pages=64)
    st = LazyState(w)
    for step in steps:
        c = _step(w, cache, st, step)
        if any(not (d.s_start == d.s_end and d.n_repl == 0) for d in step):
            assert c["stats"]["reindexed"] == 1
    cache.close()


def test_lazy_bf16_arm_exact():
    """The naive bf16 arm rounds every product; applied once it must equal the oracle's bits."""
    steps = _chain(13, 4, 3000)
    w = Workload("lazy-bf16", 2, 16, [3000], steps, seed=41)
    cache = H.make_cache(w, precision=1, flags=LAZY)
    st = LazyState(w)
    for step in steps:
        _step(w, cache, st, step, precision=1)
    cache.close()


@pytest.mark.parametrize("flags,B", [(LAZY, 16), (LAZY | REINDEX, 1)])
def test_materialize(flags, B):
    """materialize stores what a gather returned, clears the counts, and later splices build on it."""
    import torch
    steps = _chain(17, 6, 3000)
    w = Workload("lazy-mat", 3, B, [3000], steps, seed=51)
    cache = H.make_cache(w, flags=flags, slack_pages=64)
    st = LazyState(w)
    for step in steps[:3]:
        _step(w, cache, st, step)
    L = int(cache.seq_lens_host[0])
    before = H.logical_rows(cache, 0, L)
    cache.materialize(0)
    torch.cuda.synchronize()
    cache.check_status()
    assert not _pending_of(cache, 0, L).any()
    after = H.logical_rows(cache, 0, L)
    assert np.array_equal(before, after), "a gather after materialize differs from the one before"
    stored = _raw_rows(cache, 0, L)
    assert np.array_equal(stored, after)
    # the materialized bits are one rounding of the oracle's re-encoding of what was stored
    want = _want_read(w, st, 0, 0, 0)
    moved = st.pend[0] != 0
    assert np.array_equal(stored[:, ~moved], want[:, ~moved])
    H.compare_kpe(stored[:, moved, w.latent_dim:].reshape(-1, w.rope_dim),
                  want[:, moved, w.latent_dim:].reshape(-1, w.rope_dim), 0)
    st.rebase(0, stored)
    _check_read(w, cache, st, 0, 0, 0)
    for step in steps[3:]:
        _step(w, cache, st, step)
    cache.close()


@pytest.mark.parametrize("rope_dim,heads,layout,B", [(32, 2, 0, 16), (16, 4, 1, 16), (64, 1, 1, 1), (32, 2, 1, 1)])
def test_materialize_band_shapes(rope_dim, heads, layout, B):
    """Rows whose rope bands fill 128 bytes in other ways than one 64-wide band (GQA keys of
    2 x 32 or 4 x 16), both layouts: materialize stores what the gather returned (which is
    checked against the oracle), and clears every count."""
    import torch
    steps = _chain(29, 3, 1500)
    w = Workload(f"lazy-mat-{rope_dim}x{heads}", 3, B, [1500], steps, seed=81, latent_dim=128, rope_dim=rope_dim,
                 rope_heads=heads)
    cache = H.make_cache(w, pair_layout=layout, flags=LAZY, slack_pages=64)
    st = LazyState(w)
    for step in steps:
        _step(w, cache, st, step, layout=layout)
    L = int(cache.seq_lens_host[0])
    assert _pending_of(cache, 0, L).any()
    before = H.logical_rows(cache, 0, L)
    cache.materialize(0)
    torch.cuda.synchronize()
    cache.check_status()
    assert not _pending_of(cache, 0, L).any()
    assert np.array_equal(_raw_rows(cache, 0, L), before), "materialize stored other bits than the gather returned"
    cache.close()


@pytest.mark.parametrize("B", [1, 16])
def test_lazy_reindex_calls_in_flight_equal_calls_one_at_a_time(B):
    """Lazy re-index calls enqueued back to back with no synchronisation (each call's commit
    follows its prep directly: no band is turned, and at block size 1 no other fresh rows are
    written) leave exactly the stored bits, counts and tables of the same calls made one at a
    time with a synchronisation after each; those are checked against the oracle elsewhere."""
    import torch
    steps = _chain(97, 24, 1200, n_reqs=3)
    w = Workload(f"lazy-inflight-B{B}", 2, B, [1200] * 3, steps, seed=98)
    a = H.make_cache(w, flags=LAZY | REINDEX, slack_pages=64)
    b = H.make_cache(w, flags=LAZY | REINDEX, slack_pages=64)
    keep = []
    for step in steps:
        dirs, k = H.gpu_directives(w, step)
        keep.append(k)
        a.splice(dirs)  # no synchronisation
    for step in steps:
        dirs, k = H.gpu_directives(w, step)
        keep.append(k)
        b.splice(dirs)
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    a.check_status()
    b.check_status()
    for r in range(w.num_reqs):
        n = int(a.seq_lens_host[r])
        assert n == int(b.seq_lens_host[r])
        assert np.array_equal(_raw_rows(a, r, n), _raw_rows(b, r, n)), f"request {r}: stored bits differ"
        assert np.array_equal(_pending_of(a, r, n), _pending_of(b, r, n)), f"request {r}: counts differ"
    assert np.array_equal(a.table.cpu().numpy(), b.table.cpu().numpy())
    _check_free_pages_clear(a)
    del keep
    a.close()
    b.close()


def test_free_pages_clears_pending():
    import torch
    from rope_rotation_gb300 import leyline
    w = Workload("lazy-free", 1, 16, [2000, 2000], [[Dir(0, 10, 400, 3, 0), Dir(1, 5, 9, 0, 1)]], seed=61)
    cache = H.make_cache(w, flags=LAZY)
    st = LazyState(w)
    _step(w, cache, st, w.steps[0])
    L = int(cache.seq_lens_host[0])
    assert _pending_of(cache, 0, L).any()
    nb = -(-L // 16)
    pages = cache.table[0, :nb].cpu().numpy().astype(np.int32)
    leyline.leyline_free_pages(cache.pool, pages)
    torch.cuda.synchronize()
    assert not cache.pending()[torch.from_numpy(pages.astype(np.int64)).cuda()].any()
    cache.close()


def test_materialize_and_pending_refused_on_eager_pool():
    from rope_rotation_gb300 import leyline
    w = Workload("eager", 1, 16, [100], [[]], seed=1)
    cache = H.make_cache(w)
    assert leyline.leyline_pending_ptr(cache.pool) == 0
    assert cache.pending() is None
    with pytest.raises(leyline.LeylineError) as e:
        cache.materialize(0)
    assert e.value.code == leyline.LEYLINE_ERR_INVALID_ARG
    cache.close()


def test_lazy_chain_drift_single_rounding():
    """A long chain on a lazy pool: every read is one rounding of the exact re-encoding of
    the written bits, so the error does not grow with the number of splices."""
    steps = _chain(23, 24, 8192)
    w = Workload("lazy-drift", 1, 1, [8192], steps, seed=71)
    cache = H.make_cache(w, flags=LAZY | REINDEX, slack_pages=64)
    st = LazyState(w)
    rel = []
    for step in steps:
        rel.append(_step(w, cache, st, step)["rel_l2_max"])
    # against the exact re-encoding of the original rows (the definition, not the eager chain)
    L = int(cache.seq_lens_host[0])
    got = H.logical_rows(cache, 0, L)
    orig = st.origin[0]
    keep = orig >= 0
    base = synth.cache_request(w.seed, 0, w.num_layers, w.lengths[0], w.row_elems)
    bands = base[:, orig[keep], w.latent_dim:]
    shape = (w.num_layers, int(keep.sum()))
    exact = oracle.rerotate(bands, np.broadcast_to(orig[keep], shape).reshape(-1),
                            np.broadcast_to(np.arange(L)[keep], shape).reshape(-1), w.theta)
    c = H.compare_kpe(got[:, keep, w.latent_dim:].reshape(-1, w.rope_dim), exact.reshape(-1, w.rope_dim), 0)
    assert c["rel_l2"] < 1e-3 and max(rel) < 1e-3
    cache.close()


@pytest.mark.parametrize("precision,layout", [(0, 0), (0, 1), (1, 0)])
def test_large_counts_across_the_turn_table(precision, layout):
    """Counts written straight into the pending array (the pointer leyline_pending_ptr hands to
    readers), chosen across the readers' turn table: single table steps, the 2048 boundary, the
    table's last count 2048^2 - 1, the sincos path beyond it, and the int32 extremes.  A gather
    equals the oracle's re-encoding by the count within one rounding (the bf16 arm bit-exact),
    and materialize stores exactly what the gather returned."""
    import torch
    S = 2048
    counts = [0, 1, -1, 2047, S, -(S + 1), 2 * S - 1, 123456, -987654, S * S - 1, -(S * S - 1), S * S,
              -(S * S), 10 ** 7, -(10 ** 8), 2 ** 31 - 1, -(2 ** 31 - 1), -(2 ** 31)]
    L = 4 * len(counts)
    w = Workload(f"lazy-large-p{precision}-l{layout}", 2, 1, [L], [], seed=61)
    cache = H.make_cache(w, pair_layout=layout, precision=precision, flags=LAZY)
    pend_of_row = np.array([counts[t % len(counts)] for t in range(L)], dtype=np.int64)
    pages = cache.table[0, :L].long()
    cache.pending()[pages, 0] = torch.tensor(pend_of_row, dtype=torch.int32, device=cache.device)
    torch.cuda.synchronize()
    stored = _raw_rows(cache, 0, L)
    got = H.logical_rows(cache, 0, L)
    lat = w.latent_dim
    assert np.array_equal(got[:, :, :lat], stored[:, :, :lat])
    zero = pend_of_row == 0
    assert np.array_equal(got[:, zero], stored[:, zero])
    bands = stored[:, ~zero, lat:].reshape(w.num_layers, -1, w.rope_heads, w.rope_dim)
    p = np.broadcast_to(pend_of_row[~zero][None, :, None], bands.shape[:3]).reshape(-1)
    if precision == 0:
        want = oracle.rerotate(bands, 0, p, w.theta, layout)
    else:
        want = oracle.rotate_bf16only(bands, p, w.theta, layout)
    H.compare_kpe(got[:, ~zero, lat:].reshape(-1, w.rope_dim), want.reshape(-1, w.rope_dim), layout,
                  exact=precision != 0)
    cache.materialize(0)
    torch.cuda.synchronize()
    cache.check_status()
    assert not _pending_of(cache, 0, L).any()
    assert np.array_equal(_raw_rows(cache, 0, L), got), "materialize stored other bits than the gather returned"
    cache.close()


@pytest.mark.parametrize("B", [16, 1])
def test_materialize_requests_equals_one_at_a_time(B):
    """Many requests in one call turn every row exactly as materializing them one by one does
    (two pools given the same splices); a request listed twice is refused."""
    import torch
    from rope_rotation_gb300 import leyline
    rng = np.random.default_rng(71)
    n_req = 70  # more than one launch's 64 requests
    lengths = [int(rng.integers(40, 160)) for _ in range(n_req)]
    step, key = [], 0
    for r in range(n_req):
        L = lengths[r]
        if r % 9 == 4:
            continue  # a request with nothing pending
        s = int(rng.integers(0, L // 2))
        step.append(Dir(r, s, s + int(rng.integers(1, L // 3)), int(rng.integers(0, 4)), key))
        key += 1
    w = Workload(f"mat-many-B{B}", 2, B, lengths, [step], seed=72)
    one = H.make_cache(w, flags=LAZY)
    many = H.make_cache(w, flags=LAZY)
    for c in (one, many):
        dirs, keep = H.gpu_directives(w, step)
        c.splice(dirs)
        torch.cuda.synchronize()
        del keep
    order = [int(x) for x in rng.permutation(n_req)]
    for r in order:
        one.materialize(r)
    many.materialize_requests(order)
    torch.cuda.synchronize()
    one.check_status()
    many.check_status()
    for r in range(n_req):
        L = int(one.seq_lens_host[r])
        assert np.array_equal(_raw_rows(one, r, L), _raw_rows(many, r, L)), f"request {r} differs"
        assert not _pending_of(many, r, L).any()
    with pytest.raises(leyline.LeylineError):
        many.materialize_requests([3, 5, 3])
    one.close()
    many.close()
