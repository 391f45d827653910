"""Checkpoint and rollback of a pool's page accounting (needs a GPU).

A rewrite splice reads its source pages and hands them back to the free-page list
("Leyline: KV Cache Directives for Agentic Inference", section 2.3: the rotation
kernel re-indexes every downstream slot; here it writes them to fresh pages).  Until
those pages are taken again, rolling the accounting back and restoring the caller's
table gives the cache before the splice: a repeated splice is then bit-identical to
the first (the benchmark's repeats rest on this), lazy pools get their pending counts
back, and the cases a rollback cannot undo are refused with nothing changed.
"""
import numpy as np
import pytest

import splice_harness as H
from synth.configs import Dir, Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

REINDEX, LAZY = 1, 2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rope_rotation_gb300
    rope_rotation_gb300.build()


def _saved(cache):
    return cache.table.clone(), cache.seq_lens_dev.clone(), cache.seq_lens_host.copy()


def _restore(cache, saved):
    table, lens_dev, lens_host = saved
    cache.table.copy_(table)
    cache.seq_lens_dev.copy_(lens_dev)
    cache.seq_lens_host[:] = lens_host


def _all_rows(cache, w):
    return [H.logical_rows(cache, r, int(cache.seq_lens_host[r])) for r in range(w.num_reqs)]


def _splice(cache, w, step):
    dirs, keep = H.gpu_directives(w, step)
    cache.splice(dirs)
    torch.cuda.synchronize()
    cache.check_status()
    del keep


@pytest.mark.parametrize("flags,B", [(0, 16), (0, 1), (LAZY, 16), (LAZY | REINDEX, 1)])
def test_rollback_then_repeat_is_bit_identical(flags, B):
    from rope_rotation_gb300 import leyline
    step = [Dir(0, 100, 700, 9, 0), Dir(0, 900, 901, 30, 1), Dir(1, 0, 50, 0, 2), Dir(2, 333, 333, 17, 3)]
    w = Workload(f"rollback-f{flags}-B{B}", 2, B, [1500, 800, 1200], [step], seed=5)
    cache = H.make_cache(w, slack_pages=40, flags=flags)
    before = _all_rows(cache, w)
    pend0 = cache.pending().clone() if flags & LAZY else None
    free0 = cache.free_pages()
    saved = _saved(cache)
    leyline.leyline_pool_checkpoint(cache.pool)
    _splice(cache, w, step)
    first = _all_rows(cache, w)
    pend1 = cache.pending().clone() if flags & LAZY else None
    for repeat in range(2):
        leyline.leyline_pool_rollback(cache.pool)
        _restore(cache, saved)
        torch.cuda.synchronize()
        assert cache.free_pages() == free0
        for r, rows in enumerate(_all_rows(cache, w)):
            assert np.array_equal(rows, before[r]), f"request {r}: rollback did not restore the cache"
        if flags & LAZY:
            assert torch.equal(cache.pending(), pend0), "pending counts not restored"
        _splice(cache, w, step)
        for r, rows in enumerate(_all_rows(cache, w)):
            assert np.array_equal(rows, first[r]), f"request {r}: repeat {repeat} differs from the first splice"
        if flags & LAZY:
            assert torch.equal(cache.pending(), pend1), "pending counts of the repeat differ"
    cache.close()


def test_rollback_refusals():
    """No checkpoint, an unknown flag, and splices that took back pages returned since the
    checkpoint (the FIFO free list hands them out only after every page free at the
    checkpoint): each refused with nothing changed."""
    from rope_rotation_gb300 import leyline
    w = Workload("rollback-refuse", 1, 16, [400], [[Dir(0, 10, 300, 2, 0)]], seed=6)
    cache = H.make_cache(w, slack_pages=60 - H.pages_for(w))  # 60 pages: 25 held, 35 free
    assert cache.num_pages == 60 and cache.free_pages() == 35
    with pytest.raises(leyline.LeylineError) as e:
        leyline.leyline_pool_rollback(cache.pool)
    assert e.value.code == leyline.LEYLINE_ERR_INVALID_ARG
    leyline.leyline_pool_checkpoint(cache.pool)
    with pytest.raises(leyline.LeylineError) as e:
        leyline.leyline_pool_rollback(cache.pool, flags=8)
    assert e.value.code == leyline.LEYLINE_ERR_INVALID_ARG

    def rewrite_all(k):  # replaces the first block: all 25 blocks are rewritten
        step = [Dir(0, 0, 16, 16, 10 + k)]
        _splice(cache, Workload("x", 1, 16, [400], [step], seed=6), step)
        assert cache.last_stats()["pages_popped"] == 25

    rewrite_all(0)  # takes 25 of the 35 pages free at the checkpoint
    rewrite_all(1)  # takes the last 10 of them and 15 of those the first call returned
    free = cache.free_pages()
    with pytest.raises(leyline.LeylineError) as e:
        leyline.leyline_pool_rollback(cache.pool)
    assert e.value.code == leyline.LEYLINE_ERR_INVALID_ARG
    assert cache.free_pages() == free

    # one call since a new checkpoint: the rollback is allowed and gives the rows back
    saved = _saved(cache)
    rows = H.logical_rows(cache, 0, 400)
    leyline.leyline_pool_checkpoint(cache.pool)
    rewrite_all(2)
    leyline.leyline_pool_rollback(cache.pool)
    _restore(cache, saved)
    torch.cuda.synchronize()
    assert cache.free_pages() == free
    assert np.array_equal(H.logical_rows(cache, 0, 400), rows)
    cache.close()


def test_rollback_after_turning_in_place_needs_the_flag():
    """An eager re-index splice turns kept bands in place, and materialize turns stored bands:
    a rollback cannot undo either, so it is refused unless the caller accepts it."""
    from rope_rotation_gb300 import leyline
    step = [Dir(0, 100, 400, 5, 0)]
    w = Workload("rollback-turned", 2, 1, [1000], [step], seed=7)
    cache = H.make_cache(w, slack_pages=400, flags=REINDEX)
    saved = _saved(cache)
    leyline.leyline_pool_checkpoint(cache.pool)
    _splice(cache, w, step)
    assert cache.last_stats()["reindexed"] == 1
    with pytest.raises(leyline.LeylineError) as e:
        leyline.leyline_pool_rollback(cache.pool)
    assert e.value.code == leyline.LEYLINE_ERR_INVALID_ARG
    leyline.leyline_pool_rollback(cache.pool, flags=leyline.LEYLINE_ROLLBACK_ACCEPT_TURNED)
    _restore(cache, saved)
    _splice(cache, w, step)  # the same work again, on bands turned once already
    assert cache.last_stats()["reindexed"] == 1
    cache.close()

    lazy = H.make_cache(w, slack_pages=400, flags=LAZY)
    saved = _saved(lazy)
    leyline.leyline_pool_checkpoint(lazy.pool)
    _splice(lazy, w, step)
    lazy.materialize(0)
    torch.cuda.synchronize()
    with pytest.raises(leyline.LeylineError):
        leyline.leyline_pool_rollback(lazy.pool)
    leyline.leyline_pool_checkpoint(lazy.pool)  # a new checkpoint clears it
    leyline.leyline_pool_rollback(lazy.pool)
    del saved
    lazy.close()


def test_rollback_after_noalloc_splices():
    """leyline_splice_noalloc keeps the same page accounting as leyline_splice: a checkpoint
    before two no-alloc calls and a rollback after them give the rows back, and repeating the
    calls gives the same result bit for bit."""
    from rope_rotation_gb300 import leyline
    steps = [[Dir(0, 40, 130, 9, 0), Dir(1, 5, 300, 3, 1)], [Dir(0, 0, 3, 0, 2), Dir(1, 100, 101, 30, 3)]]
    w = Workload("rollback-noalloc", 2, 16, [600, 700], steps, seed=8)
    cache = H.make_cache(w, slack_pages=80)
    before = _all_rows(cache, w)
    saved = _saved(cache)
    leyline.leyline_pool_checkpoint(cache.pool)
    keep = []

    def run_steps():
        for step in steps:
            dirs, k = H.gpu_directives(w, step)
            keep.append(k)
            leyline.leyline_splice_noalloc(cache.pool, cache.tables, dirs)
        torch.cuda.synchronize()
        cache.check_status()
        return _all_rows(cache, w)

    first = run_steps()
    leyline.leyline_pool_rollback(cache.pool)
    _restore(cache, saved)
    torch.cuda.synchronize()
    for r, rows in enumerate(_all_rows(cache, w)):
        assert np.array_equal(rows, before[r]), f"request {r}: rollback did not restore the cache"
    again = run_steps()
    for r in range(w.num_reqs):
        assert np.array_equal(again[r], first[r]), f"request {r}: the repeat differs"
    del keep
    cache.close()


def test_rollback_restores_the_free_list_across_the_ring_end():
    """A rollback copies back only the free-list entries written since the checkpoint.  The
    free list is a ring of 2 * num_pages entries whose positions only grow, so the returned
    pages' region wraps past the ring's end once its positions do.  Against a twin pool that
    skips the splice and its rollback, the free list must come out identical, page for page
    in the order the pool hands pages out, at every checkpoint position tried."""
    from rope_rotation_gb300 import leyline
    step = [Dir(0, 100, 116, 16, 0)]  # rewrites blocks 6..9: takes 4 pages and returns 4
    w = Workload("rollback-ring", 2, 16, [160], [step], seed=10)
    cache = H.make_cache(w)
    twin = H.make_cache(w)
    num_pages = cache.num_pages
    free = cache.free_pages()
    assert free == twin.free_pages() and free > 4
    q_cap, tail = 2 * num_pages, num_pages  # every page was returned once at creation
    wrapped = False
    for k, advance in enumerate([free, 7, free, 3, free, 9, free, 1, free, free - 2, free, 5]):
        wrapped |= tail % q_cap + 4 > q_cap
        saved = _saved(cache)
        leyline.leyline_pool_checkpoint(cache.pool)
        _splice(cache, w, step)
        assert cache.last_stats()["pages_pushed"] == 4
        leyline.leyline_pool_rollback(cache.pool)
        _restore(cache, saved)
        torch.cuda.synchronize()
        assert cache.free_pages() == twin.free_pages() == free
        assert np.array_equal(cache.table.cpu().numpy(), twin.table.cpu().numpy())
        assert np.array_equal(H.logical_rows(cache, 0, 160), H.logical_rows(twin, 0, 160)), f"step {k}"
        # take `advance` pages from both and give them back in another order: the positions move on
        a = leyline.leyline_alloc_pages(cache.pool, advance)
        b = leyline.leyline_alloc_pages(twin.pool, advance)
        assert list(a) == list(b), f"step {k}: the free lists differ after the rollback"
        leyline.leyline_free_pages(cache.pool, a[::-1])
        leyline.leyline_free_pages(twin.pool, b[::-1])
        tail += advance
    assert wrapped, "no checkpoint put the returned pages' region across the ring's end"
    rest_a = leyline.leyline_alloc_pages(cache.pool, free)
    rest_b = leyline.leyline_alloc_pages(twin.pool, free)
    assert list(rest_a) == list(rest_b)
    cache.close()
    twin.close()
