"""Failure handling on the GPU, without any GPU fault (needs a GPU).

Refused calls (not enough free pages, FORGET, overlapping spans, bad gather
ranges) must leave the pool, the block table, the lengths and the cache bytes
unchanged.  A block table holding an id outside the pool must be caught by the
kernels' own bounds checks: the row is skipped, the status word is set, and
leyline_sync_status reports LEYLINE_ERR_DEVICE_CHECK -- nothing is read or
written out of bounds.
"""
import numpy as np
import pytest

import splice_harness as H
from synth.configs import Dir, Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rope_rotation_gb300
    rope_rotation_gb300.build()


def _snapshot(cache):
    torch.cuda.synchronize()
    return (cache.table.cpu().clone(), cache.seq_lens_dev.cpu().clone(), cache.seq_lens_host.copy(),
            cache.free_pages(), cache.kv.view(torch.int16).clone())


def _assert_unchanged(cache, snap):
    torch.cuda.synchronize()
    t, sl, slh, free, kv = snap
    assert torch.equal(cache.table.cpu(), t)
    assert torch.equal(cache.seq_lens_dev.cpu(), sl)
    assert np.array_equal(cache.seq_lens_host, slh)
    assert cache.free_pages() == free
    assert torch.equal(cache.kv.view(torch.int16), kv)


def _small_cache(free_extra: int):
    from rope_rotation_gb300.runtime import PagedCache
    from synth import fill
    B, L = 16, 200
    nb = -(-L // B)
    cache = PagedCache(2, B, nb + free_extra, 1, 32)
    cache.add_request(0, L)
    fill.fill_request(cache, 3, 0, L)
    return cache


def test_not_enough_pages_is_refused_and_changes_nothing():
    from rope_rotation_gb300 import leyline
    cache = _small_cache(free_extra=2)  # rewriting from block 1 needs 12 fresh pages
    snap = _snapshot(cache)
    with pytest.raises(leyline.LeylineError) as ei:
        cache.splice([leyline.directive(0, 20, 30, None)])
    assert ei.value.code == leyline.LEYLINE_ERR_NO_PAGES
    _assert_unchanged(cache, snap)
    cache.close()


@pytest.mark.parametrize("case", ["forget", "overlap", "past_end", "bad_request"])
def test_invalid_directives_change_nothing(case):
    from rope_rotation_gb300 import leyline
    cache = _small_cache(free_extra=40)
    snap = _snapshot(cache)
    dirs = {
        "forget": [leyline.directive(0, 20, 30, None, mode=leyline.LEYLINE_FORGET)],
        "overlap": [leyline.directive(0, 20, 30, None), leyline.directive(0, 25, 40, None)],
        "past_end": [leyline.directive(0, 150, 201, None)],
        "bad_request": [leyline.directive(1, 0, 1, None)],
    }[case]
    want = {"forget": leyline.LEYLINE_ERR_UNSUPPORTED_MODE, "overlap": leyline.LEYLINE_ERR_OVERLAP,
            "past_end": leyline.LEYLINE_ERR_INVALID_DIRECTIVE, "bad_request": leyline.LEYLINE_ERR_INVALID_DIRECTIVE}
    with pytest.raises(leyline.LeylineError) as ei:
        cache.splice(dirs)
    assert ei.value.code == want[case]
    _assert_unchanged(cache, snap)
    cache.close()


def test_gather_range_checks():
    from rope_rotation_gb300 import leyline
    cache = _small_cache(free_extra=4)
    out = torch.empty((10, cache.row), dtype=torch.bfloat16, device="cuda")
    for args in [(0, 0, 195, 205), (0, 2, 0, 10), (1, 0, 0, 10), (0, 0, 5, 4)]:
        with pytest.raises(leyline.LeylineError) as ei:
            cache.gather(*args, out=out[: max(args[3] - args[2], 0)])
        assert ei.value.code == leyline.LEYLINE_ERR_INVALID_ARG
    cache.close()


@pytest.mark.parametrize("move_kernel", ["vector", "bulk"])
def test_corrupt_table_entry_is_caught_by_device_checks(move_kernel, monkeypatch):
    """A page id outside the pool inside the live range of a request: the move kernel
    must skip the row and flag it, never dereference it."""
    monkeypatch.setenv("LEYLINE_MOVE_KERNEL", move_kernel)
    from rope_rotation_gb300 import leyline
    cache = _small_cache(free_extra=40)
    cache.table[0, 8] = cache.num_pages + 1000  # block 8 holds tokens 128..143
    torch.cuda.synchronize()
    cache.splice([leyline.directive(0, 10, 20, None)])
    with pytest.raises(leyline.LeylineError) as ei:
        cache.check_status()
    assert ei.value.code == leyline.LEYLINE_ERR_DEVICE_CHECK
    cache.check_status()  # the status word was cleared by the read
    cache.close()


def test_alloc_and_free_pages_round_trip():
    from rope_rotation_gb300 import leyline
    from rope_rotation_gb300.runtime import PagedCache
    cache = PagedCache(1, 4, 64, 1, 8)
    a = leyline.leyline_alloc_pages(cache.pool, 10)
    assert list(a) == list(range(10))
    assert cache.free_pages() == 54
    leyline.leyline_free_pages(cache.pool, a[:5])
    assert cache.free_pages() == 59
    b = leyline.leyline_alloc_pages(cache.pool, 59)  # FIFO: 10..63 first, then the returned ones
    assert list(b[:54]) == list(range(10, 64)) and sorted(b[54:]) == list(range(5))
    with pytest.raises(leyline.LeylineError) as ei:
        leyline.leyline_alloc_pages(cache.pool, 1)
    assert ei.value.code == leyline.LEYLINE_ERR_NO_PAGES
    with pytest.raises(leyline.LeylineError):
        leyline.leyline_free_pages(cache.pool, [64])
    cache.close()


def test_splices_on_two_streams_are_ordered():
    """Two consecutive splices of the same request issued on different streams: the second
    must see the first's table (the pool orders them)."""
    from rope_rotation_gb300 import leyline
    w = Workload("streams", 2, 16, [400], [[Dir(0, 30, 90, 4, 0)], [Dir(0, 10, 20, 2, 1)]], seed=9)
    cache = H.make_cache(w)
    state = H.oracle_state(w)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        H.splice_step_and_check(w, cache, state, w.steps[0], guard=False)
    with torch.cuda.stream(s2):
        H.splice_step_and_check(w, cache, state, w.steps[1], guard=False)
    cache.close()


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")  # every call was refused: nothing captured
def test_host_planned_calls_refuse_graph_capture():
    """A splice, a materialize and a checkpoint or rollback are planned on the host for the
    cache as it stands, so a CUDA graph that replayed them would apply stale plans: each
    refuses a stream under capture, before anything is enqueued or changed."""
    import torch
    from rope_rotation_gb300 import leyline
    w = Workload("capture", 1, 16, [300], [[Dir(0, 10, 40, 3, 0)]], seed=3)
    cache = H.make_cache(w, slack_pages=8)
    lazy = H.make_cache(w, slack_pages=8, flags=leyline.LEYLINE_POOL_LAZY)
    dirs, keep = H.gpu_directives(w, w.steps[0])
    leyline.leyline_pool_checkpoint(cache.pool)
    torch.cuda.synchronize()
    free, lens = cache.free_pages(), cache.seq_lens_host.copy()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    codes = []
    calls = [lambda: cache.splice(dirs, s), lambda: leyline.leyline_pool_checkpoint(cache.pool, s),
             lambda: leyline.leyline_pool_rollback(cache.pool, 0, s), lambda: lazy.materialize(0, s)]
    with torch.cuda.graph(graph, stream=s):
        for call in calls:
            try:
                call()
                codes.append(0)
            except leyline.LeylineError as e:
                codes.append(e.code)
    assert codes == [leyline.LEYLINE_ERR_INVALID_ARG] * len(calls)
    assert cache.free_pages() == free and np.array_equal(cache.seq_lens_host, lens)
    cache.splice(dirs)  # outside the capture the same call proceeds
    torch.cuda.synchronize()
    cache.check_status()
    assert int(cache.seq_lens_host[0]) == 300 - 30 + 3
    del keep
    cache.close()
    lazy.close()


def test_plans_larger_than_a_plan_slot():
    """300 one-token deletions in one call: 300 rotated segments, each with its own cos / sin,
    make a plan of about 100 KB, more than the 64 KB a plan slot starts with.  The slot's
    pinned and device buffers grow (after the pool's earlier work has ended), and the call is
    checked against the oracle like any other; later calls take the slots in turn, one of
    them the grown slot again."""
    from rope_rotation_gb300 import leyline
    L = 2000
    big = [Dir(0, 5 * k + 2, 5 * k + 3, 0, k) for k in range(300)]
    big2 = [Dir(0, 4 * k + 1, 4 * k + 2, 1 if k % 3 == 0 else 0, 300 + k) for k in range(300)]
    # 30 one-token replacements: 60 segments, more than a kernel parameter holds, so these
    # plans are uploaded too and the calls walk through all 8 slots, reusing the grown one
    mid = [Dir(0, 3 * k + 1, 3 * k + 2, 1, 700 + k) for k in range(30)]
    last = [Dir(0, 5 * k + 2, 5 * k + 3, 0, 1000 + k) for k in range(280)]  # within the shorter length
    steps = [big] + [mid] * 7 + [big2, mid, last]
    w = Workload("big-plan", 2, 16, [L], steps, seed=12)
    cache = H.make_cache(w, slack_pages=8)
    state = H.oracle_state(w)
    for step in w.steps:
        H.splice_step_and_check(w, cache, state, step)
        assert cache.last_stats()["kernels_launched"] == 3  # the plan copy, move and commit
    cache.close()
