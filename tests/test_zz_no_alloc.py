"""leyline_splice_noalloc against leyline_splice, through the C ABI (needs a GPU).

leyline_splice_noalloc exists for callers that must not allocate device memory
while they serve: for example a framework that has reserved nearly all GPU
memory in its own caching allocator, where a cudaMalloc made behind its back can
fail or fragment the memory it manages, or a process that keeps its device
footprint fixed after start-up.  It runs the same kernels with its scratch in a
static device array instead of a buffer that grows with cudaMalloc.

The test splices two identical caches, one through each entry point, for two
calls in a row, and checks that the results agree within the tolerance of the
other splice tests (latents, prefix rows, rows of R and lengths bit-exact; moved
rope bands within one bf16 step or 2^-16 of the pair norm).  It also checks that
a call whose plan exceeds the static scratch is refused without changing
anything.  This file is collected last, so a run stopped at the first failure
has already run every other test.
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


def test_noalloc_matches_splice_on_two_calls():
    from rope_rotation_gb300 import leyline
    steps = [
        [Dir(0, 40, 130, 9, 0), Dir(1, 5, 700, 3, 1), Dir(1, 800, 820, 64, 2), Dir(2, 76, 77, 1, 3)],
        [Dir(0, 0, 3, 0, 4), Dir(1, 100, 101, 30, 5), Dir(2, 10, 50, 2, 6)],
    ]
    w = Workload("noalloc", 4, 16, [300, 1000, 77], steps, seed=21)
    ref = H.make_cache(w, slack_pages=16)
    new = H.make_cache(w, slack_pages=16)
    for step in w.steps:
        dirs_ref, keep_ref = H.gpu_directives(w, step)
        dirs_new, keep_new = H.gpu_directives(w, step)
        leyline.leyline_splice(ref.pool, ref.tables, dirs_ref)
        leyline.leyline_splice_noalloc(new.pool, new.tables, dirs_new)
        torch.cuda.synchronize()
        ref.check_status()
        new.check_status()
        assert np.array_equal(ref.seq_lens_host, new.seq_lens_host)
        assert np.array_equal(ref.seq_lens_dev.cpu().numpy(), new.seq_lens_dev.cpu().numpy())
        assert ref.free_pages() == new.free_pages()
        assert H.work_stats(ref) == H.work_stats(new)
        for r in range(w.num_reqs):
            n = int(ref.seq_lens_host[r])
            a = H.logical_rows(ref, r, n)
            b = H.logical_rows(new, r, n)
            lat = w.latent_dim
            assert np.array_equal(a[:, :, :lat], b[:, :, :lat])
            H.compare_kpe(b[:, :, lat:].reshape(-1, w.rope_dim), a[:, :, lat:].reshape(-1, w.rope_dim), 0)
        del keep_ref, keep_new
    ref.close()
    new.close()


def test_noalloc_refuses_a_plan_larger_than_its_scratch():
    """20,000 one-token deletions in one request: each shifts its downstream run by a
    different Delta, so the plan carries 20,000 rotated segments with their cos/sin,
    more than the 4 MiB static scratch holds.  The call is refused and changes nothing."""
    from rope_rotation_gb300 import leyline
    from rope_rotation_gb300.runtime import PagedCache
    L, B = 100_000, 16
    nb = L // B
    cache = PagedCache(1, B, 2 * nb + 8, 1, nb + 8)
    cache.add_request(0, L)
    torch.cuda.synchronize()
    before = cache.table[0].cpu().numpy().copy()
    free = cache.free_pages()
    dirs = [leyline.directive(0, 5 * k + 2, 5 * k + 3, None) for k in range(20_000)]
    with pytest.raises(leyline.LeylineError) as ei:
        leyline.leyline_splice_noalloc(cache.pool, cache.tables, dirs)
    assert ei.value.code == leyline.LEYLINE_ERR_SCRATCH
    assert "scratch" in str(ei.value)
    assert int(cache.seq_lens_host[0]) == L and cache.free_pages() == free
    torch.cuda.synchronize()
    assert np.array_equal(cache.table[0].cpu().numpy(), before)
    cache.close()


def test_noalloc_matches_splice_in_reindex_mode():
    """The same two-call comparison on a block-size-1 pool in re-index mode, where the
    static scratch also holds the staged table entries."""
    from rope_rotation_gb300 import leyline
    steps = [[Dir(0, 40, 130, 9, 0), Dir(1, 5, 700, 3, 1), Dir(2, 76, 77, 1, 3)],
             [Dir(0, 0, 3, 0, 4), Dir(1, 100, 101, 30, 5, mode=2)]]
    w = Workload("noalloc-reindex", 3, 1, [300, 1000, 77], steps, seed=22)
    ref = H.make_cache(w, slack_pages=16, flags=leyline.LEYLINE_POOL_REINDEX)
    new = H.make_cache(w, slack_pages=16, flags=leyline.LEYLINE_POOL_REINDEX)
    for step in w.steps:
        dirs_ref, keep_ref = H.gpu_directives(w, step)
        dirs_new, keep_new = H.gpu_directives(w, step)
        leyline.leyline_splice(ref.pool, ref.tables, dirs_ref)
        leyline.leyline_splice_noalloc(new.pool, new.tables, dirs_new)
        torch.cuda.synchronize()
        ref.check_status()
        new.check_status()
        assert np.array_equal(ref.seq_lens_host, new.seq_lens_host)
        assert H.work_stats(ref) == H.work_stats(new)
        for r in range(w.num_reqs):
            n = int(ref.seq_lens_host[r])
            a = H.logical_rows(ref, r, n)
            b = H.logical_rows(new, r, n)
            assert np.array_equal(a[:, :, :w.latent_dim], b[:, :, :w.latent_dim])
            H.compare_kpe(b[:, :, w.latent_dim:].reshape(-1, w.rope_dim),
                          a[:, :, w.latent_dim:].reshape(-1, w.rope_dim), 0)
        del keep_ref, keep_new
    ref.close()
    new.close()


def test_noalloc_matches_splice_on_lazy_pools():
    """Lazy pools: both entry points move the same bits and leave the same pending counts."""
    from rope_rotation_gb300 import leyline
    steps = [[Dir(0, 40, 130, 9, 0), Dir(1, 5, 700, 3, 1)],
             [Dir(0, 0, 3, 0, 4), Dir(1, 100, 101, 30, 5, mode=2)]]
    w = Workload("noalloc-lazy", 2, 16, [300, 1000], steps, seed=23)
    ref = H.make_cache(w, slack_pages=16, flags=leyline.LEYLINE_POOL_LAZY)
    new = H.make_cache(w, slack_pages=16, flags=leyline.LEYLINE_POOL_LAZY)
    for step in w.steps:
        dirs_ref, keep_ref = H.gpu_directives(w, step)
        dirs_new, keep_new = H.gpu_directives(w, step)
        leyline.leyline_splice(ref.pool, ref.tables, dirs_ref)
        leyline.leyline_splice_noalloc(new.pool, new.tables, dirs_new)
        torch.cuda.synchronize()
        ref.check_status()
        new.check_status()
        assert np.array_equal(ref.seq_lens_host, new.seq_lens_host)
        assert H.work_stats(ref) == H.work_stats(new)
        for r in range(w.num_reqs):
            n = int(ref.seq_lens_host[r])
            assert np.array_equal(H.logical_rows(ref, r, n), H.logical_rows(new, r, n))
            nb = -(-n // w.block_size)
            pr = ref.pending()[ref.table[r, :nb].long()].reshape(-1)[:n]
            pn = new.pending()[new.table[r, :nb].long()].reshape(-1)[:n]
            assert torch.equal(pr, pn)
        del keep_ref, keep_new
    ref.close()
    new.close()


def test_noalloc_matches_splice_when_runs_shift_by_whole_blocks():
    """Re-index pool, block 16, spans off the grid with Delta a multiple of 16: kept pages,
    fresh boundary blocks and rows of R, through both entry points."""
    from rope_rotation_gb300 import leyline
    steps = [[Dir(0, 20, 54, 18, 0), Dir(1, 5, 40, 3, 1)],
             [Dir(0, 3, 19, 0, 2), Dir(1, 70, 71, 17, 3)]]
    w = Workload("noalloc-shift", 2, 16, [300, 170], steps, seed=24)
    ref = H.make_cache(w, slack_pages=16, flags=leyline.LEYLINE_POOL_REINDEX)
    new = H.make_cache(w, slack_pages=16, flags=leyline.LEYLINE_POOL_REINDEX)
    for step in w.steps:
        dirs_ref, keep_ref = H.gpu_directives(w, step)
        dirs_new, keep_new = H.gpu_directives(w, step)
        leyline.leyline_splice(ref.pool, ref.tables, dirs_ref)
        leyline.leyline_splice_noalloc(new.pool, new.tables, dirs_new)
        torch.cuda.synchronize()
        ref.check_status()
        new.check_status()
        assert H.work_stats(ref) == H.work_stats(new)
        assert ref.last_stats()["reindexed"] == 1
        for r in range(w.num_reqs):
            n = int(ref.seq_lens_host[r])
            assert np.array_equal(H.logical_rows(ref, r, n), H.logical_rows(new, r, n))
        del keep_ref, keep_new
    ref.close()
    new.close()


def test_noalloc_calls_on_two_streams_of_one_pool():
    """Consecutive no-alloc calls of one pool issued on two streams share the static scratch;
    the pool orders the second after the first (it waits for the first's completion event),
    so the results equal, bit for bit, leyline_splice's on one stream.  With kernel timing on,
    both calls are timed as leyline_splice's would be."""
    from rope_rotation_gb300 import leyline
    steps = [[Dir(0, 40, 130, 9, 0), Dir(1, 5, 700, 3, 1), Dir(2, 76, 77, 1, 3)],
             [Dir(0, 0, 3, 0, 4), Dir(1, 100, 101, 30, 5), Dir(2, 10, 50, 2, 6)]]
    w = Workload("noalloc-streams", 3, 16, [300, 1000, 77], steps, seed=25)
    ref = H.make_cache(w, slack_pages=16)
    new = H.make_cache(w, slack_pages=16)
    keep = []
    for step in w.steps:
        dirs, k = H.gpu_directives(w, step)
        keep.append(k)
        leyline.leyline_splice(ref.pool, ref.tables, dirs)
    calls = []
    for step in w.steps:
        dirs, k = H.gpu_directives(w, step)
        keep.append(k)
        calls.append(dirs)
    torch.cuda.synchronize()  # the caches and rows of R are written on the default stream
    leyline.leyline_kernel_timing_enable(new.pool, True)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for dirs, s in zip(calls, streams):
        leyline.leyline_splice_noalloc(new.pool, new.tables, dirs, s)
    ms, n = leyline.leyline_kernel_timing_read(new.pool)
    leyline.leyline_kernel_timing_enable(new.pool, False)
    assert n == 2 and ms > 0
    torch.cuda.synchronize()
    ref.check_status()
    new.check_status()
    assert np.array_equal(ref.seq_lens_host, new.seq_lens_host)
    assert ref.free_pages() == new.free_pages()
    for r in range(w.num_reqs):
        n_r = int(ref.seq_lens_host[r])
        assert np.array_equal(H.logical_rows(ref, r, n_r), H.logical_rows(new, r, n_r)), f"request {r} differs"
    del keep
    ref.close()
    new.close()
