"""Pools with the rope bands apart from the latents (LEYLINE_POOL_SPLIT_ROPE; needs a GPU).

A split pool stores latent[layer][page][slot][latent] and then rope[layer][page][slot]
[bands], the layout of paged MLA attention kernels that take a latent cache and a rope
cache.  Only addresses change, so every splice on a split pool must produce, bit for
bit, the logical rows, lengths and statistics of the same splice on a pool of whole
rows; two chains are also checked against the oracle directly.
"""
import numpy as np
import pytest

import splice_harness as H
from synth.configs import Dir, Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SPLIT, REINDEX, LAZY = 4, 1, 2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rope_rotation_gb300
    rope_rotation_gb300.build()


STEPS = [[Dir(0, 40, 130, 9, 0), Dir(1, 5, 700, 3, 1), Dir(1, 800, 820, 64, 2)],
         [Dir(0, 0, 3, 5, 3), Dir(1, 100, 101, 30, 4, mode=2)],
         [Dir(0, 17, 17, 2, 5), Dir(1, 0, 64, 0, 6)]]


def _run(w, cache):
    for step in w.steps:
        dirs, keep = H.gpu_directives(w, step)
        cache.splice(dirs)
        torch.cuda.synchronize()
        cache.check_status()
        del keep
    return H.work_stats(cache)


@pytest.mark.parametrize("B,flags,layout,precision,heads,rope", [
    (16, 0, 0, 0, 1, 64), (16, 0, 1, 0, 1, 64), (16, 0, 0, 1, 1, 64),
    (1, REINDEX, 0, 0, 1, 64), (1, REINDEX, 1, 0, 1, 64),
    (16, LAZY, 0, 0, 1, 64), (1, LAZY | REINDEX, 0, 0, 1, 64),
    (16, 0, 0, 0, 4, 128), (1, REINDEX, 1, 0, 4, 128)])
def test_split_equals_whole_rows(B, flags, layout, precision, heads, rope):
    w = Workload(f"split-B{B}-f{flags}", 3, B, [300, 1000], STEPS, seed=101, rope_dim=rope, rope_heads=heads)
    whole = H.make_cache(w, pair_layout=layout, precision=precision, slack_pages=16, flags=flags)
    split = H.make_cache(w, pair_layout=layout, precision=precision, slack_pages=16, flags=flags | SPLIT)
    assert _run(w, whole) == _run(w, split)
    for r in range(w.num_reqs):
        n = int(whole.seq_lens_host[r])
        assert n == int(split.seq_lens_host[r])
        assert np.array_equal(H.logical_rows(whole, r, n), H.logical_rows(split, r, n))
    whole.close()
    split.close()


def test_block_reindex_split_equals_whole_rows():
    lengths = [16 * 37 + 5, 16 * 20]
    steps = H.aligned_steps(111, 16, lengths, 6, evict_every=3)
    w = Workload("split-block-reindex", 3, 16, lengths, steps, seed=111)
    whole = H.make_cache(w, slack_pages=64, flags=REINDEX)
    split = H.make_cache(w, slack_pages=64, flags=REINDEX | SPLIT)
    for step in steps:
        for c in (whole, split):
            dirs, keep = H.gpu_directives(w, step)
            c.splice(dirs)
            torch.cuda.synchronize()
            c.check_status()
            del keep
        assert H.work_stats(whole) == H.work_stats(split)
    for r in range(w.num_reqs):
        n = int(whole.seq_lens_host[r])
        assert np.array_equal(H.logical_rows(whole, r, n), H.logical_rows(split, r, n))
    whole.close()
    split.close()


@pytest.mark.parametrize("B,flags", [(16, SPLIT), (1, SPLIT | REINDEX)])
def test_split_against_oracle(B, flags):
    w = Workload(f"split-oracle-B{B}", 2, B, [300, 1000], STEPS, seed=102)
    cache = H.make_cache(w, slack_pages=16, flags=flags)
    state = H.oracle_state(w)
    for step in w.steps:
        H.splice_step_and_check(w, cache, state, step)
    cache.close()


def test_split_materialize():
    w = Workload("split-materialize", 3, 1, [900], [[Dir(0, 40, 130, 9, 0)], [Dir(0, 10, 11, 0, 1)]], seed=103)
    cache = H.make_cache(w, slack_pages=16, flags=SPLIT | LAZY | REINDEX)
    _run(w, cache)
    n = int(cache.seq_lens_host[0])
    before = H.logical_rows(cache, 0, n)
    cache.materialize(0)
    torch.cuda.synchronize()
    cache.check_status()
    assert not cache.pending().any()
    assert np.array_equal(before, H.logical_rows(cache, 0, n))
    cache.close()
