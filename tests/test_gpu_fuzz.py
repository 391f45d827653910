"""Seeded random splices in every pool mode against the oracle (needs a GPU).

Each case draws request lengths, block size, layer count and 1-3 chained calls of
random directives (spans, |R|, AMORTIZE or EVICT, several per request, no-ops and
pure insertions included) from its seed, and checks every call with the oracle
through the same harness as the other parity tests.  Modes: rewrite, re-index
(block size 1 and calls on the block grid), split rope, and lazy pools against the
oracle-tracked pending counts.
"""
import numpy as np
import pytest

import splice_harness as H
from synth.configs import Dir, Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

REINDEX, LAZY, SPLIT = 1, 2, 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rope_rotation_gb300
    rope_rotation_gb300.build()


def _random_steps(rng, lengths, n_steps):
    lens = list(lengths)
    steps, key = [], 0
    for _ in range(n_steps):
        step = []
        for r, L in enumerate(lens):
            k = int(rng.integers(0, 4))
            cuts = np.sort(rng.integers(0, L + 1, size=2 * k)) if k else np.zeros(0, dtype=np.int64)
            for j in range(k):
                s, e = int(cuts[2 * j]), int(cuts[2 * j + 1])
                if j > 0 and s == int(cuts[2 * j - 2]):
                    continue  # distinct s_start
                n = int(rng.integers(0, 40))
                mode = 2 if rng.random() < 0.25 else 0
                step.append(Dir(r, s, e, n, key, mode))
                key += 1
                L = L - (e - s) + n
            lens[r] = L
        steps.append(step)
    return steps


def _case(seed):
    rng = np.random.default_rng(seed)
    n_req = int(rng.integers(1, 4))
    lengths = [int(rng.integers(0, 700)) for _ in range(n_req)]
    return rng, lengths, int(rng.integers(1, 4))


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("mode", ["rewrite", "reindex1", "split"])
def test_fuzz_eager(seed, mode):
    rng, lengths, layers = _case(1000 + seed)
    B = 1 if mode == "reindex1" else int(rng.choice([1, 2, 4, 16]))
    flags = {"rewrite": 0, "reindex1": REINDEX, "split": SPLIT | (REINDEX if seed % 2 else 0)}[mode]
    layout = int(rng.integers(0, 2))
    steps = _random_steps(rng, lengths, 3)
    w = Workload(f"fuzz-{mode}-{seed}", layers, B, lengths, steps, seed=seed)
    cache = H.make_cache(w, pair_layout=layout, slack_pages=64, flags=flags)
    state = H.oracle_state(w)
    for step in steps:
        H.splice_step_and_check(w, cache, state, step, layout=layout)
    cache.close()


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_block_grid(seed):
    rng, lengths, layers = _case(2000 + seed)
    B = int(rng.choice([2, 4, 8, 16]))
    steps = H.aligned_steps(3000 + seed, B, lengths, 3, evict_every=2)
    w = Workload(f"fuzz-grid-{seed}", layers, B, lengths, steps, seed=seed)
    cache = H.make_cache(w, slack_pages=64, flags=REINDEX | (SPLIT if seed % 2 else 0))
    state = H.oracle_state(w)
    for step in steps:
        c = H.splice_step_and_check(w, cache, state, step)
        if any(not (d.s_start == d.s_end and d.n_repl == 0) for d in step):
            assert c["stats"]["reindexed"] == 1
    cache.close()


def _shift_aligned_steps(rng, lengths, n_steps, B):
    """Random spans, with |R| chosen half the time so that Delta is a multiple of B (the
    survivors' whole blocks then keep their pages)."""
    lens = list(lengths)
    steps, key = [], 0
    for _ in range(n_steps):
        step = []
        for r, L in enumerate(lens):
            s = int(rng.integers(0, L + 1))
            e = int(rng.integers(s, min(L, s + 5 * B) + 1))
            n = int(rng.integers(0, 3 * B))
            if rng.random() < 0.5:
                n = (e - s) % B + B * int(rng.integers(0, 3))
            mode = 2 if rng.random() < 0.2 else 0
            step.append(Dir(r, s, e, n, key, mode))
            key += 1
            lens[r] = L - (e - s) + n
        steps.append(step)
    return steps


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_reindex_shift_aligned(seed):
    """Re-index pools with pages of several slots and spans off the grid: kept pages for runs
    shifted by whole blocks, fresh pages for the boundary blocks, in eager, lazy and split pools."""
    rng = np.random.default_rng(5000 + seed)
    n_req = int(rng.integers(1, 4))
    B = int(rng.choice([2, 4, 8, 16]))
    lengths = [int(rng.integers(0, 40 * B)) for _ in range(n_req)]
    layers = int(rng.integers(1, 4))
    steps = _shift_aligned_steps(rng, lengths, 3, B)
    flags = REINDEX | (SPLIT if seed % 3 == 0 else 0)
    w = Workload(f"fuzz-shift-{seed}", layers, B, lengths, steps, seed=seed)
    cache = H.make_cache(w, slack_pages=64, flags=flags | (LAZY if seed % 2 else 0))
    if seed % 2:
        import test_gpu_lazy as TL
        st = TL.LazyState(w)
        for step in steps:
            TL._step(w, cache, st, step)
    else:
        state = H.oracle_state(w)
        for step in steps:
            H.splice_step_and_check(w, cache, state, step)
    cache.close()


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_lazy(seed):
    import test_gpu_lazy as TL
    rng, lengths, layers = _case(4000 + seed)
    B = 1 if seed % 2 else int(rng.choice([2, 4, 16]))
    flags = LAZY | (REINDEX if seed % 2 else 0) | (SPLIT if seed % 3 == 0 else 0)
    steps = _random_steps(rng, lengths, 3)
    w = Workload(f"fuzz-lazy-{seed}", layers, B, lengths, steps, seed=seed)
    cache = H.make_cache(w, slack_pages=64, flags=flags)
    st = TL.LazyState(w)
    for step in steps:
        TL._step(w, cache, st, step)
    cache.close()
