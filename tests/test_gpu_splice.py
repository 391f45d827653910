"""GPU splice vs the fp64 oracle, through the C ABI (needs a GB300).

Edge cases of "Leyline: KV Cache Directives for Agentic Inference", section 2.1
(spans at the start and the end of the sequence, empty spans, pure insertions
and deletions, several directives per request, several requests per call) at
block sizes 1, 2, 4 and 16, with ragged tails; the two RoPE pair layouts; the
generic-shape kernel; the bf16-only comparison arm; and the 1-layer 4k and the
27-layer 32k workloads in full.
"""
import numpy as np
import pytest

import splice_harness as H
from synth import configs
from synth.configs import Dir, Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rope_rotation_gb300
    rope_rotation_gb300.build()


EDGE = [
    # (L, directives as (s, e, n_repl))
    (37, [(5, 20, 3)]),
    (37, [(0, 9, 2)]),             # s_start = 0
    (37, [(30, 37, 5)]),           # s_end = L, grows
    (37, [(17, 17, 6)]),           # pure insertion (Delta > 0)
    (37, [(8, 30, 0)]),            # pure deletion
    (37, [(0, 37, 4)]),            # everything replaced
    (37, [(0, 37, 0)]),            # everything deleted
    (32, [(16, 32, 0)]),           # truncation at a block boundary (B=16)
    (48, [(3, 5, 9), (20, 33, 1), (40, 41, 0)]),  # three directives
    (48, [(47, 48, 2), (1, 2, 0)]),  # unsorted input
    (64, [(10, 10, 0), (20, 30, 10)]),  # a no-op directive and Delta = 0
    (100, [(33, 71, 12)]),
]


@pytest.fixture(params=["bulk", "vector"])
def move_kernel(request, monkeypatch):
    """Both move+rotate kernels: bulk copies staged in shared memory, and vector loads."""
    monkeypatch.setenv("LEYLINE_MOVE_KERNEL", request.param)
    return request.param


@pytest.mark.parametrize("B", [1, 2, 4, 16])
def test_edge_grid(B, move_kernel):
    for i, (L, dirs) in enumerate(EDGE):
        w = Workload(f"edge{i}-B{B}", 3, B, [L], [[Dir(0, s, e, n, k) for k, (s, e, n) in enumerate(dirs)]], seed=i)
        cache = H.make_cache(w)
        state = H.oracle_state(w)
        H.splice_step_and_check(w, cache, state, w.steps[0])
        cache.close()


@pytest.mark.parametrize("B", [1, 16])
def test_many_requests_one_call_and_chained_steps(B, move_kernel):
    lengths = [70, 16, 0, 129, 33]
    steps = [
        [Dir(0, 10, 40, 3, 0), Dir(1, 0, 16, 0, 1), Dir(3, 64, 64, 20, 2), Dir(3, 100, 120, 1, 3),
         Dir(4, 32, 33, 1, 4), Dir(2, 0, 0, 5, 5)],
        [Dir(0, 0, 1, 0, 6), Dir(3, 1, 2, 2, 7), Dir(4, 0, 0, 0, 8)],
        [Dir(2, 5, 5, 17, 9), Dir(0, 30, 42, 7, 10)],
    ]
    w = Workload(f"multi-B{B}", 2, B, lengths, steps, seed=11)
    cache = H.make_cache(w, slack_pages=8)
    state = H.oracle_state(w)
    for step in w.steps:
        H.splice_step_and_check(w, cache, state, step)
    cache.close()


@pytest.mark.parametrize("layout", [0, 1])
def test_interleaved_and_half_split_layouts(layout, move_kernel):
    w = Workload(f"layout{layout}", 2, 16, [300, 211], [[Dir(0, 40, 200, 7, 0), Dir(1, 3, 50, 60, 1)]], seed=3)
    cache = H.make_cache(w, pair_layout=layout)
    H.splice_step_and_check(w, cache, H.oracle_state(w), w.steps[0], layout=layout)
    cache.close()


@pytest.mark.parametrize("layout", [0, 1])
def test_generic_shape_kernel(layout, move_kernel):
    """latent 64 + rope 16: not the MLA shape, so the generic move+rotate kernel runs."""
    w = Workload(f"generic{layout}", 3, 4, [90, 45], [[Dir(0, 20, 60, 5, 0), Dir(1, 44, 45, 3, 1)]], seed=4,
                 latent_dim=64, rope_dim=16)
    cache = H.make_cache(w, pair_layout=layout)
    H.splice_step_and_check(w, cache, H.oracle_state(w), w.steps[0], layout=layout)
    cache.close()


@pytest.mark.parametrize("layout", [0, 1])
def test_bf16_naive_arm_is_exact(layout, move_kernel):
    w = Workload(f"bf16naive{layout}", 2, 16, [500], [[Dir(0, 100, 180, 12, 0)], [Dir(0, 0, 33, 1, 1)]], seed=5)
    cache = H.make_cache(w, pair_layout=layout, precision=1)
    state = H.oracle_state(w)
    for step in w.steps:
        H.splice_step_and_check(w, cache, state, step, layout=layout, precision=1)
    cache.close()


def test_delta_zero_leaves_logical_cache_unchanged():
    """|R| = |S| with R equal to the replaced rows: every logical row keeps its bits."""
    w = Workload("delta0", 4, 16, [777], [[]], seed=6)
    cache = H.make_cache(w)
    before = H.logical_rows(cache, 0, 777)
    repl = torch.from_numpy(before[:, 100:140].copy().view(np.int16)).cuda().view(torch.bfloat16)
    from rope_rotation_gb300 import leyline
    cache.splice([leyline.directive(0, 100, 140, repl)])
    torch.cuda.synchronize()
    cache.check_status()
    after = H.logical_rows(cache, 0, 777)
    assert np.array_equal(before, after)
    cache.close()


@pytest.mark.parametrize("B", [16, 1])
def test_two_splices_equal_one_composed_splice(B):
    """Closure through the kernels ("Leyline: KV Cache Directives for Agentic Inference",
    section 2.2: R(a) R(b) = R(a + b)).  One call holding two directives turns the rows past
    both once by Delta_1 + Delta_2; the same edit as two calls (the right directive first, so
    the left one's coordinates hold) turns them by Delta_2 and then by Delta_1, rounding to
    bf16 in between.  Rows turned once (by Delta_1, with the same cos/sin) and every copied
    row must agree bit for bit; rows turned twice differ at most by the two outputs' own
    roundings (half a bf16 step each) plus the intermediate rounding turned once more:
    each element of it is at most 2^-8 of the pair norm, so at most sqrt(2) 2^-8 of the
    pair norm after the turn, plus fp32 noise."""
    import oracle
    left, right = (100, 300, 20), (500, 600, 7)
    L = 900
    # the right directive's rows of R sit at their final position in the one-call edit, and
    # one call earlier (before the left directive moves them) in the two-call edit: different
    # encodings, so they are compared with the oracle, not with each other
    one = Workload(f"closure-one-B{B}", 2, B, [L], [[Dir(0, *left, 0), Dir(0, *right, 1)]], seed=33)
    two = Workload(f"closure-two-B{B}", 2, B, [L], [[Dir(0, *right, 1)], [Dir(0, *left, 0)]], seed=33)
    ca, cb = H.make_cache(one), H.make_cache(two)
    keep = []
    for w, cache in ((one, ca), (two, cb)):
        for step in w.steps:
            dirs, k = H.gpu_directives(w, step)
            keep.append(k)
            cache.splice(dirs)
            torch.cuda.synchronize()
            cache.check_status()
    newlen, kind, idx, which = oracle.splice_map(L, [left, right])
    assert int(ca.seq_lens_host[0]) == int(cb.seq_lens_host[0]) == newlen
    a = H.logical_rows(ca, 0, newlen)
    b = H.logical_rows(cb, 0, newlen)
    lat = one.latent_dim
    assert np.array_equal(a[:, :, :lat], b[:, :, :lat]), "latent bits differ"
    right_r = (kind == 1) & (which == 1)
    twice = (kind == 0) & (idx >= right[1])
    same = ~right_r & ~twice  # prefix, the left directive's rows of R, rows turned once
    assert np.array_equal(a[:, same], b[:, same]), "rows copied or turned once differ"
    # the right directive's rows of R in the two-call edit: written, then turned by Delta_1
    d1 = left[2] - (left[1] - left[0])
    rr = b[:, right_r, lat:].reshape(-1, one.rope_dim)
    want = oracle.rerotate(a[:, right_r, lat:].reshape(-1, one.rope_dim), 0, d1, one.theta)
    H.compare_kpe(rr, want, 0)
    ga = oracle.bf16_value(a[:, twice, lat:].reshape(-1, one.rope_dim))
    gb = oracle.bf16_value(b[:, twice, lat:].reshape(-1, one.rope_dim))
    pn = H.pair_norms(ga, 0)
    bound = 0.5 * H.bf16_step(ga) + 0.5 * H.bf16_step(gb) + (np.sqrt(2.0) * 2.0 ** -8 + 2.0 ** -16) * pn
    diff = np.abs(ga - gb)
    assert np.all(diff <= bound), f"{int((diff > bound).sum())} elements beyond the two-rounding bound"
    assert np.any(diff > 0), "two roundings should leave some elements apart"
    del keep
    ca.close()
    cb.close()


def test_contiguous_4k_workload():
    w = configs.contiguous_4k()
    cache = H.make_cache(w)
    c = H.splice_step_and_check(w, cache, H.oracle_state(w), w.steps[0])
    assert c["stats"]["downstream_slots"] == 2048 and c["stats"]["repl_slots"] == 16
    cache.close()


def test_dsv2_lite_32k_workload_full(move_kernel):
    """27 layers x 32768 tokens, block 16: every row checked against the oracle."""
    w = configs.dsv2_lite_32k()
    cache = H.make_cache(w)
    c = H.splice_step_and_check(w, cache, H.oracle_state(w), w.steps[0])
    st = c["stats"]
    assert (st["downstream_slots"], st["repl_slots"], st["head_slots"]) == (6768, 12, 0)
    assert st["algorithmic_bytes"] == 2304 * 27 * (6768 + 12)
    print("cfg2 rope parity:", {k: v for k, v in c.items() if k != "stats"})
    cache.close()


# ------------------------------------------------------------------------------
# EVICT (KV-streams page: evict without resetting positions): survivors move but keep
# the positions they were encoded at; mixed with AMORTIZE, a survivor is turned by the
# AMORTIZE shifts left of it only.
MODES = [
    (60, [(5, 20, 3, 2)]),                                  # evict only: pure move
    (60, [(5, 20, 3, 2), (30, 40, 0, 0)]),                  # evict then amortize
    (60, [(5, 20, 3, 0), (30, 40, 0, 2), (50, 52, 9, 0)]),  # amortize, evict, amortize
    (48, [(0, 48, 5, 2)]),
]


@pytest.mark.parametrize("B", [1, 16])
def test_evict_and_mixed_modes(B, move_kernel):
    for i, (L, dirs) in enumerate(MODES):
        w = Workload(f"modes{i}-B{B}", 3, B, [L],
                     [[Dir(0, s, e, n, k, mode=m) for k, (s, e, n, m) in enumerate(dirs)]], seed=20 + i)
        cache = H.make_cache(w)
        H.splice_step_and_check(w, cache, H.oracle_state(w), w.steps[0])
        cache.close()


# ------------------------------------------------------------------------------
# Re-index mode (block size 1, LEYLINE_POOL_REINDEX): survivors keep their pages, only
# the table entries move and rope bands turn in place.
REINDEX = 1
LAZY = 2
SPLIT = 4


def test_reindex_edge_grid():
    for i, (L, dirs) in enumerate(EDGE + [(60, [(5, 20, 3), (30, 40, 0)])]):
        w = Workload(f"reindex{i}", 3, 1, [L], [[Dir(0, s, e, n, k) for k, (s, e, n) in enumerate(dirs)]], seed=30 + i)
        cache = H.make_cache(w, flags=REINDEX)
        c = H.splice_step_and_check(w, cache, H.oracle_state(w), w.steps[0])
        st = c["stats"]
        assert st["reindexed"] == 1
        assert st["pages_popped"] == sum(n for (_, _, n) in dirs if not (n == 0))
        cache.close()


def test_reindex_many_requests_chained_and_modes():
    lengths = [70, 16, 0, 129, 33]
    steps = [
        [Dir(0, 10, 40, 3, 0), Dir(1, 0, 16, 0, 1), Dir(3, 64, 64, 20, 2), Dir(3, 100, 120, 1, 3),
         Dir(4, 32, 33, 1, 4), Dir(2, 0, 0, 5, 5)],
        [Dir(0, 0, 1, 0, 6, mode=2), Dir(3, 1, 2, 2, 7), Dir(4, 0, 0, 0, 8)],
        [Dir(2, 5, 5, 17, 9), Dir(0, 30, 42, 7, 10), Dir(3, 40, 41, 0, 11, mode=2)],
    ]
    w = Workload("reindex-multi", 2, 1, lengths, steps, seed=12)
    cache = H.make_cache(w, slack_pages=8, flags=REINDEX)
    state = H.oracle_state(w)
    for step in w.steps:
        H.splice_step_and_check(w, cache, state, step)
    cache.close()


@pytest.mark.parametrize("layout,precision,latent,rope", [(0, 0, 512, 64), (1, 0, 512, 64), (0, 1, 512, 64),
                                                          (1, 0, 64, 16), (0, 0, 64, 128)])
def test_reindex_layouts_precisions_shapes(layout, precision, latent, rope):
    w = Workload(f"reindex-l{layout}-p{precision}-{latent}-{rope}", 2, 1, [300, 211],
                 [[Dir(0, 40, 200, 7, 0), Dir(1, 3, 50, 60, 1)], [Dir(0, 0, 5, 1, 2)]], seed=13,
                 latent_dim=latent, rope_dim=rope)
    cache = H.make_cache(w, pair_layout=layout, precision=precision, flags=REINDEX)
    state = H.oracle_state(w)
    for step in w.steps:
        H.splice_step_and_check(w, cache, state, step, layout=layout, precision=precision)
    cache.close()


def test_reindex_chain_matches_oracle_chain_call_by_call():
    """16 chained splices on 6 layers x 32768 tokens: every call checked against the oracle
    applied to its own previous state."""
    w = configs.chain_64(seed=3, num_layers=6, length=32768, n_steps=16)
    cache = H.make_cache(w, flags=REINDEX)
    state = H.oracle_state(w)
    for step in w.steps:
        c = H.splice_step_and_check(w, cache, state, step, guard=False)
        assert c["stats"]["algorithmic_bytes"] == 2 * 6 * (128 * c["stats"]["downstream_slots"] + 1152 * 12)
    cache.close()


# ------------------------------------------------------------------------------
# Re-index mode with pages of several slots: calls whose directives all lie on block
# boundaries drop, insert and shift whole pages; other calls rewrite.
@pytest.mark.parametrize("B,layout", [(16, 0), (4, 1), (2, 0)])
def test_block_reindex_aligned_chain(B, layout):
    lengths = [16 * 37 + 5, 16 * 20, 7]
    steps = H.aligned_steps(50 + B, B, lengths, 8, evict_every=3)
    w = Workload(f"block-reindex-B{B}", 3, B, lengths, steps, seed=50 + B)
    cache = H.make_cache(w, pair_layout=layout, slack_pages=64, flags=REINDEX)
    state = H.oracle_state(w)
    for step in w.steps:
        c = H.splice_step_and_check(w, cache, state, step, layout=layout)
        if any(not (d.s_start == d.s_end and d.n_repl == 0) for d in step):
            assert c["stats"]["reindexed"] == 1, "an aligned call was not re-indexed"
    cache.close()


def test_block_reindex_keeps_pages_of_runs_shifted_by_whole_blocks():
    """Block 16, directives off the block grid.  Delta = -16 keeps the pages of the survivors'
    whole blocks (the table's entries move by one block); Delta = -3 keeps nothing.  Both are
    checked against the oracle."""
    steps = [[Dir(0, 20, 54, 18, 0), Dir(1, 20, 40, 3, 1)],
             [Dir(0, 16, 48, 0, 2), Dir(1, 0, 16, 32, 3)]]
    w = Workload("block-reindex-mixed", 2, 16, [300, 170], steps, seed=60)
    cache = H.make_cache(w, slack_pages=32, flags=REINDEX)
    state = H.oracle_state(w)
    before = cache.table.cpu().numpy().copy()
    c = H.splice_step_and_check(w, cache, state, steps[0])
    assert c["stats"]["reindexed"] == 1
    after = cache.table.cpu().numpy()
    # request 0: rows from 54 on move to 38 on; new blocks 3.. hold old blocks 4.. (19 blocks
    # before, 18 after: 300 - 16 = 284 rows)
    assert np.array_equal(after[0, 3:18], before[0, 4:19])
    # request 1: Delta = -17, no block keeps its page from b0 = 1 on
    assert not (set(after[1, 1:10].tolist()) & set(before[1, 1:11].tolist()))
    assert H.splice_step_and_check(w, cache, state, steps[1])["stats"]["reindexed"] == 1
    cache.close()


# ------------------------------------------------------------------------------
# GQA/MHA rows (section 5 of the Leyline page: the directive abstraction extends to
# GQA/MHA): [V | keys of 4 heads x 128], every key band turned with the same theta_j.
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("B,flags", [(16, 0), (1, 0), (1, 1)])
def test_gqa_rows(layout, B, flags):
    steps = [[Dir(0, 20, 90, 6, 0), Dir(1, 3, 3, 9, 1, mode=2), Dir(1, 40, 41, 0, 2)],
             [Dir(0, 0, 10, 2, 3), Dir(1, 60, 70, 1, 4)]]
    w = Workload(f"gqa-l{layout}-B{B}-f{flags}", 2, B, [200, 123], steps, seed=40,
                 latent_dim=512, rope_dim=128, rope_heads=4)
    cache = H.make_cache(w, pair_layout=layout, flags=flags)
    state = H.oracle_state(w)
    for step in w.steps:
        H.splice_step_and_check(w, cache, state, step, layout=layout)
    cache.close()


# ------------------------------------------------------------------------------
# Many calls in flight: plans too large for a kernel parameter go through a ring of plan
# slots (a pinned staging buffer and a device buffer each; a kernel copies one to the
# other), so the host enqueues call after call without waiting; the final caches must
# equal, bit for bit, those of the same calls made one at a time, each of which is checked
# against the oracle at the per-splice tolerance.
@pytest.mark.parametrize("flags,batch,streams", [(0, False, 1), (REINDEX, False, 1), (0, True, 1), (REINDEX, True, 1),
                                                 (0, False, 2), (REINDEX, True, 2)])
def test_many_calls_in_flight_with_uploaded_plans(flags, batch, streams):
    """batch: the directives go in as one directive_batch() record array per call.  streams=2:
    the calls alternate between two streams (the pool orders each after the one before)."""
    import torch
    from rope_rotation_gb300 import leyline
    rng = np.random.default_rng(77)
    n_req, B = 10, 1 if flags else 16
    lengths = [int(rng.integers(200, 600)) for _ in range(n_req)]
    lens = list(lengths)
    steps, key = [], 0
    for _ in range(20):  # 20 calls, 10 requests x 2 directives each: 30+ segments per plan
        step = []
        for r in range(n_req):
            L = lens[r]
            a, b = sorted(int(x) for x in rng.integers(0, L // 2, size=2))
            c, d = sorted(int(x) for x in rng.integers(L // 2 + 1, L, size=2))
            for s, e in ((a, b), (c, d)):
                n = int(rng.integers(0, 6))
                step.append(Dir(r, s, e, n, key))
                key += 1
                L += n - (e - s)
            lens[r] = L
        steps.append(step)
    w = Workload(f"in-flight-f{flags}", 2, B, lengths, steps, seed=78)
    cache = H.make_cache(w, slack_pages=64, flags=flags)
    keep, calls = [], []
    for step in steps:
        dirs, k = H.gpu_directives(w, step)
        keep.append(k)
        if batch:
            dirs = leyline.directive_batch([d.req for d in step], [d.s_start for d in step],
                                           [d.s_end for d in step], k, n_repl=[d.n_repl for d in step],
                                           mode=[d.mode for d in step])
        calls.append(dirs)
    torch.cuda.synchronize()  # the rows of R and the cache are written on the default stream
    pick = [torch.cuda.current_stream()] if streams == 1 else [torch.cuda.Stream(), torch.cuda.Stream()]
    for i, dirs in enumerate(calls):  # no synchronisation between calls
        cache.splice(dirs, pick[i % len(pick)])
        st = cache.last_stats()  # the library's account of its host time for this call
        assert st["host_ns"] >= st["resolve_ns"] + st["plan_ns"] and st["plan_ns"] > 0
        assert st["kernels_launched"] >= 3  # the plan copy, then the splice's own kernels
    torch.cuda.synchronize()
    cache.check_status()
    # the same calls one at a time, each checked against the oracle on its own input
    want = H.checked_sequential_run(w, flags=flags, slack_pages=64)
    for r in range(w.num_reqs):
        n = int(cache.seq_lens_host[r])
        assert n == want[r].shape[1]
        assert np.array_equal(H.logical_rows(cache, r, n), want[r]), f"request {r}: calls in flight differ"
    del keep
    cache.close()


# ------------------------------------------------------------------------------
# Calls that overlap: a rewrite call's move kernel may start before the calls still running
# end, when it rewrites none of their requests and takes no page they returned.  The
# schedule below mixes calls that qualify with calls that share a request with the window
# or need pages the window returned (a tight pool); the flag each call reports must follow
# that rule, and every request must end equal, bit for bit, to the same calls made one at
# a time with each checked against the oracle.
def _run_overlapping_calls(w: Workload, flags: int, kernel: str, slack: int, window_max: int = 8) -> list:
    """Enqueue every step of w with no synchronisation, check each call's overlap flag against
    the rule, and the final caches (eager pools: equal bit for bit to the same calls made one at
    a time, each checked against the oracle; lazy pools: the stored bits and counts, exactly
    against the oracle's slot maps).  Returns the flags."""
    import torch
    B = w.block_size
    lengths = list(w.lengths)
    steps = w.steps
    n_req = w.num_reqs
    cache = H.make_cache(w, slack_pages=slack, flags=flags)
    keep, flags_seen = [], []
    # the rule, restated: the window holds the calls since the last one that waited
    q_head = sum(-(-L // B) for L in lengths)
    q_tail = cache.num_pages
    window_tail, window_reqs, window_calls, window_open = 0, set(), 0, False
    want = []
    for step in steps:
        dirs, k = H.gpu_directives(w, step)
        keep.append(k)
        cache.splice(dirs)
        st = cache.last_stats()
        rq = {d.req for d in step}
        ok = (kernel == "vector" and window_open and window_calls < window_max and not (rq & window_reqs)
              and q_head + st["pages_popped"] <= window_tail)
        want.append(int(ok))
        flags_seen.append(st["overlapped"])
        if kernel != "vector":
            window_open = False
        elif not ok:
            window_open, window_calls, window_tail, window_reqs = True, 0, q_tail, set()
        window_calls += 1
        window_reqs |= rq
        q_head += st["pages_popped"]
        q_tail += st["pages_pushed"]
    torch.cuda.synchronize()
    cache.check_status()
    assert flags_seen == want, f"overlap flags {flags_seen} != rule {want}"
    if flags & LAZY:
        # a lazy pool stores bits and counts: both exact against the oracle's slot maps
        import test_gpu_lazy as TL
        st = TL.LazyState(w)
        lens_now = np.array(w.lengths, dtype=np.int64)
        for step in steps:
            st.apply(w, step, lens_now)
            lens_now = np.array([b.shape[1] for b in st.base], dtype=np.int64)
        for r in range(n_req):
            n = int(cache.seq_lens_host[r])
            assert n == st.base[r].shape[1]
            assert np.array_equal(TL._raw_rows(cache, r, n), st.base[r]), f"request {r}: stored bits differ"
            assert np.array_equal(TL._pending_of(cache, r, n), st.pend[r]), f"request {r}: counts differ"
        TL._check_free_pages_clear(cache)
        del keep
        cache.close()
        return flags_seen
    # the same calls one at a time, each checked against the oracle on its own input
    want_rows = H.checked_sequential_run(w, flags=flags, slack_pages=slack)
    for r in range(n_req):
        n = int(cache.seq_lens_host[r])
        assert n == want_rows[r].shape[1]
        assert np.array_equal(H.logical_rows(cache, r, n), want_rows[r]), f"request {r}: overlapping calls differ"
    del keep
    cache.close()
    return flags_seen


@pytest.mark.parametrize("flags,kernel", [(0, "vector"), (LAZY, "vector"), (SPLIT, "vector"), (0, "bulk")])
def test_consecutive_calls_overlap_only_when_safe(flags, kernel, monkeypatch):
    """A fixed schedule: pairs of requests in turn, every fifth call one request of the call
    before it, a tight pool.  The bulk (TMA) move kernel always waits for the calls before it."""
    monkeypatch.setenv("LEYLINE_MOVE_KERNEL", kernel)
    rng = np.random.default_rng(91)
    n_req, B = 12, 16
    lengths = [int(rng.integers(300, 700)) for _ in range(n_req)]
    lens = list(lengths)
    steps, key = [], 0
    for c in range(24):
        reqs = [(2 * c) % n_req, (2 * c + 1) % n_req] if c % 5 != 4 else [(2 * c - 1) % n_req]
        step = []
        for r in reqs:
            L = lens[r]
            s = int(rng.integers(0, L // 2))
            e = s + int(rng.integers(20, 120))
            n = int(rng.integers(0, 5))
            step.append(Dir(r, s, e, n, key))
            key += 1
            lens[r] = L + n - (e - s)
        steps.append(step)
    w = Workload(f"overlap-f{flags}", 2, B, lengths, steps, seed=92)
    seen = _run_overlapping_calls(w, flags, kernel, slack=4)
    if kernel == "vector":
        assert 0 < sum(seen) < len(steps), "the schedule should mix overlapped and waiting calls"


@pytest.mark.parametrize("seed", range(6))
def test_overlapping_calls_fuzz(seed, monkeypatch):
    """Random schedules: 30 calls of 1-2 random requests with 1-2 directives each (so every
    plan is a kernel parameter), random block sizes, pool slack and pool modes."""
    monkeypatch.setenv("LEYLINE_MOVE_KERNEL", "vector")
    rng = np.random.default_rng(1000 + seed)
    flags = [0, LAZY, SPLIT, LAZY | SPLIT][seed % 4]
    n_req = int(rng.integers(4, 14))
    B = int(rng.choice([1, 4, 16]))
    lengths = [int(rng.integers(200, 600)) for _ in range(n_req)]
    lens = list(lengths)
    steps, key = [], 0
    for _ in range(30):
        reqs = rng.choice(n_req, size=int(rng.integers(1, 3)), replace=False)
        step = []
        for r in sorted(int(x) for x in reqs):
            L = lens[r]
            k = int(rng.integers(1, 3))
            cuts = sorted(int(x) for x in rng.choice(np.arange(1, L), size=2 * k, replace=False))
            for j in range(k):
                s, e = cuts[2 * j], cuts[2 * j + 1]
                e = min(e, s + max(L // 6, 1))
                n = int(rng.integers(0, 7))
                step.append(Dir(r, s, e, n, key))
                key += 1
                L += n - (e - s)
            lens[r] = L
        steps.append(step)
    w = Workload(f"overlap-fuzz-{seed}", int(rng.integers(1, 3)), B, lengths, steps, seed=2000 + seed)
    _run_overlapping_calls(w, flags, "vector", slack=int(rng.integers(0, 40)))
