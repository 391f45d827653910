"""The C ABI on a machine without a GPU: the library loads, exports every function
include/leyline.h declares, and its host-only planner (leyline_splice_plan)
validates directives and computes lengths and work exactly as the oracle's
logical splice does ("Leyline: KV Cache Directives for Agentic Inference",
section 2.1: D = (s_start, s_end, R, m); section 2.2: Delta = |R| - |S|).
No call here touches a device.
"""
import json
import os
import re

import numpy as np
import pytest

import oracle
from synth import configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE_DEV_PTR = 0x7F0000001000  # aligned; the dry run never dereferences it


@pytest.fixture(scope="module")
def L():
    import rope_rotation_gb300
    from rope_rotation_gb300 import leyline
    rope_rotation_gb300.build()
    leyline.load()
    return leyline


def test_exports_every_declared_symbol(L):
    header = open(os.path.join(ROOT, "include", "leyline.h")).read()
    names = set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**\s*(leyline_\w+)\s*\(", header, re.M))
    assert len(names) >= 14
    lib = L.load()
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared but not exported"
    assert "sm_103a" in L.leyline_version()


def _d(L, req, s, e, n, mode=0, reserved=0, ptr=FAKE_DEV_PTR):
    return L.Directive(req, mode, s, e, n, reserved, ptr if n > 0 else None)


def _plan(L, lens, dirs, B=16, max_blocks=None, free=-1, desc=None):
    desc = desc or L.pool_desc(4, B, 1 << 20)
    if max_blocks is None:
        max_blocks = max(-(-(x + 200) // B) for x in lens)
    return L.leyline_splice_plan(desc, np.array(lens), max_blocks, dirs, free)


@pytest.mark.parametrize("case,code", [
    ("forget", -5), ("unknown_mode", -5), ("s_gt_e", -2), ("e_gt_len", -2), ("neg_s", -2), ("bad_req", -2),
    ("overlap", -3), ("shared_start", -3), ("neg_repl", -2), ("null_repl", -1), ("misaligned_repl", -1),
    ("reserved", -1), ("capacity", -7), ("no_pages", -4),
])
def test_validation_errors(L, case, code):
    lens = [100, 50]
    dirs = {
        "forget": [_d(L, 0, 1, 5, 0, mode=1)],
        "unknown_mode": [_d(L, 0, 1, 5, 0, mode=7)],
        "s_gt_e": [_d(L, 0, 9, 5, 0)],
        "e_gt_len": [_d(L, 1, 10, 51, 0)],
        "neg_s": [_d(L, 0, -1, 5, 0)],
        "bad_req": [_d(L, 2, 1, 5, 0)],
        "overlap": [_d(L, 0, 10, 20, 1), _d(L, 0, 15, 30, 1)],
        "shared_start": [_d(L, 0, 10, 10, 1), _d(L, 0, 10, 20, 1)],
        "neg_repl": [L.Directive(0, 0, 1, 5, -1, 0, None)],
        "null_repl": [L.Directive(0, 0, 1, 5, 3, 0, None)],
        "misaligned_repl": [L.Directive(0, 0, 1, 5, 3, 0, FAKE_DEV_PTR + 2)],
        "reserved": [_d(L, 0, 1, 5, 0, reserved=1)],
        "capacity": [_d(L, 1, 0, 0, 500)],
        "no_pages": [_d(L, 0, 0, 10, 3)],
    }[case]
    kw = {"max_blocks": 10} if case == "capacity" else {}
    if case == "no_pages":
        kw["free"] = 2
    with pytest.raises(L.LeylineError) as ei:
        _plan(L, lens, dirs, **kw)
    assert ei.value.code == code
    assert L.leyline_last_error()


def test_bad_descriptors(L):
    for kw in [dict(rope_dim=8), dict(latent_dim=7), dict(block_size=0), dict(rope_theta=0.0),
               dict(pair_layout=2), dict(rotate_precision=3), dict(num_layers=0)]:
        args = dict(num_layers=2, block_size=16, num_pages=100)
        args.update(kw)
        desc = L.pool_desc(**args)
        with pytest.raises(L.LeylineError) as ei:
            L.leyline_splice_plan(desc, np.array([10]), 8, [_d(L, 0, 1, 2, 0)])
        assert ei.value.code == -1


def _expected(lens, dirs_by_req, B):
    """Lengths, downstream slots, head slots and page counts from the oracle's logical splice."""
    out = {"len": list(lens), "down": 0, "head": 0, "repl": 0, "pop": 0, "push": 0}
    for r, dirs in dirs_by_req.items():
        eff = [d for d in dirs if not (d[0] == d[1] and d[2] == 0)]
        newlen, kind, idx, _ = oracle.splice_map(lens[r], dirs)
        out["len"][r] = newlen
        if not eff:
            continue
        first_end = min(d[1] for d in eff)
        s_min = min(d[0] for d in eff)
        out["down"] += int(((kind == 0) & (idx >= first_end)).sum())
        out["repl"] += sum(d[2] for d in eff)
        b0 = s_min // B
        out["head"] += s_min - b0 * B
        out["pop"] += -(-newlen // B) - b0
        out["push"] += -(-lens[r] // B) - b0
    return out


@pytest.mark.parametrize("B", [1, 2, 16])
def test_planner_matches_oracle_on_random_directives(L, B):
    rng = np.random.default_rng(B)
    for _ in range(300):
        lens = [int(x) for x in rng.integers(0, 200, size=int(rng.integers(1, 5)))]
        dirs_by_req, dirs = {}, []
        for r, Lr in enumerate(lens):
            k = int(rng.integers(0, 4))
            cuts = sorted(int(x) for x in rng.integers(0, Lr + 1, size=2 * k))
            ds = [(cuts[2 * i], cuts[2 * i + 1], int(rng.integers(0, 20))) for i in range(k)]
            if len({d[0] for d in ds}) != len(ds):
                continue
            if ds:
                dirs_by_req[r] = ds
                dirs += [_d(L, r, s, e, n) for s, e, n in ds]
        rng.shuffle(dirs)
        st, newlens = _plan(L, lens, dirs, B=B)
        want = _expected(lens, dirs_by_req, B)
        assert list(newlens) == want["len"]
        assert st.downstream_slots == want["down"]
        assert st.repl_slots == want["repl"]
        assert st.head_slots == want["head"]
        assert st.pages_popped == want["pop"]
        assert st.pages_pushed == want["push"]
        row_bytes = 2 * 576
        assert st.algorithmic_bytes == 2 * row_bytes * 4 * (want["down"] + want["repl"])


def test_planner_matches_golden_workloads(L):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "workloads.json")))
    for name, entry in g.items():
        w = configs.by_name(name)
        lens = list(w.lengths)
        desc = L.pool_desc(w.num_layers, w.block_size, 1 << 30)
        for step, want in zip(w.steps, entry["steps"]):
            dirs = [_d(L, d.req, d.s_start, d.s_end, d.n_repl) for d in step]
            st, newlens = L.leyline_splice_plan(desc, np.array(lens), max(-(-(x + 200) // w.block_size) for x in lens),
                                                dirs)
            assert st.downstream_slots == sum(x["downstream"] for x in want), name
            for x in want:
                assert newlens[x["req"]] == x["new_len"], name
            lens = [int(v) for v in newlens]


def test_noop_directives_touch_nothing(L):
    st, newlens = _plan(L, [64, 10], [_d(L, 0, 5, 5, 0), _d(L, 1, 10, 10, 0)])
    assert list(newlens) == [64, 10]
    assert st.requests_touched == 0 and st.kernels_launched == 0 and st.pages_popped == 0


def test_reindex_keeps_pages_of_runs_shifted_by_whole_blocks(L):
    """Re-index pools with 16-slot pages keep the page of every new block whose rows all come
    from one surviving run shifted by a multiple of 16 (that old block holds exactly those
    rows); every other new block gets a fresh page and every old block not kept is returned.
    A call whose fresh pages would take more survivor and prefix rows than the kept pages
    hold is rewritten instead (same page counts when nothing is kept).  Counts worked out by
    hand for a 163-token and a 64-token request."""
    desc = L.pool_desc(4, 16, 1 << 20, flags=L.LEYLINE_POOL_REINDEX)
    lens = [16 * 10 + 3, 64]
    cases = [  # directives, re-indexed, pages popped, pages pushed
        # Delta -16: blocks 3..9 kept (old 4..10), R in fresh block 2; request 1 keeps 0..2
        ([_d(L, 0, 32, 64, 16), _d(L, 1, 0, 16, 0)], 1, 1, 3),
        ([_d(L, 0, 48, 163, 5)], 1, 1, 8),                        # to the end: block 3 fresh
        # request 1: Delta -17 keeps nothing, its 47 survivors go to 3 fresh pages; request 0
        # keeps 99 rows, so the call is re-indexed
        ([_d(L, 0, 32, 64, 16), _d(L, 1, 0, 17, 0)], 1, 4, 6),
        ([_d(L, 0, 32, 64, 3)], 0, 7, 9),                         # Delta -29: nothing kept, rewritten
        ([_d(L, 0, 40, 64, 16)], 0, 8, 9),                        # Delta -8: nothing kept, rewritten
        ([_d(L, 0, 160, 160, 16)], 1, 1, 0),                      # the partial last block moves whole
        ([_d(L, 0, 163, 163, 16)], 0, 2, 1),                      # appended inside it: rewritten
        # Delta = 18 - 34 = -16 with s_start off the grid: blocks 1 and 2 get fresh pages (head
        # rows 16..19, rows of R, survivors 38..47), blocks 3..9 keep old blocks 4..10, old
        # blocks 1..3 are returned
        ([_d(L, 0, 20, 54, 18)], 1, 2, 3),
    ]
    for dirs, reindexed, pops, pushes in cases:
        st, new = _plan(L, lens, dirs, desc=desc)
        got = (st.reindexed, st.pages_popped, st.pages_pushed)
        assert got == (reindexed, pops, pushes), [(d.s_start, d.s_end, d.n_repl) for d in dirs]
    # block size 1: every row of R gets a fresh page, every dropped token returns one; three
    # launches (prep with the rows of R, the in-place rotation, commit)
    st, _ = _plan(L, [100], [_d(L, 0, 3, 50, 7)], B=1, desc=L.pool_desc(4, 1, 1 << 20, flags=L.LEYLINE_POOL_REINDEX))
    assert (st.reindexed, st.kernels_launched, st.pages_popped, st.pages_pushed) == (1, 3, 7, 47)
    # bytes: the 50 survivors' bands turned in place (2 x 128 bytes per layer) and 7 whole rows of
    # R written (2 x 1152 bytes per layer), 4 layers; the timed kernel is the rotation alone
    assert st.algorithmic_bytes == 2 * 4 * (128 * 50 + 1152 * 7)
    assert st.timed_kernel_bytes == 2 * 4 * 128 * 50
    # a rewrite times its move+rotate kernel, which moves all of the call's bytes
    st, _ = _plan(L, [100], [_d(L, 0, 3, 50, 7)], B=1, desc=L.pool_desc(4, 1, 1 << 20))
    assert st.kernels_launched == 2 and st.timed_kernel_bytes == st.algorithmic_bytes == 2 * 4 * 1152 * (50 + 7)


def test_binding_refuses_tensors_it_cannot_pass_as_rows(L):
    """The library reads raw bf16 rows: the binding refuses other dtypes, strided views and
    an R whose row count differs from n_repl (its layer stride is n_repl rows)."""
    import torch
    good = torch.zeros((2, 3, 576), dtype=torch.bfloat16)
    assert L.directive(0, 1, 2, good).n_repl == 3
    for bad, kw in [(torch.zeros((2, 3, 576), dtype=torch.float32), {}),
                    (torch.zeros((2, 576, 3), dtype=torch.bfloat16).transpose(1, 2), {}),
                    (good, {"n_repl": 2}),
                    (torch.zeros((3, 576), dtype=torch.bfloat16), {})]:
        with pytest.raises(ValueError):
            L.directive(0, 1, 2, bad, **kw)


def test_directive_batch_is_the_c_directive_array(L):
    """directive_batch() builds the same bytes as a C array of directive() results, and the
    planner returns the same work and lengths for either form."""
    import torch
    w = configs.by_name("cfg3")
    step = w.steps[0]
    R = {d.key: torch.zeros(2, d.n_repl, 576, dtype=torch.bfloat16) for d in step if d.n_repl}
    one = [L.directive(d.req, d.s_start, d.s_end, R.get(d.key), n_repl=d.n_repl) for d in step]
    batch = L.directive_batch([d.req for d in step], [d.s_start for d in step], [d.s_end for d in step],
                              [R.get(d.key) for d in step], n_repl=[d.n_repl for d in step])
    assert batch.tobytes() == bytes((L.Directive * len(one))(*one))
    desc = L.pool_desc(w.num_layers, w.block_size, 1 << 30)
    mb = max(-(-(x + 200) // w.block_size) for x in w.lengths)
    st1, len1 = L.leyline_splice_plan(desc, np.array(w.lengths), mb, one)
    st2, len2 = L.leyline_splice_plan(desc, np.array(w.lengths), mb, batch)
    assert st1.as_dict() == st2.as_dict() and list(len1) == list(len2)
    assert st1.downstream_slots > 0
    # fields edited in place between calls: the request ids of the next batch of requests
    moved = batch.copy()
    moved["req"] += 1
    st3, len3 = L.leyline_splice_plan(desc, np.array([0] + list(w.lengths)), mb, moved)
    assert st3.downstream_slots == st1.downstream_slots and list(len3[1:]) == list(len1)
    # modes broadcast; an empty batch is a no-op
    ev = L.directive_batch([0, 1], [5, 9], [7, 9], None, mode=L.LEYLINE_EVICT)
    assert list(ev["mode"]) == [L.LEYLINE_EVICT] * 2 and list(ev["n_repl"]) == [0, 0]
    st0, len0 = L.leyline_splice_plan(desc, np.array([30, 40]), 16, L.directive_batch([], [], []))
    assert st0.requests_touched == 0 and list(len0) == [30, 40]


def test_directive_batch_refusals(L):
    import torch
    with pytest.raises(ValueError):  # rows of R must be bf16
        L.directive_batch([0], [0], [1], [torch.zeros(2, 3, 576)])
    with pytest.raises(ValueError):  # exactly n_repl rows per layer
        L.directive_batch([0], [0], [1], [torch.zeros(2, 3, 576, dtype=torch.bfloat16)], n_repl=2)
    with pytest.raises(ValueError):  # one entry of repl per directive
        L.directive_batch([0, 1], [0, 0], [1, 1], [None])
    with pytest.raises(ValueError):  # contiguous rows only
        L.directive_batch([0], [0], [1], [torch.zeros(2, 576, 3, dtype=torch.bfloat16).transpose(1, 2)])
    good = L.directive_batch([0, 1, 0, 1], [0, 0, 2, 2], [1, 1, 3, 3])
    desc = L.pool_desc(4, 16, 1 << 20)
    same_size = np.zeros(2, dtype=[(f, "<i8") for f in "abcde"])  # 40 bytes, another record
    for bad in (good[::2], same_size, np.zeros(2, dtype=np.int64)):
        with pytest.raises(ValueError):
            L.leyline_splice_plan(desc, np.array([10, 10]), 8, bad)
