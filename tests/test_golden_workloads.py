"""The stored workload shapes (tests/golden/workloads.json, written by make_golden.py from the
oracle) still come out of the generator and the oracle, and the hand-derived numbers of the two
single-directive workloads hold: Delta = |R| - |S| ("Leyline: KV Cache Directives for Agentic
Inference", section 2.2)."""
import json
import os

import oracle
from synth import configs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "workloads.json")


def test_hand_derived_single_directive_numbers():
    g = json.load(open(GOLDEN))
    c1 = g["cfg1"]["steps"][0][0]
    assert (c1["deltas"], c1["new_len"], c1["downstream"]) == ([16 - 1024], 4096 - 1008, 4096 - 2048)
    c2 = g["cfg2"]["steps"][0][0]
    assert (c2["deltas"], c2["new_len"], c2["downstream"]) == ([12 - 6000], 32768 - 5988, 32768 - 26000)
    # batched workload: the forced request has |R| = 64 over a 16-token span
    assert g["cfg3"]["steps"][0][7]["deltas"] == [48]


def test_golden_regenerates():
    g = json.load(open(GOLDEN))
    for name, entry in g.items():
        w = configs.by_name(name)
        assert (w.num_layers, w.block_size) == (entry["num_layers"], entry["block_size"])
        lengths = list(w.lengths)
        for step, want in zip(w.steps, entry["steps"]):
            got = []
            for r in range(w.num_reqs):
                dirs = [(d.s_start, d.s_end, d.n_repl) for d in step if d.req == r]
                if not dirs:
                    continue
                newlen, kind, idx, _ = oracle.splice_map(lengths[r], dirs)
                first_end = min(d[1] for d in dirs)
                got.append({"req": r, "len": lengths[r], "new_len": newlen,
                            "deltas": [n - (e - s) for s, e, n in sorted(dirs)],
                            "downstream": int(((kind == 0) & (idx >= first_end)).sum())})
                lengths[r] = newlen
            assert got == want, name
