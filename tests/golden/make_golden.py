"""Writes tests/golden/workloads.json: per workload and request, the length before and after
the splice and each directive's shift Delta = |R| - |S| ("Leyline: KV Cache Directives for
Agentic Inference", section 2.2), as computed by the oracle's logical splice (section 2.1).

Calls only ``oracle`` and the shape generator ``synth.configs``.  Run from the repo root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from synth import configs  # noqa: E402

NAMES = ["cfg1", "cfg2", "cfg3", "cfg4", "cfg5-C1-B16", "cfg5-C4-B16", "cfg5-C8-B16", "cfg5-C16-B16"]


def main():
    out = {}
    for name in NAMES:
        w = configs.by_name(name)
        lengths = list(w.lengths)
        steps = []
        for step in w.steps:
            reqs = []
            for r in range(w.num_reqs):
                dirs = [(d.s_start, d.s_end, d.n_repl) for d in step if d.req == r]
                if not dirs:
                    continue
                newlen, kind, idx, _ = oracle.splice_map(lengths[r], dirs)
                first_end = min(d[1] for d in dirs)
                downstream = int(((kind == 0) & (idx >= first_end)).sum())
                reqs.append({"req": r, "len": lengths[r], "new_len": newlen,
                             "deltas": [n - (e - s) for s, e, n in sorted(dirs)],
                             "downstream": downstream})
                lengths[r] = newlen
            steps.append(reqs)
        out[name] = {"num_layers": w.num_layers, "block_size": w.block_size, "steps": steps}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "workloads.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)
        f.write("\n")
    print(path)


if __name__ == "__main__":
    main()
