"""The full-size workloads on the GPU, through the C ABI (needs a GB300).

* batched: 8 requests, 27 layers, block 16, one directive each (one with Delta = +48);
* sweep: C in {1, 4, 8, 16} requests sharing a 61-layer pool, block 16 and block 1,
  1-3 directives per request;
* chain: 61 layers, 131072 tokens, block 1, 64 successive splices, with the drift of
  the fp32 and the bf16-only rotation against a from-scratch encoding at the final
  positions ("Leyline: KV Cache Directives for Agentic Inference", section 4.3).

At these sizes every row is checked on the device for the properties that hold at
any size (latents and unmoved rows bit-exact through the oracle's slot map, rows of
R bit-exact, RoPE pair norms preserved), and sampled rows -- every segment
boundary plus random ones -- are compared element by element with the oracle.
"""
import json
import os

import numpy as np
import pytest

import oracle
import splice_harness as H
import synth
from synth import configs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# the drift records are written where LEYLINE_RESULTS_DIR points (not written when unset)
OUT = os.environ.get("LEYLINE_RESULTS_DIR", "")


def _record(name: str, rec: dict) -> None:
    if OUT:
        os.makedirs(OUT, exist_ok=True)
        with open(os.path.join(OUT, name), "w") as f:
            json.dump(rec, f, indent=1)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rope_rotation_gb300
    rope_rotation_gb300.build()


def _release(cache):
    cache.close()
    del cache
    torch.cuda.empty_cache()


def _single_call(w, seed=0):
    cache = H.make_cache(w)
    before = cache.seq_lens_host.copy()
    dirs, keep = H.gpu_directives(w, w.steps[0])
    cache.splice(dirs)
    torch.cuda.synchronize()
    cache.check_status()
    stats = cache.last_stats()
    rng = np.random.default_rng(seed)
    samp = H.check_sampled_single_call(w, cache, w.steps[0], before, rng)
    rows = H.check_properties_all_rows(w, cache, w.steps[0], before)
    del keep
    _release(cache)
    return stats, samp, rows


def test_batched_c8():
    w = configs.batched_c8()
    stats, samp, rows = _single_call(w)
    assert stats["requests_touched"] == 8
    print("batched C8:", stats["downstream_slots"], "downstream slots;", samp, rows, "rows checked")


@pytest.mark.parametrize("B", [16, 1])
@pytest.mark.parametrize("C", [1, 4, 8, 16])
def test_sweep(C, B):
    w = configs.sweep(C, B)
    stats, samp, rows = _single_call(w, seed=C * 100 + B)
    print(f"sweep C{C} B{B}:", stats["downstream_slots"], "downstream slots;", samp, rows, "rows checked")


def _trace_back(maps, p_final):
    """Positions a final row held after each step, back to its origin.
    Returns (origin, positions) with origin ('old', t) or ('repl', step, directive row index);
    positions[j] is the position after step j for the steps since its birth."""
    pos = [p_final]
    p = p_final
    for k in range(len(maps) - 1, -1, -1):
        kind, idx = maps[k]
        if kind[p] == 1:
            return ("repl", k, int(idx[p])), pos[::-1]
        p = int(idx[p])
        pos.append(p)
    return ("old", p), pos[::-1]


def test_chain_64_drift():
    w = configs.chain_64()
    lat = w.latent_dim
    maps, L = [], w.lengths[0]
    for step in w.steps:
        d = step[0]
        L, kind, idx, _ = oracle.splice_map(L, [(d.s_start, d.s_end, d.n_repl)])
        maps.append((kind, idx))
    final_len = L
    rng = np.random.default_rng(64)
    pos = np.unique(np.concatenate([rng.integers(0, final_len, size=1200), [0, final_len - 1]]))
    layers = rng.integers(0, w.num_layers, size=pos.size)
    traces = [_trace_back(maps, int(p)) for p in pos]
    report = {"final_len": final_len, "rows": int(pos.size)}
    gpu_vals = {}
    for precision, name in ((0, "fp32"), (1, "bf16")):
        cache = H.make_cache(w, precision=precision)
        keep = []
        for step in w.steps:
            dirs, k = H.gpu_directives(w, step)
            keep.append(k)
            cache.splice(dirs)
        torch.cuda.synchronize()
        cache.check_status()
        assert int(cache.seq_lens_host[0]) == final_len
        got = H.fetch_rows(cache, 0, layers, pos)
        _release(cache)
        del keep
        chain_rows, truth_rows, moves = [], [], []
        for i, ((origin, path), layer) in enumerate(zip(traces, layers)):
            if origin[0] == "old":
                row = synth.cache_rows(w.seed, 0, int(layer), [origin[1]])[0]
                start = origin[1]
            else:
                _, k, ri = origin
                d = w.steps[k][0]
                row = synth.repl_rows(w.seed, 0, d.key, w.num_layers, d.n_repl)[layer, ri]
                start = path[0]
            assert np.array_equal(got[i, :lat], row[:lat]), "latent bits differ after the chain"
            v = row[lat:].copy()
            n = 0
            for a, b in zip(path[:-1], path[1:]):
                if a != b:
                    v = oracle.rerotate(v, a, b, w.theta) if precision == 0 else \
                        oracle.rotate_bf16only(v, b - a, w.theta)
                    n += 1
            chain_rows.append(v)
            truth_rows.append(oracle.rerotate(row[lat:], start, path[-1], w.theta))
            moves.append(n)
        chain = np.array(chain_rows)
        truth = np.array(truth_rows)
        moves = np.array(moves)
        g = oracle.bf16_value(got[:, lat:])
        c = oracle.bf16_value(chain)
        t = oracle.bf16_value(truth)
        if precision == 1:
            assert np.array_equal(got[:, lat:], chain), "bf16-only arm differs from the oracle's bf16-only chain"
        else:
            # Each step may round one element one bf16 step apart from the oracle's chain; the
            # difference of a pair then grows by at most 2^-6 of the pair norm per move.
            d = g - c
            dn = np.hypot(d[:, :32], d[:, 32:])
            pn = np.hypot(c[:, :32], c[:, 32:])
            assert np.all(dn <= moves[:, None] * 2.0 ** -6 * pn + 1e-30)
            report["fp32_vs_oracle_chain_rel_l2"] = float(np.linalg.norm(d) / np.linalg.norm(c))
        drift = float(np.linalg.norm(g - t) / np.linalg.norm(t))
        report[f"{name}_drift_rel_l2"] = drift
        report[f"{name}_oracle_chain_drift_rel_l2"] = float(np.linalg.norm(c - t) / np.linalg.norm(t))
        gpu_vals[name] = drift
    report["mean_moves"] = float(np.mean(moves))
    report["max_moves"] = int(np.max(moves))
    assert gpu_vals["fp32"] < gpu_vals["bf16"]
    assert gpu_vals["fp32"] < 2e-2
    _record("chain_drift.json", report)
    print("chain drift:", report)


def test_chain_64_lazy_drift():
    """The same 64-splice chain on a lazy pool (block 1, re-index): splices move bits and
    count turns, and each read turns the row once, so a read equals the from-scratch
    encoding at the final position within one rounding, however many splices moved it."""
    w = configs.chain_64()
    lat = w.latent_dim
    maps, L = [], w.lengths[0]
    for step in w.steps:
        d = step[0]
        L, kind, idx, _ = oracle.splice_map(L, [(d.s_start, d.s_end, d.n_repl)])
        maps.append((kind, idx))
    final_len = L
    rng = np.random.default_rng(65)
    pos = np.unique(np.concatenate([rng.integers(0, final_len, size=1200), [0, final_len - 1]]))
    layers = rng.integers(0, w.num_layers, size=pos.size)
    cache = H.make_cache(w, flags=2 | 1)
    keep = []
    for step in w.steps:
        dirs, k = H.gpu_directives(w, step)
        keep.append(k)
        cache.splice(dirs)
    torch.cuda.synchronize()
    cache.check_status()
    assert int(cache.seq_lens_host[0]) == final_len
    buf = torch.empty((1, cache.row), dtype=torch.bfloat16, device=cache.device)
    got = np.empty((pos.size, cache.row), dtype=np.uint16)
    for i, (p, layer) in enumerate(zip(pos, layers)):
        cache.gather(0, int(layer), int(p), int(p) + 1, buf)
        got[i] = buf.view(torch.int16).cpu().numpy().view(np.uint16)[0]
    stats = cache.last_stats()
    _release(cache)
    del keep
    truth, moved = [], []
    for i, p in enumerate(pos):
        origin, path = _trace_back(maps, int(p))
        layer = int(layers[i])
        if origin[0] == "old":
            row = synth.cache_rows(w.seed, 0, layer, [origin[1]])[0]
            start = origin[1]
        else:
            _, k, ri = origin
            d = w.steps[k][0]
            row = synth.repl_rows(w.seed, 0, d.key, w.num_layers, d.n_repl)[layer, ri]
            start = path[0]
        assert np.array_equal(got[i, :lat], row[:lat]), "latent bits differ after the chain"
        truth.append(oracle.rerotate(row[lat:], start, path[-1], w.theta))
        moved.append(start != path[-1])
    truth = np.array(truth)
    moved = np.array(moved)
    assert np.array_equal(got[~moved, lat:], truth[~moved])
    c = H.compare_kpe(got[moved, lat:], truth[moved], 0)
    g = oracle.bf16_value(got[:, lat:])
    t = oracle.bf16_value(truth)
    report = {"final_len": final_len, "rows": int(pos.size), "moved_rows": int(moved.sum()),
              "lazy_drift_rel_l2": float(np.linalg.norm(g - t) / np.linalg.norm(t)),
              "lazy_elements_off_by_floor_clause": c["floor_used"], "lazy_max_bf16_steps": c["max_steps"],
              "last_splice_algorithmic_bytes": int(stats["algorithmic_bytes"])}
    _record("chain_drift_lazy.json", report)
    print("lazy chain drift:", report)
    assert report["lazy_drift_rel_l2"] < 1e-3
