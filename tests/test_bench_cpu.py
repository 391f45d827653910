"""The benchmark's bookkeeping, on the CPU: the code hash that decides whether stored ncu
traffic still describes a kernel, the stored entries themselves, and the whole-job value."""
import os
import shutil

import pytest

import bench
from synth import configs


def _copy_sources(tmp_path):
    src = os.path.join(bench.ROOT, "rope_rotation_gb300", "csrc")
    dst = tmp_path / "rope_rotation_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in bench.KERNEL_COMMON + tuple(bench.KERNEL_FILES.values()):
        shutil.copy(os.path.join(src, name), dst / name)
    return dst


def test_kernel_hash_follows_code_not_comments(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = {k: bench.kernel_sha(k) for k in bench.KERNEL_FILES}
    # a comment, and a change of blank space, leave every hash alone
    move = dst / bench.KERNEL_FILES["move_rotate"]
    move.write_text(move.read_text() + "\n// a note\n/* and a block\n comment */\n\n")
    assert {k: bench.kernel_sha(k) for k in bench.KERNEL_FILES} == base
    # code in one kernel's own file changes that kernel's hash only
    move.write_text(move.read_text() + "\nnamespace { int unused_probe = 1; }\n")
    after = {k: bench.kernel_sha(k) for k in bench.KERNEL_FILES}
    assert after["move_rotate"] != base["move_rotate"]
    assert after["rotate_in_place"] == base["rotate_in_place"] and after["materialize"] == base["materialize"]
    # code in a shared header changes every hash
    hdr = dst / bench.KERNEL_COMMON[0]
    hdr.write_text(hdr.read_text() + "\nnamespace { int unused_probe_2 = 2; }\n")
    assert all(bench.kernel_sha(k) != after[k] for k in bench.KERNEL_FILES)


def test_stored_traffic_names_real_workloads_and_kernels():
    layers = {w.name: w.num_layers for w in (configs.by_name(n) for n in (
        "cfg1", "cfg2", "cfg3", "cfg5-C4-B1", "cfg5-C16-B1", "cfg5-C16-B16"))}
    for (workload, kernel), entry in bench.NCU_TRAFFIC.items():
        base = workload.split("-as-")[0]
        assert base in layers, workload
        assert kernel in ("move_rotate_vector", "rotate_in_place", "materialize"), kernel
        assert len(entry["kernel_sha256"]) == 64 and entry["bytes"] > 0
        if "scale" in entry:  # captured on fewer layers: scaled by the units of a full launch
            assert entry["scale"] == pytest.approx(layers[base] / entry["captured_layers"])


def test_resident_copies_and_units():
    # copies: one per step of a leg when they fit, at least one
    assert bench.resident_copies(10 ** 9, 25, 96.0) == 25
    assert bench.resident_copies(40 * 10 ** 9, 25, 96.0) == 2
    assert bench.resident_copies(200 * 10 ** 9, 25, 96.0) == 1
    # the CPU baseline's sample: layer-major units, every request in it, within the budget
    w = configs.by_name("cfg5-C4-B16")
    units, down = bench.oracle_units(w)
    assert len(units) == 4 * w.num_layers and sum(u[2] for u in units) == pytest.approx(down)
    pick = bench.parallel_units(units, rate_1=1e5, budget_core_s=0.0)
    assert len(pick) == 4 and {u[0] for u in pick} == {0, 1, 2, 3} and {u[1] for u in pick} == {0}
    assert len(bench.parallel_units(units, rate_1=1e12, budget_core_s=1.0)) == len(units)
    # cut to a multiple of the processes: 244 units over 16 processes -> 240
    assert len(bench.parallel_units(units, rate_1=1e12, budget_core_s=1.0, procs=16)) == 240
    assert len(bench.parallel_units(units, rate_1=1e5, budget_core_s=0.0, procs=16)) == 4  # fewer units than procs


def test_job_value_is_all_ranks_over_the_slowest():
    # 2 ranks x 10 steps x 1000 slots in 4 ms (the slowest rank) = 5M slots/s
    assert bench.job_value(1000, 10, 2, 4.0) == pytest.approx(5e6)
