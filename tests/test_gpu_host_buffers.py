"""Caller buffers in pinned host memory (needs a GPU).

On a Grace host the GPU reaches pinned host memory over NVLink-C2C, so rows of R
and gather outputs may stay in host memory: the move kernel reads the rows of R
in place and the gather writes its rows in place, with no staging copy.  These
tests check that a splice fed from pinned host rows equals one fed from device
rows bit for bit, that a gather into pinned host memory equals one into device
memory, and that pageable host memory is refused before anything changes.
"""
import ctypes
import os

import numpy as np
import pytest

import splice_harness as H
from synth import fill as sfill
from synth.configs import Dir, Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rope_rotation_gb300
    rope_rotation_gb300.build()


STEPS = [[Dir(0, 40, 130, 9, 0), Dir(1, 5, 700, 3, 1), Dir(1, 800, 820, 64, 2)],
         [Dir(0, 0, 3, 5, 3), Dir(1, 100, 101, 30, 4, mode=2)]]


def _run(w, cache, host: bool):
    from rope_rotation_gb300 import leyline
    for step in w.steps:
        keep = []
        dirs = []
        for d in step:
            r = sfill.repl_tensor(w.seed, d.req, d.key, w.num_layers, d.n_repl, w.row_elems, "cuda") \
                if d.n_repl else None
            if r is not None and host:
                r = r.cpu().pin_memory()
            keep.append(r)
            dirs.append(leyline.directive(d.req, d.s_start, d.s_end, r, n_repl=d.n_repl, mode=d.mode))
        cache.splice(dirs)
        torch.cuda.synchronize()
        cache.check_status()
        del keep


@pytest.mark.parametrize("B,flags,kernel", [(16, 0, "vector"), (16, 0, "bulk"), (1, 1, "vector"), (16, 2, "vector")])
def test_host_repl_rows_match_device_rows(B, flags, kernel, monkeypatch):
    monkeypatch.setenv("LEYLINE_MOVE_KERNEL", kernel)
    w = Workload(f"host-R-B{B}-f{flags}", 3, B, [300, 1000], STEPS, seed=81)
    ref = H.make_cache(w, slack_pages=16, flags=flags)
    new = H.make_cache(w, slack_pages=16, flags=flags)
    _run(w, ref, host=False)
    _run(w, new, host=True)
    assert H.work_stats(ref) == H.work_stats(new)
    for r in range(w.num_reqs):
        n = int(ref.seq_lens_host[r])
        assert n == int(new.seq_lens_host[r])
        assert np.array_equal(H.logical_rows(ref, r, n), H.logical_rows(new, r, n))
    ref.close()
    new.close()


def test_gather_into_pinned_host_memory():
    w = Workload("host-gather", 2, 16, [777], [STEPS[0][:1]], seed=82)
    cache = H.make_cache(w)
    _run(w, cache, host=False)
    n = int(cache.seq_lens_host[0])
    dev = torch.empty((n, cache.row), dtype=torch.bfloat16, device="cuda")
    host = torch.empty((n, cache.row), dtype=torch.bfloat16).pin_memory()
    for layer in range(w.num_layers):
        cache.gather(0, layer, 0, n, dev)
        cache.gather(0, layer, 0, n, host)
        torch.cuda.synchronize()
        assert torch.equal(dev.cpu().view(torch.int16), host.view(torch.int16))
    cache.close()


def test_pageable_host_memory_is_refused():
    from rope_rotation_gb300 import leyline
    w = Workload("host-refuse", 1, 16, [500], [[]], seed=83)
    cache = H.make_cache(w)
    torch.cuda.synchronize()
    before = cache.table.cpu().numpy().copy()
    free = cache.free_pages()
    # 16-byte aligned pageable buffer (numpy), large enough for the rows it names
    buf = np.zeros(4 * cache.row * w.num_layers + 16, dtype=np.uint16)
    addr = buf.ctypes.data
    addr += (-addr) % 16
    d = leyline.Directive(0, 0, 10, 20, 4, 0, addr)
    with pytest.raises(leyline.LeylineError) as e:
        cache.splice([d])
    assert e.value.code == leyline.LEYLINE_ERR_INVALID_ARG and "pageable" in str(e.value)
    assert int(cache.seq_lens_host[0]) == 500 and cache.free_pages() == free
    assert np.array_equal(cache.table.cpu().numpy(), before)
    out = np.zeros(10 * cache.row + 16, dtype=np.uint16)
    oaddr = out.ctypes.data
    oaddr += (-oaddr) % 16
    lib = leyline.load()
    rc = lib.leyline_gather(cache.pool, ctypes.byref(cache.tables.bt), 0, 0, 0, 10, ctypes.c_void_p(oaddr), None)
    assert rc == leyline.LEYLINE_ERR_INVALID_ARG
    assert not out.any()
    cache.close()
