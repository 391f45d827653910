"""Thin ctypes binding of libleyline.so (C ABI in include/leyline.h).

Argument marshalling only: every step of the splice runs in the library's CUDA
kernels.  Functions carry the C names and raise ``LeylineError`` on a negative
return code.  Device buffers are torch CUDA tensors (PyTorch provides device
memory and streams); the library borrows their pointers.

If the library is not built, importing works but the first call raises: there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from . import _build

LEYLINE_OK = 0
LEYLINE_ERR_INVALID_ARG = -1
LEYLINE_ERR_INVALID_DIRECTIVE = -2
LEYLINE_ERR_OVERLAP = -3
LEYLINE_ERR_NO_PAGES = -4
LEYLINE_ERR_UNSUPPORTED_MODE = -5
LEYLINE_ERR_CUDA = -6
LEYLINE_ERR_CAPACITY = -7
LEYLINE_ERR_DEVICE_CHECK = -8
LEYLINE_ERR_SCRATCH = -9

LEYLINE_PAIRS_HALF_SPLIT = 0
LEYLINE_PAIRS_INTERLEAVED = 1
LEYLINE_ROTATE_FP32 = 0
LEYLINE_ROTATE_BF16_NAIVE = 1
LEYLINE_AMORTIZE = 0
LEYLINE_FORGET = 1
LEYLINE_EVICT = 2
LEYLINE_POOL_REINDEX = 1
LEYLINE_POOL_LAZY = 2
LEYLINE_POOL_SPLIT_ROPE = 4
LEYLINE_ROLLBACK_ACCEPT_TURNED = 1


class LeylineError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"leyline error {code}: {msg}")
        self.code = code


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("latent_dim", ctypes.c_int32), ("rope_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_pages", ctypes.c_int64), ("rope_theta", ctypes.c_double),
                ("pair_layout", ctypes.c_int32), ("rotate_precision", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("rope_heads", ctypes.c_int32)]

    @property
    def row_elems(self) -> int:
        return self.latent_dim + max(self.rope_heads, 1) * self.rope_dim


class BlockTable(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("seq_lens_dev", ctypes.c_void_p), ("seq_lens_host", ctypes.c_void_p),
                ("num_reqs", ctypes.c_int32), ("max_blocks", ctypes.c_int32)]


class Directive(ctypes.Structure):
    _fields_ = [("req", ctypes.c_int32), ("mode", ctypes.c_int32), ("s_start", ctypes.c_int64),
                ("s_end", ctypes.c_int64), ("n_repl", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("repl_rows", ctypes.c_void_p)]


class Stats(ctypes.Structure):
    _fields_ = [("downstream_slots", ctypes.c_int64), ("repl_slots", ctypes.c_int64),
                ("head_slots", ctypes.c_int64), ("algorithmic_bytes", ctypes.c_int64),
                ("moved_bytes", ctypes.c_int64), ("pages_popped", ctypes.c_int64),
                ("pages_pushed", ctypes.c_int64), ("requests_touched", ctypes.c_int32),
                ("kernels_launched", ctypes.c_int32), ("reindexed", ctypes.c_int32),
                ("overlapped", ctypes.c_int32), ("host_ns", ctypes.c_int64), ("resolve_ns", ctypes.c_int64),
                ("plan_ns", ctypes.c_int64), ("timed_kernel_bytes", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_vp = ctypes.c_void_p
_SIGNATURES = {
    "leyline_pool_create": (ctypes.c_int, [ctypes.POINTER(PoolDesc), _vp, ctypes.POINTER(_vp)]),
    "leyline_pool_destroy": (ctypes.c_int, [_vp]),
    "leyline_alloc_pages": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "leyline_free_pages": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "leyline_free_page_count": (ctypes.c_int64, [_vp]),
    "leyline_pool_checkpoint": (ctypes.c_int, [_vp, _vp]),
    "leyline_pool_rollback": (ctypes.c_int, [_vp, ctypes.c_int32, _vp]),
    # the directives go in as a plain address: a ctypes array of Directive or a
    # DIRECTIVE_DTYPE record array (its data pointer)
    "leyline_splice": (ctypes.c_int, [_vp, ctypes.POINTER(BlockTable), _vp, ctypes.c_int32, _vp]),
    "leyline_splice_noalloc": (ctypes.c_int, [_vp, ctypes.POINTER(BlockTable), _vp, ctypes.c_int32, _vp]),
    "leyline_splice_plan": (ctypes.c_int, [ctypes.POINTER(PoolDesc), ctypes.POINTER(ctypes.c_int64), ctypes.c_int32,
                                           ctypes.c_int32, _vp, ctypes.c_int32, ctypes.c_int64,
                                           ctypes.POINTER(Stats), ctypes.POINTER(ctypes.c_int64)]),
    "leyline_last_stats": (ctypes.c_int, [_vp, ctypes.POINTER(Stats)]),
    "leyline_gather": (ctypes.c_int, [_vp, ctypes.POINTER(BlockTable), ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int64, ctypes.c_int64, _vp, _vp]),
    "leyline_materialize": (ctypes.c_int, [_vp, ctypes.POINTER(BlockTable), ctypes.c_int32, _vp]),
    "leyline_materialize_requests": (ctypes.c_int, [_vp, ctypes.POINTER(BlockTable), ctypes.POINTER(ctypes.c_int32),
                                                    ctypes.c_int32, _vp]),
    "leyline_pending_ptr": (ctypes.c_void_p, [_vp]),
    "leyline_sync_status": (ctypes.c_int, [_vp]),
    "leyline_kernel_timing_enable": (ctypes.c_int, [_vp, ctypes.c_int32]),
    "leyline_kernel_timing_read": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_double),
                                                  ctypes.POINTER(ctypes.c_int32)]),
    "leyline_last_error": (ctypes.c_char_p, []),
    "leyline_version": (ctypes.c_char_p, []),
}

_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libleyline.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with rope_rotation_gb300.build() "
                               "(the splice runs only in its CUDA kernels)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(rc: int) -> None:
    if rc < 0:
        msg = load().leyline_last_error().decode(errors="replace")
        raise LeylineError(rc, msg)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _tensor_ptr(t) -> int:
    return int(t.data_ptr())


def _rows_ptr(t, what: str, rows: Optional[int] = None) -> int:
    """Address of a contiguous bf16 tensor of whole rows; refuses other dtypes and strided views
    (the library reads raw bytes, so those would be read as something else)."""
    import torch
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{what}: dtype {t.dtype}, expected torch.bfloat16")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    if rows is not None and t.numel() < rows:
        raise ValueError(f"{what}: {t.numel()} elements, need {rows}")
    return int(t.data_ptr())


# ------------------------------------------------------------------ pool ----

def pool_desc(num_layers: int, block_size: int, num_pages: int, latent_dim: int = 512, rope_dim: int = 64,
              rope_theta: float = 10000.0, pair_layout: int = LEYLINE_PAIRS_HALF_SPLIT,
              rotate_precision: int = LEYLINE_ROTATE_FP32, flags: int = 0, rope_heads: int = 1) -> PoolDesc:
    return PoolDesc(num_layers, latent_dim, rope_dim, block_size, num_pages, rope_theta, pair_layout,
                    rotate_precision, flags, rope_heads)


def leyline_pool_create(desc: PoolDesc, kv) -> ctypes.c_void_p:
    """kv: torch bf16 CUDA tensor with num_layers*num_pages*block_size*row elements."""
    need = desc.num_layers * desc.num_pages * desc.block_size * desc.row_elems
    if kv.numel() != need or kv.element_size() != 2 or not kv.is_cuda or not kv.is_contiguous():
        raise LeylineError(LEYLINE_ERR_INVALID_ARG, "kv must be a contiguous 2-byte CUDA tensor of the pool's size")
    h = ctypes.c_void_p()
    _check(load().leyline_pool_create(ctypes.byref(desc), _tensor_ptr(kv), ctypes.byref(h)))
    return h


def leyline_pool_destroy(pool) -> None:
    _check(load().leyline_pool_destroy(pool))


def leyline_alloc_pages(pool, n: int) -> np.ndarray:
    ids = np.empty(max(n, 1), dtype=np.int32)
    _check(load().leyline_alloc_pages(pool, n, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
    return ids[:n]


def leyline_free_pages(pool, ids) -> None:
    a = np.ascontiguousarray(ids, dtype=np.int32)
    _check(load().leyline_free_pages(pool, a.size, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))


def leyline_free_page_count(pool) -> int:
    n = load().leyline_free_page_count(pool)
    _check(int(n) if n < 0 else 0)
    return int(n)


def leyline_pool_checkpoint(pool, stream=None) -> None:
    """Save the pool's page accounting (free-page list, positions, lazy counts) on the device."""
    _check(load().leyline_pool_checkpoint(pool, _stream_ptr(stream)))


def leyline_pool_rollback(pool, flags: int = 0, stream=None) -> None:
    """Restore the accounting saved by the last checkpoint; the caller restores its tables."""
    _check(load().leyline_pool_rollback(pool, flags, _stream_ptr(stream)))


# ----------------------------------------------------------- block table ----

class Tables:
    """Keeps the tensors behind a BlockTable alive: table int32 [R][max_blocks] and seq_lens
    int32 [R] on the device, and the int64 host mirror of the lengths."""

    def __init__(self, table, seq_lens_dev, seq_lens_host: np.ndarray):
        self.table = table
        self.seq_lens_dev = seq_lens_dev
        self.seq_lens_host = np.ascontiguousarray(seq_lens_host, dtype=np.int64)
        self.bt = BlockTable(_tensor_ptr(table), _tensor_ptr(seq_lens_dev), self.seq_lens_host.ctypes.data,
                             int(table.shape[0]), int(table.shape[1]))


def _repl_ptr(repl, n_repl: Optional[int]):
    """(n_repl, address) of a directive's rows of R, checked as the library will read them."""
    if repl is None:
        return (0 if n_repl is None else n_repl), None
    shape = repl.shape
    if n_repl is None:
        n_repl = int(shape[1]) if len(shape) == 3 else -1
    if len(shape) != 3 or int(shape[1]) < n_repl:
        raise ValueError(f"repl: shape {tuple(shape)}, expected [num_layers][>= {n_repl}][row]")
    if int(shape[1]) != n_repl:
        raise ValueError(f"repl: {int(shape[1])} rows per layer but n_repl = {n_repl}; the layer stride "
                         "of R is n_repl rows, so pass R with exactly n_repl rows per layer")
    return n_repl, _rows_ptr(repl, "repl")


def directive(req: int, s_start: int, s_end: int, repl=None, n_repl: Optional[int] = None,
              mode: int = LEYLINE_AMORTIZE) -> Directive:
    """repl: bf16 tensor [num_layers][n_repl][row], contiguous, on the pool's GPU or in pinned host
    memory (read in place by the kernel), or None."""
    n_repl, ptr = _repl_ptr(repl, n_repl)
    return Directive(req, mode, s_start, s_end, n_repl, 0, ptr)


# leyline_directive_t as a numpy record: a structured array of it is a C array of
# directives, which the splice calls take without per-element marshalling.
DIRECTIVE_DTYPE = np.dtype([("req", "<i4"), ("mode", "<i4"), ("s_start", "<i8"), ("s_end", "<i8"),
                            ("n_repl", "<i4"), ("reserved", "<i4"), ("repl_rows", "<u8")], align=True)
assert DIRECTIVE_DTYPE.itemsize == ctypes.sizeof(Directive)
assert all(DIRECTIVE_DTYPE.fields[n][1] == getattr(Directive, n).offset for n, _ in Directive._fields_)


def directive_batch(req, s_start, s_end, repl: Optional[Sequence] = None, n_repl=None,
                    mode=LEYLINE_AMORTIZE) -> np.ndarray:
    """Many directives at once: req, s_start, s_end (and n_repl, mode) are equal-length
    sequences or scalars; repl is a sequence of tensors or None, checked as directive()
    checks one.  Returns a structured array of DIRECTIVE_DTYPE that the splice calls take
    as is; its fields can be changed in place (numpy) between calls."""
    req = np.atleast_1d(np.asarray(req, dtype=np.int64))
    n = req.size
    out = np.zeros(n, dtype=DIRECTIVE_DTYPE)
    out["req"] = req
    out["s_start"] = np.broadcast_to(np.asarray(s_start, dtype=np.int64), n)
    out["s_end"] = np.broadcast_to(np.asarray(s_end, dtype=np.int64), n)
    out["mode"] = np.broadcast_to(np.asarray(mode, dtype=np.int64), n)
    rows = [None] * n if repl is None else list(repl)
    if len(rows) != n:
        raise ValueError(f"repl: {len(rows)} entries for {n} directives")
    counts = [None] * n if n_repl is None else [int(c) for c in np.broadcast_to(np.asarray(n_repl), n)]
    checked = [_repl_ptr(t, c) for t, c in zip(rows, counts)]
    out["n_repl"] = [c for c, _ in checked]
    out["repl_rows"] = [p or 0 for _, p in checked]
    return out


def _dir_array(dirs):
    """(address argument, count) for a sequence of Directive or a DIRECTIVE_DTYPE array; the
    caller keeps `dirs` alive for the call."""
    if isinstance(dirs, np.ndarray):
        if dirs.dtype != DIRECTIVE_DTYPE or dirs.ndim != 1 or not dirs.flags.c_contiguous:
            raise ValueError("directive arrays must be 1-D, contiguous and of DIRECTIVE_DTYPE")
        if dirs.size == 0:
            return (Directive * 1)(), 0
        return dirs.ctypes.data, int(dirs.size)
    return (Directive * max(len(dirs), 1))(*dirs), len(dirs)


# ---------------------------------------------------------------- splice ----

def leyline_splice(pool, tables: Tables, dirs, stream=None) -> None:
    """dirs: a sequence of Directive (directive()) or a DIRECTIVE_DTYPE array (directive_batch())."""
    arr, n = _dir_array(dirs)
    _check(load().leyline_splice(pool, ctypes.byref(tables.bt), arr, n, _stream_ptr(stream)))


def leyline_splice_noalloc(pool, tables: Tables, dirs, stream=None) -> None:
    """leyline_splice with its scratch in the library's static device array (no allocation)."""
    arr, n = _dir_array(dirs)
    _check(load().leyline_splice_noalloc(pool, ctypes.byref(tables.bt), arr, n, _stream_ptr(stream)))


def leyline_splice_plan(desc: PoolDesc, seq_lens_host, max_blocks: int, dirs: Sequence[Directive],
                        free_pages: int = -1):
    """Host-only dry run: returns (Stats, new lengths as int64 array)."""
    lens = np.ascontiguousarray(seq_lens_host, dtype=np.int64)
    out = np.empty(max(lens.size, 1), dtype=np.int64)
    st = Stats()
    arr, n = _dir_array(dirs)
    p64 = ctypes.POINTER(ctypes.c_int64)
    _check(load().leyline_splice_plan(ctypes.byref(desc), lens.ctypes.data_as(p64), lens.size, max_blocks, arr,
                                      n, free_pages, ctypes.byref(st), out.ctypes.data_as(p64)))
    return st, out[:lens.size]


def leyline_last_stats(pool) -> Stats:
    st = Stats()
    _check(load().leyline_last_stats(pool, ctypes.byref(st)))
    return st


def leyline_gather(pool, tables: Tables, req: int, layer: int, t0: int, t1: int, out, stream=None) -> None:
    """out: contiguous bf16 tensor of at least (t1 - t0) rows, on the pool's GPU or in pinned host memory."""
    ptr = _rows_ptr(out, "out") if t1 > t0 else _tensor_ptr(out)
    _check(load().leyline_gather(pool, ctypes.byref(tables.bt), req, layer, t0, t1, ptr, _stream_ptr(stream)))


def leyline_materialize(pool, tables: Tables, req: int, stream=None) -> None:
    _check(load().leyline_materialize(pool, ctypes.byref(tables.bt), req, _stream_ptr(stream)))


def leyline_materialize_requests(pool, tables: Tables, reqs, stream=None) -> None:
    """leyline_materialize for several distinct requests, in one launch per 64 of them."""
    a = np.ascontiguousarray(reqs, dtype=np.int32)
    _check(load().leyline_materialize_requests(pool, ctypes.byref(tables.bt),
                                               a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), a.size,
                                               _stream_ptr(stream)))


def leyline_pending_ptr(pool) -> int:
    """Device address of the pending counts (0 when the pool is not lazy)."""
    return load().leyline_pending_ptr(pool) or 0


def leyline_sync_status(pool) -> None:
    _check(load().leyline_sync_status(pool))


def leyline_kernel_timing_enable(pool, enable: bool = True) -> None:
    _check(load().leyline_kernel_timing_enable(pool, 1 if enable else 0))


def leyline_kernel_timing_read(pool):
    ms = ctypes.c_double()
    n = ctypes.c_int32()
    _check(load().leyline_kernel_timing_read(pool, ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def leyline_last_error() -> str:
    return load().leyline_last_error().decode(errors="replace")


def leyline_version() -> str:
    return load().leyline_version().decode()
