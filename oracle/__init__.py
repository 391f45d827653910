"""Plain fp64 CPU oracle of the Leyline AMORTIZE splice.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The GPU
library never calls it and shares no code with it; it is what the GPU results
are checked against.

The arithmetic lives in ``leyline_oracle.c`` (fp64, compiled with gcc into
``oracle/_build/liboracle.so``); this module only marshals numpy arrays.  The
pure-Python brute force in ``brute.py`` pins it on tiny inputs.

Parity status of each function (what pins it, see ``tests/test_oracle_pins.py``):
  bf16_round       pinned: torch's float32->bf16 conversion, ties, subnormals, brute force
  rope             pinned: complex exponential, matrix exponential of the rotation
                   generator, the quarter-turn textbook case, closure, norms
  rerotate         pinned: closure (equals one rotation by p - t), identity at t == p, brute force
  rotate_bf16only  pinned: quarter-turn case (exact), identity at Delta = 0, error bound
  splice_map       pinned: list-slicing brute force, sequential application, length identity
  splice_request   pinned: brute force on tiny caches; with EVICT modes: pure moves when every
                   directive evicts, one composed call equals calls applied one after another
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "leyline_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math: IEEE semantics are the point)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                        "-ffp-contract=off", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.lo_bf16_value.argtypes = [ctypes.c_uint16]
            L.lo_bf16_value.restype = ctypes.c_double
            L.lo_bf16_round.argtypes = [ctypes.c_double]
            L.lo_bf16_round.restype = ctypes.c_uint16
            L.lo_bf16_round_array.argtypes = [_f64p, ctypes.c_int64, _u16p]
            L.lo_bf16_round_array.restype = None
            L.lo_bf16_value_array.argtypes = [_u16p, ctypes.c_int64, _f64p]
            L.lo_bf16_value_array.restype = None
            L.lo_theta_j.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double]
            L.lo_theta_j.restype = ctypes.c_double
            L.lo_rope.argtypes = [_f64p, ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int, _f64p]
            L.lo_rope.restype = None
            L.lo_rerotate.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int, _i64p, _i64p, ctypes.c_double,
                                      ctypes.c_int, _u16p]
            L.lo_rerotate.restype = None
            L.lo_rotate_bf16only.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int, _i64p, ctypes.c_double,
                                             ctypes.c_int, _u16p]
            L.lo_rotate_bf16only.restype = None
            L.lo_splice_map.argtypes = [ctypes.c_int64, ctypes.c_int32, _i64p, _i64p, _i32p, ctypes.c_int64,
                                        _i32p, _i64p, _i32p]
            L.lo_splice_map.restype = ctypes.c_int64
            L.lo_splice_request.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                            ctypes.c_int, _u16p, ctypes.c_int64, ctypes.c_int32, _i64p, _i64p,
                                            _i32p, ctypes.POINTER(_u16p), _u16p, ctypes.c_int64]
            L.lo_splice_request.restype = ctypes.c_int64
            L.lo_splice_request_modes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                  ctypes.c_int, _u16p, ctypes.c_int64, ctypes.c_int32, _i64p,
                                                  _i64p, _i32p, _i32p, ctypes.POINTER(_u16p), _u16p, ctypes.c_int64]
            L.lo_splice_request_modes.restype = ctypes.c_int64
            L.lo_splice_request_heads.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_double, ctypes.c_int, _u16p, ctypes.c_int64,
                                                  ctypes.c_int32, _i64p, _i64p, _i32p, _i32p, ctypes.POINTER(_u16p),
                                                  _u16p, ctypes.c_int64]
            L.lo_splice_request_heads.restype = ctypes.c_int64
            _lib = L
    return _lib


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def bf16_round(x) -> np.ndarray:
    """Nearest bf16 bits (uint16) of each double, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().lo_bf16_round_array(_p(x, _f64p), x.size, _p(out, _u16p))
    return out


def bf16_value(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    lib().lo_bf16_value_array(_p(h, _u16p), h.size, _p(out, _f64p))
    return out


def theta_j(j: int, d: int, theta: float) -> float:
    return lib().lo_theta_j(j, d, theta)


def rope(vec, pos: float, theta: float = 10000.0, layout: int = 0) -> np.ndarray:
    """R(pos) vec in fp64 for one band of width d."""
    v = np.ascontiguousarray(vec, dtype=np.float64)
    out = np.empty_like(v)
    lib().lo_rope(_p(v, _f64p), v.shape[0], float(pos), theta, layout, _p(out, _f64p))
    return out


def rerotate(kpe: np.ndarray, from_pos, to_pos, theta: float = 10000.0, layout: int = 0) -> np.ndarray:
    """Re-encode bf16 bands [n][d] stored at positions from_pos[n] at positions to_pos[n]."""
    k = np.ascontiguousarray(kpe, dtype=np.uint16)
    shape = k.shape
    k = k.reshape(-1, shape[-1])
    n, d = k.shape
    f = np.ascontiguousarray(np.broadcast_to(np.asarray(from_pos, dtype=np.int64), (n,)))
    t = np.ascontiguousarray(np.broadcast_to(np.asarray(to_pos, dtype=np.int64), (n,)))
    out = np.empty_like(k)
    lib().lo_rerotate(_p(k, _u16p), n, d, _p(f, _i64p), _p(t, _i64p), theta, layout, _p(out, _u16p))
    return out.reshape(shape)


def rotate_bf16only(kpe: np.ndarray, delta, theta: float = 10000.0, layout: int = 0) -> np.ndarray:
    """The naive all-bf16 delta-rotation of bf16 bands [n][d] by delta[n] positions."""
    k = np.ascontiguousarray(kpe, dtype=np.uint16)
    shape = k.shape
    k = k.reshape(-1, shape[-1])
    n, d = k.shape
    dl = np.ascontiguousarray(np.broadcast_to(np.asarray(delta, dtype=np.int64), (n,)))
    out = np.empty_like(k)
    lib().lo_rotate_bf16only(_p(k, _u16p), n, d, _p(dl, _i64p), theta, layout, _p(out, _u16p))
    return out.reshape(shape)


def splice_map(L: int, dirs, cap: int | None = None):
    """Logical splice of one request.

    dirs: iterable of (s_start, s_end, n_repl).  Returns (new_len, kind, idx, which):
    kind[p] == 0 -> new position p holds original token idx[p];
    kind[p] == 1 -> it holds row idx[p] of directive which[p]'s replacement rows.
    Raises ValueError on invalid / overlapping directives.
    """
    dirs = list(dirs)
    n = len(dirs)
    s = np.array([d[0] for d in dirs] or [0], dtype=np.int64)
    e = np.array([d[1] for d in dirs] or [0], dtype=np.int64)
    r = np.array([d[2] for d in dirs] or [0], dtype=np.int32)
    if cap is None:
        cap = L + int(sum(d[2] for d in dirs))
    cap = max(cap, 1)
    kind = np.empty(cap, dtype=np.int32)
    idx = np.empty(cap, dtype=np.int64)
    which = np.empty(cap, dtype=np.int32)
    newlen = lib().lo_splice_map(L, n, _p(s, _i64p), _p(e, _i64p), _p(r, _i32p), cap,
                                 _p(kind, _i32p), _p(idx, _i64p), _p(which, _i32p))
    if newlen < 0:
        raise ValueError("invalid directives")
    return int(newlen), kind[:newlen].copy(), idx[:newlen].copy(), which[:newlen].copy()


def splice_request(cache: np.ndarray, dirs, repl: list[np.ndarray], latent_dim: int = 512,
                   theta: float = 10000.0, layout: int = 0, modes=None, rope_heads: int = 1) -> np.ndarray:
    """Splice one request's logical cache bf16 [layers][L][row] -> [layers][L'][row].

    dirs: (s_start, s_end, n_repl) per directive; repl[k]: bf16 [layers][n_repl][row].
    modes: per directive, 0 = AMORTIZE (re-encode downstream tokens), 2 = EVICT (keep their
    positions); None = all AMORTIZE.
    rope_heads: the row ends in that many RoPE bands of equal width (GQA/MHA keys); 1 for MLA.
    """
    c = np.ascontiguousarray(cache, dtype=np.uint16)
    layers, L, row = c.shape
    rope_dim = (row - latent_dim) // rope_heads
    dirs = list(dirs)
    n = len(dirs)
    s = np.array([d[0] for d in dirs] or [0], dtype=np.int64)
    e = np.array([d[1] for d in dirs] or [0], dtype=np.int64)
    r = np.array([d[2] for d in dirs] or [0], dtype=np.int32)
    cap = max(L + int(sum(d[2] for d in dirs)), 1)
    reps = [np.ascontiguousarray(x, dtype=np.uint16) for x in repl]
    for k, x in enumerate(reps):
        if x.shape != (layers, dirs[k][2], row):
            raise ValueError("replacement rows must be [layers][n_repl][row]")
    ptrs = (_u16p * max(n, 1))(*[_p(x, _u16p) for x in reps])
    out = np.zeros((layers, cap, row), dtype=np.uint16)
    if rope_heads != 1:
        m = np.array(list(modes) if modes is not None else [0] * max(n, 1), dtype=np.int32)
        if m.size == 0:
            m = np.zeros(1, dtype=np.int32)
        newlen = lib().lo_splice_request_heads(layers, latent_dim, rope_dim, rope_heads, theta, layout,
                                               _p(c, _u16p), L, n, _p(s, _i64p), _p(e, _i64p), _p(r, _i32p),
                                               _p(m, _i32p), ptrs, _p(out, _u16p), cap)
    elif modes is None:
        newlen = lib().lo_splice_request(layers, latent_dim, rope_dim, theta, layout, _p(c, _u16p), L, n,
                                         _p(s, _i64p), _p(e, _i64p), _p(r, _i32p), ptrs, _p(out, _u16p), cap)
    else:
        m = np.array(list(modes) or [0], dtype=np.int32)
        newlen = lib().lo_splice_request_modes(layers, latent_dim, rope_dim, theta, layout, _p(c, _u16p), L, n,
                                               _p(s, _i64p), _p(e, _i64p), _p(r, _i32p), _p(m, _i32p), ptrs,
                                               _p(out, _u16p), cap)
    if newlen < 0:
        raise ValueError("invalid directives")
    return np.ascontiguousarray(out[:, :newlen])
