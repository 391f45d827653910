"""Seeded synthetic inputs for the Leyline AMORTIZE splice.

This module is shared by the tests, the benchmark and the smoke check. It draws
bf16 cache rows, context lengths and directive spans, and nothing else: it holds
none of the splice's arithmetic (no rotation, no re-indexing, no shift).

Every draw is counter-based (splitmix64 of a key built from the seed and the
coordinates), so any row of any cache can be regenerated on its own, on any
machine, without replaying a sequential stream.

Cache rows.  The pages model the stored MLA key band k_pe as RoPE-rotated at its
position, with latent and k_pe values ~N(0,1).  A rotation of an isotropic
Gaussian pair is again an isotropic Gaussian pair, so the stored k_pe of a token
is drawn directly from N(0,1); the oracle treats R(-t) k_t as the token's
position-free vector.  To keep the generator cheap at tens of GB, rows are drawn
once into a table of ``BASE_ROWS`` rows of N(0,1) bf16 values, and row
(seed, stream, request, layer, token) is table row ``row_ids(...)``, a 64-bit hash
reduced modulo ``BASE_ROWS``.
"""
from __future__ import annotations

import functools

import numpy as np

BASE_ROWS = 16384
ROW_ELEMS = 576  # latent 512 + k_pe 64, bf16

STREAM_CACHE = 0  # rows of the resident cache
STREAM_REPL = 1  # replacement rows R of a directive

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(x: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser (Steele, Lea, Flood 2014) on a uint64 array; wraps mod 2**64."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _key(*parts: int) -> np.uint64:
    h = np.zeros(1, dtype=np.uint64)
    for p in parts:
        with np.errstate(over="ignore"):
            h = splitmix64(h ^ np.uint64(int(p) & 0xFFFFFFFFFFFFFFFF))
    return h[0]


def uniform01(keys: np.ndarray) -> np.ndarray:
    """53-bit uniform doubles in (0, 1) from uint64 hashes."""
    return ((keys >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


@functools.lru_cache(maxsize=4)
def base_rows(seed: int, row_elems: int = ROW_ELEMS, n_rows: int = BASE_ROWS) -> np.ndarray:
    """Table of ``n_rows`` rows of ``row_elems`` N(0,1) values as bf16 bits (uint16).

    Box-Muller on two counter-based uniforms per element.  The table is the only
    place where floating point enters the generator; both the GPU path and the
    oracle receive its bits, never its formula.
    """
    k = _key(seed, 0xB45E, row_elems, n_rows)
    n = n_rows * row_elems
    c = np.arange(n, dtype=np.uint64) * np.uint64(2)
    u1 = uniform01(splitmix64(c ^ k))
    u2 = uniform01(splitmix64((c + np.uint64(1)) ^ k))
    g = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    out = f32_to_bf16_bits(g.astype(np.float32)).reshape(n_rows, row_elems)
    out.setflags(write=False)
    return out


def row_ids(seed: int, stream: int, req: int, layer: int, tokens, n_rows: int = BASE_ROWS) -> np.ndarray:
    """Table row index for each token of (stream, request, layer); int64 in [0, n_rows)."""
    k = _key(seed, stream, req, layer)
    t = np.asarray(tokens, dtype=np.int64).astype(np.uint64)
    with np.errstate(over="ignore"):
        h = splitmix64((t * np.uint64(0xD1B54A32D192ED03)) ^ k)
    return (h % np.uint64(n_rows)).astype(np.int64)


def cache_rows(seed: int, req: int, layer: int, tokens, row_elems: int = ROW_ELEMS) -> np.ndarray:
    """bf16 bits [len(tokens)][row_elems] of the resident cache rows of one request/layer."""
    return base_rows(seed, row_elems)[row_ids(seed, STREAM_CACHE, req, layer, tokens)]


def repl_rows(seed: int, req: int, directive: int, num_layers: int, n_repl: int,
              row_elems: int = ROW_ELEMS) -> np.ndarray:
    """bf16 bits [num_layers][n_repl][row_elems] of a directive's replacement rows."""
    base = base_rows(seed, row_elems)
    out = np.empty((num_layers, n_repl, row_elems), dtype=np.uint16)
    for layer in range(num_layers):
        ids = row_ids(seed, STREAM_REPL, req * 4096 + directive, layer, np.arange(n_repl))
        out[layer] = base[ids]
    return out


def cache_request(seed: int, req: int, num_layers: int, length: int,
                  row_elems: int = ROW_ELEMS) -> np.ndarray:
    """bf16 bits [num_layers][length][row_elems]: the logical cache of one request."""
    out = np.empty((num_layers, length, row_elems), dtype=np.uint16)
    toks = np.arange(length)
    for layer in range(num_layers):
        out[layer] = cache_rows(seed, req, layer, toks, row_elems)
    return out


class Draw:
    """Counter-based integer / real draws for shapes (lengths, spans).  Stable across machines."""

    def __init__(self, seed: int, stream: int):
        self._k = _key(seed, 0x5EED, stream)
        self._i = 0

    def _next(self) -> np.uint64:
        self._i += 1
        return splitmix64(np.array([self._i], dtype=np.uint64) ^ self._k)[0]

    def integer(self, lo: int, hi: int) -> int:
        """Uniform integer in [lo, hi] (inclusive)."""
        if hi < lo:
            raise ValueError("empty range")
        return lo + int(self._next() % np.uint64(hi - lo + 1))

    def uniform(self) -> float:
        return float(uniform01(np.array([self._next()], dtype=np.uint64))[0])

    def normal(self) -> float:
        u1, u2 = self.uniform(), self.uniform()
        return float(np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2))
