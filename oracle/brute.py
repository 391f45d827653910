"""Pure-Python brute force of the Leyline AMORTIZE splice for tiny caches.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  It pins the C oracle on tiny
inputs by taking a different route to the same definition:

* the splice is literal Python list slicing, ``old[:s] + R + old[e:]``, applied
  right to left ("Leyline: KV Cache Directives for Agentic Inference", section
  2.1, mode AMORTIZE);
* each RoPE pair is a complex number and R(p) multiplies pair j by
  ``exp(i * p * theta_j)`` (section 2.2: RoPE is a unitary rotation, so applying
  R(Delta) to R(i) x equals R(i + Delta) x);
* bf16 rounding works on the integer bit pattern of the double instead of on
  frexp / nearbyint.
"""
from __future__ import annotations

import cmath
import struct


def bf16_round(x: float) -> int:
    """Nearest bf16 (ties to even) of a double, from its IEEE bit pattern."""
    if x != x:
        return 0x7FC0
    bits = struct.unpack("<Q", struct.pack("<d", x))[0]
    sign = (bits >> 63) & 1
    exp = (bits >> 52) & 0x7FF
    frac = bits & ((1 << 52) - 1)
    if exp == 0x7FF:
        return (sign << 15) | 0x7F80
    if exp == 0:  # fp64 subnormal: far below half the smallest bf16 step
        return sign << 15
    mant = (1 << 52) | frac  # value = mant * 2**(exp - 1075)
    E = exp - 1023
    normal = E >= -126
    shift = 45 if normal else 942 - exp  # keep 8 significant bits, or steps of 2**-133
    if shift >= 64:
        return sign << 15
    q, rem = divmod(mant, 1 << shift)
    half = 1 << (shift - 1)
    if rem > half or (rem == half and (q & 1)):
        q += 1
    if not normal:
        return (sign << 15) | q  # q == 128 is the smallest normal, same bits
    if q == 256:
        q, E = 128, E + 1
    field = E + 127
    if field >= 255:
        return (sign << 15) | 0x7F80
    return (sign << 15) | (field << 7) | (q - 128)


def bf16_value(h: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (h & 0xFFFF) << 16))[0]


def _pairs(d: int, layout: int):
    for j in range(d // 2):
        yield (j, j, j + d // 2) if layout == 0 else (j, 2 * j, 2 * j + 1)


def rerotate(kpe: list[int], t: int, p: int, theta: float, layout: int = 0) -> list[int]:
    """bf16 band stored at position t, re-encoded at position p (one rounding)."""
    if t == p:
        return list(kpe)
    d = len(kpe)
    out = [0] * d
    for j, ix, iy in _pairs(d, layout):
        th = theta ** (-2.0 * j / d)
        z = complex(bf16_value(kpe[ix]), bf16_value(kpe[iy]))
        z = z * cmath.exp(-1j * t * th) * cmath.exp(1j * p * th)
        out[ix] = bf16_round(z.real)
        out[iy] = bf16_round(z.imag)
    return out


def splice(rows: list[list[int]], dirs: list[tuple[int, int, list[list[int]]]],
           latent_dim: int, theta: float, layout: int = 0, modes=None, rope_heads: int = 1) -> list[list[int]]:
    """Splice one layer of one request.

    rows: bf16 rows (latent then k_pe) at positions 0..L-1.
    dirs: (s_start, s_end, R rows) with non-overlapping spans in the pre-call coordinates.
    modes: per directive, 0 = AMORTIZE (a survivor is re-encoded at its new position),
    2 = EVICT (the KV-streams page's eviction: a survivor keeps its position).  With both,
    a survivor is re-encoded at its new position minus the shift of the EVICT spans left of it.
    rope_heads: the row ends in that many RoPE bands of equal width, each re-encoded alone.
    Returns the new rows: prefix and R copied, survivors re-encoded.
    """
    modes = list(modes) if modes is not None else [0] * len(dirs)
    items = [("old", t) for t in range(len(rows))]
    for k, (s, e, R) in sorted(enumerate(dirs), key=lambda kv: -kv[1][0]):
        items = items[:s] + [("repl", (k, i)) for i in range(len(R))] + items[e:]
    out = []
    for p, (kind, v) in enumerate(items):
        if kind == "repl":
            k, i = v
            out.append(list(dirs[k][2][i]))
        else:
            row = rows[v]
            # count the index shift that EVICT spans to the left contributed, and undo it
            evict_shift = sum(len(R) - (e - s) for (s, e, R), m in zip(dirs, modes) if m == 2 and e <= v)
            band = (len(row) - latent_dim) // rope_heads
            new_row = list(row[:latent_dim])
            for h in range(rope_heads):
                lo = latent_dim + h * band
                new_row += rerotate(row[lo:lo + band], v, p - evict_shift, theta, layout)
            out.append(new_row)
    return out
