"""Fill a paged cache on the GPU with the seeded synthetic rows of ``synth``.

The rows of request r, layer l, token t are ``base_rows(seed)[row_ids(seed, 0, r, l, t)]``;
the table of base rows is uploaded once and gathered on the device, then written
through the request's block table.  Only data movement: no arithmetic of the splice.
"""
from __future__ import annotations

import functools

import numpy as np

from . import STREAM_CACHE, base_rows, repl_rows, row_ids


@functools.lru_cache(maxsize=2)
def _base_on_device(seed: int, row_elems: int, device: str):
    import torch
    b = base_rows(seed, row_elems)
    return torch.from_numpy(b.view(np.int16).copy()).to(device).view(torch.bfloat16)


def fill_request(cache, seed: int, req: int, length: int) -> None:
    """Write the synthetic rows of request `req` (tokens 0..length-1, all layers) into `cache`
    (a rope_rotation_gb300.runtime.PagedCache whose table already maps the request)."""
    import torch
    base = _base_on_device(seed, cache.row, str(cache.device))
    slots = torch.from_numpy(cache.slot_index(req, np.arange(length))).to(cache.device)
    toks = np.arange(length)
    for layer in range(cache.num_layers):
        ids = torch.from_numpy(row_ids(seed, STREAM_CACHE, req, layer, toks)).to(cache.device)
        cache.write_layer_rows(layer, slots, base.index_select(0, ids))


def repl_tensor(seed: int, req: int, key: int, num_layers: int, n_repl: int, row_elems: int, device: str):
    """Replacement rows of one directive as a bf16 CUDA tensor [num_layers][n_repl][row]."""
    import torch
    r = repl_rows(seed, req, key, num_layers, n_repl, row_elems)
    return torch.from_numpy(r.view(np.int16).copy()).to(device).view(torch.bfloat16)
