"""A paged MLA KV cache in torch device memory, driven through libleyline.so.

Plumbing for callers: it allocates the pool tensor (layout
``kv[layer][page][slot][latent + rope]``, bf16; with LEYLINE_POOL_SPLIT_ROPE the
latents ``[layer][page][slot][latent]`` followed by the rope bands
``[layer][page][slot][rope]``), the block table and the length arrays, takes pages
for new requests, and forwards splices and gathers to the C ABI.  It computes
nothing itself.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

from . import leyline


class _DeviceArray:
    """int32 device memory owned by the pool, exposed through __cuda_array_interface__."""

    def __init__(self, addr: int, n: int, device: int):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (addr, False), "version": 3}
        self.device = device


class PagedCache:
    def __init__(self, num_layers: int, block_size: int, num_pages: int, max_reqs: int, max_blocks: int,
                 latent_dim: int = 512, rope_dim: int = 64, rope_theta: float = 10000.0,
                 pair_layout: int = leyline.LEYLINE_PAIRS_HALF_SPLIT,
                 rotate_precision: int = leyline.LEYLINE_ROTATE_FP32, flags: int = 0, rope_heads: int = 1,
                 device: str = "cuda"):
        import torch
        self.torch = torch
        self.num_layers = num_layers
        self.block_size = block_size
        self.num_pages = num_pages
        self.latent_dim = latent_dim
        self.rope_dim = rope_dim
        self.rope_heads = max(rope_heads, 1)
        self.row = latent_dim + self.rope_heads * rope_dim
        self.device = torch.device(device)
        self.kv = torch.empty(num_layers * num_pages * block_size * self.row, dtype=torch.bfloat16,
                              device=self.device)
        self.desc = leyline.pool_desc(num_layers, block_size, num_pages, latent_dim, rope_dim, rope_theta,
                                      pair_layout, rotate_precision, flags, rope_heads)
        self.pool = leyline.leyline_pool_create(self.desc, self.kv)
        self.table = torch.full((max_reqs, max_blocks), -1, dtype=torch.int32, device=self.device)
        self.seq_lens_dev = torch.zeros(max_reqs, dtype=torch.int32, device=self.device)
        self.tables = leyline.Tables(self.table, self.seq_lens_dev, np.zeros(max_reqs, dtype=np.int64))

    # ------------------------------------------------------------------
    @property
    def seq_lens_host(self) -> np.ndarray:
        return self.tables.seq_lens_host

    @property
    def split(self) -> bool:
        return bool(self.desc.flags & leyline.LEYLINE_POOL_SPLIT_ROPE)

    def kv_view(self):
        """[layers][pages][block_size][row] view of a pool of whole rows."""
        if self.split:
            raise ValueError("a split-rope pool has no array of whole rows: use latent_view / rope_view")
        return self.kv.view(self.num_layers, self.num_pages, self.block_size, self.row)

    def latent_view(self):
        """[layers][pages][block_size][latent] view of the latents."""
        if not self.split:
            return self.kv_view()[..., :self.latent_dim]
        n = self.num_layers * self.num_pages * self.block_size * self.latent_dim
        return self.kv[:n].view(self.num_layers, self.num_pages, self.block_size, self.latent_dim)

    def rope_view(self):
        """[layers][pages][block_size][rope_heads * rope_dim] view of the rope bands."""
        if not self.split:
            return self.kv_view()[..., self.latent_dim:]
        n = self.num_layers * self.num_pages * self.block_size * self.latent_dim
        return self.kv[n:].view(self.num_layers, self.num_pages, self.block_size, self.row - self.latent_dim)

    def page_views(self):
        """The pool's arrays as [layers][pages][...] views, for comparing pages."""
        if not self.split:
            return [self.kv.view(self.num_layers, self.num_pages, -1)]
        return [self.latent_view().reshape(self.num_layers, self.num_pages, -1),
                self.rope_view().reshape(self.num_layers, self.num_pages, -1)]

    def read_rows(self, layers, pages, slots):
        """Stored whole rows [n][row] of (layer, page, slot) index tensors."""
        return self.torch.cat((self.latent_view()[layers, pages, slots], self.rope_view()[layers, pages, slots]), -1)

    def write_layer_rows(self, layer: int, flat_slots, rows) -> None:
        """Store whole rows [n][row] at flat slots (page * block_size + offset) of one layer."""
        if not self.split:
            flat = self.kv_view()[layer].reshape(self.num_pages * self.block_size, self.row)
            flat.index_copy_(0, flat_slots, rows)
            return
        lat = self.latent_view()[layer].reshape(self.num_pages * self.block_size, self.latent_dim)
        rope = self.rope_view()[layer].reshape(self.num_pages * self.block_size, self.row - self.latent_dim)
        lat.index_copy_(0, flat_slots, rows[:, :self.latent_dim].contiguous())
        rope.index_copy_(0, flat_slots, rows[:, self.latent_dim:].contiguous())

    def add_request(self, req: int, length: int) -> np.ndarray:
        """Take pages for a new request of `length` tokens and install its table row; returns the page ids."""
        n = -(-length // self.block_size)
        pages = leyline.leyline_alloc_pages(self.pool, n)
        row = np.full(self.table.shape[1], -1, dtype=np.int32)
        row[:n] = pages
        self.table[req].copy_(self.torch.from_numpy(row))
        self.seq_lens_dev[req] = length
        self.tables.seq_lens_host[req] = length
        return pages

    def slot_index(self, req: int, tokens) -> "np.ndarray":
        """Flat slot index page * block_size + offset of each token (host; reads the table)."""
        t = np.asarray(tokens, dtype=np.int64)
        row = self.table[req].cpu().numpy().astype(np.int64)
        return row[t // self.block_size] * self.block_size + t % self.block_size

    def splice(self, dirs, stream=None) -> None:
        """dirs: a list of leyline.directive() or one leyline.directive_batch() array."""
        leyline.leyline_splice(self.pool, self.tables, dirs, stream)

    def gather(self, req: int, layer: int, t0: int, t1: int, out=None, stream=None):
        if out is None:
            out = self.torch.empty((t1 - t0, self.row), dtype=self.torch.bfloat16, device=self.device)
        leyline.leyline_gather(self.pool, self.tables, req, layer, t0, t1, out, stream)
        return out

    def materialize(self, req: int, stream=None) -> None:
        leyline.leyline_materialize(self.pool, self.tables, req, stream)

    def materialize_requests(self, reqs, stream=None) -> None:
        """materialize several distinct requests in one launch per 64 of them."""
        leyline.leyline_materialize_requests(self.pool, self.tables, reqs, stream)

    def pending(self):
        """Pending counts [num_pages][block_size] of a lazy pool, as a torch view (None otherwise)."""
        addr = leyline.leyline_pending_ptr(self.pool)
        if not addr:
            return None
        n = self.num_pages * self.block_size
        holder = _DeviceArray(addr, n, self.device.index or 0)
        return self.torch.as_tensor(holder, device=self.device).view(self.num_pages, self.block_size)

    def free_pages(self) -> int:
        return leyline.leyline_free_page_count(self.pool)

    def last_stats(self) -> dict:
        return leyline.leyline_last_stats(self.pool).as_dict()

    def check_status(self) -> None:
        leyline.leyline_sync_status(self.pool)

    def close(self) -> None:
        if self.pool is not None:
            leyline.leyline_pool_destroy(self.pool)
            self.pool = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
