"""Paged copies of contiguous test caches: seeded block tables, packing a cache into block pools and reading it back.
Test infrastructure (the layout transform is a bijection of rows, so the oracle's contiguous results carry over)."""
from __future__ import annotations

import numpy as np
import torch

import autoregressive_video_diffusion_gb300 as dcp


class PagedCopy:
    """A PagedKVCache holding the same state as a contiguous device cache, with seeded block tables drawn as a random
    permutation of the pool's blocks; `spare` blocks are left free and filled with a canary."""

    def __init__(self, dev: dcp.KVCache, cfg: dcp.Config, block_size: int, layout: int, seed: int, spare: int = 5):
        C, bs = cfg.C, block_size
        sink = cfg.sink_chunks * C
        n_sink, n_hist, n_win = sink // bs, dev.hist_cap // bs, (cfg.window_chunks + 1) * C // bs
        n_blocks = n_sink + n_hist + n_win + spare
        perm = torch.from_numpy(np.random.default_rng(seed).permutation(n_blocks).astype(np.int32))
        self.sink_blocks = perm[:n_sink].cuda()
        self.free_blocks = perm[n_sink + n_hist + n_win:].cuda().long()
        self.cache = dcp.PagedKVCache(dev.L, dev.H, dev.D, dev.dtype, bs, layout, n_blocks, dev.hist_cap, n_win)
        self.cache.hist_blocks.copy_(perm[n_sink:n_sink + n_hist])
        self.cache.window_blocks.copy_(perm[n_sink + n_hist:n_sink + n_hist + n_win])
        self.cache.hist_len.copy_(dev.hist_len)
        self.cache.hist_t.copy_(dev.hist_t)
        self.block, self.off = dcp.paged_row_map(cfg, dev.hist_cap, bs, self.sink_blocks, self.cache.hist_blocks,
                                                 self.cache.window_blocks)
        for pool in (self.cache.k_pool, self.cache.v_pool):
            pool.view(torch.int16 if pool.element_size() == 2 else torch.int32).fill_(0x3A5C)
        self.layout = layout
        dcp.paged_pack(self.cache.k_pool, dev.k, self.block, self.off, layout)
        dcp.paged_pack(self.cache.v_pool, dev.v, self.block, self.off, layout)
        self.free0 = [self._free(pool).clone() for pool in (self.cache.k_pool, self.cache.v_pool)]

    def _free(self, pool):
        return pool[:, self.free_blocks]

    def free_blocks_untouched(self) -> bool:
        return all(torch.equal(self._free(p), f0) for p, f0 in zip((self.cache.k_pool, self.cache.v_pool), self.free0))

    def unpack_into(self, dev: dcp.KVCache) -> None:
        """Copy the paged state back into a contiguous cache (rows, hist_len, hist_t)."""
        dev.k.copy_(dcp.paged_unpack(self.cache.k_pool, self.block, self.off, self.layout))
        dev.v.copy_(dcp.paged_unpack(self.cache.v_pool, self.block, self.off, self.layout))
        dev.hist_len.copy_(self.cache.hist_len)
        dev.hist_t.copy_(self.cache.hist_t)
