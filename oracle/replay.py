"""Host replay of a workload's eviction schedule with the oracle, and ulp comparisons of stored values.

TEST INFRASTRUCTURE ONLY (tests/, __graft_entry__.smoke(), bench.py's CPU baseline).  Seeded contents come from the
``synth`` generator; every state transition here is the oracle's.
"""
from __future__ import annotations

import numpy as np

import synth
from synth.workloads import S_K, S_V, STREAM_HIST_INIT, Workload, chunk_stream

from . import OK, Cfg, HostCache, prune_step


def cfg_of(w: Workload) -> Cfg:
    return Cfg(**w.cfg_kwargs())


def _np_dtype(w: Workload):
    return np.uint16 if w.dtype == 0 else np.float32


def place_chunk(hc: HostCache, w: Workload, c: int) -> None:
    """Write chunk c's seeded K and V into its rows (the sink, or its ring slot)."""
    row0 = c * w.C if c < w.sink_chunks else w.win_row0 + w.slot_of(c) * w.C
    for arr, what in ((hc.k, S_K), (hc.v, S_V)):
        synth.fill_rows_host(arr, w.dtype, w.n_planes, w.cap, row0, w.C, w.D, w.seed, chunk_stream(c, what), w.C, 0)


def new_host_cache(w: Workload) -> HostCache:
    dt = _np_dtype(w)
    k = np.zeros((w.L, w.H, w.cap, w.D), dt)
    v = np.zeros((w.L, w.H, w.cap, w.D), dt)
    if w.hist_cap:
        for arr, s in ((k, 2 * STREAM_HIST_INIT), (v, 2 * STREAM_HIST_INIT + 1)):
            synth.fill_rows_host(arr, w.dtype, w.n_planes, w.cap, w.sink_rows, w.hist_cap, w.D, w.seed, s,
                                 w.hist_cap, 0)
    hc = HostCache(k, v, np.zeros(w.n_planes, np.int32), np.zeros(max(w.hist_cap, 1), np.int32), w.hist_cap)
    for c in range(w.sink_chunks):
        place_chunk(hc, w, c)
    return hc


def replay(w: Workload, hc: HostCache, evictions, head_is_static=None, placed=None, cfg: Cfg | None = None):
    """Run the oracle over a list of (chunk, q0_prev, q0) evictions, placing each newly generated chunk first
    (cfg: the method parameters, default those of the workload)."""
    placed = set() if placed is None else placed
    cfg = cfg_of(w) if cfg is None else cfg
    for c, q0_prev, q0 in evictions:
        for cc in w.resident_window(c):
            if cc not in placed:
                place_chunk(hc, w, cc)
                placed.add(cc)
        x0, xr = w.score_inputs(c)
        rc, _, _, _ = prune_step(hc, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, head_is_static)
        assert rc == OK, f"oracle replay refused eviction of chunk {c}: {rc}"
    return placed


def state_before_last(w: Workload, head_is_static=None, cfg: Cfg | None = None):
    """Host cache right before the workload's last eviction, and that eviction (chunk, q0_prev, q0)."""
    ev = w.evictions()
    hc = new_host_cache(w)
    placed = replay(w, hc, ev[:-1], head_is_static, cfg=cfg)
    c = ev[-1][0]
    for cc in w.resident_window(c):
        if cc not in placed:
            place_chunk(hc, w, cc)
    return hc, ev[-1]


# ------------------------------------------------------------------------------------------ comparisons
def ordered(bits: np.ndarray) -> np.ndarray:
    """Map float bit patterns (uint16 bf16 or float32) to integers whose difference counts ulps."""
    if bits.dtype == np.uint16:
        b = bits.astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    b = bits.view(np.uint32).astype(np.int64)
    return np.where(b & 0x80000000, -(b & 0x7FFFFFFF), b)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(ordered(a) - ordered(b))
