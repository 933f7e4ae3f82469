"""GPU parity of read-time re-index (reindex_mode 1) against the oracle.

Section "what differs" of the DeCoPrune page: history keys take t~(t; q0); with read-time re-index they stay at their
own frame's phase, move bitwise, and are turned once when read.  Bars: a prune step in this mode is bit-exact
(nothing rotates); a read is within 1 bf16 ulp (fp32: 2 ulp plus 2^-38 of the pair) of the oracle's fp64 turn of the
stored key, other dims bitwise, and rows past a plane's history are not written.
"""
import numpy as np
import pytest
import torch

import autoregressive_video_diffusion_gb300 as dcp
import oracle
from oracle import replay
from synth.workloads import MID, TINY, scaled
from tests import devcache
from tests.paged import PagedCopy
from tests.test_gpu_parity import _cuda, assert_key_parity, gpu_vs_oracle_step

pytestmark = pytest.mark.gpu

TINY_ROT = scaled(TINY, R=2, S=4)


def _lazy(w):
    cfg = replay.cfg_of(w)
    cfg.reindex_mode = 1
    return cfg


@pytest.mark.parametrize("w", [TINY_ROT, MID], ids=["tiny_rotating", "mid"])
def test_read_time_prune_step_is_bit_exact(gpu, w):
    hc, ev = replay.state_before_last(w, cfg=_lazy(w))
    _, _, _, inexact = gpu_vs_oracle_step(w, hc, ev, reindex_mode=1)
    assert inexact == 0


def _read(cache, gcfg, q0, plane0, n, w, ws):
    out = torch.empty((n, w.hist_cap, w.D), dtype=torch.bfloat16 if w.dtype == 0 else torch.float32, device="cuda")
    out.view(torch.int16 if w.dtype == 0 else torch.int32).fill_(0x1357)
    dcp.dcp_read_history_keys(cache, gcfg, q0, plane0, n, out, ws)
    st = dcp.dcp_get_status(cache.status)
    g = out.view(torch.int16).cpu().numpy().view(np.uint16) if w.dtype == 0 else out.cpu().numpy()
    return st, g


def _check_read(g, want, hc, plane0, w):
    canary = np.uint16(0x1357) if w.dtype == 0 else np.int32(0x1357).view(np.float32)
    for i in range(g.shape[0]):
        n = int(hc.hist_len[plane0 + i])
        assert_key_parity(g[i, :n], want[plane0 + i, :n], w.n_temporal_pairs)
        assert np.all(g[i, n:] == canary), "rows past the history must not be written"


@pytest.mark.parametrize("w,hs,planes", [(TINY_ROT, False, (0, None)), (TINY_ROT, True, (1, 2)),
                                         (MID, False, (0, None)), (MID, False, (5, 17))],
                         ids=["tiny_all", "tiny_head_specialised_range", "mid_all", "mid_range"])
def test_read_history_keys(gpu, w, hs, planes):
    hsm = (np.arange(w.L * w.H) % 3 == 1).astype(np.uint8) if hs else None
    cfg = _lazy(w)
    hc, (c, q0_prev, q0) = replay.state_before_last(w, head_is_static=hsm, cfg=cfg)
    plane0, n = planes[0], planes[1] or w.L * w.H
    want = oracle.read_history_keys(hc, cfg, q0)
    dev = devcache.to_device(hc, w)
    gcfg = devcache.dcp_config(w, reindex_mode=1)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
    st, g = _read(dev, gcfg, q0, plane0, n, w, ws)
    assert st == dcp.DCP_OK
    _check_read(g, want, hc, plane0, w)


@pytest.mark.parametrize("layout", [dcp.DCP_PAGED_HND, dcp.DCP_PAGED_NHD], ids=["hnd", "nhd"])
def test_paged_read_history_keys(gpu, layout):
    w = MID
    cfg = _lazy(w)
    hc, (c, q0_prev, q0) = replay.state_before_last(w, cfg=cfg)
    want = oracle.read_history_keys(hc, cfg, q0)
    dev = devcache.to_device(hc, w)
    gcfg = devcache.dcp_config(w, reindex_mode=1)
    pc = PagedCopy(dev, gcfg, 16, layout, seed=3)
    ws = dcp.new_workspace(dcp.dcp_paged_workspace_size(pc.cache, gcfg))
    st, g = _read(pc.cache, gcfg, q0, 0, w.L * w.H, w, ws)
    assert st == dcp.DCP_OK
    _check_read(g, want, hc, 0, w)


def test_read_time_rollout_then_read(gpu):
    """The library takes a mid-size cache through its evictions in read-time mode from the sink alone; the history
    equals the oracle's read-time replay bitwise, and reading it at the last q0 matches the oracle's read."""
    w = MID
    cfg = _lazy(w)
    o = replay.new_host_cache(w)
    dev = devcache.to_device(o, w)
    gcfg = devcache.dcp_config(w, reindex_mode=1)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
    placed = set(range(w.sink_chunks))
    for c, q0_prev, q0 in w.evictions():
        for cc in w.resident_window(c):
            if cc not in placed:
                replay.place_chunk(o, w, cc)
                placed.add(cc)
        dev2 = devcache.to_device(o, w)  # the newly placed chunks, on top of the device's own history
        dev2.hist_len.copy_(dev.hist_len)
        dev2.hist_t.copy_(dev.hist_t)
        sink = w.sink_chunks * w.C
        dev2.k[:, :, sink:sink + w.hist_cap].copy_(dev.k[:, :, sink:sink + w.hist_cap])
        dev2.v[:, :, sink:sink + w.hist_cap].copy_(dev.v[:, :, sink:sink + w.hist_cap])
        dev = dev2
        x0, xr = w.score_inputs(c)
        dcp.dcp_prune_step(dev, gcfg, _cuda(x0), _cuda(xr), w.slot_of(c), w.first_frame(c), q0_prev, q0, None, None,
                           None, ws)
        assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
        rc, _, _, _ = oracle.prune_step(o, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0)
        assert rc == oracle.OK
    g = devcache.from_device(dev, w)
    assert np.array_equal(g.hist_len, o.hist_len)
    n = int(o.hist_len.max())
    assert np.array_equal(g.hist_t[:n], o.hist_t[:n])
    sink = w.sink_chunks * w.C
    assert np.array_equal(g.k[:, :, sink:sink + n], o.k[:, :, sink:sink + n])
    q0 = w.evictions()[-1][2]
    st, gr = _read(dev, gcfg, q0, 0, w.L * w.H, w, ws)
    assert st == dcp.DCP_OK
    _check_read(gr, oracle.read_history_keys(o, cfg, q0), o, 0, w)


def test_read_refusals(gpu):
    w = TINY_ROT
    hc, (c, q0_prev, q0) = replay.state_before_last(w, cfg=_lazy(w))
    dev = devcache.to_device(hc, w)
    eager = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, eager))
    out = torch.empty((w.L * w.H, w.hist_cap, w.D), dtype=torch.float32, device="cuda")
    with pytest.raises(dcp.DcpError):
        dcp.dcp_read_history_keys(dev, eager, q0, 0, w.L * w.H, out, ws)      # eager caches are read as stored
    lazy = devcache.dcp_config(w, reindex_mode=1)
    with pytest.raises(dcp.DcpError):
        dcp.dcp_read_history_keys(dev, lazy, q0, 1, w.L * w.H, out, ws)       # plane range past the cache
    with pytest.raises(dcp.DcpError):
        dcp.dcp_read_history_keys(dev, lazy, w.max_frames + 1, 0, 1, out, ws)  # q0 past the workspace tables


def test_read_reports_history_frame_outside_table(gpu):
    """A history frame at or past q0 has no phase: the row is not written and the call reports DCP_EDEVICE."""
    w = TINY_ROT
    hc, (c, q0_prev, q0) = replay.state_before_last(w, cfg=_lazy(w))
    dev = devcache.to_device(hc, w)
    dev.hist_t[0] = q0
    gcfg = devcache.dcp_config(w, reindex_mode=1)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
    st, g = _read(dev, gcfg, q0, 0, 1, w, ws)
    assert st == dcp.DCP_EDEVICE
    assert np.all(g[0, 0] == np.int32(0x1357).view(np.float32))
    dcp.dcp_reset_status(dev.status)


@pytest.mark.parametrize("mode", [0, 1])
def test_phase_table(gpu, mode):
    """dcp_phase_table: each entry's hi + lo parts give cos / sin of theta_p (t~(t; q0) - t) (the oracle's pinned phase
    map and ladder, numpy's cos / sin) to ~2^-38; the hi parts carry at most 16 significant bits; frames that keep their
    phase get exactly {1, 0, 0, 0}."""
    w = scaled(TINY, R=2, S=4 if mode == 0 else 3, g_mode=mode)
    gcfg = devcache.dcp_config(w, reindex_mode=1)
    T_s = w.sink_chunks * w.frames_per_chunk
    q0 = 40
    n_t = w.n_temporal_pairs
    out = torch.empty((q0 - T_s) * n_t * 4, dtype=torch.float32, device="cuda")
    dcp.dcp_phase_table(gcfg, q0, T_s, q0, out)
    tab = out.view(q0 - T_s, n_t, 4).cpu().numpy().astype(np.float64)
    moved = 0
    for i, t in enumerate(range(T_s, q0)):
        tt = oracle.phase(t, q0, T_s, w.R, w.S, mode)
        for p in range(n_t):
            phi = oracle.theta(p, n_t, w.rope_base) * (tt - t)
            c, s = tab[i, p, 0] + tab[i, p, 1], tab[i, p, 2] + tab[i, p, 3]
            assert abs(c - np.cos(phi)) < 2.0 ** -38 and abs(s - np.sin(phi)) < 2.0 ** -38
            if tt == t:
                assert list(tab[i, p]) == [1.0, 0.0, 0.0, 0.0]
        moved += tt != t
    hi = out.view(q0 - T_s, n_t, 4)[..., 0::2].contiguous().view(torch.int32).cpu().numpy()
    assert np.all(hi & 0xFF == 0), "hi parts must carry at most 16 significant bits"
    assert moved > 0
    with pytest.raises(dcp.DcpError):
        dcp.dcp_phase_table(gcfg, q0, T_s, q0 + 1, out)
    with pytest.raises(dcp.DcpError):
        dcp.dcp_phase_table(gcfg, q0, T_s - 1, q0, out)
