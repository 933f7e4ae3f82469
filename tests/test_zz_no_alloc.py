"""The allocation-free prune step, dcp_prune_step_noalloc, against the workspace entry point dcp_prune_step.

Some callers of this library cannot call cudaMalloc (code inside a device allocator's callback, engines that reserve
all device memory at start-up and forbid later allocation, host programs without a device allocator of their own),
so they cannot hand dcp_prune_step a workspace.  dcp_prune_step_noalloc runs the same kernels on a fixed scratch
array compiled into the library.  These tests call it through the C ABI on two prune steps in a row and require the
same cache, lengths, frames and kept counts as the workspace entry point (the tolerance of the other GPU tests:
turned keys within 1 bf16 ulp, everything else exact), also on head-specialised steps with the kept count written to
page-locked host memory, and check that refused calls (bad arguments, a cache needing more scratch than the array
holds) change nothing.  This file is collected last so that a run stopping at its first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import autoregressive_video_diffusion_gb300 as dcp
from oracle import replay
from synth import workloads as W
from synth.workloads import MID, TINY, scaled
from tests import devcache

pytestmark = pytest.mark.gpu


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _noalloc(cache, cfg, x0, xr, slot, first, q0_prev, q0, kept, head_is_static=None, kept_host=None):
    cc, gc = cache.c(), cfg.c()
    return dcp.lib.dcp_prune_step_noalloc(ctypes.byref(cc), ctypes.byref(gc), x0.data_ptr(), xr.data_ptr(),
                                          x0.shape[1], slot, first, q0_prev, q0,
                                          None if head_is_static is None else head_is_static.data_ptr(),
                                          kept.data_ptr(), None if kept_host is None else kept_host.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)


def _two_steps(w, head_is_static=None):
    """The workload's last two evictions through both entry points, from the oracle's state before them; after each
    step the two caches, lengths, frames and kept counts must agree."""
    ev = w.evictions()
    hc = replay.new_host_cache(w)
    placed = replay.replay(w, hc, ev[:-2], head_is_static)
    for cc in w.resident_window(ev[-2][0]):
        if cc not in placed:
            replay.place_chunk(hc, w, cc)
            placed.add(cc)
    a = devcache.to_device(hc, w)          # dcp_prune_step with a caller workspace
    b = devcache.to_device(hc, w)          # dcp_prune_step_noalloc
    cfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(a, cfg))
    assert dcp.dcp_workspace_size(a, cfg) <= dcp.DCP_NOALLOC_WORKSPACE_BYTES
    hs = None if head_is_static is None else _cuda(head_is_static)
    stream = torch.cuda.current_stream().cuda_stream
    for c, q0_prev, q0 in ev[-2:]:
        new = [cc for cc in w.resident_window(c) if cc not in placed]   # the chunk generated since the last step
        for cache in (a, b):
            W.fill_device_chunks(cache.k.data_ptr(), cache.v.data_ptr(), w, new, stream)
        placed |= set(new)
        x0, xr = (_cuda(t) for t in w.score_inputs(c))
        ka = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        kb = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        kh = torch.full((1,), -1, dtype=torch.int32).pin_memory() if head_is_static is not None else None
        dcp.dcp_prune_step(a, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, hs, ka, None, ws)
        rc = _noalloc(b, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, kb, hs, kh)
        assert rc == dcp.DCP_OK, dcp.dcp_status_string(rc)
        assert dcp.dcp_get_status(a.status) == dcp.DCP_OK and dcp.dcp_get_status(b.status) == dcp.DCP_OK
        assert int(ka.item()) == int(kb.item()) > 0
        if kh is not None:  # written by the scan kernel into page-locked host memory (the stream was synchronised)
            assert int(kh.item()) == int(ka.item())
        ga, gb = devcache.from_device(a, w), devcache.from_device(b, w)
        assert np.array_equal(ga.hist_len, gb.hist_len) and np.array_equal(ga.hist_t, gb.hist_t)
        assert np.array_equal(ga.v, gb.v)
        nt2 = 2 * w.n_temporal_pairs
        assert np.array_equal(ga.k[..., nt2:], gb.k[..., nt2:])
        assert int(replay.ulp_distance(ga.k[..., :nt2], gb.k[..., :nt2]).max()) <= 1
    return a, b, cfg


def test_noalloc_matches_workspace_entry_point_two_steps(gpu):
    _two_steps(MID)


def test_noalloc_head_specialised_two_steps(gpu):
    """Head-specialised steps write the list of receiving planes into the scratch array and count them with an
    accumulator that must start each call at zero; the kept count also goes to page-locked host memory."""
    w = scaled(MID, n_static_per_layer=3)
    hsm = w.head_is_static()
    assert hsm is not None and 0 < int(hsm.sum()) < w.n_planes
    a, b, _ = _two_steps(w, hsm)
    hl = b.hist_len.cpu().numpy()
    assert np.all(hl[hsm == 1] == 0) and np.all(hl[hsm == 0] > 0)


def test_noalloc_refused_call_changes_nothing(gpu):
    """A call whose arguments fail a host check returns DCP_EINVAL, leaves the cache as it was, and the next valid
    call still gives the workspace entry point's result."""
    w = MID
    hc, (c, q0_prev, q0) = replay.state_before_last(w)
    a, b = devcache.to_device(hc, w), devcache.to_device(hc, w)
    cfg = devcache.dcp_config(w)
    x0, xr = (_cuda(t) for t in w.score_inputs(c))
    kb = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    before = devcache.from_device(b, w)
    for bad in ((w.window_chunks + 1, w.first_frame(c), q0_prev, q0),     # no such ring slot
                (w.slot_of(c), w.first_frame(c), q0_prev, w.max_frames + 1),  # q0 past the phase tables
                (w.slot_of(c), w.first_frame(c), q0 + 1, q0)):             # q0 moving backwards
        assert _noalloc(b, cfg, x0, xr, *bad, kb) == dcp.DCP_EINVAL
    torch.cuda.synchronize()
    after = devcache.from_device(b, w)
    assert int(kb.item()) == -1
    assert np.array_equal(before.k, after.k) and np.array_equal(before.v, after.v)
    assert np.array_equal(before.hist_len, after.hist_len) and np.array_equal(before.hist_t, after.hist_t)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(a, cfg))
    ka = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dcp.dcp_prune_step(a, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, None, ka, None, ws)
    assert _noalloc(b, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, kb) == dcp.DCP_OK
    assert dcp.dcp_get_status(b.status) == dcp.DCP_OK and int(kb.item()) == int(ka.item())
    ga, gb = devcache.from_device(a, w), devcache.from_device(b, w)
    assert np.array_equal(ga.hist_len, gb.hist_len) and np.array_equal(ga.v, gb.v)
    assert int(replay.ulp_distance(ga.k, gb.k).max()) <= 1


def test_noalloc_refuses_workspace_beyond_its_array(gpu):
    w = scaled(TINY, max_frames=1 << 20)   # the history phase table alone would need ~128 MB
    hc, (c, q0_prev, q0) = replay.state_before_last(scaled(TINY))
    dev = devcache.to_device(hc, w)
    cfg = devcache.dcp_config(w)
    assert dcp.dcp_workspace_size(dev, cfg) > dcp.DCP_NOALLOC_WORKSPACE_BYTES
    x0, xr = (_cuda(t) for t in w.score_inputs(c))
    kept = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = devcache.from_device(dev, w)
    rc = _noalloc(dev, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, kept)
    assert rc == dcp.DCP_EINVAL
    after = devcache.from_device(dev, w)
    assert np.array_equal(before.k, after.k) and np.array_equal(before.hist_len, after.hist_len)
