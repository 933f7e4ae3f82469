"""GPU host snapshot / restore of the pruned cache against the oracle's image (through the C ABI).

Page "기술 요약: 생성형 월드 모델을 위한 지속적 계산 상태" (gist.science/ko/paper/2607.21686), section "PCS contract":
round trip and snapshot completeness.  Bar: the image bytes are identical to the oracle's image of the same state;
a restore gives back exactly the saved rows, hist_len and hist_t and leaves every other byte of the cache as it was.
"""
import numpy as np
import pytest
import torch

import autoregressive_video_diffusion_gb300 as dcp
import oracle
from oracle import replay
from synth import workloads as W
from synth.workloads import FULL, MID, TINY, scaled
from tests import devcache

pytestmark = pytest.mark.gpu

TINY_ROT = scaled(TINY, R=2, S=4)


def _live_after(w, c):
    m = 0
    for cc in range(c + 1, c + w.window_chunks + 1):
        m |= 1 << w.slot_of(cc)
    return m


def _garbage_host(hc, seed=3):
    g = hc.copy()
    rng = np.random.default_rng(seed)
    if g.k.dtype == np.uint16:
        g.k[...] = rng.integers(0, 2 ** 16, g.k.shape, dtype=np.uint16)
        g.v[...] = rng.integers(0, 2 ** 16, g.v.shape, dtype=np.uint16)
    else:
        g.k[...] = rng.standard_normal(g.k.shape).astype(np.float32)
        g.v[...] = rng.standard_normal(g.v.shape).astype(np.float32)
    g.hist_len[...] = 0
    g.hist_t[...] = -7
    return g


def _snapshot(dev, cfg, live, q0):
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, cfg))
    img = dcp.new_snapshot_image(dcp.dcp_snapshot_max_bytes(dev, cfg, live))
    img.fill_(0xEE)
    dcp.dcp_snapshot(dev, cfg, live, q0, img, ws)
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    return img, ws


CASES = [(TINY_ROT, False), (TINY_ROT, True), (MID, False)]


@pytest.mark.parametrize("w,hs", CASES, ids=["tiny", "tiny_head_specialised", "mid"])
def test_snapshot_image_equals_oracle(gpu, w, hs):
    hsm = (np.arange(w.L * w.H) % 3 == 1).astype(np.uint8) if hs else None
    hc, (c, _, q0) = replay.state_before_last(w, head_is_static=hsm)
    live = (1 << (w.window_chunks + 1)) - 1
    want = oracle.snapshot(hc, replay.cfg_of(w), live, q0)
    dev = devcache.to_device(hc, w)
    img, _ = _snapshot(dev, devcache.dcp_config(w), live, q0)
    n = dcp.snapshot_total_bytes(img)
    assert n == want.shape[0]
    assert np.array_equal(img[:n].numpy(), want)


@pytest.mark.parametrize("w,hs", CASES, ids=["tiny", "tiny_head_specialised", "mid"])
def test_restore_equals_oracle_restore(gpu, w, hs):
    hsm = (np.arange(w.L * w.H) % 3 == 1).astype(np.uint8) if hs else None
    hc, (c, _, q0) = replay.state_before_last(w, head_is_static=hsm)
    live = _live_after(w, c)
    image = oracle.snapshot(hc, replay.cfg_of(w), live, q0)
    host = _garbage_host(hc)
    dev = devcache.to_device(host, w)
    cfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, cfg))
    img = dcp.new_snapshot_image(image.shape[0])
    img.copy_(torch.from_numpy(image))
    q0_back, live_back = dcp.dcp_restore(dev, cfg, img, ws)
    assert (q0_back, live_back) == (q0, live)
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    rc, _, _ = oracle.restore(host, replay.cfg_of(w), image)
    assert rc == oracle.OK
    g = devcache.from_device(dev, w)
    assert np.array_equal(g.hist_len, host.hist_len) and np.array_equal(g.hist_t, host.hist_t)
    assert np.array_equal(g.k, host.k) and np.array_equal(g.v, host.v)


def test_resumed_step_equals_uninterrupted(gpu):
    """Snapshot the GPU cache before an eviction, restore it into another cache, run the same prune step on both:
    the two caches end bit-identical (the page's restore experiment)."""
    w = MID
    hc, (c, q0_prev, q0) = replay.state_before_last(w)
    cfg = devcache.dcp_config(w)
    a = devcache.to_device(hc, w)
    live = (1 << (w.window_chunks + 1)) - 1
    img, ws = _snapshot(a, cfg, live, q0_prev)
    b = devcache.to_device(_garbage_host(hc), w)
    assert dcp.dcp_restore(b, cfg, img, ws) == (q0_prev, live)
    x0, xr = (torch.from_numpy(x).cuda() for x in w.score_inputs(c))
    for dev in (a, b):
        wsd = dcp.new_workspace(dcp.dcp_workspace_size(dev, cfg))
        dcp.dcp_prune_step(dev, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, None, None, None, wsd)
        assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    ga, gb = devcache.from_device(a, w), devcache.from_device(b, w)
    assert np.array_equal(ga.hist_len, gb.hist_len)
    n = int(ga.hist_len.max())
    assert np.array_equal(ga.hist_t[:n], gb.hist_t[:n])
    live_rows = np.zeros(w.cap, bool)
    live_rows[:w.sink_chunks * w.C + n] = True
    for s in range(w.window_chunks + 1):
        if (live >> s) & 1:
            r0 = w.sink_chunks * w.C + w.hist_cap + s * w.C
            live_rows[r0:r0 + w.C] = True
    assert np.array_equal(ga.k[:, :, live_rows], gb.k[:, :, live_rows])
    assert np.array_equal(ga.v[:, :, live_rows], gb.v[:, :, live_rows])


def test_image_too_small_reports_capacity(gpu):
    w = TINY_ROT
    hc, (c, _, q0) = replay.state_before_last(w)
    dev = devcache.to_device(hc, w)
    cfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, cfg))
    live = _live_after(w, c)
    need = oracle.snapshot(hc, replay.cfg_of(w), live, q0).shape[0]
    img = dcp.new_snapshot_image(need - 16)
    img.fill_(0xEE)
    dcp.dcp_snapshot(dev, cfg, live, q0, img, ws)
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_ECAPACITY
    assert dcp.snapshot_total_bytes(img) == need
    assert int(img[200]) == 0xEE, "nothing past the header is written when the image is short"
    dcp.dcp_reset_status(dev.status)


def test_refusals(gpu):
    w = TINY_ROT
    hc, (c, _, q0) = replay.state_before_last(w)
    dev = devcache.to_device(hc, w)
    cfg = devcache.dcp_config(w)
    live = _live_after(w, c)
    img, ws = _snapshot(dev, cfg, live, q0)
    pageable = torch.empty(img.numel(), dtype=torch.uint8)
    with pytest.raises(dcp.DcpError):
        dcp.dcp_snapshot(dev, cfg, live, q0, pageable, ws)
    with pytest.raises(dcp.DcpError):
        dcp.dcp_snapshot(dev, cfg, 1 << (w.window_chunks + 1), q0, img, ws)
    bad = dcp.new_snapshot_image(img.numel())
    bad.copy_(img)
    bad[0] = ord("X")
    with pytest.raises(dcp.DcpError):
        dcp.dcp_restore(dev, cfg, bad, ws)
    other_w = scaled(w, hist_cap=w.hist_cap + w.C)
    other = dcp.KVCache(other_w.L, other_w.H, other_w.D, other_w.dtype, other_w.cap, other_w.hist_cap)
    ocfg = devcache.dcp_config(other_w)
    ows = dcp.new_workspace(dcp.dcp_workspace_size(other, ocfg))
    with pytest.raises(dcp.DcpError):
        dcp.dcp_restore(other, ocfg, img, ows)
    with pytest.raises(dcp.DcpError):
        dcp.dcp_restore(dev, cfg, img[:dcp.snapshot_total_bytes(img) - 16], ws)


def test_full_depth_8_layers_sampled(gpu):
    """The bench's snapshot workload: the full-depth eviction cut to 8 layers, after its prune step (947 history
    rows per plane).  The image's header is checked in full and sampled planes row by row against the device."""
    w = scaled(FULL, L=8)
    c, q0_prev, q0 = w.evictions()[-1]
    cache = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, w.hist_cap)
    stream = torch.cuda.current_stream().cuda_stream
    W.fill_device_chunks(cache.k.data_ptr(), cache.v.data_ptr(), w, list(range(w.sink_chunks)) + w.resident_window(c),
                         stream)
    W.fill_device_history_canary(cache.k.data_ptr(), cache.v.data_ptr(), w, stream)
    cfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(cache, cfg))
    x0, xr = (torch.from_numpy(x).cuda() for x in w.score_inputs(c))
    dcp.dcp_prune_step(cache, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, None, None, None, ws)
    assert dcp.dcp_get_status(cache.status) == dcp.DCP_OK
    k = int(cache.hist_len[0].item())
    live = _live_after(w, c)
    img = dcp.new_snapshot_image(dcp.dcp_snapshot_max_bytes(cache, cfg, live))
    dcp.dcp_snapshot(cache, cfg, live, q0, img, ws)
    assert dcp.dcp_get_status(cache.status) == dcp.DCP_OK
    n_planes, sink, rb = w.L * w.H, w.sink_chunks * w.C, w.D * 2
    per_plane = sink + k + w.window_chunks * w.C
    data_off = -(-(128 + 4 * n_planes + 4 * k) // 256) * 256
    h = img[:128].numpy()
    assert bytes(h[:8]) == b"DCPSNAP1"
    assert list(h.view(np.int32)[2:6]) == [w.L, w.H, w.D, 0]
    assert list(h.view(np.int64)[3:7]) == [w.cap, w.hist_cap, sink, w.C]
    assert list(h.view(np.int32)[14:18]) == [w.window_chunks, live, q0, k]
    assert list(h.view(np.int64)[9:12]) == [rb, n_planes * per_plane, data_off + 2 * n_planes * per_plane * rb]
    assert np.all(img[128:128 + 4 * n_planes].numpy().view(np.int32) == k)
    hist_t = img[128 + 4 * n_planes:128 + 4 * n_planes + 4 * k].numpy().view(np.int32)
    assert np.array_equal(hist_t, cache.hist_t[:k].cpu().numpy())
    slots = [s for s in range(w.window_chunks + 1) if (live >> s) & 1]
    rows = np.concatenate([np.arange(sink + k)] + [np.arange(sink + w.hist_cap + s * w.C,
                                                             sink + w.hist_cap + (s + 1) * w.C) for s in slots])
    for t, tensor in enumerate((cache.k, cache.v)):
        for pl in (0, 1, 57, n_planes - 1):
            l, hh = divmod(pl, w.H)
            dev_rows = tensor[l, hh].view(torch.int16).cpu().numpy()[rows]
            off = data_off + (t * n_planes * per_plane + pl * per_plane) * rb
            got = img[off:off + per_plane * rb].numpy().view(np.int16).reshape(per_plane, w.D)
            assert np.array_equal(got, dev_rows)
