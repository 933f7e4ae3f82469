"""Pins of the oracle's host snapshot / restore of the pruned cache (no GPU).

Page "기술 요약: 생성형 월드 모델을 위한 지속적 계산 상태" (gist.science/ko/paper/2607.21686), section "PCS contract":
restore(checkpoint(s)) gives back the state (round trip), a checkpoint holds exactly the non-derivable state
(snapshot completeness), restored copies evolve independently (fork independence), and a run resumed from a
checkpoint matches the run that never stopped (the page's restore experiment: byte-identical trajectories).
"""
import numpy as np
import pytest

import oracle
from oracle import replay
from synth.workloads import TINY, scaled

W = scaled(TINY, R=2, S=4)


def _state_rows(hc, w, live):
    """(plane, row) pairs of the state: sink + history rows, then the live ring slots (derived here from the
    cache layout, independently of the oracle's image writer)."""
    sink = w.sink_chunks * w.C
    rows = []
    for p in range(w.L * w.H):
        r = list(range(sink + int(hc.hist_len[p])))
        for s in range(w.window_chunks + 1):
            if (live >> s) & 1:
                r += list(range(sink + w.hist_cap + s * w.C, sink + w.hist_cap + (s + 1) * w.C))
        rows.append(r)
    return rows


def _garbage_like(hc):
    g = hc.copy()
    rng = np.random.default_rng(11)
    g.k[...] = rng.integers(0, 2 ** 16, g.k.shape).astype(g.k.dtype) if g.k.dtype == np.uint16 else \
        rng.standard_normal(g.k.shape).astype(np.float32)
    g.v[...] = g.k[::-1].copy() if g.k.shape[0] > 1 else g.k + 1
    g.hist_len[...] = 0
    g.hist_t[...] = -7
    return g


def _live_after(w, c):
    """Ring slots holding chunks c + 1 .. c + w (the window once chunk c has left)."""
    m = 0
    for cc in range(c + 1, c + w.window_chunks + 1):
        m |= 1 << w.slot_of(cc)
    return m


def test_header_fields_and_size():
    hc, (c, _, q0) = replay.state_before_last(W)
    live = (1 << (W.window_chunks + 1)) - 1
    img = oracle.snapshot(hc, replay.cfg_of(W), live, q0)
    assert bytes(img[:8]) == b"DCPSNAP1"
    h32 = img[:128].view(np.int32)
    h64 = img[:128].view(np.int64)
    assert list(h32[2:6]) == [W.L, W.H, W.D, W.dtype]
    assert h64[3] == W.cap and h64[4] == W.hist_cap and h64[5] == W.sink_chunks * W.C and h64[6] == W.C
    assert h32[14] == W.window_chunks and h32[15] == live and h32[16] == q0 and h32[17] == int(hc.hist_len.max())
    rows = sum(len(r) for r in _state_rows(hc, W, live))
    rb = W.D * W.esize
    data_off = -(-(128 + 4 * W.L * W.H + 4 * int(hc.hist_len.max())) // 256) * 256
    assert h64[9] == rb and h64[10] == rows
    assert img.shape[0] == h64[11] == data_off + 2 * rows * rb


@pytest.mark.parametrize("hs", [False, True], ids=["dense", "head_specialised"])
def test_round_trip_restores_state_and_only_state(hs):
    hsm = None
    if hs:
        hsm = (np.arange(W.L * W.H) % 3 == 1).astype(np.uint8)
    hc, (c, q0_prev, q0) = replay.state_before_last(W, head_is_static=hsm)
    cfg = replay.cfg_of(W)
    live = _live_after(W, c - 1) | (1 << W.slot_of(c))
    img = oracle.snapshot(hc, cfg, live, q0)
    dst = _garbage_like(hc)
    before = dst.copy()
    rc, q0_back, live_back = oracle.restore(dst, cfg, img)
    assert rc == oracle.OK and q0_back == q0 and live_back == live
    assert np.array_equal(dst.hist_len, hc.hist_len)
    n = int(hc.hist_len.max())
    assert np.array_equal(dst.hist_t[:n], hc.hist_t[:n]) and np.all(dst.hist_t[n:] == -7)
    rows = _state_rows(hc, W, live)
    for p in range(W.L * W.H):
        l, h = divmod(p, W.H)
        state = np.zeros(W.cap, bool)
        state[rows[p]] = True
        assert np.array_equal(dst.k[l, h][state], hc.k[l, h][state])
        assert np.array_equal(dst.v[l, h][state], hc.v[l, h][state])
        assert np.array_equal(dst.k[l, h][~state], before.k[l, h][~state]), "free rows must not be written"
        assert np.array_equal(dst.v[l, h][~state], before.v[l, h][~state])


def test_snapshot_holds_exactly_the_state():
    """Changing a free row (past a plane's history, or in a ring slot that is not live) leaves the image as it was;
    changing any saved byte changes it."""
    hc, (c, _, q0) = replay.state_before_last(W)
    cfg = replay.cfg_of(W)
    live = _live_after(W, c)
    img = oracle.snapshot(hc, cfg, live, q0)
    sink = W.sink_chunks * W.C
    free = hc.copy()
    free.k[0, 0, sink + int(hc.hist_len[0])] += 1
    free.v[-1, -1, sink + W.hist_cap + W.slot_of(c) * W.C] += 1
    assert np.array_equal(oracle.snapshot(free, cfg, live, q0), img)
    rows = _state_rows(hc, W, live)
    rng = np.random.default_rng(5)
    for _ in range(20):
        p = int(rng.integers(W.L * W.H))
        r = rows[p][int(rng.integers(len(rows[p])))]
        d = int(rng.integers(W.D))
        m = hc.copy()
        l, h = divmod(p, W.H)
        (m.k if rng.integers(2) else m.v)[l, h, r, d] += 1
        assert not np.array_equal(oracle.snapshot(m, cfg, live, q0), img)


def test_resume_matches_uninterrupted_run_and_forks_are_independent():
    """Checkpoint after the first evictions, restore into a fresh cache, finish the schedule: the state equals the
    uninterrupted run's, byte for byte.  A second restore of the same image is not touched by the first copy's
    steps."""
    w = scaled(W, history_chunks=(1, 2, 3))
    ev = w.evictions()
    cfg = replay.cfg_of(w)
    full = replay.new_host_cache(w)
    placed = replay.replay(w, full, ev)
    part = replay.new_host_cache(w)
    placed2 = replay.replay(w, part, ev[:2])
    c_last_done = ev[1][0]
    live = _live_after(w, c_last_done)
    img = oracle.snapshot(part, cfg, live, ev[1][2])
    a, b = _garbage_like(part), _garbage_like(part)
    assert oracle.restore(a, cfg, img)[0] == oracle.OK
    assert oracle.restore(b, cfg, img)[0] == oracle.OK
    b_before = b.copy()
    replay.replay(w, a, ev[2:], placed=set(placed2))
    live_end = _live_after(w, ev[-1][0])
    assert np.array_equal(oracle.snapshot(a, cfg, live_end, ev[-1][2]), oracle.snapshot(full, cfg, live_end,
                                                                                         ev[-1][2]))
    assert np.array_equal(b.k, b_before.k) and np.array_equal(b.hist_len, b_before.hist_len)


def test_refusals():
    hc, (c, _, q0) = replay.state_before_last(W)
    cfg = replay.cfg_of(W)
    with pytest.raises(ValueError):
        oracle.snapshot(hc, cfg, 1 << (W.window_chunks + 1), q0)
    img = oracle.snapshot(hc, cfg, 1, q0)
    other = replay.new_host_cache(scaled(W, hist_cap=W.hist_cap + W.C))
    assert oracle.restore(other, replay.cfg_of(scaled(W, hist_cap=W.hist_cap + W.C)), img)[0] == oracle.EINVAL
    bad = img.copy()
    bad[0] ^= 1
    assert oracle.restore(hc.copy(), cfg, bad)[0] == oracle.EINVAL
    assert oracle.restore(hc.copy(), cfg, img[:-1])[0] == oracle.EINVAL
