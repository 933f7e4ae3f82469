"""Pins of the oracle's read-time re-index (no GPU).

Page "DeCoPrune이 디노이징 불일치로 비디오 KV 캐시를 85% 줄인다" (onedev.kr/papers/726), section "what differs": old
context keys take the temporal phase t~(t) = q0 - g(q0 - t) and only the key phase changes.  Read-time re-index keeps
each history key at its own frame's phase t and turns it once, from t to t~(t; q0), when it is read.  Expectations
here come from numpy's complex arithmetic on the raw rows, the pinned g map and the storage rounding, not from the
oracle's own rotation.
"""
import numpy as np
import pytest

import oracle
from oracle import replay
from synth.workloads import TINY, scaled

TINY_ROT = scaled(TINY, R=2, S=4)
TINY_ROT_BF16 = scaled(TINY, R=2, S=4, dtype=0)


def _lazy(w):
    cfg = replay.cfg_of(w)
    cfg.reindex_mode = 1
    return cfg


def _values(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def test_lazy_step_moves_keys_bitwise_and_leaves_history():
    w = TINY_ROT
    cfg = _lazy(w)
    hc, (c, q0_prev, q0) = replay.state_before_last(w, cfg=cfg)
    o = hc.copy()
    x0, xr = w.score_inputs(c)
    rc, _, _, idx = oracle.prune_step(o, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0)
    assert rc == oracle.OK and q0_prev != q0
    sink, n0 = w.sink_chunks * w.C, int(hc.hist_len[0])
    src = sink + w.hist_cap + w.slot_of(c) * w.C + idx
    assert np.array_equal(o.k[:, :, sink + n0:sink + n0 + len(idx)], hc.k[:, :, src]), "keys move bitwise"
    assert np.array_equal(o.k[:, :, :sink + n0], hc.k[:, :, :sink + n0]), "nothing is re-indexed"


@pytest.mark.parametrize("w", [TINY_ROT, TINY_ROT_BF16], ids=["fp32", "bf16"])
def test_read_turns_each_raw_key_once(w):
    """read(q0) row j of plane p = the raw row with pair k multiplied by exp(i theta_k (t~(t; q0) - t)), rounded once
    to the storage type (numpy complex128; within 1 ulp of the storage type for libm differences)."""
    cfg = _lazy(w)
    hc, (c, q0_prev, q0) = replay.state_before_last(w, cfg=cfg)
    got = oracle.read_history_keys(hc, cfg, q0)
    sink, nt = w.sink_chunks * w.C, w.n_temporal_pairs
    T_s = w.sink_chunks * w.frames_per_chunk
    theta = w.rope_base ** (-np.arange(nt) / nt)
    turned = 0
    for p in range(w.L * w.H):
        l, h = divmod(p, w.H)
        n = int(hc.hist_len[p])
        raw = _values(hc.k[l, h, sink:sink + n])
        t = hc.hist_t[:n].astype(np.float64)
        tt = np.array([oracle.phase(x, q0, T_s, w.R, w.S, w.g_mode) for x in t])
        z = (raw[:, 0:2 * nt:2] + 1j * raw[:, 1:2 * nt:2]) * np.exp(1j * np.outer(tt - t, theta))
        want = raw.copy()
        want[:, 0:2 * nt:2], want[:, 1:2 * nt:2] = z.real, z.imag
        if w.dtype == 0:
            want_bits = np.array([oracle.bf16_round(x) for x in want.ravel()], np.uint16).reshape(want.shape)
        else:
            want_bits = want.astype(np.float32)
        d = replay.ulp_distance(got[p, :n], want_bits)
        assert int(d.max(initial=0)) <= 1
        assert np.array_equal(got[p, :n, 2 * nt:], hc.k[l, h, sink:sink + n, 2 * nt:])
        turned += int(np.count_nonzero(tt != t))
    assert turned > 0, "the case must compress old offsets"


def test_read_is_the_raw_key_when_no_offset_is_compressed():
    """TINY keeps every offset within the span (g is the identity), so reading returns the stored keys bitwise."""
    w = TINY
    cfg = _lazy(w)
    hc, (c, q0_prev, q0) = replay.state_before_last(w, cfg=cfg)
    got = oracle.read_history_keys(hc, cfg, q0)
    sink = w.sink_chunks * w.C
    for p in range(w.L * w.H):
        l, h = divmod(p, w.H)
        n = int(hc.hist_len[p])
        assert np.array_equal(got[p, :n], hc.k[l, h, sink:sink + n])


def test_read_agrees_with_eager_re_indexing():
    """Eager re-indexing (turn at store time and at every step) and read-time re-indexing reach the same keys up to
    the rounding the eager path adds at each of its steps."""
    w = scaled(TINY_ROT, history_chunks=(1, 2, 3, 4))
    eager, (c, q0_now, _) = replay.state_before_last(w)  # eager keys are at the phase of the last step's q0
    lazy, _ = replay.state_before_last(w, cfg=_lazy(w))
    got = oracle.read_history_keys(lazy, _lazy(w), q0_now)
    sink, nt = w.sink_chunks * w.C, w.n_temporal_pairs
    steps = len(w.evictions())
    for p in range(w.L * w.H):
        l, h = divmod(p, w.H)
        n = int(eager.hist_len[p])
        assert n == int(lazy.hist_len[p])
        a, b = _values(got[p, :n]), _values(eager.k[l, h, sink:sink + n])
        assert np.array_equal(a[:, 2 * nt:], b[:, 2 * nt:])
        # each eager step rounds each component once (relative 2^-24 of the pair's length, fp32 storage)
        norm = np.repeat(np.hypot(b[:, 0:2 * nt:2], b[:, 1:2 * nt:2]), 2, axis=1)
        assert np.all(np.abs(a[:, :2 * nt] - b[:, :2 * nt]) <= 2.0 * steps * 2.0 ** -24 * norm + 1e-30)
