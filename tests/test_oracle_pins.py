"""Pins of the CPU oracle against what the page and the mathematics fix (no GPU).

Page: "DeCoPrune이 디노이징 불일치로 비디오 KV 캐시를 85% 줄인다" (onedev.kr/papers/726).  Each test names the
section its expectation comes from.  None of these expectations is produced by the oracle itself or by the CUDA
path: they are the page's printed values, hand-derived closed forms (tests/golden), invariants of the definitions,
textbook identities checked through numpy (complex rotation, nonzero), or brute force.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from oracle import replay
from synth.workloads import TINY, scaled

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ------------------------------------------------------------------------------------------ page constants
def test_page_constants():
    """Section 'premises and limits': schedule (999, 957, 899, 702), probe index 2 -> tau* = 899, gamma 0.10."""
    g = {ln[0]: ln[1:] for ln in _golden_lines("page_constants.txt")}
    sched = [int(x) for x in g["schedule"]]
    assert [oracle.lib().oracle_schedule(i) for i in range(4)] == sched
    assert oracle.lib().oracle_probe_index() == int(g["probe_index"][0])
    assert oracle.lib().oracle_schedule(oracle.lib().oracle_probe_index()) == int(g["tau_star"][0]) == 899
    assert oracle.lib().oracle_default_gamma() == np.float32(float(g["gamma"][0]))
    assert oracle.lib().oracle_schedule(4) == -1
    assert oracle.Cfg().frames_per_chunk == int(g["frames_per_chunk"][0])


# ------------------------------------------------------------------------------------------ score
def _score_rows():
    rows = []
    for ln in _golden_lines("score_example.txt"):
        if "|" in ln:
            s = " ".join(ln).split("|")
            rows.append(([float(x) for x in s[0].split()], [float(x) for x in s[1].split()], Fraction(s[2].strip())))
    return rows


def test_score_hand_example():
    """Section 'how it works': l = (1/d)||x0hat - x_final||^2 on hand-worked rows."""
    rows = _score_rows()
    x0 = np.array([r[0] for r in rows], np.float32)
    xr = np.array([r[1] for r in rows], np.float32)
    ell = oracle.score(x0, xr)
    for got, (_, _, want) in zip(ell, rows):
        assert got == np.float32(float(want))


def test_mask_direction_and_tie():
    """Section 'how it works': keep large discrepancy, drop small; the reverse criterion keeps the complement."""
    g = {ln[0]: [int(x) for x in ln[1:]] for ln in _golden_lines("score_example.txt") if "|" not in ln}
    rows = _score_rows()
    ell = oracle.score(np.array([r[0] for r in rows], np.float32), np.array([r[1] for r in rows], np.float32))
    assert oracle.keep(ell, 0.10, 0).tolist() == g["mask"]
    assert oracle.keep(ell, 0.10, 1).tolist() == g["reverse"]
    assert oracle.keep(ell, 0.25, 0).tolist() == g["mask_at_0.25"]


@pytest.mark.parametrize("d", [1, 3, 16, 64, 100])
def test_score_closed_forms(d):
    """l(x, x) = 0 and l(x + c, x) = c^2 for every d (c a power of two so both sides are exact)."""
    x = synth.normal_f32(50 * d, 7, 1).reshape(50, d)
    assert np.all(oracle.score(x, x) == 0.0)
    for c in (0.5, 2.0, 0.125):
        # x has 16 fractional bits and |x| <= 6, so x + c is exact in fp32 and every step of l is exact
        assert np.all(oracle.score((x + np.float32(c)).astype(np.float32), x) == np.float32(c * c))


def test_score_statistics():
    """x0hat = x + s*n with n ~ N(0, 1): l * d / s^2 is chi-square with d degrees of freedom (mean d, var 2d)."""
    n, d, s = 20000, 64, 0.3
    x = synth.normal_f32(n * d, 11, 1).reshape(n, d)
    z = synth.normal_f32(n * d, 11, 2).reshape(n, d)
    x0 = (x.astype(np.float64) + s * z).astype(np.float32)
    q = oracle.score(x0, x).astype(np.float64) * d / (s * s)
    assert abs(q.mean() - d) < 5 * math.sqrt(2 * d / n)
    # the generator's normals are Irwin-Hall sums of 12 uniforms: E z^4 = 2.9, so Var(z^2) = 1.9 (not 2)
    assert abs(q.var() / (1.9 * d) - 1) < 0.04


# ------------------------------------------------------------------------------------------ indices
@pytest.mark.parametrize("n,p", [(0, 0.5), (1, 1.0), (1, 0.0), (64, 0.3), (6240, 0.15), (1000, 1.0), (1000, 0.0)])
def test_indices_are_nonzero_in_order(n, p):
    """Section 'how it works': K[m], V[m] keeps the selected entries; m is the ordered list of kept positions."""
    u = synth.uniform_f64(max(n, 1), 3, 5)[:n]
    mask = (u < p).astype(np.uint8)
    idx = oracle.indices(mask) if n else np.zeros(0, np.int32)
    assert np.array_equal(idx, np.flatnonzero(mask))
    assert len(idx) == int(mask.sum())


# ------------------------------------------------------------------------------------------ g and the phase map
def test_g_and_phase_golden():
    """Section 'what differs': t~(t) = q0 - g(q0 - t) with hand-derived values of g."""
    for ln in _golden_lines("g_map.txt"):
        if ln[0] == "g":
            mode, R, S, dmax, delta = int(ln[1]), float(ln[2]), float(ln[3]), float(ln[4]), float(ln[5])
            want = float(Fraction(ln[6]))
            assert oracle.g(delta, dmax, R, S, mode) == pytest.approx(want, rel=1e-15, abs=1e-13)
        else:
            t, q0, T_s, R, S, mode = (float(x) for x in ln[1:7])
            want = float(Fraction(ln[7]))
            assert oracle.phase(t, q0, T_s, R, S, int(mode)) == pytest.approx(want, rel=1e-15, abs=1e-13)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("dmax", [10.0, 16.0, 40.0, 120.0, 300.0])
def test_g_properties(mode, dmax):
    """g is the identity on recent offsets, continuous at R, monotone, maps the oldest offset to the span end and
    never expands."""
    R, S = 12.0, 24.0
    end = S if mode == 0 else R + S
    ds = np.linspace(0.0, dmax, 997)
    gs = np.array([oracle.g(x, dmax, R, S, mode) for x in ds])
    assert np.all(gs[ds <= R] == ds[ds <= R])
    assert np.all(np.diff(gs) >= 0)
    assert np.all(gs <= ds + 1e-12)
    if dmax > end:
        assert oracle.g(dmax, dmax, R, S, mode) == pytest.approx(end, rel=1e-14)
        assert oracle.g(R + 1e-9, dmax, R, S, mode) == pytest.approx(R, abs=1e-8)
    else:
        assert np.all(gs == ds)


def test_theta_ladder():
    """theta_p = base^(-p/n_t): theta_0 = 1, theta_{n_t/2} = base^(-1/2), constant ratio between rungs."""
    assert oracle.theta(0, 22, 1e4) == 1.0
    assert oracle.theta(4, 8, 1e4) == pytest.approx(0.01, rel=1e-15)
    r = [oracle.theta(p + 1, 22, 1e4) / oracle.theta(p, 22, 1e4) for p in range(21)]
    assert np.allclose(r, 1e4 ** (-1 / 22), rtol=1e-14, atol=0)


# ------------------------------------------------------------------------------------------ rounding
def test_bf16_round_golden():
    for v, b in _golden_lines("bf16_round.txt"):
        assert oracle.bf16_round(float.fromhex(v)) == int(b, 16), v


def test_bf16_round_brute_force():
    """Nearest bf16 (ties to even) by exact rational comparison against both neighbours."""
    xs = synth.uniform_f64(3000, 5, 1) * 8.0 - 4.0
    xs = np.concatenate([xs, xs * 1e-38, xs * 1e37])
    for x in xs:
        b = oracle.bf16_round(float(x))
        got = Fraction(oracle.bf16_value(b))
        lo_bits = int((np.array([float(x)], np.float32).view(np.uint32)[0] >> 16) & 0xFFFF)
        cands = []
        for cb in (lo_bits - 1, lo_bits, lo_bits + 1, lo_bits + 2):
            cb &= 0xFFFF
            if (cb & 0x7F80) == 0x7F80:
                continue
            cands.append((abs(Fraction(oracle.bf16_value(cb)) - Fraction(float(x))), cb & 1, cb))
        best = min(cands)
        assert abs(got - Fraction(float(x))) == best[0]
        ties = [c for c in cands if c[0] == best[0]]
        if len(ties) > 1:
            assert b & 1 == 0


# ------------------------------------------------------------------------------------------ key rotation
def _rot_np(row: np.ndarray, n_t: int, base: float, dphase: float) -> np.ndarray:
    """Textbook RoPE through numpy complex arithmetic: pair (a, b) -> (a + ib) * exp(i * theta_p * dphase)."""
    out = row.astype(np.float64).copy()
    p = np.arange(n_t)
    z = (out[0:2 * n_t:2] + 1j * out[1:2 * n_t:2]) * np.exp(1j * (base ** (-p / n_t)) * dphase)
    out[0:2 * n_t:2], out[1:2 * n_t:2] = z.real, z.imag
    return out


def pair_err(got: np.ndarray, want: np.ndarray, n_t: int) -> float:
    """Largest error of a temporal component relative to the length of its pair (rotation errors scale with it)."""
    g = np.asarray(got, np.float64)[: 2 * n_t].reshape(n_t, 2)
    w = np.asarray(want, np.float64)[: 2 * n_t].reshape(n_t, 2)
    norm = np.maximum(np.hypot(w[:, 0], w[:, 1]), 1e-300)
    return float((np.abs(g - w).max(axis=1) / norm).max())


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def test_rotation_matches_complex_multiplication():
    """Section 'what differs': only the key's temporal phase changes; pairs turn like complex numbers."""
    D, n_t, base = 32, 8, 1e4
    x = synth.normal_f32(D * 40, 9, 1).reshape(40, D)
    dph = synth.uniform_f64(40, 9, 2) * 200 - 100
    for i in range(40):
        row = x[i].copy()
        oracle.rotate_key_row(row, n_t, base, float(dph[i]))
        want = _rot_np(x[i], n_t, base, float(dph[i])).astype(np.float32)
        assert np.all(replay.ulp_distance(row[:2 * n_t], want[:2 * n_t]) <= 1)
        assert np.array_equal(row[2 * n_t:], x[i][2 * n_t:]), "non-temporal dims are copied bitwise"


def test_rotation_quarter_turn_and_zero():
    row = np.array([1.0, 0.0, 0.5, 0.25], np.float32)
    r0 = row.copy()
    oracle.rotate_key_row(r0, 2, 1e4, 0.0)
    assert np.array_equal(r0, row), "a zero turn leaves the key bitwise unchanged"
    r1 = row.copy()
    oracle.rotate_key_row(r1, 1, 1e4, math.pi / 2)   # theta_0 = 1: (a, b) -> (-b, a)
    assert abs(r1[0]) < 1e-15 and r1[1] == 1.0 and np.array_equal(r1[2:], row[2:])
    r2 = np.array([0.5, 0.25], np.float32)
    oracle.rotate_key_row(r2, 1, 1e4, math.pi)
    assert np.allclose(r2, [-0.5, -0.25], atol=1e-7)


def test_rephase_equals_direct_rotation_bf16():
    """Re-phasing a rotated key from t to t~ equals rotating the raw key at t~ directly (within 1 bf16 ulp)."""
    D, n_t, base = 128, 22, 1e4
    raw = synth.normal_f32(D * 64, 4, 1).reshape(64, D).astype(np.float64)
    t = 50.0
    t_new = oracle.phase(t, 124, 4, 12, 24, 0)
    assert t_new != t
    for i in range(64):
        stored = np.array([oracle.bf16_round(v) for v in _rot_np(raw[i], n_t, base, t)], np.uint16)
        oracle.rotate_key_row(stored, n_t, base, t_new - t)
        direct = np.array([oracle.bf16_round(v) for v in _rot_np(raw[i], n_t, base, t_new)], np.uint16)
        # stored was rounded once at t, so the re-phased value may carry that rounding plus its own: <= 1 ulp of
        # the direct value for almost all entries, and never more than 2
        # stored was rounded once at t and once more after the turn: two bf16 roundings of the pair
        assert pair_err(bf16_to_f64(stored), bf16_to_f64(direct), n_t) <= 2 * 2.0 ** -8
        assert np.array_equal(stored[2 * n_t:], direct[2 * n_t:])


def test_rotation_composes():
    """Turning by phi1 then phi2 equals turning by phi1 + phi2 (fp32 storage, within 2 ulp)."""
    x = synth.normal_f32(32 * 20, 8, 3).reshape(20, 32)
    for i in range(20):
        a = x[i].copy()
        oracle.rotate_key_row(a, 8, 1e4, 3.25)
        oracle.rotate_key_row(a, 8, 1e4, -1.5)
        b = x[i].copy()
        oracle.rotate_key_row(b, 8, 1e4, 1.75)
        assert pair_err(a, b, 8) <= 3 * 2.0 ** -24
        assert np.array_equal(a[16:], b[16:])


# ------------------------------------------------------------------------------------------ compaction
def _tiny_state():
    return replay.state_before_last(TINY)


def test_compaction_invariants():
    """Section 'how it works': the kept rows move in order, one mask for all layers and heads, V copied bitwise, K
    copied bitwise outside the temporal pairs and turned to t~ inside them, sink and window untouched."""
    w = TINY
    hc, (c, q0_prev, q0) = _tiny_state()
    before = hc.copy()
    x0, xr = w.score_inputs(c)
    mask = oracle.keep(oracle.score(x0, xr))
    idx = np.flatnonzero(mask)
    rc, got_idx = oracle.compact_layers(hc, replay.cfg_of(w), w.slot_of(c), w.first_frame(c), mask, None, q0)
    assert rc == oracle.OK and np.array_equal(got_idx, idx)
    k = len(idx)
    L0 = int(before.hist_len[0])
    src0 = w.win_row0 + w.slot_of(c) * w.C
    assert np.all(hc.hist_len == L0 + k)
    assert np.array_equal(hc.hist_t[L0:L0 + k], w.first_frame(c) + idx // w.tokens_per_frame)
    n_t = w.n_temporal_pairs
    for l in range(w.L):
        for h in range(w.H):
            src_v = before.v[l, h, src0 + idx]
            assert np.array_equal(hc.v[l, h, w.sink_rows + L0: w.sink_rows + L0 + k], src_v)
            dst_k = hc.k[l, h, w.sink_rows + L0: w.sink_rows + L0 + k]
            src_k = before.k[l, h, src0 + idx]
            assert np.array_equal(dst_k[:, 2 * n_t:], src_k[:, 2 * n_t:])
            for j in range(k):
                t = w.first_frame(c) + idx[j] // w.tokens_per_frame
                want = _rot_np(src_k[j], n_t, w.rope_base, oracle.phase(t, q0, w.sink_chunks * w.F, w.R, w.S) - t)
                assert pair_err(dst_k[j], want, n_t) <= 2.0 ** -24
    keep_rows = np.ones(w.cap, bool)
    keep_rows[w.sink_rows + L0: w.sink_rows + L0 + k] = False
    assert np.array_equal(hc.k[:, :, keep_rows], before.k[:, :, keep_rows])
    assert np.array_equal(hc.v[:, :, keep_rows], before.v[:, :, keep_rows])


def test_compaction_head_specialised():
    """Section 'what differs': static heads follow Streaming (keep nothing of the leaving chunk)."""
    w = TINY
    hc, (c, q0_prev, q0) = _tiny_state()
    static = np.zeros(w.n_planes, np.uint8)
    static[1] = 1
    static[2] = 1
    hc.hist_len[static == 1] = 0
    before = hc.copy()
    mask = oracle.keep(oracle.score(*w.score_inputs(c)))
    rc, idx = oracle.compact_layers(hc, replay.cfg_of(w), w.slot_of(c), w.first_frame(c), mask, static, q0)
    assert rc == oracle.OK
    assert np.all(hc.hist_len[static == 1] == 0)
    assert np.all(hc.hist_len[static == 0] == before.hist_len[static == 0] + len(idx))
    kv = hc.k.reshape(w.n_planes, w.cap, w.D)
    assert np.array_equal(kv[static == 1], before.k.reshape(w.n_planes, w.cap, w.D)[static == 1])


def test_compaction_refusals_change_nothing():
    w = TINY
    hc, (c, q0_prev, q0) = _tiny_state()
    mask = np.ones(w.C, np.uint8)
    small = replay.HostCache(hc.k, hc.v, hc.hist_len, hc.hist_t, int(hc.hist_len[0]) + w.C - 1)
    before = small.copy()
    rc, _ = oracle.compact_layers(small, replay.cfg_of(w), w.slot_of(c), w.first_frame(c), mask, None, q0)
    assert rc == oracle.ECAPACITY
    assert np.array_equal(small.k, before.k) and np.array_equal(small.hist_len, before.hist_len)
    hc2 = hc.copy()
    hc2.hist_len[3] += 1
    before2 = hc2.copy()
    rc, _ = oracle.compact_layers(hc2, replay.cfg_of(w), w.slot_of(c), w.first_frame(c), mask, None, q0)
    assert rc == oracle.EINVAL and np.array_equal(hc2.k, before2.k)


def test_compaction_all_and_none():
    w = TINY
    for fill in (0, 1):
        hc, (c, _, q0) = _tiny_state()
        L0 = int(hc.hist_len[0])
        rc, idx = oracle.compact_layers(hc, replay.cfg_of(w), w.slot_of(c), w.first_frame(c),
                                        np.full(w.C, fill, np.uint8), None, q0)
        assert rc == oracle.OK and len(idx) == fill * w.C and np.all(hc.hist_len == L0 + fill * w.C)


# ------------------------------------------------------------------------------------------ history re-index
def test_rope_reindex_equals_direct_rotation():
    """Section 'what differs': a history key stored at phase t~(t; q0a) and re-indexed to q0b equals the raw key
    rotated directly at t~(t; q0b); values are untouched."""
    w = scaled(TINY, hist_cap=40, max_frames=512)
    D, n_t = w.D, w.n_temporal_pairs
    T_s = w.sink_chunks * w.F
    hc = replay.new_host_cache(w)
    frames = np.sort(synth.uniform_f64(40, 2, 2) * 60 + T_s).astype(np.int32)
    raw = synth.normal_f32(w.n_planes * 40 * D, 2, 3).reshape(w.n_planes, 40, D).astype(np.float64)
    q0a, q0b = 70, 80
    for p in range(w.n_planes):
        for j in range(40):
            ta = oracle.phase(float(frames[j]), q0a, T_s, w.R, w.S)
            hc.k.reshape(w.n_planes, w.cap, D)[p, w.sink_rows + j] = _rot_np(raw[p, j], n_t, w.rope_base, ta)
    hc.hist_len[:] = 40
    hc.hist_t[:40] = frames
    before = hc.copy()
    assert oracle.rope_reindex(hc, replay.cfg_of(w), q0a, q0b) == oracle.OK
    kk = hc.k.reshape(w.n_planes, w.cap, D)
    for p in range(w.n_planes):
        for j in range(40):
            tb = oracle.phase(float(frames[j]), q0b, T_s, w.R, w.S)
            want = _rot_np(raw[p, j], n_t, w.rope_base, tb)
            assert pair_err(kk[p, w.sink_rows + j], want, n_t) <= 2 * 2.0 ** -24
            assert np.array_equal(kk[p, w.sink_rows + j, 2 * n_t:], want[2 * n_t:].astype(np.float32))
    assert np.array_equal(hc.v, before.v)


def test_rope_reindex_identity_when_no_compression():
    """g is the identity when the oldest offset fits the span: nothing moves (bitwise)."""
    hc, (c, q0_prev, q0) = _tiny_state()   # q0 = 8, first non-sink frame 1: Dmax = 7 <= S = 16
    before = hc.copy()
    assert oracle.rope_reindex(hc, replay.cfg_of(TINY), q0_prev, q0) == oracle.OK
    assert np.array_equal(hc.k, before.k)


def test_prune_step_is_reindex_then_compact():
    w = scaled(TINY, R=2, S=4, hist_cap=5 * 64)   # Dmax = 7 > S, so the history does move
    a, (c, q0_prev, q0) = replay.state_before_last(w)
    b = a.copy()
    x0, xr = w.score_inputs(c)
    rc, ell, mask, idx = oracle.prune_step(a, replay.cfg_of(w), x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0)
    assert rc == oracle.OK
    assert oracle.rope_reindex(b, replay.cfg_of(w), q0_prev, q0) == oracle.OK
    rc2, idx2 = oracle.compact_layers(b, replay.cfg_of(w), w.slot_of(c), w.first_frame(c), mask, None, q0)
    assert rc2 == oracle.OK and np.array_equal(idx, idx2)
    assert np.array_equal(a.k, b.k) and np.array_equal(a.v, b.v) and np.array_equal(a.hist_len, b.hist_len)
    fresh = replay.state_before_last(w)[0]
    L0 = int(fresh.hist_len[0])
    assert not np.array_equal(a.k[:, :, w.sink_rows:w.sink_rows + L0], fresh.k[:, :, w.sink_rows:w.sink_rows + L0])


# ------------------------------------------------------------------------------------------ PR
def test_pr_brute_force_rollout():
    """Section 'how to use': PR = cumulative reduction of history KV positions visible to attention, counted per
    chunk and (layer, head), against FullKV.  Brute force: list the visible positions of every plane."""
    w = scaled(TINY, rollout_chunks=14, hist_cap=14 * 64, history_chunks=(), max_frames=64)
    hc = replay.new_host_cache(w)
    acc = [0, 0]
    brute_vis = brute_full = 0
    evictions = {c: (q0p, q0) for c, q0p, q0 in w.evictions()}
    placed = set()
    for i in range(1, w.rollout_chunks):
        # chunk i attends to everything before it that the cache still holds
        resident = [cc for cc in range(w.sink_chunks, i) if cc > i - 1 - w.window_chunks]
        for p in range(w.n_planes):
            pos = set(range(w.sink_rows)) | {("h", j) for j in range(int(hc.hist_len[p]))}
            pos |= {(cc, r) for cc in resident for r in range(w.C)}
            brute_vis += len(pos)
        brute_full += w.n_planes * i * w.C
        oracle.pr_chunk(hc.hist_len, w.sink_rows, len(resident) * w.C, i * w.C, acc)
        # chunk i is generated; if the ring is full, its oldest chunk leaves
        placed.add(i)
        c_out = i - w.window_chunks
        if c_out in evictions:
            replay.replay(w, hc, [(c_out, *evictions[c_out])], placed=placed)
    assert acc == [brute_vis, brute_full]
    pr = 1 - acc[0] / acc[1]
    assert 0.0 < pr < 1.0


def test_pr_tends_to_drop_fraction():
    """Sanity of the definition: if every leaving chunk keeps a fraction p, PR approaches 1 - p as the rollout
    grows (the page's ~85% PR pairs with ~15% kept)."""
    C, n, p = 1000, 2000, 0.15
    vis = full = 0
    hist = 0
    for i in range(1, n):
        resident = min(3, max(0, i - 1))
        vis += C + hist + resident * C
        full += i * C
        if i - 1 >= 4:
            hist += int(p * C)
    assert abs((1 - vis / full) - (1 - p)) < 0.02


# ------------------------------------------------------------------------------------------ Random ablation
def test_splitmix64_published_outputs():
    """The generator of the Random ablation reproduces the published SplitMix64 outputs for seed 1234567."""
    for seed, i, want in _golden_lines("splitmix64.txt"):
        assert oracle.splitmix64(int(seed), int(i)) == int(want)


def _ell_with_k(n, k, seed):
    rng = np.random.default_rng(seed)
    ell = rng.uniform(0.0, 0.09, n).astype(np.float32)
    ell[rng.choice(n, k, replace=False)] = rng.uniform(0.11, 2.0, k).astype(np.float32)
    return ell


@pytest.mark.parametrize("n,k", [(64, 0), (64, 64), (64, 9), (1000, 151), (6240, 947)])
def test_random_keeps_the_discrepancy_count(n, k):
    """Section 'premises and limits': Random is compared at the same compression ratio, so it keeps exactly as many
    tokens as the discrepancy rule; the kept set is the k smallest generator outputs (every kept output is below every
    dropped one), and it does not depend on which tokens have large discrepancy."""
    ell = _ell_with_k(n, k, 7 + n + k)
    stream = (0xC0FFEE << 32) | 17
    m = oracle.keep_random(ell, 0.10, stream)
    assert int(m.sum()) == k == int((ell > np.float32(0.10)).sum())
    z = np.array([oracle.splitmix64(stream, i) for i in range(n)], dtype=np.uint64)
    assert len(set(z.tolist())) == n
    if 0 < k < n:
        assert z[m == 1].max() < z[m == 0].min()
    perm = np.random.default_rng(3).permutation(n)
    assert np.array_equal(oracle.keep_random(ell[perm], 0.10, stream), m)
    assert not np.array_equal(oracle.keep_random(ell, 0.10, stream + 1), m) or k in (0, n)


def test_random_draw_is_uniform_over_subsets():
    """A uniform draw of k of n tokens without replacement: each token is kept with probability k/n and each pair
    with probability k(k-1)/(n(n-1)).  Checked over 3000 streams (n = 12, k = 4) within 5 standard deviations."""
    n, k, reps = 12, 4, 3000
    ell = _ell_with_k(n, k, 5)
    single = np.zeros(n)
    pair = np.zeros((n, n))
    for r in range(reps):
        m = oracle.keep_random(ell, 0.10, (r * 0x9E3779B1) & ((1 << 64) - 1)).astype(np.float64)
        single += m
        pair += np.outer(m, m)
    p1 = k / n
    assert np.all(np.abs(single / reps - p1) < 5 * math.sqrt(p1 * (1 - p1) / reps))
    p2 = k * (k - 1) / (n * (n - 1))
    off = pair[~np.eye(n, dtype=bool)] / reps
    assert np.all(np.abs(off - p2) < 5 * math.sqrt(p2 * (1 - p2) / reps))


def test_random_prune_step_stream():
    """A prune step under keep_rule 2 draws from the stream (random_seed << 32) | evict_first_frame and moves the
    same number of rows as the discrepancy rule."""
    w = TINY
    hc, ev = replay.state_before_last(w)
    c, q0_prev, q0 = ev
    cfg = replay.cfg_of(w)
    cfg.keep_rule, cfg.random_seed = 2, 0xABCDEF
    x0, xr = w.score_inputs(c)
    ef = w.first_frame(c)
    h2 = hc.copy()
    rc, ell, mask, idx = oracle.prune_step(h2, cfg, x0, xr, w.slot_of(c), ef, q0_prev, q0)
    assert rc == oracle.OK
    assert np.array_equal(mask, oracle.keep_random(ell, cfg.gamma, cfg.random_stream(ef)))
    assert len(idx) == int((ell > np.float32(cfg.gamma)).sum())
    assert np.array_equal(idx, np.flatnonzero(mask))
