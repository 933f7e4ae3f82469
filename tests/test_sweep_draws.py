"""The seeded geometries of the GPU sweep (tests/test_gpu_sweep.py) are valid method inputs: each one's eviction
schedule replays in the oracle with every step accepted, and the draws reach the variety the sweep claims."""
import numpy as np

from oracle import replay
import oracle
from tests.test_gpu_sweep import (BOUNDARY, N_BIG, N_BOUNDARY, N_CASES, N_EDGE, N_STAGED_TURN, N_WIDE, draw, draw_big,
                                  draw_boundary, draw_edge, draw_staged_turn, draw_wide)


def test_sweep_draws_replay_in_the_oracle():
    seen = {"bf16": 0, "fp32": 0, "vec16": 0, "paged": 0, "hs": 0, "lazy": 0, "random": 0, "reverse": 0,
            "mode1": 0, "no_sink": 0, "scalar_score": 0, "turning": 0}
    for case in range(N_CASES):
        w, over, hsm, paged = draw(case)
        cfg = replay.cfg_of(w)
        for key, val in over.items():
            setattr(cfg, key, val)
        hc = replay.new_host_cache(w)
        replay.replay(w, hc, w.evictions(), hsm, cfg=cfg)  # asserts every step returns OK
        assert int(hc.hist_len.max()) <= w.hist_cap
        seen["bf16" if w.dtype == 0 else "fp32"] += 1
        seen["vec16"] += (w.D * w.esize) % 32 != 0
        seen["paged"] += paged is not None
        seen["hs"] += hsm is not None
        seen["lazy"] += over["reindex_mode"] == 1
        seen["random"] += over["keep_rule"] == 2
        seen["reverse"] += over["keep_rule"] == 1
        seen["mode1"] += w.g_mode == 1
        seen["no_sink"] += w.sink_chunks == 0
        seen["scalar_score"] += w.d % 4 != 0
        q0_last = w.evictions()[-1][2]
        seen["turning"] += w.n_temporal_pairs > 0 and (q0_last - w.sink_chunks * w.F) > (w.S if w.g_mode == 0 else w.R + w.S)
    assert all(v > 0 for v in seen.values()), seen


def test_draws_reach_both_reindex_paths():
    """Steps that re-index a history turn it in the gather's own launch when every plane receives, and in a re-index
    kernel of its own before the gather when some heads are static: the narrow draws reach both."""
    fused = separate = 0
    for case in range(N_CASES):
        w, over, hsm, _ = draw(case)
        if over["reindex_mode"] == 1 or w.n_temporal_pairs == 0:
            continue
        T_s, end = w.sink_chunks * w.F, (w.S if w.g_mode == 0 else w.R + w.S)
        for i, (c, q0_prev, q0) in enumerate(w.evictions()):
            if i > 0 and q0 != q0_prev and (q0 - T_s > end or q0_prev - T_s > end):  # history keys turn
                separate += hsm is not None
                fused += hsm is None
    assert fused > 0 and separate > 0, (fused, separate)


def test_wide_draws_replay_in_the_oracle():
    """The wide draws (1024+ planes, rows of at most 288 bytes) replay in the oracle, and some of their steps turn no
    kept key (the staged gather) while others turn (the register-staged one)."""
    still = turning = n_paged = 0
    for case in range(N_WIDE):
        w, over, hsm, paged = draw_wide(case)
        n_paged += paged is not None
        assert w.n_planes >= 1024 and w.D * w.esize <= 288 and (w.D * w.esize) % 16 == 0
        cfg = replay.cfg_of(w)
        for key, val in over.items():
            setattr(cfg, key, val)
        hc = replay.new_host_cache(w)
        replay.replay(w, hc, w.evictions(), hsm, cfg=cfg)
        for c, _, q0 in w.evictions():
            # the leaving chunk's keys turn iff its offsets reach past R while g compresses (mode 0: q0 - T_s > S)
            turns = w.n_temporal_pairs > 0 and q0 - w.sink_chunks * w.F > w.S and q0 - c * w.F > w.R
            turning += turns
            still += not turns
    assert still > 0 and turning > 0 and n_paged > 0, (still, turning, n_paged)


def test_big_draws_replay_in_the_oracle():
    """The big-row draws are valid (rows of at most 4 KiB, the gather's table fits) and replay in the oracle."""
    sizes = set()
    for case in range(N_BIG):
        w, over, hsm, _ = draw_big(case)
        rb = w.D * w.esize
        assert 1024 <= rb <= 4096 and rb % 16 == 0 and w.F * w.n_temporal_pairs * 16 <= 100 * 1024
        sizes.add(rb)
        cfg = replay.cfg_of(w)
        for key, val in over.items():
            setattr(cfg, key, val)
        hc = replay.new_host_cache(w)
        replay.replay(w, hc, w.evictions(), hsm, cfg=cfg)
    assert len(sizes) >= 2, sizes


def test_edge_draws_replay_in_the_oracle():
    """The degenerate-chunk draws (1 to 33 tokens, score rows of 1 to 64 values) replay in the oracle."""
    for case in range(N_EDGE):
        w, over, hsm, _ = draw_edge(case)
        assert 1 <= w.C <= 33
        cfg = replay.cfg_of(w)
        for key, val in over.items():
            setattr(cfg, key, val)
        hc = replay.new_host_cache(w)
        replay.replay(w, hc, w.evictions(), hsm, cfg=cfg)


def test_boundary_draws_turn_exactly_past_the_boundary():
    """On the "at" side of each boundary the oracle's last eviction moves every kept key row bitwise (g is the
    identity on the chunk); one frame past it some kept key turns.  The GPU sweep compares both with the oracle, so a
    no-turn decision taken on the wrong side fails there."""
    for case in range(N_BOUNDARY):
        w, over, hsm, _ = draw_boundary(case)
        _, _, side = BOUNDARY[case]
        assert w.n_planes >= 1024 and w.D * w.esize <= 288
        hc, (c, q0_prev, q0) = replay.state_before_last(w)
        T_s = w.sink_chunks * w.F
        end = w.S if w.g_mode == 0 else w.R + w.S
        if BOUNDARY[case][1] == "recent":
            assert q0 - w.first_frame(c) == (w.R if side == "at" else w.R + 1) and q0 - T_s > end
        else:
            assert q0 - T_s == (end if side == "at" else end + 1) and q0 - w.first_frame(c) > w.R
        src = hc.k[:, :, w.win_row0 + w.slot_of(c) * w.C: w.win_row0 + (w.slot_of(c) + 1) * w.C].copy()
        common = int(hc.hist_len[0])
        rc, _, _, idx = oracle.prune_step(hc, replay.cfg_of(w), *w.score_inputs(c), w.slot_of(c), w.first_frame(c),
                                          q0_prev, q0)
        assert rc == oracle.OK and len(idx) > 0
        moved = hc.k[:, :, w.sink_rows + common: w.sink_rows + common + len(idx)]
        same = np.array_equal(moved, src[:, :, idx])
        assert same == (side == "at"), (case, BOUNDARY[case])


def test_staged_turn_draws_reach_the_turning_staged_gather():
    """The staged-turn draws are valid, every eviction of them turns its kept keys, and the evictions that take the
    staged gather's turning form (1024+ planes, rows of at most 288 bytes, at most 8 temporal 16-byte chunks per row;
    no history re-index in the same step, i.e. q0 unchanged, or static heads, which never fuse the re-index into the
    gather) cover both dtypes, kept counts that fill part of one 64-row block and several, and (cases 6 and up)
    static heads next to receiving ones in every layer."""
    dtypes, ks, hs_cases = set(), [], 0
    for case in range(N_STAGED_TURN):
        w, over, hsm, paged = draw_staged_turn(case)
        ppv = 4 if w.dtype == 0 else 2
        tc = -(-w.n_temporal_pairs // ppv)
        assert paged is None and w.n_planes >= 1024 and w.D * w.esize <= 288 and 1 <= tc <= 8
        assert (hsm is None) == (case < 6)
        if hsm is not None:
            per_layer = hsm.reshape(w.L, w.H).sum(axis=1)
            assert np.all(per_layer >= 1) and np.all(per_layer < w.H)
            hs_cases += 1
        cfg = replay.cfg_of(w)
        for key, val in over.items():
            setattr(cfg, key, val)
        hc = replay.new_host_cache(w)
        placed = set()
        T_s = w.sink_chunks * w.F
        staged = 0
        for c, q0_prev, q0 in w.evictions():
            for cc in w.resident_window(c):
                if cc not in placed:
                    replay.place_chunk(hc, w, cc)
                    placed.add(cc)
            assert q0 - T_s > w.S and q0 - w.first_frame(c) > w.R  # the leaving chunk's oldest frame turns
            rc, _, _, idx = oracle.prune_step(hc, cfg, *w.score_inputs(c), w.slot_of(c), w.first_frame(c), q0_prev,
                                              q0, head_is_static=hsm)
            assert rc == oracle.OK and len(idx) > 0
            if q0_prev == q0 or hsm is not None:
                staged += 1
                ks.append(len(idx))
        assert staged >= 1, case
        dtypes.add(w.dtype)
    assert dtypes == {0, 1}, dtypes
    assert hs_cases == N_STAGED_TURN - 6
    assert min(ks) < 64 < max(ks) and any(k % 64 for k in ks), ks
