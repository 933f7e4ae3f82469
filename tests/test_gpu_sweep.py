"""Seeded sweep of small geometries: every eviction of each drawn workload runs on the GPU and in the oracle from the
same host state, with the bars of test_gpu_parity.py (masks, indices, lengths, frames, values and non-temporal key
dims bit-exact; turned key dims within 1 bf16 ulp, or 2 fp32 ulp plus 2^-38 of the pair).

The draws cover what the fixed cases leave at one value: bf16 and fp32 rows of 16 to 544 bytes (16-byte vectors when a
row is not a multiple of 32 bytes), 0 to D/2 temporal pairs, ragged chunks (3 to 64 tokens per frame, 1 to 3 frames),
score rows of 3 to 64 values (scalar and vector scoring paths), 0 to 2 sink chunks, 1 to 3 window chunks, both maps
g, R and S from the identity to strong compression, the three keep rules, head-specialised steps, paged caches of
both layouts with several block sizes, and read-time re-indexing (with the final read, contiguous or paged, checked
against the oracle's).
Wide draws (1024 to 1600 planes, rows of at most 288 bytes, short chunks) run steps that turn no kept key on the
shared-memory staged gather, across row sizes and dtypes, and steps that turn on the register-staged gather; some of
them run on paged pools (HND or NHD, 8 to 32 positions per block), which take the register-staged gather.  Big
draws use rows of 1 to 4 KiB (the largest the library takes) with up to 1024 temporal pairs; edge draws use chunks of
1 to 33 tokens and score rows of 1 to 64 values.  Boundary draws put the last eviction exactly on the edge of g's
identity on the leaving chunk (where the library skips the chunk's turn) and one frame past it, for both maps g;
staged-turn draws put steps whose keys turn on the staged gather's turning form in bf16 and fp32, with and without
static heads.
"""
import numpy as np
import pytest
import torch

import autoregressive_video_diffusion_gb300 as dcp
import oracle
from oracle import replay
from synth.workloads import TINY, scaled
from tests import devcache
from tests.paged import PagedCopy
from tests.test_gpu_paged import paged_vs_oracle_step
from tests.test_gpu_parity import assert_key_parity, gpu_vs_oracle_step

pytestmark = pytest.mark.gpu

N_CASES = 128


def _clear_of_tie_band(w) -> bool:
    for c, _, _ in w.evictions():
        ell = oracle.score(*w.score_inputs(c))
        if np.min(np.abs(ell.astype(np.float64) - np.float32(w.gamma))) < 1e-6:
            return False
    return True


def draw(case: int):
    """A seeded workload and the options of one sweep case: (workload, config overrides, static-head mask or None,
    (block size, layout) or None)."""
    r = np.random.default_rng(0x5EE9 + case)
    dtype = int(r.integers(0, 2))
    D = int(r.choice([8, 16, 24, 40, 64, 72, 128, 136] if dtype == 0 else [4, 8, 12, 20, 36, 64]))
    F, T = int(r.integers(1, 4)), int(r.choice([3, 5, 8, 16, 33, 64]))
    sink, win = int(r.integers(0, 3)), int(r.integers(1, 4))
    g_mode = int(r.integers(0, 2))
    R = win * F + int(r.integers(0, 3))
    S = R + int(r.integers(0, 9)) if g_mode == 0 else int(r.integers(0, 10))
    n_ev = int(r.integers(1, 6))
    C = T * F
    last = sink + n_ev - 1
    w = scaled(TINY, name=f"sweep_{case}", index=100 + case, L=int(r.integers(1, 4)), H=int(r.integers(1, 6)), D=D,
               dtype=dtype, n_temporal_pairs=int(r.integers(0, D // 2 + 1)),
               rope_base=float(r.choice([1e4, 500.0])), tokens_per_frame=T, frames_per_chunk=F,
               d=int(r.choice([3, 8, 16, 64])), sink_chunks=sink, window_chunks=win, R=float(R), S=float(S),
               g_mode=g_mode, hist_cap=n_ev * C, max_frames=(last + win + 2) * F, evict_chunk=last,
               history_chunks=tuple(range(sink, last)), seed=5000 + case)
    if w.H > 1 and r.random() < 0.3:
        w = scaled(w, n_static_per_layer=int(r.integers(1, w.H)))
    over = {"keep_rule": int(r.choice([0, 0, 1, 2])), "random_seed": int(r.integers(0, 1 << 32)),
            "reindex_mode": int(r.random() < 0.25)}
    paged = None
    if r.random() < 0.35:
        bs = int(r.choice([b for b in (1, 2, 4, 8, 16, 32) if C % b == 0]))
        paged = (bs, int(r.integers(0, 2)))
    while not _clear_of_tie_band(w):  # keep every score clear of gamma so both sides take the same decisions
        w = scaled(w, seed=w.seed + 100)
    return w, over, w.head_is_static(), paged


def draw_wide(case: int):
    """A seeded workload of 1024 to 1600 planes with short chunks and rows of at most 288 bytes: the caches on which
    steps whose kept keys do not turn take the shared-memory staged gather."""
    r = np.random.default_rng(0x91DE + case)
    dtype = int(r.integers(0, 2))
    D = int(r.choice([8, 16, 64, 72, 128, 136] if dtype == 0 else [4, 20, 36, 64, 72]))
    F, T = int(r.integers(1, 3)), int(r.choice([3, 8, 16]))
    sink, win = int(r.integers(0, 3)), int(r.integers(1, 4))
    R = win * F + int(r.integers(0, F))  # below (w + 1) F: the leaving chunk's oldest frames lie past R
    S = R + int(r.choice([0, 2, 30]))
    n_ev = int(r.integers(1, 4))
    last = sink + n_ev - 1
    w = scaled(TINY, name=f"sweep_wide_{case}", index=200 + case, L=int(r.choice([32, 40])),
               H=int(r.choice([32, 40])), D=D, dtype=dtype, n_temporal_pairs=int(r.integers(0, D // 2 + 1)),
               tokens_per_frame=T, frames_per_chunk=F, d=int(r.choice([3, 16])), sink_chunks=sink,
               window_chunks=win, R=float(R), S=float(S), g_mode=0, hist_cap=n_ev * T * F,
               max_frames=(last + win + 2) * F, evict_chunk=last, history_chunks=tuple(range(sink, last)),
               seed=7000 + case)
    if r.random() < 0.4:
        w = scaled(w, n_static_per_layer=int(r.integers(1, w.H)))
    over = {"keep_rule": int(r.choice([0, 1, 2])), "random_seed": int(r.integers(0, 1 << 32)), "reindex_mode": 0}
    paged = None
    sizes = [b for b in (8, 16, 32) if (T * F) % b == 0]
    if sizes and r.random() < 0.5:  # paged pools of many planes
        paged = (int(r.choice(sizes)), int(r.choice([0, 0, 1])))
    while not _clear_of_tie_band(w):
        w = scaled(w, seed=w.seed + 100)
    return w, over, w.head_is_static(), paged


N_WIDE = 16


def draw_big(case: int):
    """A seeded workload with long rows (1 to 4 KiB, the largest the library takes) and long temporal parts: few
    rows per CTA in every kernel, many vectors per row."""
    r = np.random.default_rng(0xB16 + case)
    dtype = int(r.integers(0, 2))
    D = int(r.choice([512, 1024, 2048] if dtype == 0 else [256, 512, 1024]))
    F, T = int(r.integers(1, 3)), int(r.choice([4, 9, 16]))
    win = int(r.integers(1, 3))
    R = win * F + int(r.integers(0, F))
    S = R + int(r.choice([0, 3]))
    n_ev = int(r.integers(2, 5))
    last = 1 + n_ev - 1
    n_t = int(r.integers(1, min(D // 2, 1024 // F) + 1))  # the gather keeps F x n_t table entries in shared memory
    w = scaled(TINY, name=f"sweep_big_{case}", index=300 + case, L=int(r.integers(1, 3)), H=int(r.integers(1, 4)),
               D=D, dtype=dtype, n_temporal_pairs=n_t, tokens_per_frame=T, frames_per_chunk=F, d=16, sink_chunks=1,
               window_chunks=win, R=float(R), S=float(S), g_mode=0, hist_cap=n_ev * T * F,
               max_frames=(last + win + 2) * F, evict_chunk=last, history_chunks=tuple(range(1, last)),
               seed=9000 + case)
    over = {"keep_rule": 0, "random_seed": 0, "reindex_mode": int(r.random() < 0.3)}
    while not _clear_of_tie_band(w):
        w = scaled(w, seed=w.seed + 100)
    return w, over, None, None


N_BIG = 10

# degenerate chunks: (tokens per frame, frames per chunk, score width)
EDGE = [(1, 1, 1), (1, 3, 2), (2, 1, 3), (31, 1, 4), (33, 1, 5), (1, 2, 64)]


def draw_edge(case: int):
    """Chunks of 1 to 33 tokens and score rows of 1 to 64 values: a tile holds part of one warp, the ballot words a
    few bits."""
    r = np.random.default_rng(0xED6E + case)
    T, F, d = EDGE[case]
    win = int(r.integers(1, 3))
    R = win * F + int(r.integers(0, 2))
    n_ev = int(r.integers(2, 6))
    last = 1 + n_ev - 1
    w = scaled(TINY, name=f"sweep_edge_{case}", index=400 + case, L=2, H=2, D=16, dtype=int(r.integers(0, 2)),
               n_temporal_pairs=int(r.integers(1, 9)), tokens_per_frame=T, frames_per_chunk=F, d=d, sink_chunks=1,
               window_chunks=win, R=float(R), S=float(R), g_mode=0, hist_cap=n_ev * T * F,
               max_frames=(last + win + 2) * F, evict_chunk=last, history_chunks=tuple(range(1, last)),
               seed=9500 + case)
    over = {"keep_rule": int(r.choice([0, 1, 2])), "random_seed": int(r.integers(0, 1 << 32)),
            "reindex_mode": int(r.random() < 0.3)}
    while not _clear_of_tie_band(w):
        w = scaled(w, seed=w.seed + 100)
    return w, over, None, None


N_EDGE = len(EDGE)

# the host's no-turn decision (g is the identity on the leaving chunk's offsets): draws on both sides of each boundary
# (g mode, boundary, side); the chunk's oldest offset q0 - evict_first_frame is (w + 1) F for every eviction
BOUNDARY = [(m, b, side) for m in (0, 1) for b in ("recent", "span") for side in ("at", "past")]


def draw_boundary(case: int):
    """A 1024-plane cache (rows of 128 bytes, 8-token chunks) whose last eviction sits exactly on a boundary of g's
    identity or one frame past it: q0 - evict_first_frame in {R, R + 1} while g compresses, or q0 - T_s in
    {span end, span end + 1} while the chunk's oldest offset is past R.  On the "at" side no kept key turns (the staged
    gather, no cos/sin table for the chunk); one frame past it the oldest frame's keys turn (the register-staged
    gather)."""
    mode, bound, side = BOUNDARY[case]
    F, T, sink, win, n_ev = 2, 4, 1, 2, 3
    last = sink + n_ev - 1
    q0 = (last + win + 1) * F
    oldest, dmax = (win + 1) * F, q0 - sink * F          # 6 and 10
    if bound == "recent":
        R = oldest if side == "at" else oldest - 1        # offset = R, or R + 1
        S = R if mode == 0 else 1                         # span end R or R + 1: below dmax, so g compresses
    else:
        R = win * F                                       # 4 < oldest: the oldest frame lies in g's linear part
        end = dmax if side == "at" else dmax - 1
        S = end if mode == 0 else end - R
    w = scaled(TINY, name=f"sweep_boundary_{case}", index=500 + case, L=32, H=32, D=64, dtype=0,
               n_temporal_pairs=int(np.random.default_rng(0xB0D + case).integers(1, 33)), tokens_per_frame=T,
               frames_per_chunk=F, d=16, sink_chunks=sink, window_chunks=win, R=float(R), S=float(S), g_mode=mode,
               hist_cap=n_ev * T * F, max_frames=q0 + 2 * F, evict_chunk=last,
               history_chunks=tuple(range(sink, last)), seed=9700 + case)
    while not _clear_of_tie_band(w) or not np.any(oracle.score(*w.score_inputs(last)) > np.float32(w.gamma)):
        w = scaled(w, seed=w.seed + 100)  # scores clear of gamma, and at least one kept token at the last eviction
    return w, {"keep_rule": 0, "random_seed": 0, "reindex_mode": 0}, None, None


N_BOUNDARY = len(BOUNDARY)


def draw_staged_turn(case: int):
    """A 1024-plane cache (bf16 and fp32 in turn, rows of 64 to 256 bytes, 1 to 8 temporal 16-byte chunks per row)
    whose evictions all turn their kept keys.  The first eviction (q0 unchanged, nothing to re-index) takes the
    staged gather's turning form, across both dtypes (the compensated fp32 turn included), row sizes, temporal
    extents, and kept counts from part of one 64-row block to several blocks; the later ones take the fused gather +
    re-index launch.  Cases 6 and up also make 1 to 31 heads of every layer static: every eviction then takes the
    turning staged form, walking the scan's list of receiving planes instead of every plane."""
    r = np.random.default_rng(0x57A6 + case)
    dtype = case % 2
    D = int(r.choice([32, 64, 128] if dtype == 0 else [16, 32, 64]))
    ppv = 4 if dtype == 0 else 2                          # rotary pairs per 16-byte chunk
    tc = int(r.integers(1, min(8, D * (2 if dtype == 0 else 4) // 16) + 1))
    n_t = min(D // 2, tc * ppv - int(r.integers(0, ppv)))
    F, T = int(r.integers(1, 4)), int(r.choice([16, 40, 64]))
    sink, win, n_ev = 1, int(r.integers(1, 3)), int(r.integers(2, 4))
    last = sink + n_ev - 1
    R = win * F                                           # the leaving chunk's oldest offset (w + 1) F lies past R
    S = R + int(r.integers(0, 2))                         # g compresses once q0 - T_s > S
    w = scaled(TINY, name=f"sweep_staged_turn_{case}", index=600 + case, L=32, H=32, D=D, dtype=dtype,
               n_temporal_pairs=n_t, rope_base=1e4, tokens_per_frame=T, frames_per_chunk=F, d=16, sink_chunks=sink,
               window_chunks=win, R=float(R), S=float(S), g_mode=0, hist_cap=n_ev * T * F,
               max_frames=(last + win + 2) * F, evict_chunk=last, history_chunks=tuple(range(sink, last)),
               seed=9800 + case)
    while not _clear_of_tie_band(w):
        w = scaled(w, seed=w.seed + 100)
    over = {"keep_rule": int(r.choice([0, 1])), "random_seed": 0, "reindex_mode": 0}
    if case >= 6:
        w = scaled(w, n_static_per_layer=int(r.integers(1, w.H)))
    return w, over, w.head_is_static(), None


N_STAGED_TURN = 10


@pytest.mark.parametrize("case", [("narrow", i) for i in range(N_CASES)] + [("wide", i) for i in range(N_WIDE)] +
                         [("big", i) for i in range(N_BIG)] + [("edge", i) for i in range(N_EDGE)] +
                         [("boundary", i) for i in range(N_BOUNDARY)] +
                         [("staged_turn", i) for i in range(N_STAGED_TURN)],
                         ids=[f"case{i}" for i in range(N_CASES)] + [f"wide{i}" for i in range(N_WIDE)] +
                         [f"big{i}" for i in range(N_BIG)] + [f"edge{i}" for i in range(N_EDGE)] +
                         [f"boundary_m{m}_{b}_{sd}" for m, b, sd in BOUNDARY] +
                         [f"staged_turn{i}" for i in range(N_STAGED_TURN)])
def test_sweep_case(gpu, case):
    kind, case = case
    w, over, hsm, paged = {"narrow": draw, "wide": draw_wide, "big": draw_big, "edge": draw_edge,
                           "boundary": draw_boundary, "staged_turn": draw_staged_turn}[kind](case)
    ocfg = replay.cfg_of(w)
    for key, val in over.items():
        setattr(ocfg, key, val)
    hc = replay.new_host_cache(w)
    placed = set()
    for ev in w.evictions():
        for cc in w.resident_window(ev[0]):
            if cc not in placed:
                replay.place_chunk(hc, w, cc)
                placed.add(cc)
        if paged is None:
            gpu_vs_oracle_step(w, hc, ev, head_is_static=hsm, **over)
        else:
            paged_vs_oracle_step(w, hc, ev, paged[0], paged[1], head_is_static=hsm, seed=case, **over)
        replay.replay(w, hc, [ev], hsm, placed=placed, cfg=ocfg)  # the host state moves on by the oracle's step
    if over["reindex_mode"] == 1:  # the read of the final history at the last q0, contiguous or paged
        q0 = w.evictions()[-1][2]
        want = oracle.read_history_keys(hc, ocfg, q0)
        dev = devcache.to_device(hc, w)
        gcfg = devcache.dcp_config(w, **over)
        src = dev if paged is None else PagedCopy(dev, gcfg, paged[0], paged[1], seed=case + 1).cache
        size = dcp.dcp_workspace_size(dev, gcfg) if paged is None else dcp.dcp_paged_workspace_size(src, gcfg)
        ws = dcp.new_workspace(size)
        out = torch.zeros((w.n_planes, w.hist_cap, w.D), dtype=torch.bfloat16 if w.dtype == 0 else torch.float32,
                          device="cuda")
        dcp.dcp_read_history_keys(src, gcfg, q0, 0, w.n_planes, out, ws)
        assert dcp.dcp_get_status(src.status) == dcp.DCP_OK
        g = out.view(torch.int16).cpu().numpy().view(np.uint16) if w.dtype == 0 else out.cpu().numpy()
        for pl in range(w.n_planes):
            n = int(hc.hist_len[pl])
            assert_key_parity(g[pl, :n], want[pl, :n], w.n_temporal_pairs)
