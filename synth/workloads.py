"""Shapes and seeded recipes of the synthetic prune-step workloads.

The page's workload (832x480 video, 16 FPS, 4 latent frames per chunk, about one minute of context) is stood in for
by seeded synthetic tensors of that shape: 30x52 = 1560 latent tokens per frame, 6240 tokens per chunk, score rows of
d = 64 fp32 values.  The backbone's layer/head counts (40 x 40 x 128, or 40 x 8 KV heads) are the workload's own
choice; the page does not state them.  Nothing here computes any part of the prune step: the recipes only draw
numbers.  The default seed of a workload is 1000 + its index.

Stream numbering: chunk c owns streams 1000*c + {0: K, 1: V, 2: x_final, 3: noise, 4: noise-scale uniform,
5: revisit noise}; stream 7 draws the static-head set, stream 8 the revisit schedule, stream 9 the initial contents
of the history region.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import normal_f32, uniform_f64

S_K, S_V, S_XF, S_NOISE, S_SCALE, S_REVISIT = 0, 1, 2, 3, 4, 5
STREAM_STATIC, STREAM_REVISIT_PLAN, STREAM_HIST_INIT = 7, 8, 9


def chunk_stream(c: int, what: int) -> int:
    return 1000 * (c + 1) + what


@dataclass
class Workload:
    name: str
    index: int
    L: int
    H: int
    D: int
    dtype: int                  # 0 = bf16, 1 = fp32
    n_temporal_pairs: int
    rope_base: float
    tokens_per_frame: int
    frames_per_chunk: int
    d: int
    sink_chunks: int
    window_chunks: int
    gamma: float
    R: float
    S: float
    g_mode: int = 0
    hist_cap: int = 0
    max_frames: int = 0
    # one eviction: which chunk leaves the window (its successors up to evict+w are resident)
    evict_chunk: int = 0
    # chunks already compacted into the history before the timed eviction (replayed in order)
    history_chunks: tuple = ()
    # per-token noise scale s ~ LogUniform[s_lo, s_hi]; x0hat = x_final + s * N(0, 1)
    s_lo: float = 0.05
    s_hi: float = 1.0
    prefix: bool = False        # prefix pass: x0hat = x_clean + prefix_sigma * N(0, 1), xref = x_clean
    prefix_sigma: float = 0.3
    n_static_per_layer: int = 0
    rollout_chunks: int = 0
    revisit_frac: float = 0.0
    revisit_s: tuple = (0.03, 0.1)
    revisit_sigma: float = 0.01
    seed: int = field(default=-1)

    def __post_init__(self):
        if self.seed < 0:
            self.seed = 1000 + self.index

    # ------------------------------------------------------------------ layout
    @property
    def C(self) -> int:
        return self.tokens_per_frame * self.frames_per_chunk

    @property
    def F(self) -> int:
        return self.frames_per_chunk

    @property
    def sink_rows(self) -> int:
        return self.sink_chunks * self.C

    @property
    def win_row0(self) -> int:
        return self.sink_rows + self.hist_cap

    @property
    def cap(self) -> int:
        return self.sink_rows + self.hist_cap + (self.window_chunks + 1) * self.C

    @property
    def n_planes(self) -> int:
        return self.L * self.H

    @property
    def esize(self) -> int:
        return 2 if self.dtype == 0 else 4

    def slot_of(self, c: int) -> int:
        """Ring slot of non-sink chunk c."""
        assert c >= self.sink_chunks
        return (c - self.sink_chunks) % (self.window_chunks + 1)

    def first_frame(self, c: int) -> int:
        return c * self.F

    def q0_at_evict(self, c: int) -> int:
        """The next chunk to generate when chunk c leaves the window is c + w + 1."""
        return (c + self.window_chunks + 1) * self.F

    def evictions(self):
        """Eviction schedule of the workload: list of (chunk, q0_prev, q0)."""
        if self.rollout_chunks:
            chunks = list(range(self.sink_chunks, self.rollout_chunks - self.window_chunks))
        else:
            chunks = list(self.history_chunks) + [self.evict_chunk]
        out, prev = [], None
        for c in chunks:
            q0 = self.q0_at_evict(c)
            out.append((c, q0 if prev is None else prev, q0))
            prev = q0
        return out

    def resident_window(self, c_evict: int):
        """Chunks in the ring at the eviction of c_evict (c_evict and the w chunks after it)."""
        return list(range(c_evict, c_evict + self.window_chunks + 1))

    # ------------------------------------------------------------------ draws
    def _revisit_plan(self):
        """For a rollout: {chunk: earlier chunk whose x_final it revisits} for a seeded revisit_frac of chunks."""
        if not self.rollout_chunks or self.revisit_frac <= 0:
            return {}
        u = uniform_f64(2 * self.rollout_chunks, self.seed, STREAM_REVISIT_PLAN)
        plan = {}
        for c in range(self.sink_chunks + 1, self.rollout_chunks):
            if u[2 * c] < self.revisit_frac:
                plan[c] = self.sink_chunks + int(u[2 * c + 1] * (c - self.sink_chunks))
        return plan

    def _x_final(self, c: int, plan) -> np.ndarray:
        C, d = self.C, self.d
        if c in plan:
            base = self._x_final(plan[c], plan).astype(np.float64)
            return (base + self.revisit_sigma * normal_f32(C * d, self.seed, chunk_stream(c, S_REVISIT)).reshape(C, d)
                    ).astype(np.float32)
        return normal_f32(C * d, self.seed, chunk_stream(c, S_XF)).reshape(C, d)

    def score_inputs(self, c: int):
        """(x0hat, xref) fp32 [C][d] for chunk c (the leaving chunk of an eviction)."""
        C, d = self.C, self.d
        noise = normal_f32(C * d, self.seed, chunk_stream(c, S_NOISE)).reshape(C, d).astype(np.float64)
        if self.prefix:
            xref = normal_f32(C * d, self.seed, chunk_stream(c, S_XF)).reshape(C, d)
            x0 = (xref.astype(np.float64) + self.prefix_sigma * noise).astype(np.float32)
            return x0, xref
        plan = self._revisit_plan()
        xref = self._x_final(c, plan)
        lo, hi = (self.revisit_s if c in plan else (self.s_lo, self.s_hi))
        u = uniform_f64(C, self.seed, chunk_stream(c, S_SCALE))
        s = lo * np.exp(u * math.log(hi / lo))
        x0 = (xref.astype(np.float64) + s[:, None] * noise).astype(np.float32)
        return x0, xref

    def head_is_static(self):
        """uint8 [L*H]: a seeded n_static_per_layer heads of each layer follow the Streaming policy."""
        if self.n_static_per_layer <= 0:
            return None
        u = uniform_f64(self.L * self.H, self.seed, STREAM_STATIC).reshape(self.L, self.H)
        out = np.zeros((self.L, self.H), np.uint8)
        for l in range(self.L):
            out[l, np.argsort(u[l], kind="stable")[: self.n_static_per_layer]] = 1
        return out.reshape(-1)

    def cfg_kwargs(self):
        return dict(gamma=self.gamma, keep_rule=0, sink_chunks=self.sink_chunks, window_chunks=self.window_chunks,
                    tokens_per_frame=self.tokens_per_frame, frames_per_chunk=self.frames_per_chunk,
                    n_temporal_pairs=self.n_temporal_pairs, rope_base=self.rope_base, g_recent_R=self.R,
                    g_span_S=self.S, g_mode=self.g_mode)

    def algorithmic_bytes(self, k: int, n_dynamic: int, hist_rows_changed: int) -> int:
        """Bytes the step must move: score rows read, kept K and V rows read and written, the temporal part of each
        re-phased history key read and written, the mask/index lists."""
        score = 2 * self.C * self.d * 4
        gather = k * n_dynamic * 2 * (self.D * self.esize) * 2
        rephase = hist_rows_changed * 2 * (2 * self.n_temporal_pairs * self.esize)
        lists = self.C * (1 + 4)
        return score + gather + rephase + lists


def _logu_hi_for_fraction(lo: float, gamma: float, frac: float) -> float:
    """Upper end b of s ~ LogU[lo, b] such that P(s > sqrt(gamma)) = frac (the chi-square spread of l around s^2 is
    ignored; the realised kept fraction is reported by the bench)."""
    a = math.log(math.sqrt(gamma))
    return math.exp((a - frac * math.log(lo)) / (1.0 - frac))


TINY = Workload(name="tiny_fp32_single_prune", index=0, L=2, H=2, D=32, dtype=1, n_temporal_pairs=8, rope_base=1e4,
                tokens_per_frame=64, frames_per_chunk=1, d=16, sink_chunks=1, window_chunks=2, gamma=0.10, R=8, S=16,
                hist_cap=5 * 64, max_frames=64, evict_chunk=5, history_chunks=(1, 2, 3, 4))

MID = Workload(name="mid_bf16_single_eviction", index=1, L=4, H=8, D=128, dtype=0, n_temporal_pairs=22,
               rope_base=1e4, tokens_per_frame=1560, frames_per_chunk=4, d=64, sink_chunks=1, window_chunks=3,
               gamma=0.10, R=12, S=24, hist_cap=3 * 6240, max_frames=64, evict_chunk=6,
               history_chunks=(1, 2, 3, 4, 5))

FULL = Workload(name="full_depth_bf16_single_eviction", index=2, L=40, H=40, D=128, dtype=0, n_temporal_pairs=22,
                rope_base=1e4, tokens_per_frame=1560, frames_per_chunk=4, d=64, sink_chunks=1, window_chunks=3,
                gamma=0.10, R=12, S=24, hist_cap=6240, max_frames=256, evict_chunk=1, history_chunks=(),
                s_lo=0.05, s_hi=_logu_hi_for_fraction(0.05, 0.10, 0.1575))

# Same shapes as FULL with frame indices as if 27 chunks had already passed (q0 = 124): the fused re-phase turns
# every gathered key by a nonzero angle.  History empty.
FULL_ROTATED = Workload(name="full_depth_bf16_single_eviction_rotated", index=2, L=40, H=40, D=128, dtype=0,
                        n_temporal_pairs=22, rope_base=1e4, tokens_per_frame=1560, frames_per_chunk=4, d=64,
                        sink_chunks=1, window_chunks=3, gamma=0.10, R=12, S=24, hist_cap=6240, max_frames=256,
                        evict_chunk=27, history_chunks=(), s_lo=0.05,
                        s_hi=_logu_hi_for_fraction(0.05, 0.10, 0.1575))

ROLLOUT = Workload(name="minute_rollout_gqa8", index=3, L=40, H=8, D=128, dtype=0, n_temporal_pairs=22,
                   rope_base=1e4, tokens_per_frame=1560, frames_per_chunk=4, d=64, sink_chunks=1, window_chunks=3,
                   gamma=0.10, R=12, S=24, hist_cap=56 * 6240, max_frames=256, rollout_chunks=60, s_lo=0.03,
                   s_hi=1.0, revisit_frac=0.2)

HS_PREFIX = Workload(name="head_specialised_prefix", index=4, L=40, H=40, D=128, dtype=0, n_temporal_pairs=22,
                     rope_base=1e4, tokens_per_frame=1560, frames_per_chunk=4, d=64, sink_chunks=1, window_chunks=3,
                     gamma=0.10, R=12, S=24, hist_cap=2 * 6240, max_frames=64, evict_chunk=2, history_chunks=(1,),
                     prefix=True, prefix_sigma=0.3, n_static_per_layer=20)

ALL = {w.name: w for w in (TINY, MID, FULL, FULL_ROTATED, ROLLOUT, HS_PREFIX)}


def scaled(w: Workload, **over) -> Workload:
    """A copy of workload w with some fields replaced (smaller parity cases of the same recipe)."""
    import dataclasses
    return dataclasses.replace(w, **over)


def chunk_row0(w: Workload, c: int) -> int:
    """First cache row of chunk c: the sink rows for sink chunks, else its ring slot."""
    return c * w.C if c < w.sink_chunks else w.win_row0 + w.slot_of(c) * w.C


def fill_device_chunks(k_ptr: int, v_ptr: int, w: Workload, chunks, cuda_stream: int, planes=None) -> None:
    """Write the seeded K and V of each chunk in `chunks` into its rows of a device cache [L][H][cap][D].

    `planes` (optional list of original plane indices) fills a cache that holds only those planes, in that order,
    with the values they have in the full workload."""
    from . import fill_rows_device
    for c in chunks:
        row0 = chunk_row0(w, c)
        for ptr, what in ((k_ptr, S_K), (v_ptr, S_V)):
            if planes is None:
                fill_rows_device(ptr, w.dtype, w.n_planes, w.cap, row0, w.C, w.D, w.seed, chunk_stream(c, what),
                                 w.C, 0, cuda_stream)
            else:
                for i, p in enumerate(planes):
                    fill_rows_device(ptr + i * w.cap * w.D * w.esize, w.dtype, 1, w.cap, row0, w.C, w.D, w.seed,
                                     chunk_stream(c, what), w.C, p * w.C, cuda_stream)


def fill_device_history_canary(k_ptr: int, v_ptr: int, w: Workload, cuda_stream: int, planes=None) -> None:
    """Seeded contents of the (not yet used) history rows, so stray writes show up."""
    from . import fill_rows_device
    if not w.hist_cap:
        return
    for ptr, s in ((k_ptr, 2 * STREAM_HIST_INIT), (v_ptr, 2 * STREAM_HIST_INIT + 1)):
        if planes is None:
            fill_rows_device(ptr, w.dtype, w.n_planes, w.cap, w.sink_rows, w.hist_cap, w.D, w.seed, s, w.hist_cap, 0,
                             cuda_stream)
        else:
            for i, p in enumerate(planes):
                fill_rows_device(ptr + i * w.cap * w.D * w.esize, w.dtype, 1, w.cap, w.sink_rows, w.hist_cap, w.D,
                                 w.seed, s, w.hist_cap, p * w.hist_cap, cuda_stream)


def host_chunk_rows(w: Workload, c: int, plane: int, what: int, rows) -> np.ndarray:
    """Host copy of rows `rows` (positions inside chunk c) of one plane's K (what=S_K) or V (S_V)."""
    from . import fill_rows_host
    dt = np.uint16 if w.dtype == 0 else np.float32
    out = np.empty((len(rows), w.D), dt)
    tmp = np.empty((1, w.D), dt)
    for i, r in enumerate(rows):
        fill_rows_host(tmp, w.dtype, 1, 1, 0, 1, w.D, w.seed, chunk_stream(c, what), w.C, plane * w.C + int(r))
        out[i] = tmp[0]
    return out
