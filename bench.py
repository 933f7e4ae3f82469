"""Benchmark of the DeCoPrune history-KV prune step on GB300 (one JSON line on rank 0).

One step = one full prune step (score + threshold + index scan + fused K/V gather with key re-phase + history
re-index) of the full-depth eviction workload: 40 layers x 40 KV heads x head_dim 128 bf16 cache (sink chunk, three
dense window chunks and the leaving chunk resident, ~31 GB with the history region), 6240 tokens per chunk, score rows
of 64 fp32 values, ~15% of tokens kept.  Inputs are seeded synthetic tensors of that shape, resident in HBM before
the timed region; L2 (129 MB) is flushed between steps by writing a 256 MB buffer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dcp|reference] [--no-extra]

`value` is the step's algorithmic bytes (what the method must read and write) divided by the device time of the step
(CUDA events on the launching stream, max over ranks), summed over ranks.  With N > 1 every rank runs its own replica
of the workload on its own GPU (the step has no exchange: "weak" scaling).  `--impl reference` times the CPU oracle on
a bounded sample of the same workload (the only other thing this script may run).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "history-KV prune step GB/s (score+scan+gather+RoPE) & % of GB300 HBM peak"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# DRAM bytes (read + write) of one full-depth gather launch (gather_staged_kernel<false>), scaled from ncu captures of
# dram__bytes_read.sum and dram__bytes_write.sum on two reduced cases of the same workload (156 and 312 tokens per
# frame): reads scale with the algorithmic reads (1.0005x), writes are the algorithmic writes less the ~50 MB still
# dirty in L2 when the launch ends.  They describe the kernel code they were taken on (gather.cu and the shared
# header, `//` comments and blank lines aside): when that code differs, the bench reports no traffic figure.
GATHER_TRAFFIC_BYTES = 1_501_515_005
GATHER_TRAFFIC_CODE_SHA256 = "ee4f66eb6fef98f507fc0ed766e666329eb2664c565babdde24abc59bae80072"


def _code_only(text: str) -> str:
    """Source text without its // comments, trailing blanks and empty lines (the kernel sources hold no // inside a
    string literal and no block comments)."""
    lines = (ln.split("//", 1)[0].rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def _gather_traffic():
    import hashlib
    h = hashlib.sha256()
    for f in ("gather.cu", "dcp_internal.cuh"):
        with open(os.path.join(ROOT, "autoregressive_video_diffusion_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return GATHER_TRAFFIC_BYTES if h.hexdigest() == GATHER_TRAFFIC_CODE_SHA256 else None


def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part", "hardware")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------------------------------ clocks
class _Nvml:
    """Reads (never sets) one GPU's SM clock, its maximum and the active clock-event reasons through NVML."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, local: int):
        import ctypes
        import torch
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(local)
        uuid = getattr(props, "uuid", None)
        if uuid is not None:  # the physical GPU behind this process's device (CUDA_VISIBLE_DEVICES may renumber)
            rc = lib.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(), ctypes.byref(self.h))
        else:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(local, ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle")
        self.lib = lib
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_mhz = self._clock(lib.nvmlDeviceGetMaxClockInfo)

    def _clock(self, fn):
        v = self.ct.c_uint()
        if fn(self.h, 1, self.ct.byref(v)) != 0:  # NVML_CLOCK_SM
            raise OSError("clock query failed")
        return float(v.value)

    def read(self):
        r = self.ct.c_ulonglong()
        if self.reasons_fn(self.h, self.ct.byref(r)) != 0:
            raise OSError("reason query failed")
        return self._clock(self.lib.nvmlDeviceGetClockInfo), self.max_mhz, \
            {n for b, n in self.REASONS.items() if r.value & b}


class ClockSampler:
    """SM clock and throttle reasons while the bench runs: NVML polled every 2 ms (reads only), so that the short
    timed region gets samples of its own; nvidia-smi's 50 ms loop where NVML cannot be loaded."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    SMI_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.rows = []  # (time, sm MHz, max MHz, set of active reasons)
        self.marks = []
        self.source = None
        self._stop = threading.Event()

    def start(self):
        try:
            nv = _Nvml(self.gpu_index)
            self.source = "nvml, 2 ms"
            threading.Thread(target=self._poll, args=(nv,), daemon=True).start()
            return
        except (OSError, AttributeError):
            pass
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu_index), "-lms", "50"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, 50 ms"
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _poll(self, nv):
        while not self._stop.is_set():
            try:
                sm, mx, reasons = nv.read()
            except OSError:
                return
            self.rows.append((time.time(), sm, mx, reasons))
            time.sleep(0.002)

    def _read(self):
        for ln in self.proc.stdout:
            parts = [x.strip() for x in ln.strip().split(",")]
            if len(parts) < 9:
                continue
            try:
                row = (time.time(), float(parts[1]), float(parts[2]),
                       {n for n, v in zip(self.SMI_REASONS, parts[5:9]) if v.lower() == "active"})
            except ValueError:
                continue
            self.rows.append(row)

    def mark(self, name):
        self.marks.append((name, time.time()))

    def stop(self):
        self._stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = list(self.rows)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        use = inside if len(inside) >= 3 else [r for r in rows if r[0] <= t1]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"], "samples": 0}
        reasons = set()
        for r in use:
            reasons |= r[3]
        return {"sm_mhz": float(np.median([r[1] for r in use])), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(use), "samples_in_timed_region": len(inside),
                "source": self.source}


# ------------------------------------------------------------------------------------------ distributed
_BACKEND = {"name": None}


def dist_setup(backend: str | None = None):
    """Join the process group the launcher set up (RANK / WORLD_SIZE / LOCAL_RANK / MASTER_*).  NCCL on GPUs; gloo
    for the CPU tests of this logic.  Returns (world, rank, local_rank)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = backend or "nccl"
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
        _BACKEND["name"] = backend
    return world, rank, local


def dist_max(x: float, world: int) -> float:
    """Max of x over the ranks (the step time the whole job waited for)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if _BACKEND["name"] == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_throughput(bytes_per_rank_step: int, ms_max: float, world: int) -> float:
    """Whole-job GB/s: every rank moves its own replica's bytes; the job waits for the slowest rank."""
    return world * bytes_per_rank_step / (ms_max * 1e-3) / 1e9


# ------------------------------------------------------------------------------------------ GPU arm
class FullDepthStep:
    """Device state of one eviction of a full-size workload, ready to be pruned repeatedly."""

    def __init__(self, w, keep_rule: int = 0, random_seed: int = 0):
        import torch

        import autoregressive_video_diffusion_gb300 as dcp
        from synth import workloads as W
        self.w, self.dcp = w, dcp
        c, q0_prev, q0 = w.evictions()[-1]
        self.c, self.q0_prev, self.q0 = c, q0_prev, q0
        stream = torch.cuda.current_stream().cuda_stream
        self.cache = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, w.hist_cap)
        W.fill_device_chunks(self.cache.k.data_ptr(), self.cache.v.data_ptr(), w,
                             list(range(w.sink_chunks)) + w.resident_window(c), stream)
        W.fill_device_history_canary(self.cache.k.data_ptr(), self.cache.v.data_ptr(), w, stream)
        self.cfg = dcp.Config(gamma=w.gamma, keep_rule=keep_rule, sink_chunks=w.sink_chunks,
                              window_chunks=w.window_chunks, tokens_per_frame=w.tokens_per_frame,
                              frames_per_chunk=w.frames_per_chunk, n_temporal_pairs=w.n_temporal_pairs,
                              rope_base=w.rope_base, g_recent_R=w.R, g_span_S=w.S, g_mode=w.g_mode,
                              max_frames=w.max_frames, random_seed=random_seed)
        self.ws = dcp.new_workspace(dcp.dcp_workspace_size(self.cache, self.cfg))
        x0, xr = w.score_inputs(c)
        self.x0_host = torch.from_numpy(x0).pin_memory()
        self.xr_host = torch.from_numpy(xr).pin_memory()
        self.x0 = self.x0_host.cuda()
        self.xr = self.xr_host.cuda()
        self.kept = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.kept_host = torch.zeros(1, dtype=torch.int32).pin_memory()
        self.hist_len0 = self.cache.hist_len.clone()
        self.hist_t0 = self.cache.hist_t.clone()
        self.flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.drain_buf = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()

    def restore(self):
        self.cache.hist_len.copy_(self.hist_len0)
        self.cache.hist_t.copy_(self.hist_t0)

    def flush_l2(self):
        """Evict the L2 (129 MB) before a timed step: write a 256 MB buffer, then read another 256 MB buffer so the
        dirty lines of the write are drained to HBM here rather than inside the timed step."""
        self.flush_buf.fill_(1)
        self.drain_sum = self.drain_buf.sum()

    def step(self, x0=None, xr=None, kept_host=None):
        w = self.w
        self.dcp.dcp_prune_step(self.cache, self.cfg, self.x0 if x0 is None else x0, self.xr if xr is None else xr,
                                w.slot_of(self.c), w.first_frame(self.c), self.q0_prev, self.q0, None, self.kept,
                                kept_host, self.ws)

    def launches_per_step(self):
        """The scan, then one launch that moves the kept rows (with the history re-index folded in when there is one:
        no static heads here)."""
        return 2


class PagedFullDepthStep(FullDepthStep):
    """The same eviction on a paged copy of the cache: block pools of `block_size` positions (HND or NHD) and
    block tables drawn as a seeded permutation of the pool's blocks."""

    def __init__(self, w, block_size: int, layout: int):
        import torch
        super().__init__(w)
        dcp, cfg, bs = self.dcp, self.cfg, block_size
        C, sink = w.C, w.sink_chunks * w.C
        n_sink, n_hist, n_win = sink // bs, w.hist_cap // bs, (w.window_chunks + 1) * C // bs
        n_blocks = n_sink + n_hist + n_win
        perm = torch.from_numpy(np.random.default_rng(0xB10C).permutation(n_blocks).astype(np.int32)).cuda()
        pc = dcp.PagedKVCache(w.L, w.H, w.D, w.dtype, bs, layout, n_blocks, w.hist_cap, n_win)
        pc.hist_blocks.copy_(perm[n_sink:n_sink + n_hist])
        pc.window_blocks.copy_(perm[n_sink + n_hist:])
        block, off = dcp.paged_row_map(cfg, w.hist_cap, bs, perm[:n_sink], pc.hist_blocks, pc.window_blocks)
        dcp.paged_pack(pc.k_pool, self.cache.k, block, off, layout)
        dcp.paged_pack(pc.v_pool, self.cache.v, block, off, layout)
        pc.hist_len.copy_(self.cache.hist_len)
        pc.hist_t.copy_(self.cache.hist_t)
        self.cache = pc  # the contiguous tensors are released here
        self.ws = dcp.new_workspace(dcp.dcp_paged_workspace_size(pc, cfg))
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    def step(self, x0=None, xr=None, kept_host=None):
        w = self.w
        self.dcp.dcp_paged_prune_step(self.cache, self.cfg, self.x0 if x0 is None else x0,
                                      self.xr if xr is None else xr, w.slot_of(self.c), w.first_frame(self.c),
                                      self.q0_prev, self.q0, None, self.kept, kept_host, self.ws)


def run_gpu(w, steps: int, warmup: int, world: int, rank: int, local: int, clocks: ClockSampler | None,
            e2e_steps: int, preroll_s: float = 1.0, keep_rule: int = 0, paged=None):
    import torch

    import autoregressive_video_diffusion_gb300 as dcp
    s = FullDepthStep(w, keep_rule=keep_rule, random_seed=0x5EED) if paged is None else PagedFullDepthStep(w, *paged)
    stream = torch.cuda.current_stream()
    ev_scan, ev_gather = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_scan.record(stream)
    ev_gather.record(stream)
    torch.cuda.synchronize()
    # warm-up, and a short sustained pre-roll so the clock sampler sees the part under this load
    for _ in range(warmup):
        s.restore()
        s.step()
    torch.cuda.synchronize()
    pre_t = time.time()
    while time.time() - pre_t < preroll_s:
        s.restore()
        s.flush_l2()
        s.step()
        torch.cuda.synchronize()
    st = dcp.dcp_get_status(s.cache.status)
    if st != dcp.DCP_OK:
        raise RuntimeError(f"prune step reported {dcp.dcp_status_string(st)}")
    k = int(s.kept.item())
    n_dyn = w.n_planes
    hist_rows_changed = 0
    alg_bytes = w.algorithmic_bytes(k, n_dyn, hist_rows_changed)
    gather_bytes = k * n_dyn * 2 * (w.D * w.esize) * 2

    # the timed region: exactly `steps` prune steps on the library's normal launch path
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    dist_barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark("timed_start")
    t_wall0 = time.time()
    for i in range(steps):
        s.restore()
        s.flush_l2()
        starts[i].record(stream)
        s.step()
        ends[i].record(stream)
        ends[i].synchronize()
    torch.cuda.synchronize()
    dist_barrier(world)
    t_wall1 = time.time()
    if clocks:
        clocks.mark("timed_end")
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = float(np.mean(step_ms))
    ms_max = dist_max(ms, world)

    # per-kernel times: the same steps again with CUDA events recorded by the library between its kernels (an event
    # between two kernels stops the second from launching early, so these steps are not the timed ones)
    scan_ms, gather_ms = [], []
    dcp.dcp_set_phase_events(ev_scan, ev_gather)
    for i in range(steps):
        s.restore()
        s.flush_l2()
        starts[i].record(stream)
        s.step()
        ends[i].record(stream)
        ends[i].synchronize()
        scan_ms.append(starts[i].elapsed_time(ev_scan))
        gather_ms.append(ev_scan.elapsed_time(ev_gather))
    dcp.dcp_set_phase_events(None, None)
    torch.cuda.synchronize()

    # end to end through the public API: the score inputs sit in page-locked host memory and the step reads them
    # over the host link (the scan kernel's loads); the kept count comes back to page-locked host memory, written by
    # the scan kernel.  For comparison, the same with explicit copies of the inputs into device buffers first.
    e2e_ms, copy_e2e_ms, h2d_ms = [], [], []
    if e2e_steps:  # untimed: the first device access to the page-locked inputs sets up their mappings (~0.4 ms)
        s.restore()
        s.step(x0=s.x0_host, xr=s.xr_host, kept_host=s.kept_host)
        torch.cuda.synchronize()
    for _ in range(e2e_steps):
        s.restore()
        s.flush_l2()
        s.kept_host.fill_(-1)
        a, b = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        a.record(stream)
        s.step(x0=s.x0_host, xr=s.xr_host, kept_host=s.kept_host)
        b.record(stream)
        b.synchronize()
        assert int(s.kept_host.item()) == k
        e2e_ms.append(a.elapsed_time(b))
    for _ in range(e2e_steps):
        s.restore()
        s.flush_l2()
        s.kept_host.fill_(-1)
        a, m, b = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        s.x0.copy_(s.x0_host, non_blocking=True)
        s.xr.copy_(s.xr_host, non_blocking=True)
        m.record(stream)
        s.step(kept_host=s.kept_host)
        b.record(stream)
        b.synchronize()
        assert int(s.kept_host.item()) == k
        copy_e2e_ms.append(a.elapsed_time(b))
        h2d_ms.append(a.elapsed_time(m))
    e2e = float(np.mean(e2e_ms)) if e2e_ms else None
    e2e_max = dist_max(e2e, world) if e2e is not None else None

    res = dict(k=k, alg_bytes=alg_bytes, gather_bytes=gather_bytes, ms=ms, ms_max=ms_max,
               ms_median=float(np.median(step_ms)), scan_ms=float(np.mean(scan_ms)),
               gather_ms=float(np.mean(gather_ms)), e2e_ms=e2e_max, wall=(t_wall0, t_wall1),
               e2e_median_ms=float(np.median(e2e_ms)) if e2e_ms else None,
               h2d_ms=float(np.median(h2d_ms)) if h2d_ms else None,
               copy_e2e_ms=float(np.median(copy_e2e_ms)) if copy_e2e_ms else None,
               launches=steps * s.launches_per_step(), h2d=2 * s.x0.numel() * 4, d2h=4)
    del s
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------------------------ the other workloads
class DeviceRollout:
    """A device cache taken through a workload's eviction schedule by the library itself: each newly generated
    chunk's K/V is written on the device by the seeded generator and its score inputs staged (untimed), then the prune
    step runs.  Used for the workloads whose history matters (mid eviction, head-specialised prefix pass, rollout)."""

    def __init__(self, w, head_is_static=None, reindex_mode: int = 0):
        import torch

        import autoregressive_video_diffusion_gb300 as dcp
        from synth import workloads as W
        self.w, self.dcp, self.W, self.torch = w, dcp, W, torch
        self.reindex_mode = reindex_mode
        self.stream = torch.cuda.current_stream()
        self.cache = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, w.hist_cap)
        s = self.stream.cuda_stream
        W.fill_device_history_canary(self.cache.k.data_ptr(), self.cache.v.data_ptr(), w, s)
        W.fill_device_chunks(self.cache.k.data_ptr(), self.cache.v.data_ptr(), w, list(range(w.sink_chunks)), s)
        self.placed = set(range(w.sink_chunks))
        self.cfg = dcp.Config(gamma=w.gamma, keep_rule=0, sink_chunks=w.sink_chunks,
                              window_chunks=w.window_chunks, tokens_per_frame=w.tokens_per_frame,
                              frames_per_chunk=w.frames_per_chunk, n_temporal_pairs=w.n_temporal_pairs,
                              rope_base=w.rope_base, g_recent_R=w.R, g_span_S=w.S, g_mode=w.g_mode,
                              max_frames=w.max_frames, reindex_mode=reindex_mode)
        self.ws = dcp.new_workspace(dcp.dcp_workspace_size(self.cache, self.cfg))
        self.static = head_is_static
        self.hs = None if head_is_static is None else torch.from_numpy(head_is_static).cuda()
        self.n_dyn = w.n_planes if head_is_static is None else int((head_is_static == 0).sum())
        self.kept = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.drain_buf = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")
        self.inputs = {}

    def prepare(self, c):
        """Write the chunks resident when chunk c leaves, and stage c's score inputs on the device (untimed)."""
        new = [cc for cc in self.w.resident_window(c) if cc not in self.placed]
        self.W.fill_device_chunks(self.cache.k.data_ptr(), self.cache.v.data_ptr(), self.w, new,
                                  self.stream.cuda_stream)
        self.placed |= set(new)
        x0, xr = self.w.score_inputs(c)
        self.inputs[c] = (self.torch.from_numpy(x0).cuda(), self.torch.from_numpy(xr).cuda())

    def step(self, c, q0_prev, q0):
        w = self.w
        x0, xr = self.inputs[c]
        self.dcp.dcp_prune_step(self.cache, self.cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, self.hs,
                                self.kept, None, self.ws)

    def timed_step(self, c, q0_prev, q0) -> float:
        """One prune step between CUDA events on the stream, after an L2 flush; returns ms."""
        torch = self.torch
        self.flush_buf.fill_(1)
        self.drain_sum = self.drain_buf.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(self.stream)
        self.step(c, q0_prev, q0)
        b.record(self.stream)
        b.synchronize()
        return a.elapsed_time(b)

    def rows_rephased(self, q0_prev, q0, hist_len_sum) -> int:
        """History rows whose key phase moves: every history row once the span compresses (history frames are all
        older than the dense window, so they all lie in g's linear part), none while g is the identity."""
        w = self.w
        T_s = w.sink_chunks * w.F
        end = w.S if w.g_mode == 0 else w.R + w.S
        moves = q0 != q0_prev and (q0 - T_s > end or q0_prev - T_s > end) and self.reindex_mode == 0
        return hist_len_sum if moves else 0

    def check(self):
        st = self.dcp.dcp_get_status(self.cache.status)
        if st != self.dcp.DCP_OK:
            raise RuntimeError(f"{self.w.name}: prune step reported {self.dcp.dcp_status_string(st)}")


def run_last_eviction(w, reps: int):
    """History built by the library over the earlier evictions; the last eviction timed `reps` times, restoring the
    history lengths, frames and key rows between repetitions (untimed)."""
    import torch
    r = DeviceRollout(w)
    ev = w.evictions()
    for c, q0p, q0 in ev[:-1]:
        r.prepare(c)
        r.step(c, q0p, q0)
    c, q0p, q0 = ev[-1]
    r.prepare(c)
    H0 = w.sink_rows
    hl0, ht0 = r.cache.hist_len.clone(), r.cache.hist_t.clone()
    khist0 = r.cache.k[:, :, H0:H0 + w.hist_cap].clone()
    hist_sum = int(hl0.sum().item())
    times = []
    for _ in range(reps):
        r.cache.hist_len.copy_(hl0)
        r.cache.hist_t.copy_(ht0)
        r.cache.k[:, :, H0:H0 + w.hist_cap].copy_(khist0)
        times.append(r.timed_step(c, q0p, q0))
    r.check()
    k = int(r.kept.item())
    ms = float(np.median(times))
    nbytes = w.algorithmic_bytes(k, r.n_dyn, r.rows_rephased(q0p, q0, hist_sum))
    out = {"workload": w.name, "kept": k, "history_rows_before": int(hl0[0].item()), "q0_prev": q0p, "q0": q0,
           "us_per_step": ms * 1e3, "algorithmic_bytes": nbytes, "GB_per_s": nbytes / (ms * 1e-3) / 1e9, "reps": reps}
    del r, khist0
    torch.cuda.empty_cache()
    return out


def run_graph_replay(w, reps: int):
    """The workload's last eviction from an idle GPU, host submission included: the direct call against the same
    call recorded in a CUDA graph and replayed (the history restored, untimed, between repetitions)."""
    import torch

    import autoregressive_video_diffusion_gb300 as dcp
    r = DeviceRollout(w)
    ev = w.evictions()
    for c, q0p, q0 in ev[:-1]:
        r.prepare(c)
        r.step(c, q0p, q0)
    c, q0p, q0 = ev[-1]
    r.prepare(c)
    H0 = w.sink_rows
    hl0, ht0 = r.cache.hist_len.clone(), r.cache.hist_t.clone()
    kh0 = r.cache.k[:, :, H0:H0 + w.hist_cap].clone()

    def restore():
        r.cache.hist_len.copy_(hl0)
        r.cache.hist_t.copy_(ht0)
        r.cache.k[:, :, H0:H0 + w.hist_cap].copy_(kh0)

    restore()
    r.step(c, q0p, q0)  # the first call sets up the launch attributes outside capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    x0, xr = r.inputs[c]
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dcp.dcp_prune_step(r.cache, r.cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0p, q0, None, r.kept, None,
                               r.ws, stream=s)

    def timed(fn):
        out = []
        for _ in range(reps):
            restore()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            out.append(a.elapsed_time(b))
        return float(np.median(out[3:]))

    direct = timed(lambda: r.step(c, q0p, q0))
    graph = timed(lambda: g.replay())
    r.check()
    del g, r
    torch.cuda.empty_cache()
    return {"workload": w.name, "direct_us": direct * 1e3, "graph_replay_us": graph * 1e3,
            "note": "idle GPU before each step, host submission included"}


def run_head_specialised(w, reps: int):
    """Prefix pass with 20 static heads per layer: both evictions of the pass, each timed; `reps` passes."""
    import torch
    per = []
    for _ in range(reps):
        r = DeviceRollout(w, w.head_is_static())
        row = []
        for c, q0p, q0 in w.evictions():
            r.prepare(c)
            hist_sum = int(r.cache.hist_len.sum().item())
            ms = r.timed_step(c, q0p, q0)
            k = int(r.kept.item())
            nbytes = w.algorithmic_bytes(k, r.n_dyn, r.rows_rephased(q0p, q0, hist_sum))
            row.append((ms, k, nbytes))
        r.check()
        per.append(row)
        del r
        torch.cuda.empty_cache()
    out = {"workload": w.name, "dynamic_planes": int((w.head_is_static() == 0).sum()), "evictions": []}
    for i, (c, q0p, q0) in enumerate(w.evictions()):
        ms = float(np.median([p[i][0] for p in per]))
        k, nbytes = per[0][i][1], per[0][i][2]
        out["evictions"].append({"chunk": c, "q0": q0, "kept": k, "us_per_step": ms * 1e3,
                                 "GB_per_s": nbytes / (ms * 1e-3) / 1e9})
    return out


DRIFT_PLANES = (0, 1, 77, 160, 319)  # sampled planes of the 320-plane rollout cache for the drift report


def _bits_as_ordered(t):
    """bf16 / fp32 bit patterns as integers whose differences count ulps (torch, on the device)."""
    import torch
    if t.dtype == torch.bfloat16:
        b = t.view(torch.int16).to(torch.int64)
        return torch.where(b < 0, -(b & 0x7FFF), b)
    b = t.view(torch.int32).to(torch.int64)
    return torch.where(b < 0, -(b & 0x7FFFFFFF), b)


def run_rollout(w, reindex_mode: int = 0, eager_keys=None):
    """The minute-long rollout: every chunk generated in turn, a prune step after each one that leaves the window;
    per-step times, and the cumulative PR against FullKV kept by the library's host counter.  With read-time
    re-index (reindex_mode 1) the steps re-index nothing, and the read of the final history at the final q0
    (dcp_read_history_keys of every plane) is timed as well."""
    import torch

    import autoregressive_video_diffusion_gb300 as dcp
    r = DeviceRollout(w, reindex_mode=reindex_mode)
    pr = dcp.DcpPrCounter(0, 0)
    ev = {c: (q0p, q0) for c, q0p, q0 in w.evictions()}
    steps = []
    for i in range(1, w.rollout_chunks):
        hist_sum = int(r.cache.hist_len.sum().item())
        window = min(w.window_chunks, max(0, i - w.sink_chunks)) * w.C
        dcp.dcp_pr_add_chunk(pr, w.n_planes, hist_sum, min(w.sink_chunks, i) * w.C, window, i * w.C)
        c = i - w.window_chunks            # the chunk that leaves once chunk i is generated
        if c in ev:
            q0p, q0 = ev[c]
            r.prepare(c)
            ms = r.timed_step(c, q0p, q0)
            k = int(r.kept.item())
            nbytes = w.algorithmic_bytes(k, r.n_dyn, r.rows_rephased(q0p, q0, hist_sum))
            steps.append((ms, nbytes, k, hist_sum // w.n_planes))
    r.check()
    ms = np.array([s[0] for s in steps])
    nb = np.array([s[1] for s in steps], dtype=np.float64)
    out = {"workload": w.name, "prune_steps": len(steps), "mean_us_per_step": float(ms.mean() * 1e3),
           "median_us_per_step": float(np.median(ms) * 1e3), "max_us_per_step": float(ms.max() * 1e3),
           "last10_mean_us": float(ms[-10:].mean() * 1e3), "GB_per_s": float(nb.sum() / (ms.sum() * 1e-3) / 1e9),
           "last10_GB_per_s": float(nb[-10:].sum() / (ms[-10:].sum() * 1e-3) / 1e9),
           "final_history_rows": int(r.cache.hist_len[0].item()), "cumulative_PR": dcp.dcp_pr_value(pr),
           "kept_fraction_mean": float(np.mean([s[2] for s in steps]) / w.C),
           "curve_us": [round(float(x) * 1e3, 1) for x in ms], "reindex_mode": reindex_mode}
    if reindex_mode == 1:
        q0_last = w.evictions()[-1][2]
        out_keys = torch.empty((w.n_planes, w.hist_cap, w.D), dtype=r.cache.k.dtype, device="cuda")
        rows = int(r.cache.hist_len.sum().item())
        times = []
        for _ in range(5):
            r.flush_buf.fill_(1)
            r.drain_sum = r.drain_buf.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(r.stream)
            dcp.dcp_read_history_keys(r.cache, r.cfg, q0_last, 0, w.n_planes, out_keys, r.ws)
            b.record(r.stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        r.check()
        rms = float(np.median(times))
        nbytes = rows * w.D * w.esize * 2
        out["read_history_keys"] = {"rows": rows, "q0": q0_last, "us": rms * 1e3, "bytes": nbytes,
                                    "GB_per_s": nbytes / (rms * 1e-3) / 1e9}
        if eager_keys is not None:
            # drift of the eager path: its keys were turned and rounded at every step; the read turns the raw key
            # once (within 1 ulp of the exact turn), so their difference is the accumulated rounding
            n = int(r.cache.hist_len[0].item())
            nt2 = 2 * w.n_temporal_pairs
            read = out_keys[list(DRIFT_PLANES), :n].float()
            eager = eager_keys[:, :n].float()
            ulps = (_bits_as_ordered(out_keys[list(DRIFT_PLANES), :n, :nt2]) -
                    _bits_as_ordered(eager_keys[:, :n, :nt2])).abs()
            pair = torch.sqrt(eager[..., 0:nt2:2] ** 2 + eager[..., 1:nt2:2] ** 2).repeat_interleave(2, dim=-1)
            rel = (read[..., :nt2] - eager[..., :nt2]).abs() / pair.clamp_min(1e-30)
            out["drift_eager_vs_read_time"] = {
                "planes": list(DRIFT_PLANES), "rows": n, "steps": len(steps),
                "entries_differing": int((ulps > 0).sum().item()), "entries": int(ulps.numel()),
                "max_ulp": int(ulps.max().item()), "max_of_pair_length": float(rel.max().item()),
                "non_temporal_bitwise": bool(torch.equal(out_keys[list(DRIFT_PLANES), :n, nt2:],
                                                         eager_keys[:, :n, nt2:]))}
        del out_keys
    else:
        out["_final_keys"] = r.cache.k.view(w.n_planes, w.cap, w.D)[list(DRIFT_PLANES), w.sink_rows:
                                                                    w.sink_rows + w.hist_cap].clone()
    del r
    torch.cuda.empty_cache()
    return out


def run_snapshot(w, reps: int):
    """Host snapshot and restore (dcp_snapshot / dcp_restore) of the state left by the full-depth eviction, cut to
    w.L layers: sink, 947 history rows and the three live window chunks of every plane.  Compared with a plain copy
    of the same byte count between the same page-locked buffer and the device (the link's own rate)."""
    import torch

    import autoregressive_video_diffusion_gb300 as dcp
    from synth import workloads as W
    c, q0_prev, q0 = w.evictions()[-1]
    stream = torch.cuda.current_stream()
    cache = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, w.hist_cap)
    W.fill_device_chunks(cache.k.data_ptr(), cache.v.data_ptr(), w,
                         list(range(w.sink_chunks)) + w.resident_window(c), stream.cuda_stream)
    W.fill_device_history_canary(cache.k.data_ptr(), cache.v.data_ptr(), w, stream.cuda_stream)
    cfg = dcp.Config(gamma=w.gamma, sink_chunks=w.sink_chunks, window_chunks=w.window_chunks,
                     tokens_per_frame=w.tokens_per_frame, frames_per_chunk=w.frames_per_chunk,
                     n_temporal_pairs=w.n_temporal_pairs, rope_base=w.rope_base, g_recent_R=w.R, g_span_S=w.S,
                     g_mode=w.g_mode, max_frames=w.max_frames)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(cache, cfg))
    x0, xr = (torch.from_numpy(x).cuda() for x in w.score_inputs(c))
    dcp.dcp_prune_step(cache, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, None, None, None, ws)
    live = 0
    for cc in range(c + 1, c + w.window_chunks + 1):
        live |= 1 << w.slot_of(cc)
    img = dcp.new_snapshot_image(dcp.dcp_snapshot_max_bytes(cache, cfg, live))
    dcp.dcp_snapshot(cache, cfg, live, q0, img, ws)
    torch.cuda.synchronize()
    if dcp.dcp_get_status(cache.status) != dcp.DCP_OK:
        raise RuntimeError("snapshot reported an error")
    n = dcp.snapshot_total_bytes(img)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn):
        out = []
        for _ in range(reps):
            ev[0].record(stream)
            fn()
            ev[1].record(stream)
            ev[1].synchronize()
            out.append(ev[0].elapsed_time(ev[1]))
        return float(np.median(out))

    snap_ms = timed(lambda: dcp.dcp_snapshot(cache, cfg, live, q0, img, ws))
    rest_ms = timed(lambda: dcp.dcp_restore(cache, cfg, img, ws))
    if dcp.dcp_get_status(cache.status) != dcp.DCP_OK:
        raise RuntimeError("restore reported an error")
    dev_buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    host = img[:n]
    d2h_ms = timed(lambda: host.copy_(dev_buf, non_blocking=True))
    h2d_ms = timed(lambda: dev_buf.copy_(host, non_blocking=True))
    gbs = lambda ms: n / (ms * 1e-3) / 1e9  # noqa: E731
    out = {"workload": f"{w.name} cut to {w.L} layers, after its eviction", "image_bytes": n,
           "history_rows_per_plane": int(cache.hist_len[0].item()), "live_window_chunks": w.window_chunks,
           "snapshot_us": snap_ms * 1e3, "snapshot_GB_per_s": gbs(snap_ms),
           "restore_us": rest_ms * 1e3, "restore_GB_per_s": gbs(rest_ms),
           "plain_copy_d2h_GB_per_s": gbs(d2h_ms), "plain_copy_h2d_GB_per_s": gbs(h2d_ms),
           "frac_of_plain_copy": {"snapshot": d2h_ms / snap_ms, "restore": h2d_ms / rest_ms},
           "gpu_launches_per_call": 2}
    del cache, dev_buf, img, host, ws
    torch.cuda.empty_cache()
    return out


def run_entry_case(case: str, steps: int, warmup: int):
    """Single entry points on their own (one GPU), for per-kernel measurement and profiling captures:
    reindex: dcp_rope_reindex of a bf16 cache of 64 planes x 90,000 history rows (frames 4-219, ~417 rows per frame,
             D 128, n_t 22) moved from q0 220 to 224 (then 224 -> 228, ...); algorithmic bytes 2 x 88 B per row.
    score:   dcp_score_mask of the full-depth workload's 6240 x 64 score inputs; algorithmic bytes 2 x 6240 x 64 x 4.
    read:    dcp_read_history_keys (read-time re-index) of the same 64-plane, 90,000-row history at q0 224, 228, ...
             into a [64][100000][128] buffer; algorithmic bytes 2 x 256 B per row.
    random:  dcp_score_mask under keep rule 2 (Random at the discrepancy rule's count) of the full-depth chunk."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import autoregressive_video_diffusion_gb300 as dcp
    from synth.workloads import FULL
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    drain = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")
    if case in ("reindex", "read"):
        L, H, D, C, hist_cap, rows = 8, 8, 128, 6240, 100000, 90000
        cache = dcp.KVCache(L, H, D, dcp.DCP_BF16, C + hist_cap + 4 * C, hist_cap)
        cache.k.normal_(generator=torch.Generator(device="cuda").manual_seed(1234))
        cache.v.zero_()
        cache.hist_len.fill_(rows)
        frames = (4 + np.arange(rows) * 216 // rows).astype(np.int32)
        cache.hist_t[:rows].copy_(torch.from_numpy(frames))
        cfg = dcp.Config(max_frames=1024, reindex_mode=1 if case == "read" else 0)
        ws = dcp.new_workspace(dcp.dcp_workspace_size(cache, cfg))
        status = cache.status
        if case == "reindex":
            def call(i):
                dcp.dcp_rope_reindex(cache, cfg, 220 + 4 * i, 224 + 4 * i, ws)
            nbytes = L * H * rows * 2 * 88
        else:
            out = torch.empty((L * H, hist_cap, D), dtype=torch.bfloat16, device="cuda")

            def call(i):
                dcp.dcp_read_history_keys(cache, cfg, 224 + 4 * i, 0, L * H, out, ws)
            nbytes = L * H * rows * 2 * D * 2
    else:
        c = FULL.evictions()[-1][0]
        x0, xr = (torch.from_numpy(a).cuda() for a in FULL.score_inputs(c))
        n = FULL.C
        ws = dcp.new_workspace(dcp.dcp_score_workspace_size(n))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kept = torch.zeros(1, dtype=torch.int32, device="cuda")
        idx = torch.empty(n, dtype=torch.int32, device="cuda")

        rule = 2 if case == "random" else 0

        def call(i):
            dcp.dcp_score_mask(x0, xr, FULL.gamma, rule, None, None, idx, kept, status, ws, random_stream=i)
        nbytes = 2 * n * FULL.d * 4
    for i in range(warmup):
        call(i)
    times = []
    for i in range(steps):
        flush.fill_(1)
        _ = drain.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call(warmup + i)
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    st = dcp.dcp_get_status(status)
    ms = float(np.median(times))
    print(json.dumps({"case": case, "us_per_call": ms * 1e3, "algorithmic_bytes": nbytes,
                      "GB_per_s": nbytes / (ms * 1e-3) / 1e9, "steps": steps, "status": dcp.dcp_status_string(st)}))


# ------------------------------------------------------------------------------------------ CPU oracle (baseline)
class OracleSample:
    """The CPU oracle's prune step on a bounded sample of the workload: the whole score / threshold / index scan of
    the chunk plus the gather and re-phase of `n_planes` of its planes (a host cache holding only those planes, with
    the values they have in the full workload)."""

    def __init__(self, w, n_planes: int):
        import oracle
        import synth
        from oracle import replay
        from synth import workloads as W
        self.oracle, self.w = oracle, w
        self.c, self.q0_prev, self.q0 = w.evictions()[-1]
        self.planes = list(range(0, w.n_planes, max(1, w.n_planes // n_planes)))[:n_planes]
        dt = np.uint16 if w.dtype == 0 else np.float32
        k_arr = np.zeros((1, len(self.planes), w.cap, w.D), dt)
        v_arr = np.zeros((1, len(self.planes), w.cap, w.D), dt)
        for cc in list(range(w.sink_chunks)) + w.resident_window(self.c):
            row0 = W.chunk_row0(w, cc)
            for i, p in enumerate(self.planes):
                for arr, what in ((k_arr, W.S_K), (v_arr, W.S_V)):
                    synth.fill_rows_host(arr[0, i:i + 1], w.dtype, 1, w.cap, row0, w.C, w.D, w.seed,
                                         W.chunk_stream(cc, what), w.C, p * w.C)
        self.hc = oracle.HostCache(k_arr, v_arr, np.zeros(len(self.planes), np.int32),
                                   np.zeros(max(w.hist_cap, 1), np.int32), w.hist_cap)
        self.x0, self.xr = w.score_inputs(self.c)
        self.cfg = replay.cfg_of(w)
        self.k = 0

    def step(self) -> float:
        """One timed oracle prune step; returns seconds."""
        w = self.w
        self.hc.hist_len[:] = 0
        t0 = time.perf_counter()
        rc, _, _, idx = self.oracle.prune_step(self.hc, self.cfg, self.x0, self.xr, w.slot_of(self.c),
                                               w.first_frame(self.c), self.q0_prev, self.q0)
        sec = time.perf_counter() - t0
        assert rc == self.oracle.OK
        self.k = len(idx)
        return sec

    def bytes_per_step(self) -> int:
        w = self.w
        return 2 * w.C * w.d * 4 + self.k * len(self.planes) * 2 * (w.D * w.esize) * 2 + w.C * 5

    def describe(self, reps: int) -> str:
        return (f"oracle prune step of {self.w.name}: full score/mask/index scan of {self.w.C} tokens + gather and "
                f"re-phase of {len(self.planes)} of {self.w.n_planes} planes (k={self.k}), {reps} timed step(s), "
                f"one thread")


# ------------------------------------------------------------------------------------------ the JSON line
L2_NOTE = "flushed between GPU steps (256 MB write, then 256 MB read to drain dirty lines); cache 30.7 GB >> L2"
COMPUTE_NOTE = "fp32 score, fp32 compensated rotation, bf16 storage (the CPU oracle: fp64, rounded once to bf16)"


def line_config(w, k: int) -> dict:
    """The `config` object of the JSON line, the same for the GPU arm and the reference (CPU oracle) arm: the workload
    and its step's kept count and algorithmic bytes (history empty: nothing is re-indexed)."""
    return {"workload": w.name, "L": w.L, "H": w.H, "D": w.D, "tokens_per_chunk": w.C, "d": w.d, "kept": k,
            "evicting_chunk": w.evictions()[-1][0], "q0": w.evictions()[-1][2],
            "algorithmic_bytes_per_step": w.algorithmic_bytes(k, w.n_planes, 0), "l2": L2_NOTE}


def _rate(us: float, nbytes: int, peak: float) -> dict:
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us_per_step": round(us, 1), "GB_per_s": round(gbs) if gbs >= 100 else round(gbs, 2),
            "frac": round(gbs / peak, 3) if gbs >= 100 else round(gbs / peak, 5)}


def compact_extra(d: dict, peak: float) -> dict:
    """Every extra workload as a short {us_per_step, GB_per_s, frac} object (frac of the measured copy peak), so that
    the whole summary sits in the last part of the line."""
    out = {}

    def put(name, src, us_key="us_per_step", bytes_key=None):
        if src is None:
            return
        nbytes = src[bytes_key] if bytes_key else src["GB_per_s"] * 1e9 * src[us_key] * 1e-6
        out[name] = _rate(src[us_key], nbytes, peak)
    put("full_rotated_2r", d.get("full_depth_rotated"))
    if "full_depth_rotated" in d:
        out["full_rotated_2r"]["gather_us"] = round(d["full_depth_rotated"]["gather_us"], 1)
    put("random_ablation", d.get("full_depth_random_ablation"))
    put("paged_hnd", d.get("full_depth_paged_hnd"))
    put("paged_nhd", d.get("full_depth_paged_nhd"))
    put("paged_hnd_2r", d.get("full_depth_rotated_paged_hnd"))
    put("tiny_fp32", d.get("tiny_fp32_single_prune"), bytes_key="algorithmic_bytes")
    put("mid_bf16", d.get("mid_bf16_single_eviction"), bytes_key="algorithmic_bytes")
    hs = d.get("head_specialised_prefix")
    if hs:
        for i, e in enumerate(hs["evictions"]):
            put(f"hs_prefix_ev{i + 1}", e)
    for name, key in (("rollout_eager", "minute_rollout_gqa8"),
                      ("rollout_read_time", "minute_rollout_gqa8_read_time_reindex")):
        r = d.get(key)
        if r:
            gbs = r["GB_per_s"]
            out[name] = {"us_per_step": round(r["mean_us_per_step"], 1), "GB_per_s": round(gbs),
                         "frac": round(gbs / peak, 3), "last10_us": round(r["last10_mean_us"], 1),
                         "PR": round(r["cumulative_PR"], 4)}
            if "read_history_keys" in r:
                rh = r["read_history_keys"]
                out["read_final_history"] = _rate(rh["us"], rh["bytes"], peak)
            if "drift_eager_vs_read_time" in r:
                out[name]["drift_of_pair"] = round(r["drift_eager_vs_read_time"]["max_of_pair_length"], 4)
    g = d.get("cuda_graph_replay")
    if g:
        out["graph_replay_us"] = {x["workload"].split("_")[0]: [round(x["direct_us"], 1), round(x["graph_replay_us"], 1)]
                                  for x in g}
    sn = d.get("host_snapshot_restore")
    if sn:
        out["host_snapshot"] = {"GB_per_s": round(sn["snapshot_GB_per_s"], 1),
                                "frac_of_link": round(sn["frac_of_plain_copy"]["snapshot"], 3)}
        out["host_restore"] = {"GB_per_s": round(sn["restore_GB_per_s"], 1),
                               "frac_of_link": round(sn["frac_of_plain_copy"]["restore"], 3)}
    return out


# ------------------------------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="dcp", choices=["dcp", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the rotated full-depth line and the CPU baseline")
    ap.add_argument("--oracle-planes", type=int, default=64)
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling captures only: the same workload with fewer layers (a few GB on the device)")
    ap.add_argument("--tokens-per-frame", type=int, default=0,
                    help="profiling captures only: the same workload with shorter chunks (every plane kept, a few GB)")
    ap.add_argument("--rotated", action="store_true",
                    help="profiling captures only: the rotated full-depth eviction (every kept key turns) instead")
    ap.add_argument("--preroll", type=float, default=1.0, help="seconds of untimed steps before the timed region")
    ap.add_argument("--detail", default="", help="write the full result of every extra workload (curves, per-kernel "
                                                 "times) as JSON to this file; the line carries a compact summary")
    ap.add_argument("--case", default="step",
                    choices=["step", "reindex", "score", "random", "read", "snapshot", "paged-hnd", "paged-nhd", "mid",
                             "rollout-late"],
                    help="step: the prune step (default); reindex: dcp_rope_reindex of a 64-plane cache with 90,000 "
                         "history rows per plane; score: dcp_score_mask of one full-depth chunk (random: under "
                         "keep rule 2); read: dcp_read_history_keys of the re-index case's history; snapshot: "
                         "dcp_snapshot / dcp_restore of the state after the full-depth eviction cut to --layers "
                         "(default 8) layers; paged-hnd / paged-nhd: the full-depth step on a paged copy of the "
                         "cache (16-position blocks); mid: the mid bf16 eviction (history of five chunks built by the "
                         "library, re-indexed 36 -> 40 in the gather's launch), --steps repetitions; rollout-late: the "
                         "last eviction of the eager minute rollout cut to --layers (default 4) layers, its history "
                         "built by the library over the 55 earlier evictions, --steps repetitions")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.case == "snapshot":
        import __graft_entry__
        __graft_entry__.build()
        from synth.workloads import FULL, scaled
        print(json.dumps({"case": "snapshot", **run_snapshot(scaled(FULL, L=args.layers or 8), reps=args.steps)}))
        return
    if args.case.startswith("paged-"):
        import __graft_entry__
        __graft_entry__.build()
        import autoregressive_video_diffusion_gb300 as dcp
        from synth.workloads import FULL, scaled
        wp = FULL if args.layers <= 0 else scaled(FULL, L=args.layers, name=f"{FULL.name}_L{args.layers}")
        layout = dcp.DCP_PAGED_HND if args.case == "paged-hnd" else dcp.DCP_PAGED_NHD
        r = run_gpu(wp, args.steps, args.warmup, 1, 0, 0, None, e2e_steps=0, preroll_s=args.preroll,
                    paged=(16, layout))
        print(json.dumps({"case": args.case, "workload": wp.name, "block_size": 16, "kept": r["k"],
                          "us_per_step": r["ms"] * 1e3, "GB_per_s": r["alg_bytes"] / (r["ms"] * 1e-3) / 1e9,
                          "gather_us": r["gather_ms"] * 1e3,
                          "gather_GB_per_s": r["gather_bytes"] / (r["gather_ms"] * 1e-3) / 1e9}))
        return
    if args.case == "mid":
        import __graft_entry__
        __graft_entry__.build()
        from synth.workloads import MID
        print(json.dumps({"case": "mid", **run_last_eviction(MID, reps=args.steps)}))
        return
    if args.case == "rollout-late":
        import __graft_entry__
        __graft_entry__.build()
        from synth.workloads import ROLLOUT, scaled
        wr = scaled(ROLLOUT, L=args.layers or 4, name=f"{ROLLOUT.name}_L{args.layers or 4}")
        print(json.dumps({"case": "rollout-late", **run_last_eviction(wr, reps=args.steps)}))
        return
    if args.case != "step":
        run_entry_case(args.case, args.steps, args.warmup)
        return

    from synth.workloads import FULL, FULL_ROTATED, scaled
    base = FULL_ROTATED if args.rotated else FULL
    w = base if args.layers <= 0 else scaled(base, L=args.layers, name=f"{base.name}_L{args.layers}")
    if args.tokens_per_frame > 0:
        T = args.tokens_per_frame
        w = scaled(w, tokens_per_frame=T, hist_cap=4 * T, name=f"{w.name}_T{T}")
    world, rank, local = dist_setup() if args.impl == "dcp" else (int(os.environ.get("WORLD_SIZE", "1")),
                                                                 int(os.environ.get("RANK", "0")), 0)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()

    if args.impl == "reference":
        if rank != 0:
            return
        # the CPU oracle and the input generator only: the product library is neither built nor loaded here
        import oracle
        import synth
        oracle.build()
        synth.build()
        sample = OracleSample(w, args.oracle_planes)
        for _ in range(args.warmup):
            sample.step()
        secs = [sample.step() for _ in range(args.steps)]
        value = sample.bytes_per_step() / float(np.mean(secs)) / 1e9
        desc = sample.describe(args.steps)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": float(np.mean(secs)) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": line_config(w, sample.k), "compute": COMPUTE_NOTE,
                "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
                "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    dist_barrier(world)
    import autoregressive_video_diffusion_gb300  # noqa: F401
    torch.cuda.set_device(local)
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    res = run_gpu(w, args.steps, args.warmup, world, rank, local, clocks, e2e_steps=max(3, args.steps),
                  preroll_s=args.preroll)
    if clocks:
        clocks.stop()
        clk = clocks.summary(*res["wall"])
    extra = {}
    if not args.no_extra:
        r2 = run_gpu(FULL_ROTATED, max(5, args.steps // 2), args.warmup, world, rank, local, None, e2e_steps=0)
        extra["full_depth_rotated"] = {
            "workload": FULL_ROTATED.name, "q0": FULL_ROTATED.evictions()[-1][2], "kept": r2["k"],
            "us_per_step": r2["ms_max"] * 1e3, "GB_per_s": r2["alg_bytes"] / (r2["ms_max"] * 1e-3) / 1e9,
            "gather_us": r2["gather_ms"] * 1e3,
            "gather_GB_per_s": r2["gather_bytes"] / (r2["gather_ms"] * 1e-3) / 1e9}
        r3 = run_gpu(FULL, max(5, args.steps // 2), args.warmup, world, rank, local, None, e2e_steps=0, keep_rule=2)
        extra["full_depth_random_ablation"] = {
            "workload": FULL.name, "keep_rule": 2, "kept": r3["k"], "us_per_step": r3["ms_max"] * 1e3,
            "GB_per_s": r3["alg_bytes"] / (r3["ms_max"] * 1e-3) / 1e9, "scan_us": r3["scan_ms"] * 1e3,
            "gather_us": r3["gather_ms"] * 1e3,
            "note": "Random at the discrepancy rule's kept count (radix select of SplitMix64 priorities in the scan)"}
        import autoregressive_video_diffusion_gb300 as dcp
        for name, wl, layout in (("full_depth_paged_hnd", FULL, dcp.DCP_PAGED_HND),
                                 ("full_depth_paged_nhd", FULL, dcp.DCP_PAGED_NHD),
                                 ("full_depth_rotated_paged_hnd", FULL_ROTATED, dcp.DCP_PAGED_HND)):
            rp = run_gpu(wl, max(5, args.steps // 2), args.warmup, world, rank, local, None, e2e_steps=0,
                         paged=(16, layout))
            extra[name] = {"workload": wl.name, "block_size": 16, "layout": "HND" if layout == 0 else "NHD",
                           "kept": rp["k"], "us_per_step": rp["ms_max"] * 1e3,
                           "GB_per_s": rp["alg_bytes"] / (rp["ms_max"] * 1e-3) / 1e9,
                           "gather_us": rp["gather_ms"] * 1e3,
                           "gather_GB_per_s": rp["gather_bytes"] / (rp["gather_ms"] * 1e-3) / 1e9}
        from synth.workloads import HS_PREFIX, MID, ROLLOUT, TINY
        extra["tiny_fp32_single_prune"] = run_last_eviction(TINY, reps=20)
        extra["mid_bf16_single_eviction"] = run_last_eviction(MID, reps=20)
        extra["cuda_graph_replay"] = [run_graph_replay(TINY, reps=23), run_graph_replay(MID, reps=23)]
        extra["head_specialised_prefix"] = run_head_specialised(HS_PREFIX, reps=3)
        extra["minute_rollout_gqa8"] = run_rollout(ROLLOUT)
        eager_keys = extra["minute_rollout_gqa8"].pop("_final_keys")
        extra["minute_rollout_gqa8_read_time_reindex"] = run_rollout(ROLLOUT, reindex_mode=1, eager_keys=eager_keys)
        del eager_keys
        from synth.workloads import scaled
        extra["host_snapshot_restore"] = run_snapshot(scaled(FULL, L=8), reps=5)
    if rank != 0:
        return
    peak, peak_kind = _peaks()
    value = job_throughput(res["alg_bytes"], res["ms_max"], world)
    gather_gbs = res["gather_bytes"] / (res["gather_ms"] * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_max"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": line_config(w, res["k"]), "compute": COMPUTE_NOTE,
        "us_per_step": res["ms_max"] * 1e3,
        "pct_of_nominal_hbm": 100.0 * (value / world) / NOMINAL_HBM_GBS,
        "pct_of_measured_hbm": 100.0 * (value / world) / peak,
        "roofline": {"bound": "hbm", "kernel": "gather_staged_kernel" if w is FULL else "gather", "achieved": gather_gbs,
                     "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": gather_gbs / peak,
                     "traffic": _gather_traffic() if w is FULL else None,
                     "algorithmic_bytes_per_launch": res["gather_bytes"]},
        "phases_us": {"scan": res["scan_ms"] * 1e3, "gather": res["gather_ms"] * 1e3,
                      "note": "per-kernel events from a second loop of the same steps"},
        "gpu_launches": res["launches"],
        "clocks": clk,
    }
    if res["e2e_ms"] is not None:
        line["e2e"] = {"value": job_throughput(res["alg_bytes"], res["e2e_ms"], world), "unit": "GB/s",
                       "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                       "us_per_step": res["e2e_ms"] * 1e3, "median_us_per_step": res["e2e_median_ms"] * 1e3,
                       "inputs": "page-locked host memory read by the scan kernel over the host link; kept count "
                                 "written to page-locked host memory by the scan kernel",
                       "with_explicit_copies": {"median_us_per_step": res["copy_e2e_ms"] * 1e3,
                                                "h2d_copy_us_median": res["h2d_ms"] * 1e3}}
    if not args.no_extra:
        sample = OracleSample(w, args.oracle_planes)
        sample.step()
        secs = [sample.step() for _ in range(5)]
        line["cpu_baseline"] = {"value": sample.bytes_per_step() / float(np.mean(secs)) / 1e9, "unit": "GB/s",
                                "cores": 1, "kind": "oracle", "sample": sample.describe(5),
                                "host_cores_available": cores, "host_cpu": _cpu_model()}
    if extra:
        if args.detail:
            with open(args.detail, "w") as f:
                json.dump(extra, f)
        line["extra"] = compact_extra(extra, peak)  # last: the end of the line holds every workload's summary
    print(json.dumps(line))


if __name__ == "__main__":
    main()
