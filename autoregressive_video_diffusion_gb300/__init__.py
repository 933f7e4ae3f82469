"""Python binding of libdcp, the GB300 (sm_103a) DeCoPrune history-KV prune step.

Argument marshalling only: every function here passes tensor addresses and sizes to the C ABI declared in
``include/dcp.h`` (same names) on torch's current CUDA stream, and raises :class:`DcpError` on a non-zero status.
Every step of the prune runs in the library's CUDA kernels; there is no CPU or PyTorch fallback, and importing this
package fails if ``libdcp.so`` has not been built (``python autoregressive_video_diffusion_gb300/build.py``).

The method (page "DeCoPrune이 디노이징 불일치로 비디오 KV 캐시를 85% 줄인다", onedev.kr/papers/726): score each
token of the chunk that leaves the dense window by l = (1/d)||x0hat(tau*) - x_final||^2, keep the tokens with
l > gamma (one mask for every layer), physically gather K[m], V[m] into the compacted history, and re-index the
temporal RoPE phase of history keys to t~(t) = q0 - g(q0 - t).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdcp.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python autoregressive_video_diffusion_gb300/build.py` "
                      "(nvcc, sm_103a).  There is no fallback implementation.")

lib = ctypes.CDLL(LIB_PATH)

DCP_OK, DCP_EINVAL, DCP_ECAPACITY, DCP_ECUDA, DCP_ETIMEOUT, DCP_EDEVICE = range(6)
DCP_BF16, DCP_F32 = 0, 1

# The page's fixed choices (section "premises and limits"): 4-step schedule, probe at zero-based index 2, gamma.
SCHEDULE = (999, 957, 899, 702)
PROBE_INDEX = 2
TAU_STAR = SCHEDULE[PROBE_INDEX]
GAMMA = 0.10


class DcpCacheC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("L", ctypes.c_int32), ("H", ctypes.c_int32),
                ("D", ctypes.c_int32), ("dtype", ctypes.c_int32), ("cap", ctypes.c_int64),
                ("hist_cap", ctypes.c_int64), ("hist_len", ctypes.c_void_p), ("hist_t", ctypes.c_void_p),
                ("status", ctypes.c_void_p)]


class DcpConfigC(ctypes.Structure):
    _fields_ = [("gamma", ctypes.c_float), ("keep_rule", ctypes.c_int32), ("sink_chunks", ctypes.c_int32),
                ("window_chunks", ctypes.c_int32), ("tokens_per_frame", ctypes.c_int32),
                ("frames_per_chunk", ctypes.c_int32), ("n_temporal_pairs", ctypes.c_int32),
                ("pair_layout", ctypes.c_int32), ("rope_base", ctypes.c_double), ("g_recent_R", ctypes.c_double),
                ("g_span_S", ctypes.c_double), ("g_mode", ctypes.c_int32), ("rephase_sink", ctypes.c_int32),
                ("max_frames", ctypes.c_int32), ("random_seed", ctypes.c_uint32), ("reindex_mode", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class DcpPagedCacheC(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("L", ctypes.c_int32),
                ("H", ctypes.c_int32), ("D", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("layout", ctypes.c_int32), ("n_blocks", ctypes.c_int64),
                ("hist_cap", ctypes.c_int64), ("hist_blocks", ctypes.c_void_p), ("window_blocks", ctypes.c_void_p),
                ("hist_len", ctypes.c_void_p), ("hist_t", ctypes.c_void_p), ("status", ctypes.c_void_p)]


class DcpPrCounter(ctypes.Structure):
    _fields_ = [("visible", ctypes.c_int64), ("full", ctypes.c_int64)]


_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_pc, _pg = ctypes.POINTER(DcpCacheC), ctypes.POINTER(DcpConfigC)
_SIGS = {
    "dcp_workspace_size": ([_pc, _pg], _sz),
    "dcp_score_workspace_size": ([_i32], _sz),
    "dcp_workspace_init": ([_vp, _sz, _vp], _i32),
    "dcp_score_mask": ([_vp, _vp, _i32, _i32, _f32, _i32, ctypes.c_uint64, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                        _vp], _i32),
    "dcp_compact_layers": ([_pc, _pg, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _sz, _vp], _i32),
    "dcp_rope_reindex": ([_pc, _pg, _i32, _i32, _vp, _sz, _vp], _i32),
    "dcp_prune_step": ([_pc, _pg, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "dcp_workspace_outputs": ([_pc, _pg, _vp, _vp, _vp, _vp], _i32),
    "dcp_get_status": ([_vp, _vp], _i32),
    "dcp_reset_status": ([_vp, _vp], _i32),
    "dcp_status_string": ([_i32], ctypes.c_char_p),
    "dcp_pr_add_chunk": ([ctypes.POINTER(DcpPrCounter), _i64, _i64, _i64, _i64, _i64], None),
    "dcp_pr_value": ([ctypes.POINTER(DcpPrCounter)], ctypes.c_double),
    "dcp_abi_struct_sizes": ([], ctypes.c_uint32),
    "dcp_set_phase_events": ([_vp, _vp], _i32),
    "dcp_prune_step_noalloc": ([_pc, _pg, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp], _i32),
    "dcp_paged_workspace_size": ([ctypes.POINTER(DcpPagedCacheC), _pg], _sz),
    "dcp_paged_prune_step": ([ctypes.POINTER(DcpPagedCacheC), _pg, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp,
                              _vp, _vp, _sz, _vp], _i32),
    "dcp_abi_paged_cache_size": ([], ctypes.c_uint32),
    "dcp_read_history_keys": ([_pc, _pg, _i32, _i32, _i32, _vp, _vp, _sz, _vp], _i32),
    "dcp_phase_table": ([_pg, _i32, _i32, _i32, _vp, _vp], _i32),
    "dcp_paged_read_history_keys": ([ctypes.POINTER(DcpPagedCacheC), _pg, _i32, _i32, _i32, _vp, _vp, _sz, _vp],
                                    _i32),
    "dcp_snapshot_max_bytes": ([_pc, _pg, ctypes.c_uint32], _sz),
    "dcp_snapshot": ([_pc, _pg, ctypes.c_uint32, _i32, _vp, _sz, _vp, _sz, _vp], _i32),
    "dcp_restore": ([_pc, _pg, _vp, _sz, ctypes.POINTER(_i32), ctypes.POINTER(ctypes.c_uint32), _vp, _sz, _vp],
                    _i32),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res

_sizes = lib.dcp_abi_struct_sizes()
if (_sizes >> 16) != ctypes.sizeof(DcpCacheC) or (_sizes & 0xFFFF) != ctypes.sizeof(DcpConfigC) or \
        lib.dcp_abi_paged_cache_size() != ctypes.sizeof(DcpPagedCacheC):
    raise ImportError("libdcp struct layout does not match the binding")


class DcpError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: {dcp_status_string(status)} ({status})")
        self.status = status


def dcp_status_string(status: int) -> str:
    return lib.dcp_status_string(status).decode()


def _check(rc: int, what: str) -> None:
    if rc != DCP_OK:
        raise DcpError(what, rc)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


@dataclass
class Config:
    """Method parameters (dcp_config)."""
    gamma: float = GAMMA
    keep_rule: int = 0
    sink_chunks: int = 1
    window_chunks: int = 3
    tokens_per_frame: int = 1560
    frames_per_chunk: int = 4
    n_temporal_pairs: int = 22
    rope_base: float = 10000.0
    g_recent_R: float = 12.0
    g_span_S: float = 24.0
    g_mode: int = 0
    max_frames: int = 256
    pair_layout: int = 0
    rephase_sink: int = 0
    random_seed: int = 0
    reindex_mode: int = 0

    @property
    def C(self) -> int:
        return self.tokens_per_frame * self.frames_per_chunk

    def c(self) -> DcpConfigC:
        return DcpConfigC(self.gamma, self.keep_rule, self.sink_chunks, self.window_chunks, self.tokens_per_frame,
                          self.frames_per_chunk, self.n_temporal_pairs, self.pair_layout, self.rope_base,
                          self.g_recent_R, self.g_span_S, self.g_mode, self.rephase_sink, self.max_frames,
                          self.random_seed & 0xFFFFFFFF, self.reindex_mode, 0)

    def random_stream(self, evict_first_frame: int) -> int:
        """SplitMix64 seed a prune step under keep_rule 2 draws from (as dcp_prune_step forms it)."""
        return ((self.random_seed & 0xFFFFFFFF) << 32) | (evict_first_frame & 0xFFFFFFFF)


class KVCache:
    """Device tensors of one KV cache in the sink | history | window-ring layout (dcp_cache)."""

    def __init__(self, L: int, H: int, D: int, dtype: int, cap: int, hist_cap: int, device="cuda"):
        tdt = torch.bfloat16 if dtype == DCP_BF16 else torch.float32
        self.L, self.H, self.D, self.dtype, self.cap, self.hist_cap = L, H, D, dtype, cap, hist_cap
        self.k = torch.empty((L, H, cap, D), dtype=tdt, device=device)
        self.v = torch.empty((L, H, cap, D), dtype=tdt, device=device)
        self.hist_len = torch.zeros(L * H, dtype=torch.int32, device=device)
        self.hist_t = torch.zeros(max(hist_cap, 1), dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def c(self) -> DcpCacheC:
        return DcpCacheC(_ptr(self.k), _ptr(self.v), self.L, self.H, self.D, self.dtype, self.cap, self.hist_cap,
                         _ptr(self.hist_len), _ptr(self.hist_t), _ptr(self.status))


def dcp_workspace_size(cache: KVCache, cfg: Config) -> int:
    cc, gc = cache.c(), cfg.c()
    n = lib.dcp_workspace_size(ctypes.byref(cc), ctypes.byref(gc))
    if n == 0:
        raise DcpError("dcp_workspace_size", DCP_EINVAL)
    return n


def dcp_score_workspace_size(n_tok: int) -> int:
    return lib.dcp_score_workspace_size(n_tok)


def dcp_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(lib.dcp_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "dcp_workspace_init")


def new_workspace(nbytes: int, device="cuda", stream=None) -> torch.Tensor:
    """A zero-initialised, 256-byte aligned device workspace (torch allocation; not on the hot path)."""
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + nbytes]
    dcp_workspace_init(ws, stream)
    return ws


def dcp_score_mask(x0hat: torch.Tensor, xref: torch.Tensor, gamma: float, keep_rule: int, ell, mask, idx, kept,
                   status: torch.Tensor, ws: torch.Tensor, stream=None, random_stream: int = 0) -> None:
    n_tok, d = x0hat.shape
    _check(lib.dcp_score_mask(_ptr(x0hat), _ptr(xref), n_tok, d, gamma, keep_rule, random_stream, _ptr(ell),
                              _ptr(mask), _ptr(idx), _ptr(kept), _ptr(status), _ptr(ws), ws.numel(), _stream(stream)),
           "dcp_score_mask")


def dcp_compact_layers(cache: KVCache, cfg: Config, evict_slot: int, evict_first_frame: int, mask: torch.Tensor,
                       head_is_static, q0: int, kept, ws: torch.Tensor, stream=None) -> None:
    cc, gc = cache.c(), cfg.c()
    _check(lib.dcp_compact_layers(ctypes.byref(cc), ctypes.byref(gc), evict_slot, evict_first_frame, _ptr(mask),
                                  _ptr(head_is_static), q0, _ptr(kept), _ptr(ws), ws.numel(), _stream(stream)),
           "dcp_compact_layers")


def dcp_rope_reindex(cache: KVCache, cfg: Config, q0_prev: int, q0: int, ws: torch.Tensor, stream=None) -> None:
    cc, gc = cache.c(), cfg.c()
    _check(lib.dcp_rope_reindex(ctypes.byref(cc), ctypes.byref(gc), q0_prev, q0, _ptr(ws), ws.numel(),
                                _stream(stream)), "dcp_rope_reindex")


def dcp_prune_step(cache: KVCache, cfg: Config, x0hat: torch.Tensor, xref: torch.Tensor, evict_slot: int,
                   evict_first_frame: int, q0_prev: int, q0: int, head_is_static, kept_dev, kept_host_pinned,
                   ws: torch.Tensor, stream=None) -> None:
    cc, gc = cache.c(), cfg.c()
    _check(lib.dcp_prune_step(ctypes.byref(cc), ctypes.byref(gc), _ptr(x0hat), _ptr(xref), x0hat.shape[1],
                              evict_slot, evict_first_frame, q0_prev, q0, _ptr(head_is_static), _ptr(kept_dev),
                              _ptr(kept_host_pinned), _ptr(ws), ws.numel(), _stream(stream)), "dcp_prune_step")


DCP_NOALLOC_WORKSPACE_BYTES = 4 << 20


def dcp_prune_step_noalloc(cache: KVCache, cfg: Config, x0hat: torch.Tensor, xref: torch.Tensor, evict_slot: int,
                           evict_first_frame: int, q0_prev: int, q0: int, head_is_static, kept_dev, kept_host_pinned,
                           stream=None) -> None:
    """dcp_prune_step without a workspace, for callers that cannot allocate device memory: the library's own fixed
    scratch array (DCP_NOALLOC_WORKSPACE_BYTES per GPU) is used instead.  Calls that overlap on the GPU race."""
    cc, gc = cache.c(), cfg.c()
    _check(lib.dcp_prune_step_noalloc(ctypes.byref(cc), ctypes.byref(gc), _ptr(x0hat), _ptr(xref), x0hat.shape[1],
                                      evict_slot, evict_first_frame, q0_prev, q0, _ptr(head_is_static),
                                      _ptr(kept_dev), _ptr(kept_host_pinned), _stream(stream)),
           "dcp_prune_step_noalloc")


def dcp_workspace_outputs(cache: KVCache, cfg: Config, ws: torch.Tensor):
    """Views of the workspace where the last prune/compact call left l (fp32), the mask (uint8), the index list."""
    cc, gc = cache.c(), cfg.c()
    pe, pm, pi = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
    _check(lib.dcp_workspace_outputs(ctypes.byref(cc), ctypes.byref(gc), _ptr(ws), ctypes.byref(pe),
                                     ctypes.byref(pm), ctypes.byref(pi)), "dcp_workspace_outputs")
    C, base = cfg.C, ws.data_ptr()
    ell = ws[pe.value - base: pe.value - base + 4 * C].view(torch.float32)
    mask = ws[pm.value - base: pm.value - base + C]
    idx = ws[pi.value - base: pi.value - base + 4 * C].view(torch.int32)
    return ell, mask, idx


def dcp_get_status(status: torch.Tensor, stream=None) -> int:
    return lib.dcp_get_status(_ptr(status), _stream(stream))


def dcp_reset_status(status: torch.Tensor, stream=None) -> None:
    _check(lib.dcp_reset_status(_ptr(status), _stream(stream)), "dcp_reset_status")


def dcp_pr_add_chunk(acc: DcpPrCounter, n_planes: int, hist_len_sum: int, sink_visible: int, window_visible: int,
                     prior_tokens: int) -> None:
    lib.dcp_pr_add_chunk(ctypes.byref(acc), n_planes, hist_len_sum, sink_visible, window_visible, prior_tokens)


def dcp_pr_value(acc: DcpPrCounter) -> float:
    return lib.dcp_pr_value(ctypes.byref(acc))


def dcp_set_phase_events(ev_after_scan, ev_after_gather) -> None:
    """Record torch.cuda.Event objects (or None) after the scan and gather kernels of each dcp_prune_step."""
    a = None if ev_after_scan is None else ev_after_scan.cuda_event
    b = None if ev_after_gather is None else ev_after_gather.cuda_event
    _check(lib.dcp_set_phase_events(a, b), "dcp_set_phase_events")


# ------------------------------------------------------------------------------------------ host snapshot
def dcp_snapshot_max_bytes(cache: KVCache, cfg: Config, live_slots: int) -> int:
    cc, gc = cache.c(), cfg.c()
    n = lib.dcp_snapshot_max_bytes(ctypes.byref(cc), ctypes.byref(gc), live_slots)
    if n == 0:
        raise DcpError("dcp_snapshot_max_bytes", DCP_EINVAL)
    return n


def new_snapshot_image(nbytes: int) -> torch.Tensor:
    """Page-locked, 256-byte aligned host buffer for a snapshot image (torch allocation; not on the hot path)."""
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, pin_memory=True)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + nbytes]


def snapshot_total_bytes(image: torch.Tensor) -> int:
    """Size written by the snapshot held in `image` (its header's total_bytes; read after the stream synced)."""
    return int(image[88:96].view(torch.int64).item())


def dcp_snapshot(cache: KVCache, cfg: Config, live_slots: int, q0: int, image: torch.Tensor, ws: torch.Tensor,
                 stream=None) -> None:
    cc, gc = cache.c(), cfg.c()
    _check(lib.dcp_snapshot(ctypes.byref(cc), ctypes.byref(gc), live_slots, q0, _ptr(image), image.numel(),
                            _ptr(ws), ws.numel(), _stream(stream)), "dcp_snapshot")


def dcp_restore(cache: KVCache, cfg: Config, image: torch.Tensor, ws: torch.Tensor, stream=None):
    """Returns (q0, live_slots) of the image."""
    cc, gc = cache.c(), cfg.c()
    q0, live = ctypes.c_int32(0), ctypes.c_uint32(0)
    _check(lib.dcp_restore(ctypes.byref(cc), ctypes.byref(gc), _ptr(image), image.numel(), ctypes.byref(q0),
                           ctypes.byref(live), _ptr(ws), ws.numel(), _stream(stream)), "dcp_restore")
    return q0.value, live.value


# ------------------------------------------------------------------------------------------ paged variant
DCP_PAGED_HND, DCP_PAGED_NHD = 0, 1


class PagedKVCache:
    """Device block pools and block tables of one paged KV cache (dcp_paged_cache).

    Pools are [L][n_blocks][H][block_size][D] (HND) or [L][n_blocks][block_size][H][D] (NHD); hist_blocks and
    window_blocks are int32 device tensors the caller fills (block ids of the history positions and of the ring
    slots, slot s owning entries [s * C / block_size, (s + 1) * C / block_size))."""

    def __init__(self, L: int, H: int, D: int, dtype: int, block_size: int, layout: int, n_blocks: int,
                 hist_cap: int, n_window_blocks: int, device="cuda"):
        tdt = torch.bfloat16 if dtype == DCP_BF16 else torch.float32
        shape = (L, n_blocks, H, block_size, D) if layout == DCP_PAGED_HND else (L, n_blocks, block_size, H, D)
        self.L, self.H, self.D, self.dtype = L, H, D, dtype
        self.block_size, self.layout, self.n_blocks, self.hist_cap = block_size, layout, n_blocks, hist_cap
        self.k_pool = torch.empty(shape, dtype=tdt, device=device)
        self.v_pool = torch.empty(shape, dtype=tdt, device=device)
        self.hist_blocks = torch.zeros(max(hist_cap // block_size, 1), dtype=torch.int32, device=device)
        self.window_blocks = torch.zeros(max(n_window_blocks, 1), dtype=torch.int32, device=device)
        self.hist_len = torch.zeros(L * H, dtype=torch.int32, device=device)
        self.hist_t = torch.zeros(max(hist_cap, 1), dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def c(self) -> DcpPagedCacheC:
        return DcpPagedCacheC(_ptr(self.k_pool), _ptr(self.v_pool), self.L, self.H, self.D, self.dtype,
                              self.block_size, self.layout, self.n_blocks, self.hist_cap, _ptr(self.hist_blocks),
                              _ptr(self.window_blocks), _ptr(self.hist_len), _ptr(self.hist_t), _ptr(self.status))


def dcp_paged_workspace_size(cache: PagedKVCache, cfg: Config) -> int:
    cc, gc = cache.c(), cfg.c()
    n = lib.dcp_paged_workspace_size(ctypes.byref(cc), ctypes.byref(gc))
    if n == 0:
        raise DcpError("dcp_paged_workspace_size", DCP_EINVAL)
    return n


def dcp_paged_prune_step(cache: PagedKVCache, cfg: Config, x0hat: torch.Tensor, xref: torch.Tensor, evict_slot: int,
                         evict_first_frame: int, q0_prev: int, q0: int, head_is_static, kept, kept_host,
                         ws: torch.Tensor, stream=None) -> None:
    cc, gc = cache.c(), cfg.c()
    _check(lib.dcp_paged_prune_step(ctypes.byref(cc), ctypes.byref(gc), _ptr(x0hat), _ptr(xref), x0hat.shape[1],
                                    evict_slot, evict_first_frame, q0_prev, q0, _ptr(head_is_static), _ptr(kept),
                                    _ptr(kept_host), _ptr(ws), ws.numel(), _stream(stream)), "dcp_paged_prune_step")


def paged_row_map(cfg: Config, hist_cap: int, block_size: int, sink_blocks: torch.Tensor, hist_blocks: torch.Tensor,
                  window_blocks: torch.Tensor):
    """(block, row-in-block) of every row of the contiguous layout sink | history | ring, as int64 tensors on the
    tables' device.  For moving caches between the two layouts (set-up and checks; not on the prune path)."""
    C = cfg.C
    sink = cfg.sink_chunks * C
    dev = hist_blocks.device
    pos = torch.arange(sink + hist_cap + (cfg.window_chunks + 1) * C, device=dev)
    block = torch.empty_like(pos)
    region = [(0, sink, sink_blocks), (sink, sink + hist_cap, hist_blocks),
              (sink + hist_cap, pos.numel(), window_blocks)]
    for lo, hi, tbl in region:
        i = pos[lo:hi] - lo
        if hi > lo:
            block[lo:hi] = tbl.to(device=dev, dtype=torch.int64)[i // block_size]
    return block, pos % block_size


def paged_pack(pool: torch.Tensor, t: torch.Tensor, block: torch.Tensor, off: torch.Tensor, layout: int) -> None:
    """Write a contiguous [L][H][rows][D] tensor into a block pool through a row map."""
    if layout == DCP_PAGED_HND:
        pool[:, block, :, off, :] = t.permute(2, 0, 1, 3)
    else:
        pool[:, block, off] = t.permute(0, 2, 1, 3)


def paged_unpack(pool: torch.Tensor, block: torch.Tensor, off: torch.Tensor, layout: int) -> torch.Tensor:
    """Read a block pool back into a contiguous [L][H][rows][D] tensor through a row map."""
    if layout == DCP_PAGED_HND:
        return pool[:, block, :, off, :].permute(1, 2, 0, 3).contiguous()
    return pool[:, block, off].permute(0, 2, 1, 3).contiguous()


# ------------------------------------------------------------------------------------------ read-time re-index
def dcp_read_history_keys(cache, cfg: Config, q0: int, plane0: int, n_planes: int, out: torch.Tensor,
                          ws: torch.Tensor, stream=None) -> None:
    """History keys of planes [plane0, plane0 + n_planes) turned to t~(t; q0) into out [n_planes][hist_cap][D]
    (reindex_mode 1).  `cache` is a KVCache or a PagedKVCache."""
    cc, gc = cache.c(), cfg.c()
    fn = lib.dcp_paged_read_history_keys if isinstance(cache, PagedKVCache) else lib.dcp_read_history_keys
    _check(fn(ctypes.byref(cc), ctypes.byref(gc), q0, plane0, n_planes, _ptr(out), _ptr(ws), ws.numel(),
              _stream(stream)), "dcp_read_history_keys")


def dcp_phase_table(cfg: Config, q0: int, frame_lo: int, frame_hi: int, out: torch.Tensor, stream=None) -> None:
    """cos/sin entries {c_hi, c_lo, s_hi, s_lo} of the turn t -> t~(t; q0) for frames [frame_lo, frame_hi) and every
    temporal pair, into out (float32 [(frame_hi - frame_lo) * n_t * 4], device)."""
    gc = cfg.c()
    _check(lib.dcp_phase_table(ctypes.byref(gc), q0, frame_lo, frame_hi, _ptr(out), _stream(stream)),
           "dcp_phase_table")
