"""ctypes wrapper of the plain C++ CPU oracle (``dcp_oracle.cpp``).  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline/reference leg use this package.  The
product path (``autoregressive_video_diffusion_gb300``) never imports it.

Every array is a numpy array on the host.  Caches are [L][H][cap][D] arrays of uint16 (bf16 bits) or float32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dcp_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, EINVAL, ECAPACITY = 0, 1, 2


def build_cmd():
    return ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-o", _LIB, _SRC]


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.run(build_cmd(), check=True)
    return _LIB


class OracleCache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("L", ctypes.c_int32), ("H", ctypes.c_int32),
                ("D", ctypes.c_int32), ("dtype", ctypes.c_int32), ("cap", ctypes.c_int64),
                ("hist_cap", ctypes.c_int64), ("hist_len", ctypes.c_void_p), ("hist_t", ctypes.c_void_p)]


class OracleConfig(ctypes.Structure):
    _fields_ = [("gamma", ctypes.c_float), ("keep_rule", ctypes.c_int32), ("sink_chunks", ctypes.c_int32),
                ("window_chunks", ctypes.c_int32), ("tokens_per_frame", ctypes.c_int32),
                ("frames_per_chunk", ctypes.c_int32), ("n_temporal_pairs", ctypes.c_int32),
                ("rope_base", ctypes.c_double), ("g_recent_R", ctypes.c_double), ("g_span_S", ctypes.c_double),
                ("g_mode", ctypes.c_int32), ("random_seed", ctypes.c_uint32), ("reindex_mode", ctypes.c_int32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i32, i64, f32, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        pc, pcfg = ctypes.POINTER(OracleCache), ctypes.POINTER(OracleConfig)
        sig = {
            "oracle_schedule": ([i32], i32),
            "oracle_probe_index": ([], i32),
            "oracle_default_gamma": ([], f32),
            "oracle_score": ([vp, vp, i64, i32, vp], None),
            "oracle_keep": ([vp, i64, f32, i32, vp], None),
            "oracle_splitmix64": ([ctypes.c_uint64, i64], ctypes.c_uint64),
            "oracle_keep_random": ([vp, i64, f32, ctypes.c_uint64, vp], None),
            "oracle_indices": ([vp, i64, vp], i64),
            "oracle_g": ([f64, f64, f64, f64, i32], f64),
            "oracle_phase": ([f64, f64, f64, f64, f64, i32], f64),
            "oracle_theta": ([i32, i32, f64], f64),
            "oracle_bf16_value": ([ctypes.c_uint16], f64),
            "oracle_bf16_round": ([f64], ctypes.c_uint16),
            "oracle_rotate_key_row": ([vp, i32, i32, i32, f64, f64], None),
            "oracle_gather_key_row": ([vp, vp, pc, pcfg, i32, i32], None),
            "oracle_compact_layers": ([pc, pcfg, i32, i32, vp, vp, i32, vp, vp], i32),
            "oracle_rope_reindex": ([pc, pcfg, i32, i32], i32),
            "oracle_prune_step": ([pc, pcfg, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp], i32),
            "oracle_pr_chunk": ([vp, i64, i64, i64, i64, vp, vp], None),
            "oracle_read_history_keys": ([pc, pcfg, i32, vp], None),
            "oracle_snapshot_size": ([pc, pcfg, ctypes.c_uint32], i64),
            "oracle_snapshot": ([pc, pcfg, ctypes.c_uint32, i32, vp, i64], i32),
            "oracle_restore": ([pc, pcfg, vp, i64, vp, vp], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous numpy"
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Cfg:
    """Method parameters; the readings of the points the page leaves open are listed at the top of dcp_oracle.cpp."""
    gamma: float = 0.10
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
    random_seed: int = 0
    reindex_mode: int = 0

    def c(self) -> OracleConfig:
        return OracleConfig(self.gamma, self.keep_rule, self.sink_chunks, self.window_chunks, self.tokens_per_frame,
                            self.frames_per_chunk, self.n_temporal_pairs, self.rope_base, self.g_recent_R,
                            self.g_span_S, self.g_mode, self.random_seed, self.reindex_mode)

    def random_stream(self, evict_first_frame: int) -> int:
        """The SplitMix64 stream a prune step of the Random ablation (keep_rule 2) draws from."""
        return ((self.random_seed & 0xFFFFFFFF) << 32) | (evict_first_frame & 0xFFFFFFFF)


class HostCache:
    """Host arrays of one KV cache in the sink | history | window-ring layout the oracle works on."""

    def __init__(self, k: np.ndarray, v: np.ndarray, hist_len: np.ndarray, hist_t: np.ndarray, hist_cap: int):
        assert k.shape == v.shape and k.ndim == 4 and k.dtype == v.dtype
        self.k, self.v = k, v
        self.hist_len = hist_len.astype(np.int32, copy=False)
        self.hist_t = hist_t.astype(np.int32, copy=False)
        self.hist_cap = hist_cap
        self.dtype = 0 if k.dtype == np.uint16 else 1

    def c(self) -> OracleCache:
        L, H, cap, D = self.k.shape
        return OracleCache(_p(self.k), _p(self.v), L, H, D, self.dtype, cap, self.hist_cap, _p(self.hist_len),
                           _p(self.hist_t))

    def copy(self) -> "HostCache":
        return HostCache(self.k.copy(), self.v.copy(), self.hist_len.copy(), self.hist_t.copy(), self.hist_cap)


def score(x0hat: np.ndarray, xref: np.ndarray) -> np.ndarray:
    n, d = x0hat.shape
    out = np.empty(n, np.float32)
    lib().oracle_score(_p(np.ascontiguousarray(x0hat, np.float32)), _p(np.ascontiguousarray(xref, np.float32)), n,
                       d, _p(out))
    return out


def keep(ell: np.ndarray, gamma: float = 0.10, keep_rule: int = 0) -> np.ndarray:
    out = np.empty(ell.shape[0], np.uint8)
    lib().oracle_keep(_p(np.ascontiguousarray(ell, np.float32)), ell.shape[0], gamma, keep_rule, _p(out))
    return out


def splitmix64(stream: int, i: int) -> int:
    return lib().oracle_splitmix64(stream, i)


def keep_random(ell: np.ndarray, gamma: float, stream: int) -> np.ndarray:
    """Random ablation: as many tokens as ell > gamma would keep, drawn uniformly from the SplitMix64 stream."""
    out = np.empty(ell.shape[0], np.uint8)
    lib().oracle_keep_random(_p(np.ascontiguousarray(ell, np.float32)), ell.shape[0], gamma, stream, _p(out))
    return out


def indices(mask: np.ndarray) -> np.ndarray:
    idx = np.empty(mask.shape[0], np.int32)
    k = lib().oracle_indices(_p(np.ascontiguousarray(mask, np.uint8)), mask.shape[0], _p(idx))
    return idx[:k].copy()


def g(delta, delta_max, R, S, mode=0) -> float:
    return lib().oracle_g(delta, delta_max, R, S, mode)


def phase(t, q0, T_s, R, S, mode=0) -> float:
    return lib().oracle_phase(t, q0, T_s, R, S, mode)


def theta(p, n_t, base) -> float:
    return lib().oracle_theta(p, n_t, base)


def bf16_round(x: float) -> int:
    return lib().oracle_bf16_round(x)


def bf16_value(b: int) -> float:
    return lib().oracle_bf16_value(b)


def rotate_key_row(row: np.ndarray, n_t: int, base: float, dphase: float) -> None:
    dtype = 0 if row.dtype == np.uint16 else 1
    lib().oracle_rotate_key_row(_p(row), dtype, row.shape[-1], n_t, base, dphase)


def gather_key_row(src: np.ndarray, cache: HostCache, cfg: Cfg, t: int, q0: int) -> np.ndarray:
    dst = np.empty_like(src)
    cc, oc = cache.c(), cfg.c()
    lib().oracle_gather_key_row(_p(src), _p(dst), ctypes.byref(cc), ctypes.byref(oc), t, q0)
    return dst


def compact_layers(cache: HostCache, cfg: Cfg, evict_slot: int, evict_first_frame: int, mask: np.ndarray,
                   head_is_static, q0: int):
    C = cfg.tokens_per_frame * cfg.frames_per_chunk
    idx = np.empty(C, np.int32)
    k = ctypes.c_int64(0)
    cc, oc = cache.c(), cfg.c()
    hs = None if head_is_static is None else np.ascontiguousarray(head_is_static, np.uint8)
    rc = lib().oracle_compact_layers(ctypes.byref(cc), ctypes.byref(oc), evict_slot, evict_first_frame,
                                     _p(np.ascontiguousarray(mask, np.uint8)), _p(hs), q0, _p(idx), ctypes.byref(k))
    return rc, idx[:k.value].copy()


def rope_reindex(cache: HostCache, cfg: Cfg, q0_prev: int, q0: int) -> int:
    cc, oc = cache.c(), cfg.c()
    return lib().oracle_rope_reindex(ctypes.byref(cc), ctypes.byref(oc), q0_prev, q0)


def prune_step(cache: HostCache, cfg: Cfg, x0hat: np.ndarray, xref: np.ndarray, evict_slot: int,
               evict_first_frame: int, q0_prev: int, q0: int, head_is_static=None):
    """Returns (rc, ell, mask, idx)."""
    C = cfg.tokens_per_frame * cfg.frames_per_chunk
    assert x0hat.shape[0] == C
    d = x0hat.shape[1]
    ell = np.empty(C, np.float32)
    mask = np.empty(C, np.uint8)
    idx = np.empty(C, np.int32)
    k = ctypes.c_int64(0)
    cc, oc = cache.c(), cfg.c()
    hs = None if head_is_static is None else np.ascontiguousarray(head_is_static, np.uint8)
    rc = lib().oracle_prune_step(ctypes.byref(cc), ctypes.byref(oc), _p(np.ascontiguousarray(x0hat, np.float32)),
                                 _p(np.ascontiguousarray(xref, np.float32)), d, evict_slot, evict_first_frame,
                                 q0_prev, q0, _p(hs), _p(ell), _p(mask), _p(idx), ctypes.byref(k))
    return rc, ell, mask, idx[:k.value].copy()


def pr_chunk(hist_len: np.ndarray, sink_visible: int, window_visible: int, prior: int, acc):
    """acc = [visible, full] (python ints), updated in place."""
    v, f = ctypes.c_int64(acc[0]), ctypes.c_int64(acc[1])
    hl = np.ascontiguousarray(hist_len, np.int32)
    lib().oracle_pr_chunk(_p(hl), hl.shape[0], sink_visible, window_visible, prior, ctypes.byref(v), ctypes.byref(f))
    acc[0], acc[1] = v.value, f.value


def snapshot(cache: HostCache, cfg: Cfg, live_slots: int, q0: int) -> np.ndarray:
    """Host image of the cache's non-derivable state (sink, history rows, live ring slots, hist_len, hist_t, q0)."""
    cc, oc = cache.c(), cfg.c()
    n = lib().oracle_snapshot_size(ctypes.byref(cc), ctypes.byref(oc), live_slots)
    if n < 0:
        raise ValueError("snapshot refused")
    out = np.empty(n, np.uint8)
    rc = lib().oracle_snapshot(ctypes.byref(cc), ctypes.byref(oc), live_slots, q0, _p(out), n)
    if rc != OK:
        raise ValueError(f"snapshot refused: {rc}")
    return out


def restore(cache: HostCache, cfg: Cfg, image: np.ndarray):
    """Restore an image into the cache in place; returns (rc, q0, live_slots)."""
    cc, oc = cache.c(), cfg.c()
    q0, live = ctypes.c_int32(0), ctypes.c_uint32(0)
    img = np.ascontiguousarray(image, np.uint8)
    rc = lib().oracle_restore(ctypes.byref(cc), ctypes.byref(oc), _p(img), img.shape[0], ctypes.byref(q0),
                              ctypes.byref(live))
    return rc, q0.value, live.value


def read_history_keys(cache: HostCache, cfg: Cfg, q0: int) -> np.ndarray:
    """Keys of a read-time re-indexed cache as attention at q0 sees them: [planes][hist_cap][D] (rows past a plane's
    history are zero)."""
    L, H, cap, D = cache.k.shape
    out = np.zeros((L * H, cache.hist_cap, D), cache.k.dtype)
    cc, oc = cache.c(), cfg.c()
    lib().oracle_read_history_keys(ctypes.byref(cc), ctypes.byref(oc), q0, _p(out))
    return out
