"""Seeded synthetic inputs for the DeCoPrune prune step (shared by the oracle's tests, the CUDA tests and the bench).

This module draws numbers; it computes nothing of the prune step itself. Every value is a pure function of
(seed, stream, index) — see ``synth.cu`` for the exact definitions — so the host can regenerate any row of a
cache that the device filled, bit for bit.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cu")
_LIB = os.path.join(_HERE, "libsynth.so")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def build_cmd():
    return [NVCC, *ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-ffp-contract=off",
            "-o", _LIB, _SRC]


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.run(build_cmd(), check=True)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, u64, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
        L.synth_stream_key.argtypes = [u64, u64]
        L.synth_stream_key.restype = u64
        L.synth_word.argtypes = [u64, u64]
        L.synth_word.restype = u64
        L.synth_normal_f32.argtypes = [vp, i64, u64, u64, i64]
        L.synth_uniform_f64.argtypes = [vp, i64, u64, u64, i64]
        L.synth_fill_rows_host.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, i64, u64, u64, i64, i64]
        L.synth_fill_rows_device.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, i64, u64, u64, i64, i64, vp]
        L.synth_fill_rows_device.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def normal_f32(n: int, seed: int, stream: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().synth_normal_f32(_ptr(out), n, seed, stream, offset)
    return out


def uniform_f64(n: int, seed: int, stream: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().synth_uniform_f64(_ptr(out), n, seed, stream, offset)
    return out


DT_BF16, DT_F32 = 0, 1


def fill_rows_host(out: np.ndarray, dtype: int, planes: int, plane_stride_rows: int, row0: int, rows: int, D: int,
                   seed: int, stream: int, key_rows_per_plane: int, key_row0: int = 0) -> None:
    """Write normal(stream) values into rows [row0, row0+rows) of each plane of a [planes][stride][D] array.

    The counter of element e of row (row0 + r) of plane p is ((p*key_rows_per_plane) + key_row0 + r)*D + e.
    ``out`` is uint16 (bf16 bits) for dtype 0 and float32 for dtype 1.
    """
    assert out.dtype == (np.uint16 if dtype == DT_BF16 else np.float32)
    assert out.size >= planes * plane_stride_rows * D
    lib().synth_fill_rows_host(_ptr(out), dtype, planes, plane_stride_rows, row0, rows, D, seed, stream,
                               key_rows_per_plane, key_row0)


def fill_rows_device(ptr: int, dtype: int, planes: int, plane_stride_rows: int, row0: int, rows: int, D: int,
                     seed: int, stream: int, key_rows_per_plane: int, key_row0: int, cuda_stream: int) -> None:
    """Device version of :func:`fill_rows_host` (same values, bit for bit) into device memory at ``ptr``."""
    rc = lib().synth_fill_rows_device(ctypes.c_void_p(ptr), dtype, planes, plane_stride_rows, row0, rows, D, seed,
                                      stream, key_rows_per_plane, key_row0, ctypes.c_void_p(cuda_stream))
    if rc != 0:
        raise RuntimeError("synth_fill_rows_device failed")


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)
