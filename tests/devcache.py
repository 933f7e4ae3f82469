"""Host <-> device copies of caches for the GPU tests and smoke(): the oracle's host arrays on one side, the
library's KVCache tensors on the other.  Test infrastructure."""
from __future__ import annotations

import numpy as np
import torch

import autoregressive_video_diffusion_gb300 as dcp
from oracle import HostCache
from synth.workloads import Workload


def dcp_config(w: Workload, **over) -> dcp.Config:
    kw = dict(gamma=w.gamma, keep_rule=0, sink_chunks=w.sink_chunks, window_chunks=w.window_chunks,
              tokens_per_frame=w.tokens_per_frame, frames_per_chunk=w.frames_per_chunk,
              n_temporal_pairs=w.n_temporal_pairs, rope_base=w.rope_base, g_recent_R=w.R, g_span_S=w.S,
              g_mode=w.g_mode, max_frames=w.max_frames)
    kw.update(over)
    return dcp.Config(**kw)


def _to_torch(a: np.ndarray, w: Workload) -> torch.Tensor:
    if w.dtype == 0:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def to_device(hc: HostCache, w: Workload) -> dcp.KVCache:
    dev = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, w.hist_cap)
    dev.k.copy_(_to_torch(hc.k, w))
    dev.v.copy_(_to_torch(hc.v, w))
    dev.hist_len.copy_(torch.from_numpy(hc.hist_len))
    dev.hist_t.copy_(torch.from_numpy(hc.hist_t))
    return dev


def from_device(dev: dcp.KVCache, w: Workload) -> HostCache:
    if w.dtype == 0:
        k = dev.k.view(torch.int16).cpu().numpy().view(np.uint16)
        v = dev.v.view(torch.int16).cpu().numpy().view(np.uint16)
    else:
        k = dev.k.cpu().numpy()
        v = dev.v.cpu().numpy()
    return HostCache(k, v, dev.hist_len.cpu().numpy(), dev.hist_t.cpu().numpy(), w.hist_cap)
