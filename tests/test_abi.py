"""The C ABI of libdcp on the host: every declared symbol is exported, struct layouts match the binding, and
host-side validation rejects bad arguments before any CUDA call.  No GPU is used: the rejected calls return before
they touch a device, and the cases that would need a device are skipped when one is present (the GPU tests cover
them with real buffers)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import autoregressive_video_diffusion_gb300 as dcp
from tests.conftest import has_gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dcp.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(dcp_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", dcp.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\sT\s(dcp_\w+)$", out.stdout, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(dcp.lib, n)


def test_struct_layout_matches_binding():
    sizes = dcp.lib.dcp_abi_struct_sizes()
    assert sizes >> 16 == ctypes.sizeof(dcp.DcpCacheC) == 72
    assert sizes & 0xFFFF == ctypes.sizeof(dcp.DcpConfigC) == 80
    assert dcp.lib.dcp_abi_paged_cache_size() == ctypes.sizeof(dcp.DcpPagedCacheC) == 96


def test_status_strings():
    assert dcp.dcp_status_string(dcp.DCP_OK) == "ok"
    for s in range(1, 6):
        assert dcp.dcp_status_string(s) not in ("ok", "unknown status")
    assert dcp.dcp_status_string(99) == "unknown status"


def test_page_constants_in_binding():
    assert dcp.SCHEDULE == (999, 957, 899, 702) and dcp.TAU_STAR == 899 and dcp.GAMMA == 0.10


# ------------------------------------------------------------------------------------------ host validation
FAKE = 1 << 40  # aligned, never dereferenced: every call below is rejected before any launch


def _cache(**over):
    kw = dict(k=FAKE, v=FAKE + (1 << 36), L=2, H=2, D=128, dtype=dcp.DCP_BF16, cap=6240 * 6, hist_cap=6240,
              hist_len=FAKE + (2 << 36), hist_t=FAKE + (3 << 36), status=FAKE + (4 << 36))
    kw.update(over)
    return dcp.DcpCacheC(**kw)


def _cfg(**over):
    c = dcp.Config(max_frames=256)
    for k, v in over.items():
        setattr(c, k, v)
    return c.c()


def _ws_size(cache, cfg):
    return dcp.lib.dcp_workspace_size(ctypes.byref(cache), ctypes.byref(cfg))


def test_workspace_size():
    n = _ws_size(_cache(), _cfg())
    assert n > 0 and n % 256 == 0
    assert dcp.lib.dcp_score_workspace_size(6240) > 0
    assert dcp.lib.dcp_score_workspace_size(0) == 0


@pytest.mark.parametrize("bad", [
    dict(k=0), dict(v=0), dict(hist_len=0), dict(hist_t=0), dict(status=0), dict(k=FAKE + 8), dict(L=0), dict(H=0),
    dict(D=0), dict(D=127), dict(D=4), dict(D=2056), dict(dtype=7), dict(cap=6240 * 5), dict(hist_cap=-1)])
def test_invalid_cache_rejected(bad):
    assert _ws_size(_cache(**bad), _cfg()) == 0


@pytest.mark.parametrize("bad", [
    dict(tokens_per_frame=0), dict(frames_per_chunk=0), dict(window_chunks=-1), dict(sink_chunks=-1),
    dict(n_temporal_pairs=65), dict(n_temporal_pairs=-1), dict(pair_layout=1), dict(rephase_sink=1),
    dict(rope_base=0.0), dict(rope_base=float("nan")), dict(g_recent_R=11.0), dict(g_span_S=11.5),
    dict(g_mode=2), dict(g_mode=1, g_span_S=-1.0), dict(keep_rule=3), dict(keep_rule=-1),
    dict(gamma=float("inf")), dict(max_frames=0), dict(reindex_mode=2), dict(reindex_mode=-1)])
def test_invalid_config_rejected(bad):
    assert _ws_size(_cache(), _cfg(**bad)) == 0


def _prune(cache, cfg, ws=FAKE, ws_bytes=None, slot=0, eff=4, q0_prev=20, q0=20, x0=FAKE, xr=FAKE, d=64):
    if ws_bytes is None:
        ws_bytes = max(_ws_size(cache, cfg), 1)
    return dcp.lib.dcp_prune_step(ctypes.byref(cache), ctypes.byref(cfg), x0, xr, d, slot, eff, q0_prev, q0, None,
                                  None, None, ws, ws_bytes, None)


@pytest.mark.skipif(has_gpu(), reason="rejected-argument calls use fake device addresses; GPU tests cover these")
@pytest.mark.parametrize("case", [
    dict(slot=4), dict(slot=-1), dict(eff=3), dict(q0=7), dict(q0=300), dict(q0_prev=21), dict(q0_prev=3),
    dict(ws=0), dict(ws=FAKE + 16), dict(ws_bytes=16), dict(x0=0), dict(xr=0), dict(d=0), dict(x0=FAKE + 2)])
def test_invalid_prune_arguments_rejected(case):
    assert _prune(_cache(), _cfg(), **case) == dcp.DCP_EINVAL


@pytest.mark.skipif(has_gpu(), reason="rejected-argument calls use fake device addresses; GPU tests cover these")
def test_invalid_other_entry_points_rejected():
    c, g = _cache(), _cfg()
    n = _ws_size(c, g)
    L = dcp.lib
    assert L.dcp_compact_layers(ctypes.byref(c), ctypes.byref(g), 0, 4, None, None, 20, None, FAKE, n, None) == 1
    assert L.dcp_compact_layers(ctypes.byref(c), ctypes.byref(g), 9, 4, FAKE, None, 20, None, FAKE, n, None) == 1
    assert L.dcp_rope_reindex(ctypes.byref(c), ctypes.byref(g), 30, 20, FAKE, n, None) == 1
    assert L.dcp_rope_reindex(ctypes.byref(c), ctypes.byref(g), 20, 999, FAKE, n, None) == 1
    assert L.dcp_score_mask(None, FAKE, 64, 16, 0.1, 0, 0, None, None, None, None, FAKE, FAKE, 1 << 20, None) == 1
    assert L.dcp_score_mask(FAKE, FAKE, 0, 16, 0.1, 0, 0, None, None, None, None, FAKE, FAKE, 1 << 20, None) == 1
    assert L.dcp_score_mask(FAKE, FAKE, 64, 16, 0.1, 3, 0, None, None, None, None, FAKE, FAKE, 1 << 20, None) == 1
    assert L.dcp_score_mask(FAKE, FAKE, 64, 16, 0.1, 0, 0, None, None, None, None, None, FAKE, 1 << 20, None) == 1
    assert L.dcp_score_mask(FAKE, FAKE, 64, 16, 0.1, 0, 0, None, None, None, None, FAKE, FAKE, 8, None) == 1
    assert L.dcp_workspace_init(None, 1024, None) == 1
    assert L.dcp_get_status(None, None) == 1
    assert L.dcp_reset_status(None, None) == 1


def test_seeded_inputs_clear_of_tie_band():
    """Every seeded score input of the workloads keeps |l - gamma| >= 1e-6, so the kernel's fp32 sum and the
    oracle's double sum take the same keep decision and masks can be compared exactly."""
    import oracle
    from synth.workloads import ALL
    for w in ALL.values():
        for c, _, _ in w.evictions()[:8]:
            ell = oracle.score(*w.score_inputs(c))
            assert np.min(np.abs(ell.astype(np.float64) - np.float32(w.gamma))) >= 1e-6, (w.name, c)
