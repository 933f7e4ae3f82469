"""GPU parity: the CUDA prune step (through the C ABI) against the CPU oracle on the same seeded inputs.

Bars: masks, index lists, kept counts, hist_len, hist_t, every value row and every non-temporal key dim are bit-exact;
l is within 1e-5 relative; re-phased keys are within 1 bf16 ulp (fp32 keys: 2 ulp plus 2^-38 of the pair's |a| + |b|)
of the oracle's fp64 rotation rounded once.  The masks are compared exactly because every seeded input keeps
|l - gamma| >= 1e-6 (checked on the CPU in test_abi.py).
"""
import numpy as np
import pytest
import torch

import autoregressive_video_diffusion_gb300 as dcp
import oracle
import synth
from oracle import replay
from synth import workloads as W
from synth.workloads import FULL, FULL_ROTATED, HS_PREFIX, MID, ROLLOUT, TINY, scaled
from tests import devcache

pytestmark = pytest.mark.gpu

TINY_ROT = scaled(TINY, R=2, S=4)                       # the oldest history offsets are compressed: keys turn
TINY_MODE1 = scaled(TINY, R=2, S=3, g_mode=1)


def _cuda(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_score_parity(g_ell, ell, g_mask, mask, g_idx, idx, kept):
    g_ell = g_ell.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(g_ell, ell.astype(np.float64), rtol=1e-5, atol=0)
    assert np.array_equal(g_mask.cpu().numpy(), mask)
    assert kept == len(idx)
    assert np.array_equal(g_idx[:kept].cpu().numpy(), idx)


FP32_TURN_ABS = 2.0 ** -38  # absolute error of the fp32 turn, in units of the pair's |a| + |b|


def assert_key_parity(g: np.ndarray, o: np.ndarray, n_t: int) -> int:
    """Temporal dims within 1 bf16 ulp of the oracle (bf16 keys), or within 2 fp32 ulp plus 2^-38 of the pair's
    |a| + |b| (fp32 keys); the rest bitwise.  Returns the count of entries that are not bit-exact.

    The fp32 bound is the turn's own error: the cos/sin table carries ~40 significant bits, so an output that nearly
    cancels (a cos - b sin far below the pair's length) keeps an absolute error of ~2^-40 of the pair, which is many
    of its own ulps; elsewhere the relative error of the few rounded operations stays within 2 ulp."""
    nt2 = 2 * n_t
    assert np.array_equal(g[..., nt2:], o[..., nt2:]), "non-temporal key dims must be copied bitwise"
    d = replay.ulp_distance(g[..., :nt2], o[..., :nt2])
    if g.dtype == np.uint16:
        assert int(d.max(initial=0)) <= 1, f"re-phased key off by {int(d.max())} ulp"
    else:
        gv = g[..., :nt2].view(np.float32).astype(np.float64)
        ov = o[..., :nt2].view(np.float32)
        pair = np.abs(ov.astype(np.float64)).reshape(ov.shape[:-1] + (n_t, 2)).sum(-1).repeat(2, axis=-1)
        bound = 2 * np.spacing(np.abs(ov)).astype(np.float64) + FP32_TURN_ABS * pair
        err = np.abs(gv - ov.astype(np.float64))
        bad = err > bound
        assert not bad.any(), (f"re-phased fp32 key off by {int(d[bad].max())} ulp, "
                               f"{(err[bad] / pair[bad]).max():.3g} of the pair's |a| + |b|")
    return int(np.count_nonzero(d))


def assert_cache_parity(g: oracle.HostCache, o: oracle.HostCache, w) -> int:
    assert np.array_equal(g.hist_len, o.hist_len)
    assert np.array_equal(g.hist_t, o.hist_t)
    assert np.array_equal(g.v, o.v), "values must match bitwise everywhere"
    return assert_key_parity(g.k, o.k, w.n_temporal_pairs)


def gpu_vs_oracle_step(w, hc, ev, head_is_static=None, **cfg_over):
    """Run one prune step on the GPU and in the oracle from the same host state; compare everything."""
    c, q0_prev, q0 = ev
    x0, xr = w.score_inputs(c)
    ocfg = replay.cfg_of(w)
    for key, val in cfg_over.items():
        setattr(ocfg, key, val)
    dev = devcache.to_device(hc, w)
    gcfg = devcache.dcp_config(w, **cfg_over)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
    kept = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    hs = None if head_is_static is None else _cuda(head_is_static)
    dcp.dcp_prune_step(dev, gcfg, _cuda(x0), _cuda(xr), w.slot_of(c), w.first_frame(c), q0_prev, q0, hs, kept, None,
                       ws)
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    o = hc.copy()
    rc, ell, mask, idx = oracle.prune_step(o, ocfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0,
                                           head_is_static)
    assert rc == oracle.OK
    g_ell, g_mask, g_idx = dcp.dcp_workspace_outputs(dev, gcfg, ws)
    assert_score_parity(g_ell, ell, g_mask, mask, g_idx, idx, int(kept.item()))
    g = devcache.from_device(dev, w)
    inexact = assert_cache_parity(g, o, w)
    return o, g, idx, inexact


# ------------------------------------------------------------------------------------------ small full compares
@pytest.mark.parametrize("w", [TINY, TINY_ROT, TINY_MODE1], ids=["tiny", "tiny_rotating", "tiny_mode1"])
def test_tiny_prune_step(gpu, w):
    hc, ev = replay.state_before_last(w)
    o, g, idx, _ = gpu_vs_oracle_step(w, hc, ev)
    assert 0 < len(idx) < w.C


def test_mid_prune_step(gpu):
    """Mid bf16 eviction (4 x 8 x 128, 6240 tokens, history of 5 compacted chunks re-indexed from q0 36 to 40)."""
    hc, ev = replay.state_before_last(MID)
    assert ev[1] != ev[2]
    o, g, idx, inexact = gpu_vs_oracle_step(MID, hc, ev)
    print(f"mid: kept {len(idx)}, re-phased key entries not bit-exact: {inexact}")


@pytest.mark.parametrize("gamma,expect", [(-1.0, "all"), (1e9, "none")])
def test_all_or_nothing_kept(gpu, gamma, expect):
    w = scaled(TINY_ROT, gamma=gamma, hist_cap=6 * 64)
    hc, ev = replay.state_before_last(w)
    _, _, idx, _ = gpu_vs_oracle_step(w, hc, ev)
    assert len(idx) == (w.C if expect == "all" else 0)


def test_reverse_criterion(gpu):
    hc, ev = replay.state_before_last(TINY_ROT)
    gpu_vs_oracle_step(TINY_ROT, hc, ev, keep_rule=1)


@pytest.mark.parametrize("seed", [0, 0x5EED1234])
def test_random_ablation_step(gpu, seed):
    """Random at the discrepancy rule's kept count (section 'premises and limits'): the same rows move, bit-exact, as
    in the oracle drawing from the same SplitMix64 stream."""
    hc, ev = replay.state_before_last(TINY_ROT)
    o, g, idx, _ = gpu_vs_oracle_step(TINY_ROT, hc, ev, keep_rule=2, random_seed=seed)
    assert 0 < len(idx) < TINY_ROT.C


def test_random_ablation_mid(gpu):
    """Random ablation on the mid bf16 eviction (6240 tokens: the radix select runs several passes)."""
    hc, ev = replay.state_before_last(MID)
    gpu_vs_oracle_step(MID, hc, ev, keep_rule=2, random_seed=77)


@pytest.mark.parametrize("w", [TINY_ROT, MID], ids=["tiny_rotating", "mid"])
def test_host_resident_score_inputs(gpu, w):
    """Score rows in page-locked host memory are read by the scan kernel over the host link: the step equals the one
    on device rows, bit for bit; the kept count lands in page-locked host memory; pageable host memory is refused."""
    hc, (c, q0_prev, q0) = replay.state_before_last(w)
    x0, xr = w.score_inputs(c)
    cfg = devcache.dcp_config(w)
    a, b = devcache.to_device(hc, w), devcache.to_device(hc, w)
    ws_a = dcp.new_workspace(dcp.dcp_workspace_size(a, cfg))
    ws_b = dcp.new_workspace(dcp.dcp_workspace_size(b, cfg))
    kept_host = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    args = (w.slot_of(c), w.first_frame(c), q0_prev, q0, None)
    dcp.dcp_prune_step(a, cfg, _cuda(x0), _cuda(xr), *args, None, None, ws_a)
    dcp.dcp_prune_step(b, cfg, torch.from_numpy(x0).pin_memory(), torch.from_numpy(xr).pin_memory(), *args, None,
                       kept_host, ws_b)
    torch.cuda.synchronize()
    assert dcp.dcp_get_status(b.status) == dcp.DCP_OK
    ga, gb = devcache.from_device(a, w), devcache.from_device(b, w)
    assert np.array_equal(ga.k, gb.k) and np.array_equal(ga.v, gb.v)
    assert np.array_equal(ga.hist_len, gb.hist_len) and np.array_equal(ga.hist_t, gb.hist_t)
    assert int(kept_host.item()) == int(gb.hist_len.max()) - int(hc.hist_len.max())
    with pytest.raises(dcp.DcpError):
        dcp.dcp_prune_step(b, cfg, torch.from_numpy(x0), _cuda(xr), *args, None, None, ws_b)
    with pytest.raises(dcp.DcpError):
        dcp.dcp_prune_step(b, cfg, _cuda(x0), _cuda(xr), *args, None, torch.zeros(1, dtype=torch.int32), ws_b)


@pytest.mark.parametrize("w", [TINY_ROT, MID], ids=["tiny_rotating", "mid"])
def test_prune_step_in_cuda_graph(gpu, w):
    """A prune step recorded by stream capture and replayed gives the same cache, bit for bit, as the direct call."""
    hc, (c, q0_prev, q0) = replay.state_before_last(w)
    x0, xr = (_cuda(a) for a in w.score_inputs(c))
    cfg = devcache.dcp_config(w)
    a, b = devcache.to_device(hc, w), devcache.to_device(hc, w)
    ws_a = dcp.new_workspace(dcp.dcp_workspace_size(a, cfg))
    ws_b = dcp.new_workspace(dcp.dcp_workspace_size(b, cfg))
    args = (w.slot_of(c), w.first_frame(c), q0_prev, q0, None, None, None)
    dcp.dcp_prune_step(a, cfg, x0, xr, *args, ws_a)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dcp.dcp_prune_step(b, cfg, x0, xr, *args, ws_b, stream=s)
    torch.cuda.synchronize()
    gb0 = devcache.from_device(b, w)
    assert np.array_equal(gb0.hist_len, hc.hist_len), "capture must not run the step"
    g.replay()
    torch.cuda.synchronize()
    assert dcp.dcp_get_status(b.status) == dcp.DCP_OK
    ga, gb = devcache.from_device(a, w), devcache.from_device(b, w)
    assert np.array_equal(ga.k, gb.k) and np.array_equal(ga.v, gb.v)
    assert np.array_equal(ga.hist_len, gb.hist_len) and np.array_equal(ga.hist_t, gb.hist_t)


def test_fp32_rows_not_power_of_two(gpu):
    """fp32 keys with D = 36 (144-byte rows, 9 vectors per row) take the general index path."""
    w = scaled(TINY_ROT, D=36, n_temporal_pairs=7, d=10)
    hc, ev = replay.state_before_last(w)
    gpu_vs_oracle_step(w, hc, ev)


def test_bf16_small_head_dim(gpu):
    w = scaled(TINY_ROT, D=64, dtype=0, n_temporal_pairs=3, d=128)
    hc, ev = replay.state_before_last(w)
    gpu_vs_oracle_step(w, hc, ev)


# ------------------------------------------------------------------------------------------ standalone entry points
@pytest.mark.parametrize("n_tok,d", [(1, 16), (64, 16), (6240, 64), (100003, 64), (777, 128), (500, 10), (300, 3)])
@pytest.mark.parametrize("keep_rule", [0, 1, 2])
def test_score_mask(gpu, n_tok, d, keep_rule):
    x = synth.normal_f32(n_tok * d, 31, 1).reshape(n_tok, d)
    z = synth.normal_f32(n_tok * d, 31, 2).reshape(n_tok, d)
    s = 0.05 * np.exp(synth.uniform_f64(n_tok, 31, 3) * np.log(20.0))
    x0 = (x.astype(np.float64) + s[:, None] * z).astype(np.float32)
    ell = oracle.score(x0, x)
    stream = (0xD1CE << 32) | n_tok
    mask = oracle.keep_random(ell, 0.10, stream) if keep_rule == 2 else oracle.keep(ell, 0.10, keep_rule)
    idx = oracle.indices(mask)
    band = np.abs(ell.astype(np.float64) - np.float32(0.10)) < 1e-6
    ws = dcp.new_workspace(dcp.dcp_score_workspace_size(n_tok))
    g_ell = torch.empty(n_tok, dtype=torch.float32, device="cuda")
    g_mask = torch.empty(n_tok, dtype=torch.uint8, device="cuda")
    g_idx = torch.empty(n_tok, dtype=torch.int32, device="cuda")
    kept = torch.empty(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # the workspace must come back ready for the next call
        dcp.dcp_score_mask(_cuda(x0), _cuda(x), 0.10, keep_rule, g_ell, g_mask, g_idx, kept, status, ws,
                           random_stream=stream)
        assert dcp.dcp_get_status(status) == dcp.DCP_OK
        if band.any():
            pytest.skip("seeded input lands in the tie band")
        assert_score_parity(g_ell, ell, g_mask, mask, g_idx, idx, int(kept.item()))


def test_compact_layers_and_rope_reindex(gpu):
    """The two halves of the step on their own, each against the oracle's same half."""
    w = TINY_ROT
    hc, (c, q0_prev, q0) = replay.state_before_last(w)
    ocfg = replay.cfg_of(w)
    gcfg = devcache.dcp_config(w)
    # re-index first
    dev = devcache.to_device(hc, w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
    dcp.dcp_rope_reindex(dev, gcfg, q0_prev, q0, ws)
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    o = hc.copy()
    assert oracle.rope_reindex(o, ocfg, q0_prev, q0) == oracle.OK
    g = devcache.from_device(dev, w)
    assert not np.array_equal(o.k, hc.k)
    assert_cache_parity(g, o, w)
    # then compaction with the oracle's mask
    mask = oracle.keep(oracle.score(*w.score_inputs(c)))
    kept = torch.zeros(1, dtype=torch.int32, device="cuda")
    dcp.dcp_compact_layers(dev, gcfg, w.slot_of(c), w.first_frame(c), _cuda(mask), None, q0, kept, ws)
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    rc, idx = oracle.compact_layers(o, ocfg, w.slot_of(c), w.first_frame(c), mask, None, q0)
    assert rc == oracle.OK and int(kept.item()) == len(idx)
    assert_cache_parity(devcache.from_device(dev, w), o, w)
    # re-index with nothing to do leaves the cache bitwise alone
    before = devcache.from_device(dev, w)
    dcp.dcp_rope_reindex(dev, gcfg, q0, q0, ws)
    after = devcache.from_device(dev, w)
    assert np.array_equal(before.k, after.k)


def test_head_specialised_small(gpu):
    w = TINY_ROT
    static = np.zeros(w.n_planes, np.uint8)
    static[[0, 3]] = 1
    hc, ev = replay.state_before_last(w, head_is_static=static)
    assert np.all(hc.hist_len[static == 1] == 0)
    o, g, idx, _ = gpu_vs_oracle_step(w, hc, ev, head_is_static=static)
    assert np.all(g.hist_len[static == 1] == 0)


# ------------------------------------------------------------------------------------------ device-side errors
def test_capacity_error_leaves_cache(gpu):
    w = scaled(TINY_ROT, gamma=-1.0)                   # keep all 64 tokens
    hc, (c, q0_prev, q0) = replay.state_before_last(scaled(TINY_ROT, gamma=-1.0, hist_cap=5 * 64))
    x0, xr = w.score_inputs(c)
    dev = devcache.to_device(hc, w)
    tight = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, int(hc.hist_len[0]) + w.C - 1)
    tight.k, tight.v, tight.hist_len, tight.hist_t = dev.k, dev.v, dev.hist_len, dev.hist_t
    gcfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(tight, gcfg))
    before = devcache.from_device(dev, w)
    dcp.dcp_prune_step(tight, gcfg, _cuda(x0), _cuda(xr), w.slot_of(c), w.first_frame(c), q0_prev, q0, None, None,
                       None, ws)
    assert dcp.dcp_get_status(tight.status) == dcp.DCP_ECAPACITY
    after = devcache.from_device(dev, w)
    assert np.array_equal(before.k, after.k) and np.array_equal(before.hist_len, after.hist_len)


def test_history_filled_exactly(gpu):
    """Every token kept at every eviction with a history region of exactly the rows they need: the last step fills it
    to hist_cap and is accepted (the capacity bound is inclusive)."""
    w = scaled(TINY_ROT, gamma=-1.0, hist_cap=5 * 64)
    hc, ev = replay.state_before_last(w)
    assert int(hc.hist_len[0]) + w.C == w.hist_cap
    o, g, idx, _ = gpu_vs_oracle_step(w, hc, ev)
    assert len(idx) == w.C and int(g.hist_len[0]) == w.hist_cap


def test_inconsistent_lengths_detected(gpu):
    w = TINY_ROT
    hc, (c, q0_prev, q0) = replay.state_before_last(w)
    hc.hist_len[2] -= 1
    dev = devcache.to_device(hc, w)
    gcfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
    x0, xr = w.score_inputs(c)
    before = devcache.from_device(dev, w)
    dcp.dcp_prune_step(dev, gcfg, _cuda(x0), _cuda(xr), w.slot_of(c), w.first_frame(c), q0_prev, q0, None, None, None,
                       ws)
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_EDEVICE
    after = devcache.from_device(dev, w)
    assert np.array_equal(before.k, after.k) and np.array_equal(before.hist_len, after.hist_len)


def test_corrupt_history_detected(gpu):
    """A history length outside [0, hist_cap] or a history frame outside the phase table is reported as
    DCP_EDEVICE and nothing moves (no trap)."""
    w = TINY_ROT
    hc, (c, q0_prev, q0) = replay.state_before_last(w)
    x0, xr = w.score_inputs(c)
    for corrupt in ("len", "frame"):
        bad = hc.copy()
        if corrupt == "len":
            bad.hist_len[:] = w.hist_cap + 1
        else:
            bad.hist_t[0] = q0 + 5   # a frame that is not even in the past
        dev = devcache.to_device(bad, w)
        gcfg = devcache.dcp_config(w)
        ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
        before = devcache.from_device(dev, w)
        dcp.dcp_prune_step(dev, gcfg, _cuda(x0), _cuda(xr), w.slot_of(c), w.first_frame(c), q0_prev, q0, None, None,
                           None, ws)
        assert dcp.dcp_get_status(dev.status) == dcp.DCP_EDEVICE, corrupt
        after = devcache.from_device(dev, w)
        if corrupt == "len":
            assert np.array_equal(before.k, after.k) and np.array_equal(before.hist_len, after.hist_len)
        else:
            # only the row whose frame is outside the table is left alone by the re-index; the rest proceeds
            assert np.array_equal(before.k[:, :, w.sink_rows], after.k[:, :, w.sink_rows])


def test_one_workspace_serves_every_entry_point(gpu):
    """The workspace comes back ready after every call: score-only, re-index, compaction and full steps interleaved
    on one workspace give the oracle's results."""
    w = TINY_ROT
    hc, (c, q0_prev, q0) = replay.state_before_last(w)
    dev = devcache.to_device(hc, w)
    gcfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
    x0, xr = w.score_inputs(c)
    n = w.C
    kept = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.zeros(n, dtype=torch.int32, device="cuda")
    ref_idx = oracle.indices(oracle.keep(oracle.score(x0, xr)))
    for _ in range(3):
        dcp.dcp_score_mask(_cuda(x0), _cuda(xr), w.gamma, 0, None, None, idx, kept, dev.status, ws)
        assert int(kept.item()) == len(ref_idx) and np.array_equal(idx[: len(ref_idx)].cpu().numpy(), ref_idx)
    o = hc.copy()
    dcp.dcp_rope_reindex(dev, gcfg, q0_prev, q0, ws)
    assert oracle.rope_reindex(o, replay.cfg_of(w), q0_prev, q0) == oracle.OK
    dcp.dcp_score_mask(_cuda(x0), _cuda(xr), w.gamma, 0, None, None, idx, kept, dev.status, ws)
    mask = oracle.keep(oracle.score(x0, xr))
    dcp.dcp_compact_layers(dev, gcfg, w.slot_of(c), w.first_frame(c), _cuda(mask), None, q0, kept, ws)
    rc, _ = oracle.compact_layers(o, replay.cfg_of(w), w.slot_of(c), w.first_frame(c), mask, None, q0)
    assert rc == oracle.OK and dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    assert_cache_parity(devcache.from_device(dev, w), o, w)


# ------------------------------------------------------------------------------------------ full-size single eviction
def _full_size_eviction(w, sample_planes, paged=None):
    """Full-size eviction on the GPU; paged = (block_size, layout) runs it on a paged copy of the cache (read back
    into the contiguous cache for the checks)."""
    c, q0_prev, q0 = w.evictions()[-1]
    stream = torch.cuda.current_stream().cuda_stream
    dev = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, w.hist_cap)
    W.fill_device_chunks(dev.k.data_ptr(), dev.v.data_ptr(), w, list(range(w.sink_chunks)) + w.resident_window(c),
                         stream)
    W.fill_device_history_canary(dev.k.data_ptr(), dev.v.data_ptr(), w, stream)
    k0, v0 = dev.k.clone(), dev.v.clone()
    gcfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
    x0, xr = w.score_inputs(c)
    kept = torch.zeros(1, dtype=torch.int32, device="cuda")
    if paged:
        from tests.paged import PagedCopy
        pc = PagedCopy(dev, gcfg, paged[0], paged[1], seed=7)
        pws = dcp.new_workspace(dcp.dcp_paged_workspace_size(pc.cache, gcfg))
        dcp.dcp_paged_prune_step(pc.cache, gcfg, _cuda(x0), _cuda(xr), w.slot_of(c), w.first_frame(c), q0_prev, q0,
                                 None, kept, None, pws)
        assert dcp.dcp_get_status(pc.cache.status) == dcp.DCP_OK
        assert pc.free_blocks_untouched()
        pc.unpack_into(dev)
        ws = pws
        del pc
        torch.cuda.empty_cache()
    else:
        dcp.dcp_prune_step(dev, gcfg, _cuda(x0), _cuda(xr), w.slot_of(c), w.first_frame(c), q0_prev, q0, None, kept,
                           None, ws)
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    ell = oracle.score(x0, xr)
    mask = oracle.keep(ell, w.gamma)
    idx = oracle.indices(mask)
    k = len(idx)
    g_ell, g_mask, g_idx = dcp.dcp_workspace_outputs(dev, gcfg, ws)
    assert_score_parity(g_ell, ell, g_mask, mask, g_idx, idx, int(kept.item()))
    assert torch.all(dev.hist_len == k)
    assert np.array_equal(dev.hist_t[:k].cpu().numpy(), w.first_frame(c) + idx // w.tokens_per_frame)
    # copy properties over every plane
    H0, src0 = w.sink_rows, w.win_row0 + w.slot_of(c) * w.C
    it = torch.from_numpy(idx.astype(np.int64)).cuda() + src0
    nt2 = 2 * w.n_temporal_pairs
    for l in range(w.L):
        assert torch.equal(dev.v[l, :, H0:H0 + k], v0[l][:, it]), "V rows must be moved bitwise"
        assert torch.equal(dev.k[l, :, H0:H0 + k, nt2:], k0[l][:, it][..., nt2:]), "non-temporal K dims bitwise"
        for t_new, t_old in ((dev.k, k0), (dev.v, v0)):
            assert torch.equal(t_new[l, :, :H0], t_old[l, :, :H0]), "sink must stay untouched"
            assert torch.equal(t_new[l, :, H0 + k:], t_old[l, :, H0 + k:]), "window and free history untouched"
    # re-phased temporal dims on sampled planes against the oracle, one row at a time
    probe = oracle.HostCache(np.zeros((1, 1, 1, w.D), np.uint16), np.zeros((1, 1, 1, w.D), np.uint16),
                             np.zeros(1, np.int32), np.zeros(1, np.int32), 0)
    ocfg = replay.cfg_of(w)
    inexact = 0
    kh = dev.k.view(torch.int16)
    for p in sample_planes:
        l, h = divmod(p, w.H)
        src = W.host_chunk_rows(w, c, p, W.S_K, idx)
        got = kh[l, h, H0:H0 + k].cpu().numpy().view(np.uint16)
        want = np.stack([oracle.gather_key_row(src[j], probe, ocfg, w.first_frame(c) + int(idx[j]) //
                                               w.tokens_per_frame, q0) for j in range(k)])
        inexact += assert_key_parity(got, want, w.n_temporal_pairs)
    return k, inexact


@pytest.mark.parametrize("w", [FULL, FULL_ROTATED], ids=["full_depth", "full_depth_rotated"])
def test_full_depth_eviction(gpu, w):
    planes = [0, 1, 39, 40, 777, 800, 1201, 1599]
    k, inexact = _full_size_eviction(w, planes)
    assert 0.13 * w.C < k < 0.17 * w.C
    print(f"{w.name}: kept {k}; sampled re-phased entries not bit-exact: {inexact}")


# ------------------------------------------------------------------------------------------ head-specialised + prefix
def _subset_host_cache(w, planes, chunks):
    """Host cache holding only `planes` (as a [1][len(planes)] cache) with their full-workload contents."""
    dt = np.uint16 if w.dtype == 0 else np.float32
    n = len(planes)
    k = np.zeros((1, n, w.cap, w.D), dt)
    v = np.zeros((1, n, w.cap, w.D), dt)
    hc = oracle.HostCache(k, v, np.zeros(n, np.int32), np.zeros(max(w.hist_cap, 1), np.int32), w.hist_cap)
    _subset_place(hc, w, planes, chunks)
    for i, p in enumerate(planes):
        for arr, s in ((k, 2 * W.STREAM_HIST_INIT), (v, 2 * W.STREAM_HIST_INIT + 1)):
            synth.fill_rows_host(arr[0, i:i + 1], w.dtype, 1, w.cap, w.sink_rows, w.hist_cap, w.D, w.seed, s,
                                 w.hist_cap, p * w.hist_cap)
    return hc


def _subset_place(hc, w, planes, chunks):
    for c in chunks:
        row0 = W.chunk_row0(w, c)
        for i, p in enumerate(planes):
            for arr, what in ((hc.k, W.S_K), (hc.v, W.S_V)):
                synth.fill_rows_host(arr[0, i:i + 1], w.dtype, 1, w.cap, row0, w.C, w.D, w.seed,
                                     W.chunk_stream(c, what), w.C, p * w.C)


# the same prefix pass with a span that compresses (S = 14 < q0 - T_s): both evictions turn their kept keys, and the
# second re-indexes the first one's history, on the staged gather's turning form over the receiving-plane list
HS_PREFIX_TURNING = scaled(HS_PREFIX, name="head_specialised_prefix_turning", S=14)


@pytest.mark.parametrize("w", [HS_PREFIX, HS_PREFIX_TURNING], ids=["identity", "turning"])
def test_head_specialised_prefix_pass(gpu, w):
    """Config of 40 x 40 heads, 20 static per layer (Streaming), prefix pruning over 6 observed chunks (x0hat = the
    clean chunk re-noised at tau*, scored against the clean chunk); chunks 1 and 2 leave the window.  Sampled planes
    are replayed by the oracle as a cache of their own (planes are independent once the mask is fixed)."""
    static = w.head_is_static()
    assert static.reshape(w.L, w.H).sum(axis=1).tolist() == [20] * w.L
    stream = torch.cuda.current_stream().cuda_stream
    dev = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, w.hist_cap)
    W.fill_device_history_canary(dev.k.data_ptr(), dev.v.data_ptr(), w, stream)
    gcfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
    hs = _cuda(static)
    planes = [int(p) for p in np.flatnonzero(static)[:4]] + [int(p) for p in np.flatnonzero(static == 0)[:4]] + [1599]
    sub = _subset_host_cache(w, planes, [0])
    placed = {0}
    W.fill_device_chunks(dev.k.data_ptr(), dev.v.data_ptr(), w, [0], stream)
    ocfg = replay.cfg_of(w)
    ks = []
    for c, q0_prev, q0 in w.evictions():
        new = [cc for cc in w.resident_window(c) if cc not in placed]
        W.fill_device_chunks(dev.k.data_ptr(), dev.v.data_ptr(), w, new, stream)
        _subset_place(sub, w, planes, new)
        placed |= set(new)
        x0, xr = w.score_inputs(c)
        kept = torch.zeros(1, dtype=torch.int32, device="cuda")
        dcp.dcp_prune_step(dev, gcfg, _cuda(x0), _cuda(xr), w.slot_of(c), w.first_frame(c), q0_prev, q0, hs, kept,
                           None, ws)
        assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
        rc, ell, mask, idx = oracle.prune_step(sub, ocfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0,
                                               static[planes])
        assert rc == oracle.OK and int(kept.item()) == len(idx)
        ks.append(len(idx))
    hl = dev.hist_len.cpu().numpy()
    assert np.all(hl[static == 1] == 0) and np.all(hl[static == 0] == sum(ks))
    kh, vh = dev.k.view(torch.int16), dev.v.view(torch.int16)
    for i, p in enumerate(planes):
        l, h = divmod(p, w.H)
        assert np.array_equal(vh[l, h].cpu().numpy().view(np.uint16), sub.v[0, i])
        assert_key_parity(kh[l, h].cpu().numpy().view(np.uint16), sub.k[0, i], w.n_temporal_pairs)
    assert 0.2 < ks[0] / w.C < 0.3
    # the turning variant really turns: a receiving plane's first history row differs from its source key row in the
    # temporal dims (and only there)
    i = 4                                   # the first receiving plane of the sample
    assert static[planes[i]] == 0
    c1 = w.evictions()[0][0]
    src = np.zeros((1, w.cap, w.D), np.uint16)
    synth.fill_rows_host(src, w.dtype, 1, w.cap, W.chunk_row0(w, c1), w.C, w.D, w.seed, W.chunk_stream(c1, W.S_K),
                         w.C, planes[i] * w.C)
    first = W.chunk_row0(w, c1) + int(oracle.indices(oracle.keep(oracle.score(*w.score_inputs(c1)), w.gamma))[0])
    row, raw = sub.k[0, i, w.sink_rows], src[0, first]
    nt2 = 2 * w.n_temporal_pairs
    assert np.array_equal(row[nt2:], raw[nt2:])
    assert np.array_equal(row[:nt2], raw[:nt2]) == (w is HS_PREFIX)


# ------------------------------------------------------------------------------------------ rollout
ROLL_SMALL = scaled(ROLLOUT, L=2, H=2, rollout_chunks=14, hist_cap=10 * 6240)


def test_rollout_per_step(gpu):
    """Every eviction of a 14-chunk rollout (GQA-sized cache cut to 4 planes): the GPU step, started from the
    oracle's own pre-step state, matches the oracle's post-step state."""
    w = ROLL_SMALL
    hc = replay.new_host_cache(w)
    placed = set(range(w.sink_chunks))
    worst = 0
    for ev in w.evictions():
        for cc in w.resident_window(ev[0]):
            if cc not in placed:
                replay.place_chunk(hc, w, cc)
                placed.add(cc)
        o, g, idx, inexact = gpu_vs_oracle_step(w, hc, ev)
        worst = max(worst, inexact)
        hc = o
    print(f"rollout: final hist_len {int(hc.hist_len[0])}, worst per-step inexact entries {worst}")


def test_rollout_gpu_trajectory(gpu):
    """The GPU runs the whole rollout on its own state (chunks written on the device); at the end it agrees with the
    oracle's trajectory: lengths, frames and values exactly, non-temporal key dims bitwise, temporal key dims within a
    drift that grows with the steps (each side rounds every turned key once per step): at most steps * 2^-8 of the
    pair's length, and on at most 1e-4 of the entries."""
    w = ROLL_SMALL
    stream = torch.cuda.current_stream().cuda_stream
    dev = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, w.hist_cap)
    W.fill_device_history_canary(dev.k.data_ptr(), dev.v.data_ptr(), w, stream)
    W.fill_device_chunks(dev.k.data_ptr(), dev.v.data_ptr(), w, list(range(w.sink_chunks)), stream)
    gcfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, gcfg))
    hc = replay.new_host_cache(w)
    placed = set(range(w.sink_chunks))
    for c, q0_prev, q0 in w.evictions():
        new = [cc for cc in w.resident_window(c) if cc not in placed]
        W.fill_device_chunks(dev.k.data_ptr(), dev.v.data_ptr(), w, new, stream)
        x0, xr = w.score_inputs(c)
        dcp.dcp_prune_step(dev, gcfg, _cuda(x0), _cuda(xr), w.slot_of(c), w.first_frame(c), q0_prev, q0, None, None,
                           None, ws)
        replay.replay(w, hc, [(c, q0_prev, q0)], placed=placed)
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    g = devcache.from_device(dev, w)
    assert np.array_equal(g.hist_len, hc.hist_len) and np.array_equal(g.hist_t, hc.hist_t)
    assert np.array_equal(g.v, hc.v)
    nt2 = 2 * w.n_temporal_pairs
    assert np.array_equal(g.k[..., nt2:], hc.k[..., nt2:])
    d = replay.ulp_distance(g.k[..., :nt2], hc.k[..., :nt2])
    # A one-ulp difference in the large component of a pair turns, at the next re-index, into an error of the same
    # absolute size in the other component, which can be many of its own ulps when that component is near zero.
    # So drift is bounded relative to the pair's length: at most one bf16 rounding (2^-8) per step.
    gf = synth.bf16_bits_to_f32(g.k[..., :nt2]).astype(np.float64).reshape(-1, w.n_temporal_pairs, 2)
    of = synth.bf16_bits_to_f32(hc.k[..., :nt2]).astype(np.float64).reshape(-1, w.n_temporal_pairs, 2)
    rel = np.abs(gf - of).max(axis=2) / np.maximum(np.hypot(of[..., 0], of[..., 1]), 1e-30)
    steps = len(w.evictions())
    print(f"rollout drift over {steps} steps: {int(np.count_nonzero(d))} of {d.size} entries differ, max "
          f"{int(d.max())} ulp of the entry, max {rel.max():.3g} of the pair length")
    assert rel.max() <= steps * 2.0 ** -8
    assert np.count_nonzero(d) <= 1e-4 * d.size
