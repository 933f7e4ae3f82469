"""The minute-long rollout at its full size against the oracle: 40 layers x 8 KV heads x head_dim 128 bf16, 60 chunks
of 6240 tokens, a prune step after each chunk that leaves the window (56 steps), the history growing to about 92k rows
per plane.  This is the workload the bench times, so the re-index, gather and read kernels run the launch
configuration (their division of 320 planes x ~92k rows over the CTAs) the bench reports.

Planes are independent once the chunk's mask is fixed (the page's shared mask), so the oracle replays a sample of
eight planes, each as a one-plane cache of its own with the values that plane has in the full workload, stepped in
threads (the oracle's C calls release the interpreter lock).

* Read-time re-index (keys keep their own frame; nothing is re-indexed per step): the GPU runs the whole trajectory
  on its own state.  At the end the history lengths and frames of every plane, and every byte of each sampled plane
  (keys move bitwise in this mode), equal the oracle's; the read of all 320 planes' history at the final q0 is within
  1 bf16 ulp of the oracle's read on the sampled planes and writes nothing past a plane's history; and the library's
  cumulative PR counter, fed the GPU's history lengths, equals the oracle's count over the same rollout.
* Eager re-index (history keys turned at every step): at every step the GPU starts from the oracle's own pre-step
  state of the sampled planes, replicated over all 320 planes (plane (l, h) holds sampled plane h's state), runs the
  step, and every plane must match the oracle's post-step state of its sampled plane: values, non-temporal key dims
  and untouched rows bitwise, turned key dims within 1 bf16 ulp.  The PR counters agree here too.
"""
from concurrent.futures import ThreadPoolExecutor
from functools import lru_cache

import numpy as np
import pytest
import torch

import autoregressive_video_diffusion_gb300 as dcp
import oracle
from oracle import replay
from synth import workloads as W
from synth.workloads import ROLLOUT
from tests import devcache
from tests.test_gpu_parity import _subset_host_cache, _subset_place, assert_key_parity

pytestmark = pytest.mark.gpu

PLANES = (0, 1, 47, 77, 160, 203, 254, 319)   # sampled (layer, head) planes of the 320; eight of them, one per head


@lru_cache(maxsize=None)
def _inputs(c: int):
    return ROLLOUT.score_inputs(c)


def _cuda(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _i16(a: np.ndarray) -> torch.Tensor:
    """uint16 (bf16 bits) host array -> int16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


class _Oracle:
    """The oracle's rollout on the sampled planes: one single-plane host cache per plane, stepped in threads."""

    def __init__(self, w, reindex_mode: int):
        self.w = w
        self.cfg = replay.cfg_of(w)
        self.cfg.reindex_mode = reindex_mode
        self.caches = [_subset_host_cache(w, [p], list(range(w.sink_chunks))) for p in PLANES]
        self.placed = set(range(w.sink_chunks))
        self.pool = ThreadPoolExecutor(len(PLANES))
        self.pr = [0, 0]

    def place(self, chunks):
        new = [c for c in chunks if c not in self.placed]
        list(self.pool.map(lambda i: _subset_place(self.caches[i], self.w, [PLANES[i]], new), range(len(PLANES))))
        self.placed |= set(new)
        return new

    def step(self, c, q0_prev, q0):
        w = self.w
        x0, xr = _inputs(c)

        def one(hc):
            return oracle.prune_step(hc, self.cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0)
        out = list(self.pool.map(one, self.caches))
        for rc, _, _, idx in out:
            assert rc == oracle.OK
            assert np.array_equal(idx, out[0][3])
        return out[0][3]

    def hist_len(self) -> int:
        lens = {int(hc.hist_len[0]) for hc in self.caches}
        assert len(lens) == 1
        return lens.pop()

    def add_pr_chunk(self, sink_visible, window_visible, prior):
        oracle.pr_chunk(np.full(self.w.n_planes, self.hist_len(), np.int32), sink_visible, window_visible, prior,
                        self.pr)


def _schedule(w):
    """(generated chunk i, its PR terms, the chunk that leaves after it or None) over the whole rollout."""
    ev = {c: (q0p, q0) for c, q0p, q0 in w.evictions()}
    for i in range(1, w.rollout_chunks):
        window = min(w.window_chunks, max(0, i - w.sink_chunks)) * w.C
        c = i - w.window_chunks
        yield (min(w.sink_chunks, i) * w.C, window, i * w.C), ((c,) + ev[c] if c in ev else None)


def _ordered_i32(t: torch.Tensor) -> torch.Tensor:
    """bf16 bit patterns (int16 tensor) as integers whose differences count ulps."""
    b = t.to(torch.int32)
    return torch.where(b < 0, -(b & 0x7FFF), b)


def test_minute_rollout_read_time_full_size(gpu):
    w = ROLLOUT
    stream = torch.cuda.current_stream().cuda_stream
    dev = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, w.hist_cap)
    W.fill_device_history_canary(dev.k.data_ptr(), dev.v.data_ptr(), w, stream)
    W.fill_device_chunks(dev.k.data_ptr(), dev.v.data_ptr(), w, list(range(w.sink_chunks)), stream)
    cfg = devcache.dcp_config(w, reindex_mode=1)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, cfg))
    kept = torch.zeros(1, dtype=torch.int32, device="cuda")
    orc = _Oracle(w, reindex_mode=1)
    pr = dcp.DcpPrCounter(0, 0)
    steps = 0
    for (sink_vis, win_vis, prior), ev in _schedule(w):
        dcp.dcp_pr_add_chunk(pr, w.n_planes, int(dev.hist_len.sum().item()), sink_vis, win_vis, prior)
        orc.add_pr_chunk(sink_vis, win_vis, prior)
        if ev is None:
            continue
        c, q0_prev, q0 = ev
        new = orc.place(w.resident_window(c))
        W.fill_device_chunks(dev.k.data_ptr(), dev.v.data_ptr(), w, new, stream)
        x0, xr = (_cuda(a) for a in _inputs(c))
        dcp.dcp_prune_step(dev, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, None, kept, None, ws)
        idx = orc.step(c, q0_prev, q0)
        assert int(kept.item()) == len(idx), f"chunk {c}"
        steps += 1
    assert steps == len(w.evictions()) == 56
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    n = orc.hist_len()
    assert n > 80_000
    assert torch.all(dev.hist_len == n)
    assert np.array_equal(dev.hist_t[:n].cpu().numpy(), orc.caches[0].hist_t[:n])
    assert (pr.visible, pr.full) == tuple(orc.pr), "library PR counter vs the oracle's count"
    kh, vh = dev.k.view(w.n_planes, w.cap, w.D).view(torch.int16), dev.v.view(w.n_planes, w.cap, w.D).view(torch.int16)
    for i, p in enumerate(PLANES):  # every row of the plane: sink, history (moved bitwise), ring, free rows
        assert np.array_equal(kh[p].cpu().numpy().view(np.uint16), orc.caches[i].k[0, 0]), f"K of plane {p}"
        assert np.array_equal(vh[p].cpu().numpy().view(np.uint16), orc.caches[i].v[0, 0]), f"V of plane {p}"
    # the read of every plane's history at the final q0 (the launch the bench times), sampled planes checked
    q0 = w.evictions()[-1][2]
    out = torch.empty((w.n_planes, w.hist_cap, w.D), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    dcp.dcp_read_history_keys(dev, cfg, q0, 0, w.n_planes, out, ws)
    assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
    want = list(orc.pool.map(lambda hc: oracle.read_history_keys(hc, orc.cfg, q0), orc.caches))
    oh = out.view(torch.int16)
    inexact = 0
    for i, p in enumerate(PLANES):
        got = oh[p].cpu().numpy().view(np.uint16)
        inexact += assert_key_parity(got[:n], want[i][0, :n], w.n_temporal_pairs)
        assert np.all(got[n:] == 0xFFFF), "nothing written past the plane's history"
    print(f"read-time rollout: {steps} steps, history {n} rows, PR {dcp.dcp_pr_value(pr):.4f}, read entries not "
          f"bit-exact on {len(PLANES)} planes: {inexact}")


def test_minute_rollout_eager_per_step_full_size(gpu):
    w = ROLLOUT
    nt2 = 2 * w.n_temporal_pairs
    H0 = w.sink_rows
    orc = _Oracle(w, reindex_mode=0)
    dev = dcp.KVCache(w.L, w.H, w.D, w.dtype, w.cap, w.hist_cap)
    cfg = devcache.dcp_config(w)
    ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, cfg))
    kept = torch.zeros(1, dtype=torch.int32, device="cuda")
    pr = dcp.DcpPrCounter(0, 0)
    assert w.H == len(PLANES)
    # the oracle's state of the sampled planes on the device, [8][cap][D]; plane (l, h) of the GPU cache gets row h
    st_k = torch.stack([_i16(hc.k[0, 0]) for hc in orc.caches])
    st_v = torch.stack([_i16(hc.v[0, 0]) for hc in orc.caches])
    dk = dev.k.view(torch.int16)  # [L][H][cap][D]
    dv = dev.v.view(torch.int16)

    def upload_rows(r0, r1):
        """Rows [r0, r1) of every sampled plane, from the oracle's host caches into the device copy."""
        for h, hc in enumerate(orc.caches):
            st_k[h, r0:r1].copy_(_i16(hc.k[0, 0, r0:r1]))
            st_v[h, r0:r1].copy_(_i16(hc.v[0, 0, r0:r1]))

    steps = worst = 0
    for (sink_vis, win_vis, prior), ev in _schedule(w):
        orc.add_pr_chunk(sink_vis, win_vis, prior)
        if ev is None:
            dcp.dcp_pr_add_chunk(pr, w.n_planes, w.n_planes * orc.hist_len(), sink_vis, win_vis, prior)
            continue
        c, q0_prev, q0 = ev
        for cc in orc.place(w.resident_window(c)):      # the chunks generated since the last step, into their slots
            r0 = W.chunk_row0(w, cc)
            upload_rows(r0, r0 + w.C)
        # the oracle's pre-step state on every plane of the GPU cache
        n0 = orc.hist_len()
        dk.copy_(st_k.unsqueeze(0).expand_as(dk))
        dv.copy_(st_v.unsqueeze(0).expand_as(dv))
        dev.hist_len.fill_(n0)
        dev.hist_t.copy_(torch.from_numpy(orc.caches[0].hist_t))
        dcp.dcp_pr_add_chunk(pr, w.n_planes, int(dev.hist_len.sum().item()), sink_vis, win_vis, prior)
        x0, xr = (_cuda(a) for a in _inputs(c))
        dcp.dcp_prune_step(dev, cfg, x0, xr, w.slot_of(c), w.first_frame(c), q0_prev, q0, None, kept, None, ws)
        idx = orc.step(c, q0_prev, q0)
        assert dcp.dcp_get_status(dev.status) == dcp.DCP_OK
        assert int(kept.item()) == len(idx), f"chunk {c}"
        n1 = orc.hist_len()
        assert n1 == n0 + len(idx) and torch.all(dev.hist_len == n1)
        assert np.array_equal(dev.hist_t[:n1].cpu().numpy(), orc.caches[0].hist_t[:n1])
        upload_rows(H0, H0 + n1)                        # the oracle's post-step history rows
        for h in range(w.H):                            # the 40 planes holding sampled plane h
            want_k, want_v = st_k[h].expand(w.L, -1, -1), st_v[h].expand(w.L, -1, -1)
            assert torch.equal(dv[:, h], want_v), f"values, head {h}, chunk {c}"
            assert torch.equal(dk[:, h, :, nt2:], want_k[..., nt2:]), f"non-temporal key dims, head {h}, chunk {c}"
            assert torch.equal(dk[:, h, :H0, :nt2], want_k[:, :H0, :nt2]), "sink keys untouched"
            assert torch.equal(dk[:, h, H0 + n1:, :nt2], want_k[:, H0 + n1:, :nt2]), "ring and free rows untouched"
            d = (_ordered_i32(dk[:, h, H0:H0 + n1, :nt2]) - _ordered_i32(want_k[:, H0:H0 + n1, :nt2])).abs_()
            assert int(d.max().item()) <= 1, f"turned keys off by more than 1 ulp, head {h}, chunk {c}"
            worst = max(worst, int(torch.count_nonzero(d).item()))
        steps += 1
    assert steps == 56
    assert (pr.visible, pr.full) == tuple(orc.pr), "library PR counter vs the oracle's count"
    print(f"eager rollout per step: {steps} steps on 320 planes, final history {orc.hist_len()} rows, PR "
          f"{dcp.dcp_pr_value(pr):.4f}, worst per-step entries not bit-exact (40 planes): {worst}")
