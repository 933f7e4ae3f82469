"""The library's host PR bookkeeping (dcp_pr_add_chunk / dcp_pr_value) against the oracle's per-plane count and
a direct sum.  Page "DeCoPrune이 디노이징 불일치로 비디오 KV 캐시를 85% 줄인다" (onedev.kr/papers/726), section
'how to use': PR is the cumulative reduction of visible history KV positions, per chunk, layer and head, against
FullKV."""
import numpy as np

import autoregressive_video_diffusion_gb300 as dcp
import oracle
import synth


def test_pr_counter_matches_oracle():
    n_planes, C = 320, 6240
    acc = dcp.DcpPrCounter(0, 0)
    ref = [0, 0]
    u = synth.uniform_f64(60 * n_planes, 21, 1)
    hist = np.zeros(n_planes, np.int64)
    for i in range(1, 60):
        window = min(3, i - 1) * C
        dcp.dcp_pr_add_chunk(acc, n_planes, int(hist.sum()), C, window, i * C)
        oracle.pr_chunk(hist.astype(np.int32), C, window, i * C, ref)
        hist += (u[i * n_planes:(i + 1) * n_planes] * 0.4 * C).astype(np.int64) * (i > 4)
    assert (acc.visible, acc.full) == tuple(ref)
    assert dcp.dcp_pr_value(acc) == 1 - ref[0] / ref[1]


def test_pr_value_empty():
    assert dcp.dcp_pr_value(dcp.DcpPrCounter(0, 0)) == 0.0
