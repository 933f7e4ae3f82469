"""Host threads calling the library at the same time, each on its own cache, workspace and stream, in a fresh process
(so the per-kernel launch set-up is first made while both threads launch): every result equals the oracle's."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent('''
    import threading
    import numpy as np
    import torch
    import autoregressive_video_diffusion_gb300 as dcp
    import oracle
    from oracle import replay
    from synth.workloads import MID, TINY, scaled
    from tests import devcache
    from tests.test_gpu_parity import assert_cache_parity

    torch.cuda.set_device(0)
    cases = [scaled(TINY, R=2, S=4), MID, scaled(TINY, R=2, S=3, g_mode=1), scaled(MID, n_static_per_layer=3)]
    jobs = []
    for w in cases:
        hsm = w.head_is_static()
        hc, (c, q0p, q0) = replay.state_before_last(w, head_is_static=hsm)
        x0, xr = w.score_inputs(c)
        o = hc.copy()
        rc, _, _, _ = oracle.prune_step(o, replay.cfg_of(w), x0, xr, w.slot_of(c), w.first_frame(c), q0p, q0, hsm)
        assert rc == oracle.OK
        dev = devcache.to_device(hc, w)
        cfg = devcache.dcp_config(w)
        ws = dcp.new_workspace(dcp.dcp_workspace_size(dev, cfg))
        jobs.append(dict(w=w, o=o, dev=dev, cfg=cfg, ws=ws, ev=(c, q0p, q0),
                         x0=torch.from_numpy(x0).cuda(), xr=torch.from_numpy(xr).cuda(),
                         hs=None if hsm is None else torch.from_numpy(hsm).cuda(),
                         kept=torch.zeros(1, dtype=torch.int32, device="cuda"), stream=torch.cuda.Stream()))
    torch.cuda.synchronize()
    start = threading.Barrier(len(jobs))
    errors = []

    def run(j):
        try:
            w, (c, q0p, q0) = j["w"], j["ev"]
            start.wait()
            dcp.dcp_prune_step(j["dev"], j["cfg"], j["x0"], j["xr"], w.slot_of(c), w.first_frame(c), q0p, q0,
                               j["hs"], j["kept"], None, j["ws"], stream=j["stream"])
            j["stream"].synchronize()
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for j in jobs:
        assert dcp.dcp_get_status(j["dev"].status) == dcp.DCP_OK
        assert_cache_parity(devcache.from_device(j["dev"], j["w"]), j["o"], j["w"])
    print("threads ok", len(jobs))
''')


def test_concurrent_host_threads(gpu):
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    assert "threads ok 4" in r.stdout
