"""The bench's reference arm (the CPU oracle on a bounded sample) prints the contract's JSON line; under a multi-rank
launch only rank 0 runs it.  No GPU needed."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_line():
    r = _run({"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["higher_is_better"] is True and line["steps"] == 1 and line["warmup"] == 3
    assert line["config"]["workload"] == "full_depth_bf16_single_eviction"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_loads_no_product_library():
    """The reference arm runs the oracle and the input generator only: the product package is never imported and
    its shared library never mapped into the process."""
    code = ("import runpy, sys; sys.argv = ['bench.py', '--impl', 'reference', '--steps', '1', '--warmup', '3']; "
            "runpy.run_path('bench.py', run_name='__main__'); "
            "assert 'autoregressive_video_diffusion_gb300' not in sys.modules; "
            "assert 'libdcp.so' not in open('/proc/self/maps').read(); print('clean')")
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().splitlines()[-1] == "clean"


def test_both_arms_share_the_config():
    """The GPU arm's config is line_config(workload, kept); the reference arm prints the same object."""
    import bench
    from synth.workloads import FULL
    r = _run({"RANK": "0", "WORLD_SIZE": "1"})
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["config"] == bench.line_config(FULL, line["config"]["kept"])
    assert line["config"]["kept"] == 947


def test_compact_extra_fits_the_kept_tail():
    """Every extra workload's summary is a short object; with the CPU baseline before it the end of the line holds
    all of them within 1500 characters."""
    import bench
    us = lambda x: {"us_per_step": x, "GB_per_s": 6000.0}  # noqa: E731
    roll = {"mean_us_per_step": 670.0, "last10_mean_us": 1100.0, "GB_per_s": 4600.0, "cumulative_PR": 0.638}
    detail = {
        "full_depth_rotated": dict(us(255.0), gather_us=240.0), "full_depth_random_ablation": us(252.0),
        "full_depth_paged_hnd": us(251.0), "full_depth_paged_nhd": us(255.0), "full_depth_rotated_paged_hnd": us(262.0),
        "tiny_fp32_single_prune": {"us_per_step": 22.0, "algorithmic_bytes": 52000},
        "mid_bf16_single_eviction": {"us_per_step": 40.0, "algorithmic_bytes": 146_000_000},
        "head_specialised_prefix": {"evictions": [us(205.0), us(203.0)]},
        "minute_rollout_gqa8": dict(roll),
        "minute_rollout_gqa8_read_time_reindex": dict(roll, read_history_keys={"us": 2450.0, "bytes": 15_033_958_400},
                                                      drift_eager_vs_read_time={"max_of_pair_length": 0.153}),
        "cuda_graph_replay": [{"workload": "tiny_fp32_single_prune", "direct_us": 36.0, "graph_replay_us": 21.7},
                              {"workload": "mid_bf16_single_eviction", "direct_us": 67.0, "graph_replay_us": 51.0}],
        "host_snapshot_restore": {"snapshot_GB_per_s": 192.3, "restore_GB_per_s": 210.5,
                                  "frac_of_plain_copy": {"snapshot": 0.994, "restore": 0.996}},
    }
    ex = bench.compact_extra(detail, 6774.9)
    for key in ("full_rotated_2r", "random_ablation", "paged_hnd", "paged_nhd", "paged_hnd_2r", "tiny_fp32",
                "mid_bf16", "hs_prefix_ev1", "hs_prefix_ev2", "rollout_eager", "rollout_read_time",
                "read_final_history", "graph_replay_us", "host_snapshot", "host_restore"):
        assert key in ex, key
    for key in ("full_rotated_2r", "mid_bf16", "rollout_eager"):
        assert set(ex[key]) >= {"us_per_step", "GB_per_s", "frac"}
    assert abs(ex["mid_bf16"]["GB_per_s"] - 146e6 / 40e-6 / 1e9) <= 1
    text = json.dumps({"cpu_baseline": {"value": 1.07, "unit": "GB/s", "cores": 1, "kind": "oracle"}, "extra": ex})
    assert len(text) < 1400, len(text)


def test_traffic_figure_keyed_to_code_not_comments():
    """The bench keeps its DRAM-traffic figure only while the gather's code is the one the counters were taken on; the
    key drops // comments and blank lines, which is sound only while the keyed sources hold no // inside a string
    literal and no block comment."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench._code_only("a = 1;  // x\n\n  // y\n  b(2);   \n") == "a = 1;\n  b(2);"
    for f in ("gather.cu", "dcp_internal.cuh"):
        with open(os.path.join(ROOT, "autoregressive_video_diffusion_gb300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        assert "/*" not in text, f
        for ln in text.splitlines():
            code = ln.split("//", 1)[0]
            assert code.count('"') % 2 == 0, (f, ln)  # every string literal closes before a // on its line
