"""bench.py's reference arm (the float64 oracle on host cores) keeps the
one-JSON-line contract, on a small workload so it runs in seconds; under
torchrun only rank 0 prints."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ, **(extra_env or {}))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32", "--steps", "2",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [l for l in r.stdout.splitlines() if l.strip()]


def test_reference_arm_line():
    lines = _run()
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_fp32"
    # the same config object as the GPU arm's line, so the two lines compare
    sys.path.insert(0, ROOT)
    import bench
    from tensor_transformer_layer_03_b300 import inputs as I
    assert d["config"] == bench.workload_config("tiny_fp32", I.WORKLOADS["tiny_fp32"], 1)
    assert d["cpu_baseline"]["sample"].startswith("the whole workload (1 x 64 tokens)")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_silent():
    assert _run({"RANK": "1"}) == []


def test_clock_sampler_window_and_reasons():
    """The clocks summary covers only samples inside [mark_start, mark_end]
    (median SM clock, max clock, union of throttle reasons, sample count),
    and marks can be set again for the next measured window."""
    sys.path.insert(0, ROOT)
    import bench
    cs = bench.ClockSampler(0)
    assert cs.summary()["samples"] == 0
    cs.samples = [(1.0, 1000, 2032, 500.0, []), (2.0, 1900, 2032, 900.0, ["sw_power_cap"]),
                  (3.0, 2000, 2032, 950.0, []), (4.0, 2032, 2032, 300.0, ["hw_slowdown"])]
    cs.t0, cs.t1 = (1.5, None), (3.5, None)
    s = cs.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 1950.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_median"] == 925.0
    cs.t0, cs.t1 = (3.5, None), (4.5, None)
    s = cs.summary()
    assert s["samples"] == 1 and s["reasons"] == ["hw_slowdown"]


def test_reference_sample_sizing():
    """The reference arm runs the whole sequence per step when warm-up plus
    steps fit its time budget, else the longest 64-token-multiple prefix that
    does (at least 64 tokens)."""
    sys.path.insert(0, ROOT)
    import bench
    from tensor_transformer_layer_03_b300 import inputs as I
    wl = I.WORKLOADS["llama7b_prefill"]
    per_token = 1.0 / 760.0  # the oracle's rate on a 16-core host
    assert bench.reference_sample(wl, 20, 5, per_token) == wl.seq            # 25 x 2.7 s < 150 s
    n = bench.reference_sample(wl, 1000, 5, per_token)                        # the default step count
    assert n == 64
    n = bench.reference_sample(wl, 80, 5, per_token)                          # 85 x 2.7 s > 150 s
    assert n % 64 == 0 and 64 <= n < wl.seq and 85 * n * per_token <= bench.REF_BUDGET_S
    assert 85 * (n + 64) * per_token > bench.REF_BUDGET_S
    c = bench.workload_config("llama7b_prefill", wl, 4)
    assert c["parallelism"] == "replicas4" and c["seq"] == 2048 and c["tp_degree"] == 4 and "l2" in c
