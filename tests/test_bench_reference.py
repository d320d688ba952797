"""The reference arm of bench.py (the CPU oracle, timed): its one JSON line
carries the contract's keys, and under several ranks only rank 0 runs."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# the routing workload scaled to 32 experts (146 tokens): well under a second
CMD = [sys.executable, "bench.py", "--impl", "reference", "--workload", "route_qb", "--experts", "32",
       "--steps", "1", "--warmup", "3"]


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run(CMD, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    out = _run({})
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["unit"] == "routed tokens/s"
    # the same metric and config as the GPU arm's routing line
    assert d["metric"] == bench.ROUTE_METRIC and d["dtype"] == "f32"
    assert d["config"]["workload"] == "route_qb_T4096_scaled_n32_jacobi"
    assert d["config"]["n_experts"] == 32 and d["config"]["T"] == 146
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    out = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out.returncode == 0, out.stderr[-2000:]
    assert not [ln for ln in out.stdout.splitlines() if ln.startswith("{")]


def test_cpu_route_baseline_times_the_oracle_on_the_given_logits():
    import numpy as np
    logits = np.random.default_rng(0).standard_normal((64, 16)).astype(np.float32)
    for gs, runs_at_least in ((True, 1), (False, 2)):
        cb = bench.cpu_route_baseline(logits, 4, gs)
        assert cb["kind"] == "oracle" and cb["unit"] == "routed tokens/s" and cb["cores"] >= 1
        assert cb["value"] > 0
        assert ("gauss_seidel" if gs else "jacobi") in cb["sample"] and "64 x 16" in cb["sample"]
        runs = int(cb["sample"].split(" run(s)")[0].rsplit(" ", 1)[1])
        assert runs >= runs_at_least and (runs == 1 or not gs)
