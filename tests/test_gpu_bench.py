"""bench.py end to end on the tiny workload: one JSON line with the fields the
benchmark contract names, for the plain step and for the hybrid options (the
zero-copy commit and the gated delta rule)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--config", "tiny", "--steps", "3", "--warmup", "3",
           "--cpu-seconds", "2", *args]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("extra", [(), ("--commit", "select", "--gdn-verify")], ids=["plain", "select_gdn"])
def test_bench_line_fields(sv, extra):
    d = _bench(*extra)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks",
                "gpu_launches", "acceptance_rate", "mean_accept_len"):
        assert key in d, key
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["steps"] == 3 and d["warmup"] == 3
    assert d["config"]["workload"] == "tiny"
    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["peak"] > 0 and roof["achieved"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    kernels = d["kernels"]
    assert {"attention", "accept", "commit"} <= set(kernels)
    plan = kernels["attention"]["plan"]  # the kernel instance the attention call ran
    assert set(plan) == {"kernel", "m_tiles", "keys_per_tile", "stages", "p_buffers", "ctas_per_sm"}
    assert plan["kernel"] == "mma" and plan["m_tiles"] == 1  # tiny: head dim 64, 16 packed rows
    launches_per_step = 3
    if extra:
        assert kernels["commit"]["kind"] == "select" and "gdn_verify" in kernels
        assert d["config"]["commit"].startswith("select") and "gdn_verify" in d["config"]
        launches_per_step = 4
    assert d["gpu_launches"] == launches_per_step * d["steps"]
