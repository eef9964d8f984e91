"""bench.py's native arm end to end on a small truncation of the Llama-3-8B
layout (the leading tensors, ~20M params; the other configurations are left
out at such sizes): one JSON line with the contract's keys, a positive
throughput, the roofline fraction of a kernel that does its work, the e2e
leg with its link rates and copies-only pipeline, clock samples taken within
the timed region (where nvidia-smi runs), and no device error."""
import json
import os
import subprocess
import sys

import pytest

from gpu_util import torch_cuda

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_native_arm_small():
    torch_cuda()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--params", "20000000", "--steps", "3",
                        "--warmup", "3"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["gpu_launches"] == 3
    assert d["gpu_launch_kinds"] == {"adamw_pipelined": 3}, d["gpu_launch_kinds"]
    assert 0 < d["config"]["params_per_gpu"] <= 20_000_000
    assert d["value"] > 0 and d["ms_per_step"] > 0
    roof = d["roofline"]
    assert roof["bound"] == "hbm" and 0.05 < roof["frac"] < 1.5, roof
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] == 2 * d["config"]["params_per_gpu"]
    assert e2e["copies_only_gparams_s"] > 0 and set(e2e["link_gbs"]) == {"h2d", "d2h", "both"}
    assert e2e["small_footprint_copies_gparams_s"] > 0
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["all_cores"]["cores"] >= 1
    clk = d["clocks"]
    assert clk is None or (clk["window"] == "timed region" and clk["samples"] >= 1 and clk["sm_mhz"] > 0), clk
