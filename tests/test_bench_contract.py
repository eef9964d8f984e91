"""The reference arm of bench.py runs on the CPU: its one JSON line carries
the keys the benchmark contract asks for, with the native arm's workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["params_per_gpu"] == 8_030_261_248 and d["config"]["tensors"] == 291
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


def test_a_device_error_stops_the_bench_without_a_line(capsys):
    """A kernel that reports a wait that gave up (error word != 0) makes the
    bench exit non-zero and print no JSON line; a clean word lets it go on."""
    import pytest
    import bench
    bench.require_no_device_error(lambda: 0, "timed device-resident steps")
    with pytest.raises(SystemExit) as e:
        bench.require_no_device_error(lambda: 1, "timed device-resident steps")
    assert e.value.code != 0
    out = capsys.readouterr()
    assert out.out == "" and "0x1" in out.err


def test_every_timed_region_is_checked_before_the_line_is_printed():
    """In the native arm, the error word is read after the warm-up, the timed
    device-resident steps and the timed end-to-end steps, and all of that
    before the result line is printed."""
    import ast
    import inspect
    import bench
    tree = ast.parse(inspect.getsource(bench.run_gpu))
    checks, prints = [], []
    for node in ast.walk(tree):
        if isinstance(node, ast.Call) and isinstance(node.func, ast.Name):
            if node.func.id == "require_no_device_error":
                checks.append((node.lineno, node.args[1].value))
            if node.func.id == "print":
                prints.append(node.lineno)
    regions = {r for _, r in checks}
    assert {"warm-up steps", "timed device-resident steps", "timed end-to-end steps"} <= regions
    assert prints and max(l for l, _ in checks) < min(prints)


def test_clock_summary_keeps_the_samples_of_the_timed_region():
    """The clock record covers the timed region only: samples outside the
    host-clock window are dropped (an idle clock before the region must not
    set the median), reasons are those seen inside it, and a region shorter
    than the sampling period gets the sample nearest its middle."""
    import datetime

    import bench
    base = datetime.datetime(2026, 1, 5, 10, 0, 0)

    def line(ms, sm, reason="Not Active", pcap="Not Active"):
        ts = (base + datetime.timedelta(milliseconds=ms)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, 0, {sm}, 2070, 300.5, 0x0, {reason}, Not Active, Not Active, {pcap}"

    lines = [line(0, 990), line(50, 990, reason="Active"), line(100, 2070), line(150, 2055, pcap="Active"),
             line(200, 2070), line(250, 1200), "garbage", ""]
    rows = bench.ClockSampler.parse(lines)
    assert len(rows) == 6
    t = lambda ms: (base + datetime.timedelta(milliseconds=ms)).timestamp()
    s = bench.ClockSampler.summarize(rows, t(90), t(210))
    assert s["samples"] == 3 and s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    one = bench.ClockSampler.summarize(rows, t(40), t(45))
    assert one["samples"] == 1 and one["reasons"] == ["hw_slowdown"] and one["sm_mhz"] == 990
    assert s["window"] == "timed region"
    assert bench.ClockSampler.summarize(rows)["samples"] == 6
    odd = bench.ClockSampler.parse(["12:00:01 PM, 0, 1980, 2070, 300.5, 0x0, Not Active, Not Active, "
                                    "Not Active, Not Active"])
    s = bench.ClockSampler.summarize(rows + odd, t(90), t(210))
    assert s["samples"] == 7 and s["window"] == "all samples"
    assert bench.ClockSampler.summarize([], t(0), t(1)) is None


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """Launched the way multi-GPU runs are (torchrun, two ranks, loopback
    rendezvous), the reference arm prints exactly one JSON line -- rank 0's,
    with n_gpus = 2 -- and every rank exits 0."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["config"]["params_per_gpu"] == 8_030_261_248
