"""Benchmark of the fused AdamW-SR step on the Llama-3-8B parameter set.

One step = one fused AdamW step with stochastic bf16 write-back over all 291
tensors (8,030,261,248 parameters; bf16 params and grads, f32 moments), i.e.
one multi-tensor C-ABI call.  The working set (176.7 GB of traffic per step)
is far larger than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  ``value`` is device-resident throughput (params/s over
the timed steps, CUDA events); ``e2e`` repeats the measurement with the
step's gradients copied from pinned host memory before, and the updated bf16
params copied back after, every step (chunks of consecutive tensors pipelined
over three streams so both copy directions overlap the compute).  ``--impl reference`` times the CPU
oracle (single core) on a bounded sample of the same workload instead.
Multi-GPU (torchrun): each rank updates its own full 8B-parameter shard of an
N x 8B flat parameter vector (its base_index offset by rank), no collective on
the data path: weak scaling.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "AdamW-SR step Gparams/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "Gparams/s"
BYTES_PER_PARAM = 22          # bf16 p r/w (2+2), bf16 g r (2), f32 m r/w (4+4), f32 v r/w (4+4)
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
NOMINAL_HBM_GBS = 8000.0
# the device code of the AdamW-SR kernel: traffic figures are valid while
# these files are unchanged
KERNEL_SRC = [os.path.join(ROOT, "stochastic_rounding_gb300", "csrc", f)
              for f in ("common.cuh", "pipeline.cuh", "adamw_kernels.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")

CPU_SAMPLE_ELEMS = 1 << 24     # oracle sample per step (one core)
E2E_CHUNK = 1 << 28            # params per chunk of the end-to-end pipeline


def require_no_device_error(take_error, region):
    """Read (and clear) the library's device error word after a timed region,
    outside it.  A set bit means a kernel's pipeline wait gave up and left
    work undone, which would make the step look faster than it is: the
    benchmark then stops with a non-zero exit and prints no result line."""
    bits = take_error()
    if bits:
        print(f"bench.py: device error bits {bits:#x} after the {region}: a kernel left work undone; "
              "no result is reported", file=sys.stderr, flush=True)
        raise SystemExit(3)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_sha():
    h = hashlib.sha256()
    for path in KERNEL_SRC:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_per_param():
    """DRAM bytes per parameter from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        if d.get("source_sha256") == source_sha():
            return float(d["dram_bytes_per_param"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples (every 50 ms, time-stamped) around the
    timed region; `mark_start`/`mark_end` bracket the region on the host clock,
    and `summary` keeps the samples taken inside it (the nearest one if the
    region is shorter than the sampling period)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    @staticmethod
    def parse(lines):
        """Rows of the CSV lines nvidia-smi wrote (malformed lines skipped)."""
        import datetime
        rows = []
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                row = dict(sm=float(parts[2]), smax=float(parts[3]), power=float(parts[4]),
                           hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9])
            except ValueError:
                continue
            row["t"] = None
            for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
                try:
                    row["t"] = datetime.datetime.strptime(parts[0], fmt).timestamp()
                    break
                except ValueError:
                    pass
            rows.append(row)
        return rows

    @staticmethod
    def summarize(rows, t0=None, t1=None):
        """Median SM clock, max clock, active slowdown reasons and peak power
        over the rows taken within [t0, t1] (all rows without a window or
        with an unreadable timestamp; the row nearest the window's middle if
        none falls inside it)."""
        if not rows:
            return None
        inside, window = rows, "all samples"
        if t0 is not None and t1 is not None and all(r["t"] is not None for r in rows):
            window = "timed region"
            inside = [r for r in rows if t0 <= r["t"] <= t1]
            if not inside:
                mid = 0.5 * (t0 + t1)
                inside = [min(rows, key=lambda r: abs(r["t"] - mid))]
        reasons = set()
        for r in inside:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["smax"] for r in inside), "reasons": sorted(reasons),
                "samples": len(inside), "period_ms": ClockSampler.PERIOD_MS, "window": window,
                "power_w_max": max(r["power"] for r in inside)}

    def summary(self):
        if self.proc is None or not self.path:
            return None
        with open(self.path) as f:
            rows = self.parse(f)
        os.remove(self.path)
        return self.summarize(rows, self.t0, self.t1)


def cpu_oracle_sample(steps, sample_elems=CPU_SAMPLE_ELEMS, seed=0):
    """Time the C oracle (one core) on a sample of the 8B workload: windows of
    the 8B layout at their true base indices, bf16 p/g, f32 m/v.  Returns
    (params/s per step list, description)."""
    import numpy as np

    import oracle
    from stochastic_rounding_gb300 import workloads as W
    o = oracle.get()
    table = W.param_table(W.LLAMA_8B)
    starts, _ = W.offsets(table)
    big = [i for i, (_, n, norm) in enumerate(table) if not norm]
    rng = np.random.default_rng(seed)
    pieces = 8
    per = sample_elems // pieces
    windows = []
    for t in rng.choice(big, pieces, replace=False):
        s = int(rng.integers(0, table[t][1] - per)) & ~7
        windows.append(int(starts[t]) + s)
    hr = W.host_rng(seed, 1)
    data = []
    for base in windows:
        data.append([W.to_bf16_bits(W.normal_f32(hr, per, 0.02)), W.to_bf16_bits(W.normal_f32(hr, per, 1e-3)),
                     np.zeros(per, np.float32), np.zeros(per, np.float32), base])
    rates = []
    for step in range(1, steps + 1):
        t0 = time.perf_counter()
        for p, g, m, v, base in data:
            o.adamw_step(p, g, m, v, step=step, seed=0, base_index=base, **HP)
        dt = time.perf_counter() - t0
        rates.append(pieces * per / dt)
    desc = (f"{pieces} windows x {per} params of the Llama-3-8B layout (bf16 p/g, f32 m/v, true base "
            f"indices), C oracle single thread, per step")
    return rates, desc


def host_link_rates(dev, nbytes=1 << 30, reps=3):
    """GB/s of this machine's host link with page-locked host memory, measured
    outside the timed steps: one nbytes host-to-device copy, one
    device-to-host copy, and one of each at once on two streams (aggregate
    bytes / time); best of ``reps`` each, CUDA events."""
    import torch
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed(fn):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s1)
            s2.wait_stream(s1)
            fn()
            s1.wait_stream(s2)
            e1.record(s1)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)

    def both():
        h2d()
        d2h()
    rates = {"h2d": nbytes / (timed(h2d) / 1e3) / 1e9, "d2h": nbytes / (timed(d2h) / 1e3) / 1e9,
             "both": 2 * nbytes / (timed(both) / 1e3) / 1e9}
    del h_in, h_out, d_in, d_out
    return rates


def ring_copies_seconds(g_dev, p_dev, n, dev, steps, chunk=1 << 26, slots=2):
    """Seconds per step of the end-to-end leg's transfers alone (2 B per param in,
    2 B out, contiguous chunk-element ranges, host-to-device on one stream and
    device-to-host of each range after its own host-to-device on another)
    through a small ring of page-locked staging buffers -- ``slots`` per
    direction, 512 MB in all by default -- instead of host buffers for the
    whole set.  Measured outside the timed steps, after one untimed pass: on
    hosts whose page-locked transfers stall in proportion to the page-locked
    footprint it shows what the link gives the same bytes without that."""
    import torch
    g_ring = [torch.empty(chunk, dtype=g_dev.dtype, pin_memory=True) for _ in range(slots)]
    p_ring = [torch.empty(chunk, dtype=p_dev.dtype, pin_memory=True) for _ in range(slots)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    main = torch.cuda.current_stream(dev)
    ranges = [(lo, min(n, lo + chunk)) for lo in range(0, n, chunk)]

    def one_pass():
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        for c, (lo, hi) in enumerate(ranges):
            with torch.cuda.stream(s_in):
                g_dev[lo:hi].copy_(g_ring[c % slots][:hi - lo], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev)
                p_ring[c % slots][:hi - lo].copy_(p_dev[lo:hi], non_blocking=True)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    one_pass()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for _ in range(steps):
        one_pass()
    e1.record(main)
    torch.cuda.synchronize(dev)
    seconds = e0.elapsed_time(e1) / 1e3 / steps
    del g_ring, p_ring
    return seconds


def e2e_chunks(tensors, max_params=E2E_CHUNK):
    """The chunks the end-to-end pipeline forms: consecutive tensors grouped
    while they hold at most max_params (a larger tensor is a chunk of its
    own), the rule asr_adamw_sr_multi_tensor_host applies.  Each chunk is the
    contiguous range [lo, hi) of the flat buffers its tensors span."""
    groups, group, count = [], [], 0
    for t in tensors:
        n_t = t[0].numel()
        if group and count + n_t > max_params:
            groups.append(group)
            group, count = [], 0
        group.append(t)
        count += n_t
    if group:
        groups.append(group)
    return [(grp[0][4], grp[-1][4] + grp[-1][0].numel()) for grp in groups]


def _oracle_shard_worker(args):
    """One process of the all-cores oracle run: its own window of the 8B
    layout, one step, timed inside the process."""
    shard, per, seed = args
    import numpy as np

    import oracle
    from stochastic_rounding_gb300 import workloads as W
    o = oracle.get()
    table = W.param_table(W.LLAMA_8B)
    starts, _ = W.offsets(table)
    big = [i for i, (_, n, norm) in enumerate(table) if not norm]
    t = big[shard % len(big)]
    base = int(starts[t]) + (shard // len(big)) * per
    hr = W.host_rng(seed, 100 + shard)
    p = W.to_bf16_bits(W.normal_f32(hr, per, 0.02))
    g = W.to_bf16_bits(W.normal_f32(hr, per, 1e-3))
    m = np.zeros(per, np.float32)
    v = np.zeros(per, np.float32)
    t0 = time.perf_counter()
    o.adamw_step(p, g, m, v, step=1, seed=0, base_index=base, **HP)
    return per, time.perf_counter() - t0


def start_oracle_pool():
    """A spawn-started pool over the process's CPU affinity set (started
    before the first GPU call, as forked children of a CUDA process hang)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    return mp.get_context("spawn").Pool(cores), cores


def cpu_oracle_all_cores(pool, cores, per=1 << 23):
    """The same oracle, unchanged, one shard (a window of the 8B layout at its
    true base index) per core, all cores at once: params/s over the wall time
    of the slowest shard."""
    results = pool.map(_oracle_shard_worker, [(i, per, 0) for i in range(cores)])
    wall = max(dt for _, dt in results)
    return {"value": sum(n for n, _ in results) / wall / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes x {per} params (one window of the 8B layout each), one step, "
                      f"the oracle unchanged, sharded by base index"}


def measure_configs(asr, W, dev, steps, warmup, peak):
    """The other synthetic configurations, each timed with CUDA events after
    warm-up: Gparams/s and algorithmic GB/s against the measured copy peak."""
    import torch
    out = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)

    def timed(fn, reps=steps):
        for t in range(1, warmup + 1):
            fn(t)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for t in range(warmup + 1, warmup + reps + 1):
            fn(t)
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    def single(name, n, pdt, gdt, bpp, note):
        p = W.device_normal_(torch.empty(n, dtype=pdt, device=dev), gen, 0.02)
        g = W.device_normal_(torch.empty(n, dtype=gdt, device=dev), gen, 1e-3)
        m = torch.zeros(n, device=dev)
        v = torch.zeros(n, device=dev)
        # steps of a millisecond or less: at least 50 timed launches, so the
        # host's gap before the first one (the GPU idles while the call is
        # prepared) is spread thin
        reps = max(steps, 50)
        ms = timed(lambda t: asr.asr_adamw_sr_step(p, g, m, v, step=t, seed=0, **HP), reps)
        gbs = bpp * n / ms / 1e6
        out[name] = {"params": n, "ms_per_step": ms, "gparams_per_s": n / ms / 1e6, "bytes_per_param": bpp,
                     "gbs": gbs, "frac_of_measured_copy": gbs / peak, "timed_steps": reps, "note": note}
        del p, g, m, v

    single("single_65536_bf16", 65536, torch.bfloat16, torch.bfloat16, BYTES_PER_PARAM,
           "1.4 MB: L2-resident and launch-bound")
    out["single_65536_bf16"]["host_us_per_call"] = binding_host_cost(asr, W, dev, gen)
    out["single_65536_bf16"]["graph_us_per_step"] = graph_step_cost(asr, W, dev, gen)
    single("fp32_16777216", 16777216, torch.float32, torch.float32, 28, "fp32 params and grads")
    single("bf16_268435456", 268435456, torch.bfloat16, torch.bfloat16, BYTES_PER_PARAM, "one tensor")
    ps = W.DeviceParamSet(W.LLAMA_1B, device=dev, seed=2)
    from stochastic_rounding_gb300 import _lib
    table = _lib.make_table(ps.tensors())
    ms = timed(lambda t: asr.asr_adamw_sr_multi_tensor(table, step=t, seed=0, device=dev, **HP))
    gbs = BYTES_PER_PARAM * ps.numel / ms / 1e6
    out["llama_16L_h2048_147t"] = {"params": ps.numel, "ms_per_step": ms, "gparams_per_s": ps.numel / ms / 1e6,
                                   "bytes_per_param": BYTES_PER_PARAM, "gbs": gbs,
                                   "frac_of_measured_copy": gbs / peak, "note": "147 tensors, one launch"}
    del ps
    torch.cuda.empty_cache()
    # the stand-alone kernels of the library, each a few seconds at most
    for m, n, k, budget in ((8192, 8192, 8192, 1e9), (8192, 8192, 1024, 2.5e8), (8192, 8192, 512, 2.5e8)):
        out[f"gemm_{m}x{n}x{k}"] = gemm_measure(asr, dev, m, n, k, steps, warmup, budget)
    out["sr_op_1073741824"] = elementwise_measure(asr, dev, "sr", 1 << 30, steps, warmup)
    out["philox_268435456"] = elementwise_measure(asr, dev, "philox", 1 << 28, steps, warmup)
    out["subulp_demo"] = subulp_demo(asr, dev)
    out["fp32_vs_torch_adamw"] = fp32_vs_torch_adamw(asr, W, dev)
    out["shard_invariance_268m"] = shard_invariance(asr, W, dev)
    torch.cuda.empty_cache()
    return out


def shard_invariance(asr, W, dev, n=268_435_456, shards=8):
    """The pages' shard invariance: one bf16 tensor of n params (~U(-1, 1)
    params, ~N(0, 1e-2) grads, seed 1234, step 7) updated whole and as
    `shards` contiguous shards (one of them cut off a multiple of 4, each
    with its own base index), compared bit for bit."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    p = W.device_uniform_(torch.empty(n, device=dev), gen, -1.0, 1.0).to(torch.bfloat16)
    g = W.device_normal_(torch.empty(n, device=dev), gen, 1e-2).to(torch.bfloat16)
    whole = [p.clone(), g, torch.zeros(n, device=dev), torch.zeros(n, device=dev)]
    split = [p, g, torch.zeros(n, device=dev), torch.zeros(n, device=dev)]
    asr.asr_adamw_sr_step(*whole, base_index=0, step=7, seed=1234, **HP)
    cuts = [n * k // shards for k in range(shards + 1)]
    cuts[1] += 3                                   # one cut off a multiple of 4
    asr.asr_adamw_sr_multi_tensor([(split[0][a:b], split[1][a:b], split[2][a:b], split[3][a:b], a)
                                   for a, b in zip(cuts, cuts[1:])], step=7, seed=1234, **HP)
    torch.cuda.synchronize(dev)
    same = (torch.equal(whole[0].view(torch.int16), split[0].view(torch.int16))
            and torch.equal(whole[2], split[2]) and torch.equal(whole[3], split[3]))
    require_no_device_error(asr.asr_take_device_error, "shard invariance")
    return {"what": "one 268M-param bf16 tensor updated whole and as 8 shards with their base indices",
            "params": n, "shards": shards, "cuts": cuts, "bitwise_equal": bool(same)}


def fp32_vs_torch_adamw(asr, W, dev, n=16_777_216, steps=100):
    """The pages' accuracy criterion: fp32 parameters updated by the library
    stay within 1e-4 of torch.optim.AdamW (its plain per-parameter form) run
    on the same gradients, over 100 steps; n params ~N(0, 0.02), grads
    ~N(0, 1e-3) drawn fresh every step.  Reports the largest absolute
    difference at the end."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(20240)
    p = W.device_normal_(torch.empty(n, device=dev), gen, 0.02)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    tp = torch.nn.Parameter(p.clone())
    opt = torch.optim.AdamW([tp], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"], foreach=False, fused=False)
    g = torch.empty(n, device=dev)
    for step in range(1, steps + 1):
        W.device_normal_(g, gen, 1e-3)
        asr.asr_adamw_sr_step(p, g, m, v, step=step, seed=0, **HP)
        tp.grad = g
        opt.step()
    torch.cuda.synchronize(dev)
    diff = float((p.double() - tp.detach().double()).abs().max())
    require_no_device_error(asr.asr_take_device_error, "fp32 comparison with torch.optim.AdamW")
    return {"what": "max |p - torch.optim.AdamW p| after 100 steps, fp32 params and grads, same grads",
            "params": n, "steps": steps, "max_abs_diff": diff, "criterion": 1e-4, "within": diff < 1e-4}


SUBULP_STEPS, SUBULP_LR, SUBULP_TARGET = 6000, 1e-4, 1.5


def subulp_demo(asr, dev, n=65536):
    """The pages' sub-ULP demonstration through the library: AdamW on the
    loss (w - 1.5)^2 from w = 1.0, bf16 weights and no fp32 master copy, lr
    1e-4 (a fortieth of the bf16 spacing below 1.0), 6,000 steps, for n
    weights at once, with nearest and with stochastic rounding, and the
    stochastic run repeated.  Reports the mean weights, whether nearest
    rounding moved any weight, the same optimisation in binary64 without
    rounding, and whether the rerun gave the same bits."""
    import math
    import time as _time

    import torch
    hp = dict(lr=SUBULP_LR, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)

    def run(rounding):
        w = torch.ones(n, dtype=torch.bfloat16, device=dev)
        m = torch.zeros(n, device=dev)
        v = torch.zeros(n, device=dev)
        for k in range(1, SUBULP_STEPS + 1):
            g = 2.0 * (w.float() - SUBULP_TARGET)
            asr.asr_adamw_sr_step(w, g, m, v, step=k, seed=7, rounding=rounding, **hp)
        torch.cuda.synchronize(dev)
        return w

    t0 = _time.time()
    w_rn = run("rne")
    w_sr = run("sr")
    w_sr2 = run("sr")
    seconds = _time.time() - t0
    ref, m, v = 1.0, 0.0, 0.0
    for k in range(1, SUBULP_STEPS + 1):
        g = 2.0 * (ref - SUBULP_TARGET)
        m = 0.9 * m + 0.1 * g
        v = 0.999 * v + 0.001 * g * g
        ref -= SUBULP_LR * (m / (1 - 0.9 ** k)) / (math.sqrt(v / (1 - 0.999 ** k)) + 1e-8)
    require_no_device_error(asr.asr_take_device_error, "sub-ULP demonstration")
    return {"what": "AdamW on (w - 1.5)^2 from w = 1.0, bf16 weights, no fp32 master, lr 1e-4, 6,000 steps",
            "params": n, "steps": SUBULP_STEPS, "rn_mean": float(w_rn.float().mean()),
            "rn_moved": bool((w_rn.float() != 1.0).any()), "sr_mean": float(w_sr.float().mean()),
            "unrounded_binary64": ref, "sr_rerun_bitwise": bool(torch.equal(w_sr.view(torch.int16),
                                                                            w_sr2.view(torch.int16))),
            "seconds": seconds}


def optimizer_step_time(asr, tensors, dev, steps, warmup, n):
    """The user-facing optimizer (AdamWSR.step()) on the same 8B set: wall
    time per step over `steps` steps after `warmup`, with the blocking and
    with the deferred device-error check.  Its moments are the set's own
    buffers (placed in the optimizer state as a loaded checkpoint would be),
    so no memory is added."""
    import torch
    params = []
    for p, g, m, v, base in tensors:
        prm = torch.nn.Parameter(p)
        prm.grad = g
        params.append(prm)
    out = {}
    for mode in (True, "deferred"):
        opt = asr.AdamWSR(params, lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                          weight_decay=HP["weight_decay"], seed=0, check_errors=mode)
        for prm, (p, g, m, v, base) in zip(params, tensors):
            opt.state[prm] = {"step": 0, "exp_avg": m, "exp_avg_sq": v}
        for _ in range(warmup):
            opt.step()
        opt.poll_errors(wait=True)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(steps):
            opt.step()
        opt.poll_errors(wait=True)
        torch.cuda.synchronize(dev)
        ms = (time.perf_counter() - t0) / steps * 1e3
        out["blocking_check" if mode is True else "deferred_check"] = {
            "ms_per_step": ms, "gparams_per_s": n / ms / 1e6}
        del opt
    out["note"] = ("AdamWSR.step() on the 8B set (291 parameters), wall clock with a synchronize at the end; "
                   "the blocking check waits for each step, the deferred one reads the error word one step late")
    return out


def graph_step_cost(asr, W, dev, gen, n=65536, steps=50):
    """GPU time per step of the small single-tensor step when its launches
    come from a CUDA graph (50 consecutive steps captured once after an
    ordinary call, then replayed): the cost of the step itself, without the
    host's per-call work."""
    import torch
    p = W.device_normal_(torch.empty(n, dtype=torch.bfloat16, device=dev), gen, 0.02)
    g = W.device_normal_(torch.empty(n, dtype=torch.bfloat16, device=dev), gen, 1e-3)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    asr.asr_adamw_sr_step(p, g, m, v, step=1, seed=0, **HP)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for t in range(2, steps + 2):
            asr.asr_adamw_sr_step(p, g, m, v, step=t, seed=0, **HP)
    graph.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    require_no_device_error(asr.asr_take_device_error, "graph-replayed steps")
    return e0.elapsed_time(e1) / steps * 1e3


def binding_host_cost(asr, W, dev, gen, n=65536, calls=200):
    """Host time per call (microseconds) to enqueue one single-tensor step:
    through the C ABI directly (ctypes, arguments marshalled once) and
    through the Python binding (tensor checks, hyperparameter struct, stream
    lookup every call).  Few enough calls that the launch queue never fills,
    so the host loop is not held up by the GPU."""
    import ctypes
    import torch
    from stochastic_rounding_gb300 import _lib
    p = W.device_normal_(torch.empty(n, dtype=torch.bfloat16, device=dev), gen, 0.02)
    g = W.device_normal_(torch.empty(n, dtype=torch.bfloat16, device=dev), gen, 1e-3)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    L = _lib.lib()
    sh = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    hps = [_lib.make_hparams(step=t, seed=0, **HP) for t in range(1, calls + 1)]
    args = (ctypes.c_void_p(p.data_ptr()), _lib.ASR_BF16, ctypes.c_void_p(g.data_ptr()), _lib.ASR_BF16,
            ctypes.c_void_p(m.data_ptr()), ctypes.c_void_p(v.data_ptr()), n, 0)
    res = {}
    for rep in range(2):                     # the first pass warms both paths up
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for h in hps:
            if L.asr_adamw_sr_step(*args, ctypes.byref(h), sh) != _lib.ASR_OK:
                raise RuntimeError("asr_adamw_sr_step failed")
        res["c_abi"] = (time.perf_counter() - t0) / calls * 1e6
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for t in range(1, calls + 1):
            asr.asr_adamw_sr_step(p, g, m, v, step=t, seed=0, **HP)
        res["python_binding"] = (time.perf_counter() - t0) / calls * 1e6
        torch.cuda.synchronize(dev)
    require_no_device_error(asr.asr_take_device_error, "binding cost calls")
    return res


def step_config(n, tensors, truncated, world):
    """The `config` of the AdamW-SR step lines (both arms)."""
    return {"workload": ("llama3-8b" if not truncated else f"llama3-8b truncated to {n:,} params")
                        + f": fused AdamW-SR multi-tensor step, {tensors} tensors, {n:,} params per GPU",
            "params_per_gpu": n, "tensors": tensors,
            "param_dtype": "bf16", "grad_dtype": "bf16", "state_dtype": "f32",
            "rounding": "stochastic (Philox4x32-10)", "bytes_per_param": BYTES_PER_PARAM,
            "l2": "inputs larger than L2 (176.7 GB moved per step)",
            "parallelism": f"shard{world}" if world > 1 else "single"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from stochastic_rounding_gb300 import workloads as W
    rates, desc = cpu_oracle_sample(args.warmup + args.steps)
    timed = rates[args.warmup:]
    value = statistics.median(timed) / 1e9
    ms = CPU_SAMPLE_ELEMS / (value * 1e9) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        # the native arm's workload; each step of this arm times the oracle on
        # a bounded sample of it (params/s is per sampled parameter)
        "config": step_config(sum(n for _, n, _ in W.param_table(W.LLAMA_8B)), len(W.param_table(W.LLAMA_8B)),
                              0, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    rank, world, local = dist_env()
    pool = None
    if rank == 0:
        pool, pool_cores = start_oracle_pool()
    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from __graft_entry__ import build
    build()
    import stochastic_rounding_gb300 as asr
    from stochastic_rounding_gb300 import _lib
    from stochastic_rounding_gb300 import workloads as W

    ps = W.DeviceParamSet(W.LLAMA_8B, device=dev, seed=rank, max_params=args.params)
    tensors = ps.tensors()
    # rank r owns parameters [r*N, (r+1)*N) of an N x 8B flat vector
    offset = rank * ps.numel
    table = _lib.make_table([(p, g, m, v, base + offset) for p, g, m, v, base in tensors])
    stream = torch.cuda.Stream(device=dev)
    n = ps.numel

    def step(t):
        asr.asr_adamw_sr_multi_tensor(table, step=t, seed=0, stream=stream, device=dev, **HP)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def max_over_ranks(x):
        if world == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())

    t_global = 0
    for _ in range(args.warmup):
        t_global += 1
        step(t_global)
    torch.cuda.synchronize(dev)
    require_no_device_error(asr.asr_take_device_error, "warm-up steps")

    # ---- device-resident timed region
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    counts_before = asr.asr_kernel_launches()
    with ClockSampler(local) as clocks:
        all_start = torch.cuda.Event(enable_timing=True)
        all_end = torch.cuda.Event(enable_timing=True)
        clocks.mark_start()
        all_start.record(stream)
        for k in range(args.steps):
            t_global += 1
            starts[k].record(stream)
            step(t_global)
            ends[k].record(stream)
        all_end.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark_end()
    counts_after = asr.asr_kernel_launches()
    barrier()
    require_no_device_error(asr.asr_take_device_error, "timed device-resident steps")
    total_ms = max_over_ranks(all_start.elapsed_time(all_end))
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    launch_ms = statistics.mean(per_launch_ms)
    clock = clocks.summary()
    # the library's own launch counters over the timed region (one
    # multi-tensor launch per step expected)
    launches = sum(counts_after[k] - counts_before[k] for k in counts_after)
    launch_kinds = {k: counts_after[k] - counts_before[k] for k in counts_after if counts_after[k] != counts_before[k]}

    value = world * n * args.steps / (total_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    achieved = BYTES_PER_PARAM * n / (launch_ms / 1e3) / 1e9
    tpp = traffic_per_param()

    # ---- end to end through the C ABI with host buffers: every step is one
    # asr_adamw_sr_multi_tensor_host call, which copies the grads in from
    # page-locked host memory, steps, and copies the updated bf16 params back
    # out, pipelined in the library over chunks of consecutive tensors and
    # three streams (copies of chunk c+1 in and c-1 out overlap the step on
    # chunk c).
    chunks = e2e_chunks(tensors)
    # one pinned host buffer per chunk (a contiguous range [lo, hi) of the
    # flat layout), each tensor a view of its chunk's buffer: torch's pinned
    # allocator rounds each request up to a power of two, which for two whole
    # 16 GB buffers would double the host memory taken; per ~512 MB chunk the
    # rounding wastes ~10 %
    g_host = [torch.empty(hi - lo, dtype=torch.bfloat16, pin_memory=True) for lo, hi in chunks]
    p_host = [torch.empty(hi - lo, dtype=torch.bfloat16, pin_memory=True) for lo, hi in chunks]
    for (lo, hi), gh in zip(chunks, g_host):
        gh.copy_(ps.g[lo:hi])
    rows, c = [], 0
    for p_t, g_t, m_t, v_t, base in tensors:
        while base >= chunks[c][1]:
            c += 1
        a = base - chunks[c][0]
        k = p_t.numel()
        rows.append((p_t, g_t, m_t, v_t, base + offset, g_host[c][a:a + k], p_host[c][a:a + k]))
    host_table = _lib.make_host_table(rows)
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)

    def e2e_steps(count):
        nonlocal t_global
        for _ in range(count):
            t_global += 1
            asr.asr_adamw_sr_multi_tensor_host(host_table, step=t_global, seed=0, chunk_elems=E2E_CHUNK,
                                               stream=stream, copy_in=s_in, copy_out=s_out, device=dev, **HP)
        stream.wait_stream(s_out)            # the last params out are part of the step

    def copies_steps(count):
        """The same transfers with no step: per chunk, grads in on s_in and
        params out on s_out after that chunk's grads are in."""
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for _ in range(count):
            for c, (lo, hi) in enumerate(chunks):
                with torch.cuda.stream(s_in):
                    ps.g[lo:hi].copy_(g_host[c], non_blocking=True)
                    ev_in = torch.cuda.Event()
                    ev_in.record(s_in)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_in)
                    p_host[c].copy_(ps.p[lo:hi], non_blocking=True)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    e2e_steps(args.warmup)                   # untimed, like the device-resident leg
    torch.cuda.synchronize(dev)
    e_steps = max(1, args.steps)
    barrier()
    e_counts_before = asr.asr_kernel_launches()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    e2e_steps(e_steps)
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    e_counts_after = asr.asr_kernel_launches()
    barrier()
    launches_e2e = sum(e_counts_after[k] - e_counts_before[k] for k in e_counts_after)
    require_no_device_error(asr.asr_take_device_error, "timed end-to-end steps")
    e_ms = max_over_ranks(e_start.elapsed_time(e_end))
    e2e_value = world * n * e_steps / (e_ms / 1e3) / 1e9
    # the same transfers with the steps left out, outside the timed region:
    # what this machine's host link allows for them
    c_start = torch.cuda.Event(enable_timing=True)
    c_end = torch.cuda.Event(enable_timing=True)
    c_start.record(stream)
    copies_steps(e_steps)
    c_end.record(stream)
    torch.cuda.synchronize(dev)
    copies_value = world * n * e_steps / (max_over_ranks(c_start.elapsed_time(c_end)) / 1e3) / 1e9
    del g_host, p_host
    ring_value = world * n / max_over_ranks(ring_copies_seconds(ps.g, ps.p, n, dev, e_steps)) / 1e9
    link = host_link_rates(dev)
    # the copies alone bound the end-to-end step: 2n bytes in and 2n out
    floor_s = max(2 * n / (link["h2d"] * 1e9), 2 * n / (link["d2h"] * 1e9), 4 * n / (link["both"] * 1e9))

    others = None
    if rank == 0 and not args.params:
        others = {"optimizer_class_8b": optimizer_step_time(asr, tensors, dev, args.steps, args.warmup, n)}
        others.update(measure_configs(asr, W, dev, args.steps, args.warmup, peak))

    cpu = None
    if rank == 0:
        rates, desc = cpu_oracle_sample(steps=3)
        cpu = {"value": statistics.median(rates) / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": desc + ", median of 3 steps"}
        cpu["all_cores"] = cpu_oracle_all_cores(pool, pool_cores)
        pool.close()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": step_config(n, len(tensors), args.params, world),
            "achieved_gbs": achieved, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": tpp * n if tpp is not None else None,
                         "kernel": ("adamw_sr_tma_kernel<bf16,bf16,SR,512>" if "adamw_pipelined" in launch_kinds
                                    else "adamw_sr_kernel<bf16,bf16,SR,vector,512>"),
                         "launch_ms_mean": launch_ms},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 2 * n,
                    "d2h_bytes_per_step": 2 * n, "steps": e_steps, "chunks": len(chunks),
                    "gpu_launches": launches_e2e,
                    "link_gbs": link, "link_floor_gparams_s": n / floor_s / 1e9,
                    "frac_of_link_floor": e2e_value / world / (n / floor_s / 1e9),
                    "copies_only_gparams_s": copies_value, "frac_of_copies_only": e2e_value / copies_value,
                    "small_footprint_copies_gparams_s": ring_value,
                    "what": "one asr_adamw_sr_multi_tensor_host call per step: bf16 grads H2D from "
                            "pinned host, step, bf16 params D2H to pinned host, pipelined in the library "
                            "over chunks of consecutive tensors and three streams; host buffers hold the "
                            "whole set (copies_only: the same transfers per chunk without the steps; "
                            "small_footprint_copies: the same bytes through a 512 MB page-locked "
                            "staging ring, no steps)"},
            "gpu_launches": launches,
            "gpu_launch_kinds": launch_kinds,
            "configs": others,
            "clocks": clock,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def gemm_cpu_baseline(a, b, m, n, k, budget_macs=6e9):
    """The oracle's GEMM (binary64 sums of the exact products, one rounding
    to binary32, the per-element stochastic rounding), single-threaded C,
    timed on the first rows of the same operands: as many rows as fit in
    about budget_macs multiply-adds."""
    import numpy as np
    import torch
    import oracle
    o = oracle.get()
    rows = int(max(1, min(m, budget_macs // (n * k))))
    a_h = a[:rows].cpu().view(torch.int16).numpy().view(np.uint16)
    b_h = b.cpu().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    o.gemm_bf16(a_h, b_h, step=1, seed=0)
    dt = time.perf_counter() - t0
    return {"value": 2.0 * rows * n * k / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"{rows} of {m} rows x {n} columns x K={k}, C oracle single thread, {dt:.1f} s"}


def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


# The SR epilogue's integer-multiply ceiling.  Each output element takes a
# quarter of a Philox4x32-10 call: 10 rounds x 2 products (32 x 32 -> 64 bits)
# / 4 outputs = 5 products, i.e. 10 32-bit multiply results (low and high
# halves).  The public CUDA throughput table gives 64 32-bit integer
# multiply(-add) results per clock per SM.
EPILOGUE_MUL_RESULTS_PER_OUTPUT = 10
INT_MUL_RESULTS_PER_CLK_PER_SM = 64


def gemm_measure(asr, dev, m, n, k, steps, warmup, cpu_budget_macs):
    """The tcgen05 GEMM with the stochastic-rounding epilogue (and with the
    round-to-nearest epilogue, and torch.matmul = cuBLAS, for context) on
    one m x n x k problem: TFLOP/s by CUDA events over the timed launches,
    against the measured bf16 tensor peak; beside it the epilogue's
    integer-multiply rate against the SMs' integer-multiply ceiling at the
    maximum SM clock (the bound that matters at small K)."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    a = torch.randn(m, k, device=dev, generator=g).to(torch.bfloat16)
    b = torch.randn(n, k, device=dev, generator=g).to(torch.bfloat16)
    c = torch.empty(m, n, device=dev, dtype=torch.bfloat16)
    flops = 2.0 * m * n * k
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps

    t_sr = timed(lambda: asr.asr_gemm_bf16_sr(a, b, c, rounding="sr", step=1, seed=0))
    t_rn = timed(lambda: asr.asr_gemm_bf16_sr(a, b, c, rounding="rne"))
    require_no_device_error(asr.asr_take_device_error, f"timed GEMM {m}x{n}x{k}")
    t_cublas = timed(lambda: torch.matmul(a, b.t()))
    peak, kind = bf16_peak()
    tf = flops / (t_sr / 1e3) / 1e12
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            clk_mhz = float(json.load(f)["sm_max_mhz"])
    except Exception:
        clk_mhz = 2070.0
    mul_rate = EPILOGUE_MUL_RESULTS_PER_OUTPUT * m * n / (t_sr / 1e3)
    mul_peak = sms * clk_mhz * 1e6 * INT_MUL_RESULTS_PER_CLK_PER_SM
    entry = {"workload": f"gemm {m}x{n}x{k} bf16, f32 accumulate, C = A.B^T, SR epilogue",
             "ms": t_sr, "tflops": tf,
             "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                          "peak_kind": kind},
             "epilogue_int_mul": {"achieved": mul_rate / 1e12, "peak": mul_peak / 1e12,
                                  "unit": "T multiply results/s", "frac": mul_rate / mul_peak,
                                  "per_output": EPILOGUE_MUL_RESULTS_PER_OUTPUT,
                                  "peak_basis": f"{sms} SMs x {clk_mhz:.0f} MHz x "
                                                f"{INT_MUL_RESULTS_PER_CLK_PER_SM}/clk/SM"},
             "rne_epilogue_tflops": flops / (t_rn / 1e3) / 1e12,
             "cublas_torch_matmul_tflops": flops / (t_cublas / 1e3) / 1e12,
             "steps": steps, "warmup": warmup}
    if cpu_budget_macs:
        entry["cpu_baseline"] = gemm_cpu_baseline(a, b, m, n, k, cpu_budget_macs)
    del a, b, c
    return entry


def run_gemm(args):
    """One GEMM problem (--gemm M N K) as its own JSON line."""
    import torch
    from __graft_entry__ import build
    build()
    import stochastic_rounding_gb300 as asr
    m, n, k = args.gemm
    dev = torch.device("cuda", 0)
    e = gemm_measure(asr, dev, m, n, k, args.steps, args.warmup, 6e9)
    line = {"metric": "bf16 GEMM with stochastic-rounding epilogue TFLOP/s", "value": e["tflops"],
            "unit": "TFLOP/s", "ms": e["ms"], "config": {"workload": e["workload"]},
            "roofline": e["roofline"], "epilogue_int_mul": e["epilogue_int_mul"],
            "rne_epilogue_tflops": e["rne_epilogue_tflops"],
            "cublas_torch_matmul_tflops": e["cublas_torch_matmul_tflops"],
            "cpu_baseline": e["cpu_baseline"], "steps": args.steps, "warmup": args.warmup}
    print(json.dumps(line), flush=True)
    return 0


def elementwise_measure(asr, dev, kind, n, steps, warmup, sample=1 << 22):
    """The stand-alone rounding op (kind "sr": float32 -> bf16 with Philox
    bits, 6 B per element) or the Philox op (kind "philox": n counters, 16 B
    written each) over n elements resident in HBM (larger than L2), by CUDA
    events over the timed launches, against the measured copy bandwidth; the
    oracle on a ``sample``-element sample beside it."""
    import torch
    import oracle
    if kind == "sr":
        unit_bytes, what = 6, "stand-alone stochastic rounding float32 -> bf16"
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        x = torch.randn(n, device=dev, generator=g)
        out = torch.empty(n, device=dev, dtype=torch.bfloat16)
        fn = lambda: asr.asr_stochastic_round_bf16(x, out, base_index=0, step=1, seed=0)  # noqa: E731
    else:
        unit_bytes, what = 16, "Philox4x32-10 counters, four words each"
        x = None
        out = torch.empty(4 * n, device=dev, dtype=torch.int32)
        fn = lambda: asr.asr_philox4x32(out, n, 0, 1, 0, 0)  # noqa: E731
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    require_no_device_error(asr.asr_take_device_error, f"timed {kind} launches")
    peak, pkind = measured_peak()
    gbs = unit_bytes * n / (ms / 1e3) / 1e9
    o = oracle.get()
    t0 = time.perf_counter()
    if kind == "sr":
        o.sr_fill(x[:sample].cpu().numpy(), 0, 1, 0)
    else:
        o.philox_fill(sample, 0, 1, 0, 0)
    dt = time.perf_counter() - t0
    unit = "Gelem/s" if kind == "sr" else "Gctr/s"
    del x, out
    return {"workload": f"{what}, {n:,} {'elements' if kind == 'sr' else 'counters'}", "what": what,
            "value": n / (ms / 1e3) / 1e9, "unit": unit, "ms": ms,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "peak_kind": pkind, "bytes_per_unit": unit_bytes},
            "cpu_baseline": {"value": sample / dt / 1e9, "unit": unit, "cores": 1, "kind": "oracle",
                             "sample": f"{sample:,} {'elements' if kind == 'sr' else 'counters'}, "
                                       f"C oracle single thread"},
            "steps": steps, "warmup": warmup}


def run_elementwise(args):
    """The stand-alone rounding op (--sr N) or the Philox op (--philox N) as
    its own JSON line."""
    import torch
    from __graft_entry__ import build
    build()
    import stochastic_rounding_gb300 as asr
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kind, n = ("sr", args.sr) if args.sr else ("philox", args.philox)
    e = elementwise_measure(asr, dev, kind, n, args.steps, args.warmup)
    line = {"metric": f"{e['what']} {e['unit']}", "value": e["value"], "unit": e["unit"], "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": e["ms"], "higher_is_better": True,
            "dtype": "f32->bf16" if kind == "sr" else "u32", "data": "synthetic",
            "config": {"workload": e["workload"], "l2": "inputs and outputs larger than L2"},
            "roofline": e["roofline"], "cpu_baseline": e["cpu_baseline"], "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--params", type=int, default=0,
                    help="keep only the tensors of the 8B layout that fit in this many params "
                         "(a small case for profiling); 0 = the full set")
    ap.add_argument("--gemm", type=int, nargs=3, metavar=("M", "N", "K"), default=None,
                    help="time the tensor-core GEMM with the stochastic-rounding epilogue instead")
    ap.add_argument("--sr", type=int, default=0, metavar="N",
                    help="time the stand-alone stochastic-rounding op on N float32 elements instead")
    ap.add_argument("--philox", type=int, default=0, metavar="N",
                    help="time the Philox op on N counters instead")
    args = ap.parse_args()
    if args.gemm:
        return run_gemm(args)
    if args.sr or args.philox:
        return run_elementwise(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
