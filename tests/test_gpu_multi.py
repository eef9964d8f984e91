"""GPU parity of the multi-tensor launch: bitwise equal to per-tensor calls
and to the oracle; Llama-shaped parameter sets checked on sampled windows."""
import numpy as np
import pytest

from gpu_util import assert_same_bits, dev, host, pick_windows, torch_cuda
from stochastic_rounding_gb300 import workloads as W

pytestmark = pytest.mark.gpu
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@pytest.fixture(scope="module")
def asr():
    torch_cuda()
    from stochastic_rounding_gb300 import build
    build.build()
    import stochastic_rounding_gb300 as m
    m.lib()
    return m


def _random_set(rng, count, max_n, offsets=(0, 0, 0, 1, 3)):
    """Host arrays and device slices of ``count`` tensors with mixed dtypes,
    some starting off a 16-byte boundary, bases cumulative with gaps."""
    host_t, base = [], 5
    for i in range(count):
        n = int(rng.integers(0, max_n))
        pdt = rng.choice(["bf16", "f32"])
        gdt = rng.choice(["bf16", "f32"])
        off = int(rng.choice(offsets))
        p = W.normal_f32(rng, n + off, 0.02)
        g = W.normal_f32(rng, n + off, 1e-3)
        if pdt == "bf16":
            p = W.to_bf16_bits(p)
        if gdt == "bf16":
            g = W.to_bf16_bits(g)
        m = W.normal_f32(rng, n + off, 1e-4)
        v = np.abs(W.normal_f32(rng, n + off, 1e-6))
        host_t.append(([p, g, m, v], off, base))
        base += n + int(rng.integers(0, 3))
    return host_t


def _dev_set(host_t):
    out = []
    for arrs, off, base in host_t:
        ts = [dev(a)[off:] for a in arrs]
        out.append((ts[0], ts[1], ts[2], ts[3], base))
    return out


@pytest.mark.parametrize("rounding", ["sr", "rne"])
def test_multi_equals_per_tensor_and_oracle(asr, orc, rounding):
    import torch
    rng = np.random.default_rng(21 if rounding == "sr" else 22)
    hs = _random_set(rng, 37, 20000)
    a = _dev_set(hs)
    b = _dev_set(hs)
    for step in (1, 2):
        asr.asr_adamw_sr_multi_tensor(a, step=step, seed=2**35 + 1, rounding=rounding, **HP)
        for p, g, m, v, base in b:
            asr.asr_adamw_sr_step(p, g, m, v, base_index=base, step=step, seed=2**35 + 1,
                                  rounding=rounding, **HP)
        for arrs, off, base in hs:
            p, g, m, v = (x[off:].copy() for x in arrs)
            orc.adamw_step(p, g, m, v, step=step, seed=2**35 + 1, base_index=base,
                           rounding=0 if rounding == "sr" else 1, **HP)
            for x, y in zip(arrs, (p, g, m, v)):
                x[off:] = y
    torch.cuda.synchronize()
    for i, ((arrs, off, base), ta, tb) in enumerate(zip(hs, a, b)):
        for k in (0, 2, 3):
            assert np.array_equal(host(ta[k]).view(np.uint8), host(tb[k]).view(np.uint8)), \
                f"tensor {i}: multi-tensor differs from per-tensor calls"
            assert_same_bits(host(ta[k]), arrs[k][off:], f"tensor {i} buffer {k}")


def test_more_tensors_than_one_launch_holds(asr, orc):
    """1,100 small tensors (more than one launch's table) in one call."""
    import torch
    rng = np.random.default_rng(23)
    hs = _random_set(rng, 1100, 300, offsets=(0,))
    a = _dev_set(hs)
    asr.asr_adamw_sr_multi_tensor(a, step=3, seed=4, **HP)
    torch.cuda.synchronize()
    for i, ((arrs, off, base), t) in enumerate(zip(hs, a)):
        p, g, m, v = (x.copy() for x in arrs)
        orc.adamw_step(p, g, m, v, step=3, seed=4, base_index=base, **HP)
        assert_same_bits(host(t[0]), p, f"tensor {i} p")
        assert_same_bits(host(t[2]), m, f"tensor {i} m")
        assert_same_bits(host(t[3]), v, f"tensor {i} v")


def _check_windows(asr, orc, ps, table, windows, step, seed):
    """One multi-tensor step, with the windows checked against the oracle."""
    import torch
    before = []
    for t, s, n in windows:
        a = ps.starts[t] + s
        before.append([host(x[a:a + n]) for x in (ps.p, ps.g, ps.m, ps.v)])
    asr.asr_adamw_sr_multi_tensor(table, step=step, seed=seed, device=ps.device, **HP)
    torch.cuda.synchronize()
    for (t, s, n), (p, g, m, v) in zip(windows, before):
        a = ps.starts[t] + s
        orc.adamw_step(p, g, m, v, step=step, seed=seed, base_index=a, **HP)
        assert_same_bits(host(ps.p[a:a + n]), p, f"{ps.table[t][0]}[{s}:{s + n}] p step {step}")
        assert_same_bits(host(ps.m[a:a + n]), m, f"{ps.table[t][0]}[{s}:{s + n}] m step {step}")
        assert_same_bits(host(ps.v[a:a + n]), v, f"{ps.table[t][0]}[{s}:{s + n}] v step {step}")


def _host_view(t):
    """A host copy of a device tensor as a numpy array (bf16 as uint16
    patterns), without a second copy."""
    import torch
    a = t.detach().cpu()
    if a.dtype == torch.bfloat16:
        return a.view(torch.int16).numpy().view(np.uint16)
    return a.numpy()


def _mem_available():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


@pytest.mark.parametrize("shape,steps", [(W.LLAMA_1B, (1, 2)), (W.LLAMA_8B, (1,))],
                         ids=["llama-1.5B-147t", "llama3-8B-291t"])
def test_llama_param_set_every_element(asr, orc, shape, steps):
    """Every element of every tensor of a Llama-shaped set, after one
    multi-tensor launch per step, equals the oracle run at the tensor's base
    index (host threads, each on a contiguous chunk; the oracle call releases
    the interpreter lock).  Moments start from nonzero values so each term of
    the update is exercised from the first step.  Skipped where the host lacks
    the memory for one host copy of the set."""
    import concurrent.futures
    import os

    import torch
    from stochastic_rounding_gb300 import _lib
    table = W.param_table(shape)
    _, total = W.offsets(table)
    need = total * 12 + max(n for _, n, _ in table) * 10
    if _mem_available() < need * 1.25 + (8 << 30):
        pytest.skip(f"host memory: {need / 2**30:.0f} GiB for one copy of the set")
    ps = W.DeviceParamSet(shape, seed=5)
    W.device_normal_(ps.m, ps.gen, 1e-4)
    W.device_normal_(ps.v, ps.gen, 1e-6)
    ps.v.abs_()
    dev_table = _lib.make_table(ps.tensors())
    workers = max(1, len(os.sched_getaffinity(0)))
    chunk = 1 << 24
    jobs = [(s + a, min(s + n, s + a + chunk)) for s, n in zip(ps.starts, ps.sizes) for a in range(0, n, chunk)]
    with concurrent.futures.ThreadPoolExecutor(workers) as pool:
        for k, step in enumerate(steps):
            if k > 0:
                ps.new_grads()
            torch.cuda.synchronize()
            p, g, m, v = (_host_view(x) for x in (ps.p, ps.g, ps.m, ps.v))
            asr.asr_adamw_sr_multi_tensor(dev_table, step=step, seed=0, device=ps.device, **HP)

            def run(lo_hi, step=step):
                lo, hi = lo_hi
                orc.adamw_step(p[lo:hi], g[lo:hi], m[lo:hi], v[lo:hi], step=step, seed=0, base_index=lo, **HP)

            list(pool.map(run, jobs))
            torch.cuda.synchronize()
            for (name, n, _), s in zip(ps.table, ps.starts):
                for got, want, what in ((ps.p, p, "p"), (ps.m, m, "m"), (ps.v, v, "v")):
                    gh = _host_view(got[s:s + n])
                    w = want[s:s + n]
                    u = np.uint16 if w.dtype == np.uint16 else np.uint32
                    if not np.array_equal(gh.view(u), w.view(u)):
                        assert_same_bits(gh, w, f"{name} {what} step {step}")
            del p, g, m, v
    del ps, dev_table
    torch.cuda.empty_cache()


@pytest.mark.parametrize("shape,steps,checked", [(W.LLAMA_1B, 20, (1, 2, 20)), (W.LLAMA_8B, 10, (1, 10))],
                         ids=["llama-1.5B-147t-20steps", "llama3-8B-291t-10steps"])
def test_llama_param_set_sampled(asr, orc, shape, steps, checked):
    """The Llama-shaped sets in one multi-tensor launch per step: norm tensors
    whole, every other tensor's head, tail and two random unaligned windows
    checked against the oracle at the listed steps."""
    import torch
    from stochastic_rounding_gb300 import _lib
    ps = W.DeviceParamSet(shape, seed=0)
    table = _lib.make_table(ps.tensors())
    rng = np.random.default_rng(31)
    windows = pick_windows(rng, ps.sizes, per_tensor=2, length=2048)
    for step in range(1, steps + 1):
        if step > 1:
            ps.new_grads()
        if step in checked:
            _check_windows(asr, orc, ps, table, windows, step, seed=0)
        else:
            asr.asr_adamw_sr_multi_tensor(table, step=step, seed=0, device=ps.device, **HP)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(ps.p[:1 << 20].float()).all())
    del ps
    torch.cuda.empty_cache()


def test_llama_set_at_positions_off_a_multiple_of_4(asr, orc):
    """A Llama-shaped set (the leading tensors of the 1.5B layout, ~300M
    params, 16-byte-aligned buffers) whose global positions are shifted by
    1, 2 or 3 per tensor, as when an odd-sized parameter comes earlier in a
    model: every tensor then takes the pipelined kernel that draws three
    Philox counters per 8-element unit.  Sampled windows of every tensor
    equal the oracle at steps 1 and 3."""
    import torch
    from stochastic_rounding_gb300 import _lib
    ps = W.DeviceParamSet(W.LLAMA_1B, seed=5, max_params=300_000_000)
    shift = [1 + (t % 3) for t in range(len(ps.sizes))]
    tensors = [(p, g, m, v, base + shift[t]) for t, (p, g, m, v, base) in enumerate(ps.tensors())]
    assert all(b % 4 != 0 for *_, b in tensors)
    table = _lib.make_table(tensors)
    rng = np.random.default_rng(32)
    windows = pick_windows(rng, ps.sizes, per_tensor=2, length=2048)
    for step in (1, 2, 3):
        if step > 1:
            ps.new_grads()
        before = []
        if step != 2:
            for t, st, n in windows:
                a = ps.starts[t] + st
                before.append([host(x[a:a + n]) for x in (ps.p, ps.g, ps.m, ps.v)])
        asr.asr_adamw_sr_multi_tensor(table, step=step, seed=9, device=ps.device, **HP)
        torch.cuda.synchronize()
        for (t, st, n), (p, g, m, v) in zip(windows, before):
            a = ps.starts[t] + st
            orc.adamw_step(p, g, m, v, step=step, seed=9, base_index=a + shift[t], **HP)
            where = f"{ps.table[t][0]}[{st}:{st + n}] step {step}"
            assert_same_bits(host(ps.p[a:a + n]), p, where + " p")
            assert_same_bits(host(ps.m[a:a + n]), m, where + " m")
            assert_same_bits(host(ps.v[a:a + n]), v, where + " v")
    assert asr.asr_take_device_error() == 0
    del ps
    torch.cuda.empty_cache()


def test_concurrent_calls_from_threads_and_streams(asr, orc):
    """Two host threads, each with its own stream and its own tensor set,
    issue 5 multi-tensor steps each with no synchronisation between them (the
    library's entry points may run concurrently on disjoint buffers): both
    sets end bit-equal to the oracle run step by step."""
    import threading
    import torch
    from stochastic_rounding_gb300 import _lib
    rng = np.random.default_rng(40)
    sets = [_random_set(rng, 60, 40000), _random_set(rng, 45, 70000)]
    devs = [_dev_set(s) for s in sets]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    errors = []

    def worker(k):
        try:
            table = _lib.make_table(devs[k])
            for step in range(1, 6):
                asr.asr_adamw_sr_multi_tensor(table, step=step, seed=11 + k, stream=streams[k], **HP)
        except Exception as e:          # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for k, host_t in enumerate(sets):
        for (arrs, off, base), (pd, gd, md, vd, _) in zip(host_t, devs[k]):
            p, g, m, v = (a[off:].copy() for a in arrs)
            for step in range(1, 6):
                orc.adamw_step(p, g, m, v, step=step, seed=11 + k, base_index=base, **HP)
            assert_same_bits(host(pd), p, f"set {k} base {base} p")
            assert_same_bits(host(md), m, f"set {k} base {base} m")
            assert_same_bits(host(vd), v, f"set {k} base {base} v")
    assert asr.asr_take_device_error() == 0
