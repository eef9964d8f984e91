"""GPU parity of the single-tensor fused AdamW-SR step through the C ABI
against the oracle: bit-exact params (bf16 or f32) and f32 moments."""
import numpy as np
import pytest

from gpu_util import assert_same_bits, dev, host, torch_cuda
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


def _make(rng, n, pdt, gdt, states=True, pscale=0.02, gscale=1e-3):
    p = W.normal_f32(rng, n, pscale)
    g = W.normal_f32(rng, n, gscale)
    if pdt == "bf16":
        p = W.to_bf16_bits(p)
    if gdt == "bf16":
        g = W.to_bf16_bits(g)
    if states:
        m = W.normal_f32(rng, n, 1e-4)
        v = np.abs(W.normal_f32(rng, n, 1e-6))
    else:
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
    return p, g, m, v


# Steps of at most 128 MiB of traffic whose buffers are aligned (and whose
# bases are multiples of 4, where bits are drawn) take the register kernel.
# To put a small tensor through the pipelined kernel instead, a test steps
# it in one multi-tensor call with a ballast tensor of the same dtypes that
# takes the launch group past that size (its elements stay zero: p, g, m
# and v all 0 give 0 again).
BALLAST = 8_000_000
_ballast_cache = {}


def _ballast(pd, gd):
    import torch
    key = (pd.dtype, gd.dtype)
    if key not in _ballast_cache:
        _ballast_cache[key] = (torch.zeros(BALLAST, dtype=pd.dtype, device="cuda"),
                               torch.zeros(BALLAST, dtype=gd.dtype, device="cuda"),
                               torch.zeros(BALLAST, device="cuda"), torch.zeros(BALLAST, device="cuda"),
                               2**36)
    return _ballast_cache[key]


def _step_both(asr, orc, h, d, via="alone", **kw):
    """One step on the GPU and in the oracle.  via="alone": the tensor by
    itself (asr_adamw_sr_step); via="pipelined": together with the ballast in
    one multi-tensor call, so the tensor's launch group is large enough for
    the pipelined kernel whatever its own size."""
    p, g, m, v = h
    pd, gd, md, vd = d
    base = kw.pop("base_index", 0)
    if via == "pipelined":
        asr.asr_adamw_sr_multi_tensor([(pd, gd, md, vd, base), _ballast(pd, gd)], **kw)
    else:
        asr.asr_adamw_sr_step(pd, gd, md, vd, base_index=base, **kw)
    orc.adamw_step(p, g, m, v, base_index=base, rounding=0 if kw.get("rounding", "sr") == "sr" else 1,
                   **{k: val for k, val in kw.items() if k != "rounding"})


def _check(h, d, what):
    for name, a, t in zip("pmv", (h[0], h[2], h[3]), (d[0], d[2], d[3])):
        assert_same_bits(host(t), a, f"{what} {name}")


def test_single_tensor_65536_bf16_10_steps(asr, orc):
    """65,536 bf16 params ~N(0,0.02), bf16 grads ~N(0,1e-3) drawn per
    (seed, step), m = v = 0, seed 0, 10 steps: bit-exact after every step."""
    n, seed = 65536, 0
    p = W.to_bf16_bits(W.normal_f32(W.host_rng(seed, 0), n, 0.02))
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    d = [dev(p), None, dev(m), dev(v)]
    for step in range(1, 11):
        g = W.to_bf16_bits(W.normal_f32(W.host_rng(seed, step), n, 1e-3))
        d[1] = dev(g)
        asr.asr_adamw_sr_step(d[0], d[1], d[2], d[3], step=step, seed=seed, **HP)
        orc.adamw_step(p, g, m, v, step=step, seed=seed, **HP)
        _check((p, g, m, v), d, f"step {step}")


@pytest.mark.parametrize("pdt,gdt,rounding", [("bf16", "bf16", "sr"), ("bf16", "bf16", "rne"),
                                              ("bf16", "f32", "sr"), ("bf16", "f32", "rne"),
                                              ("f32", "bf16", "sr"), ("f32", "f32", "sr")])
@pytest.mark.parametrize("base", [0, 5, 2**33 + 2, 2**40 + 3])
@pytest.mark.parametrize("via", ["alone", "pipelined"])
def test_dtype_combinations_ragged(asr, orc, pdt, gdt, rounding, base, via):
    n = 3 * 4096 + 13
    rng = np.random.default_rng(hash((pdt, gdt, rounding, base)) % 2**32)
    h = _make(rng, n, pdt, gdt)
    d = [dev(a) for a in h]
    for step in (1, 2, 3):
        _step_both(asr, orc, h, d, via=via, step=step, seed=2**40 + 17, base_index=base, rounding=rounding, **HP)
        _check(h, d, f"{pdt}/{gdt}/{rounding} base {base} step {step} {via}")


def _kinds_launched(asr, fn):
    """The library's kernel launches fn made, by kind (its launch counters)."""
    before = asr.asr_kernel_launches()
    fn()
    after = asr.asr_kernel_launches()
    return {k: after[k] - before[k] for k in after if after[k] != before[k]}


def test_launch_group_size_picks_the_kernel(asr):
    """Aligned tensors whose launch group moves at most 128 MiB take the
    register kernel's vector units, larger groups (the ballast the tests use
    included) the pipelined kernel; bf16 tensors at bases off a multiple of
    4 take the pipelined kernel at any size; a view one element into its
    storage is split into scalar units for its head and vector units for the
    rest."""
    import torch
    rng = np.random.default_rng(31)
    h = _make(rng, 65536, "bf16", "bf16")
    d = [dev(a) for a in h]
    assert _kinds_launched(asr, lambda: asr.asr_adamw_sr_step(*d, step=1, seed=0, **HP)) == {"adamw_vector": 1}
    assert _kinds_launched(asr, lambda: asr.asr_adamw_sr_multi_tensor(
        [(*d, 0), _ballast(d[0], d[1])], step=2, seed=0, **HP)) == {"adamw_pipelined": 1}
    assert _kinds_launched(asr, lambda: asr.asr_adamw_sr_step(*d, base_index=3, step=3, seed=0, **HP)) == \
        {"adamw_pipelined_any_base": 1}
    views = [t[1:] for t in d]                 # first common aligned element: 7; base 1 + 7 = 8
    assert _kinds_launched(asr, lambda: asr.asr_adamw_sr_step(*views, base_index=1, step=4, seed=0, **HP)) == \
        {"adamw_scalar": 1, "adamw_vector": 1}
    for pdt, gdt in (("f32", "f32"), ("bf16", "f32"), ("f32", "bf16")):
        p = torch.zeros(65536, dtype=torch.float32 if pdt == "f32" else torch.bfloat16, device="cuda")
        g = torch.zeros(65536, dtype=torch.float32 if gdt == "f32" else torch.bfloat16, device="cuda")
        m, v = torch.zeros(65536, device="cuda"), torch.zeros(65536, device="cuda")
        assert _kinds_launched(asr, lambda: asr.asr_adamw_sr_multi_tensor(
            [(p, g, m, v, 0), _ballast(p, g)], step=1, seed=0, **HP)) == {"adamw_pipelined": 1}, (pdt, gdt)
        # base 2: no bits drawn for f32 params; bf16 params need a multiple of 4
        base = 2 if pdt == "f32" else 4
        assert _kinds_launched(asr, lambda: asr.asr_adamw_sr_step(p, g, m, v, base_index=base, step=1, seed=0,
                                                                  **HP)) == {"adamw_vector": 1}, (pdt, gdt)
    torch.cuda.synchronize()


@pytest.mark.parametrize("off", [1, 2, 3])
@pytest.mark.parametrize("via", ["alone", "pipelined"])
def test_unaligned_buffers(asr, orc, off, via):
    """Buffers that start off a 16-byte boundary by the same element offset
    (slices) are split at the first element where all four are aligned: a
    scalar head, then the vector kernels (the register kernel alone, the
    pipelined kernel in a large launch group).  Bit-exact; nothing outside
    the slice is written."""
    import torch
    n = 4096 * 2 + 77
    rng = np.random.default_rng(off)
    h = _make(rng, n + off, "bf16", "bf16")
    full = [dev(a) for a in h]
    d = [t[off:] for t in full]
    hs = [a[off:].copy() for a in h]
    guard = [host(t)[:off].copy() for t in full]
    _step_both(asr, orc, hs, d, via=via, step=4, seed=3, base_index=10 + off, **HP)
    _check(hs, d, f"offset {off} {via}")
    for g0, t in zip(guard, full):
        assert np.array_equal(host(t)[:off], g0)
    torch.cuda.synchronize()


@pytest.mark.parametrize("pdt,gdt", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16"), ("f32", "f32")])
@pytest.mark.parametrize("offs", [(1, 1, 1, 1), (3, 3, 3, 3), (7, 7, 7, 7), (1, 3, 1, 1), (1, 1, 2, 2), (0, 0, 1, 1),
                                  (2, 2, 3, 3)])
@pytest.mark.parametrize("via", ["alone", "pipelined"])
def test_unaligned_views(asr, orc, pdt, gdt, offs, via):
    """p, g, m, v each a view some elements into its storage, in every dtype
    combination: where some element puts all four on a 16-byte boundary the
    tensor is split there (scalar head, vector rest: alone, or in a launch
    group large enough for the pipelined kernel), where none does it takes
    the plain kernel's scalar units -- either way bit-exact against the
    oracle, with guard words before and after every view untouched."""
    import torch
    rng = np.random.default_rng(sum(offs) + 7)
    n = 2 * 8192 + 45
    h = _make(rng, n, pdt, gdt)
    fulls, views = [], []
    for a, off in zip(h, offs):
        guard = np.full(off + 9, 0x7E, a.dtype)
        full = dev(np.concatenate([guard[:off], a, guard[off:]]))
        fulls.append((full, off))
        views.append(full[off:off + n])
    for base in (12, 13):
        _step_both(asr, orc, h, views, via=via, step=2, seed=8, base_index=base, **HP)
        _check(h, views, f"{pdt}/{gdt} offsets {offs} base {base} {via}")
    for full, off in fulls:
        t = host(full)
        assert np.all(t[:off] == 0x7E) and np.all(t[off + n:] == 0x7E), f"offsets {offs}: wrote outside the view"
    torch.cuda.synchronize()


# Edges of the pipelined kernel's tiles: 256 elements per consumer warp and
# unit, 3,072 to 8,192 elements by dtype combination (multiples of 1,024
# from 3,072 to 6,144 and 8,192 cover every shape in use or in the sweeps);
# one and two tiles, +-1.
TILE_EDGES = sorted({t * k + d for t in (3072, 4096, 5120, 6144, 8192) for k in (1, 2) for d in (-1, 0, 1)})


@pytest.mark.parametrize("pdt,gdt", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16"), ("f32", "f32")])
@pytest.mark.parametrize("via", ["alone", "pipelined"])
def test_small_and_boundary_sizes(asr, orc, pdt, gdt, via):
    """Sizes 0-33 and the pipelined kernel's tile edges, bases 0, 1 and 3,
    alone (the register kernel, or the pipelined one at bases off a
    multiple of 4 with bits drawn) and in a launch group large enough for
    the pipelined kernel; guard words after every buffer."""
    import torch
    rng = np.random.default_rng(11)
    sizes = list(range(0, 34)) if pdt == gdt == "bf16" else list(range(0, 34, 7))
    for n in sizes + TILE_EDGES:
        for base in (0, 1, 3):
            h = _make(rng, n, pdt, gdt)
            # guard bands after the buffers
            full = [dev(np.concatenate([a, np.full(9, 0x7E, a.dtype)])) for a in h]
            d = [t[:n] for t in full]
            _step_both(asr, orc, h, d, via=via, step=2, seed=5, base_index=base, **HP)
            _check(h, d, f"{pdt}/{gdt} n={n} base={base} {via}")
            for t, a in zip(full, h):
                assert np.all(host(t)[n:] == 0x7E), f"{pdt}/{gdt} n={n}: wrote past the end"
    torch.cuda.synchronize()


def test_special_values(asr, orc):
    """Inf/NaN/zero/denormal params and grads; tiny and huge moments.  NaN
    results compare as 'both NaN' (CPU and GPU NaN payloads differ)."""
    rng = np.random.default_rng(12)
    n = 4096 + 100
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-40, 3e38, -3e38, 1e-20], np.float32)
    for pdt in ("bf16", "f32"):
        p = W.normal_f32(rng, n, 1.0)
        g = W.normal_f32(rng, n, 1.0)
        p[rng.integers(0, n, 300)] = rng.choice(specials, 300)
        g[rng.integers(0, n, 300)] = rng.choice(specials, 300)
        m = W.normal_f32(rng, n, 1.0)
        v = np.abs(W.normal_f32(rng, n, 1.0))
        v[:50] = 0.0
        m[:50] = 0.0
        if pdt == "bf16":
            p = W.to_bf16_bits(p)
        for via in ("alone", "pipelined"):
            h = [a.copy() for a in (p, g, m, v)]
            d = [dev(a) for a in h]
            for eps in (1e-8, 0.0):
                _step_both(asr, orc, h, d, via=via, step=3, seed=8, lr=1e-2, beta1=0.9, beta2=0.999, eps=eps,
                           weight_decay=0.1)
                _check(h, d, f"specials {pdt} eps={eps} {via}")


def test_reproducible_and_keyed(asr):
    """Same (seed, step) -> identical step; another seed or step changes the
    bf16 params but not the moments."""
    import torch
    rng = np.random.default_rng(13)
    h = _make(rng, 100000, "bf16", "bf16")
    outs = {}
    for key in ((1, 1), (1, 1), (2, 1), (1, 2)):
        d = [dev(a) for a in h]
        asr.asr_adamw_sr_step(d[0], d[1], d[2], d[3], step=key[1], seed=key[0], **HP)
        outs.setdefault(key, []).append([host(t) for t in d])
    torch.cuda.synchronize()
    a, b = outs[(1, 1)]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert not np.array_equal(outs[(2, 1)][0][0], a[0])
    assert np.array_equal(outs[(2, 1)][0][2], a[2])
    assert not np.array_equal(outs[(1, 2)][0][0], a[0])


def test_checkpoint_resume(asr):
    """10 steps straight == 5 steps, copy every buffer to the host and back,
    5 more steps (the generator is stateless, keyed by seed and step)."""
    rng = np.random.default_rng(14)
    n = 50000
    h = _make(rng, n, "bf16", "bf16", states=False)
    grads = [W.to_bf16_bits(W.normal_f32(rng, n, 1e-3)) for _ in range(10)]
    a = [dev(x) for x in h]
    for t in range(1, 11):
        asr.asr_adamw_sr_step(a[0], dev(grads[t - 1]), a[2], a[3], step=t, seed=21, **HP)
    b = [dev(x) for x in h]
    for t in range(1, 6):
        asr.asr_adamw_sr_step(b[0], dev(grads[t - 1]), b[2], b[3], step=t, seed=21, **HP)
    saved = [host(x) for x in b]
    b = [dev(x) for x in saved]
    for t in range(6, 11):
        asr.asr_adamw_sr_step(b[0], dev(grads[t - 1]), b[2], b[3], step=t, seed=21, **HP)
    for x, y in zip(a, b):
        if x is not None:
            assert np.array_equal(host(x), host(y))


def test_runs_on_the_given_stream(asr, orc):
    import torch
    rng = np.random.default_rng(15)
    h = _make(rng, 1 << 20, "bf16", "bf16")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = [dev(a) for a in h]
        asr.asr_adamw_sr_step(d[0], d[1], d[2], d[3], step=1, seed=1, **HP)
    s.synchronize()
    orc.adamw_step(h[0], h[1], h[2], h[3], step=1, seed=1, **HP)
    _check(h, d, "side stream")


def test_fp32_params_16m_100_steps(asr, orc):
    """One f32 tensor of 16,777,216 elements ~N(0,0.02), f32 grads ~N(0,1e-3)
    fresh per step, f32 moments, 100 steps: bit-exact with the oracle, and
    within the page's 1e-4 of torch.optim.AdamW run on the same grads."""
    import torch
    n, steps = 16_777_216, 100
    gen = torch.Generator(device="cuda")
    gen.manual_seed(20240)
    p = W.device_normal_(torch.empty(n, device="cuda"), gen, 0.02)
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    hp_ = host(p)
    hm = np.zeros(n, np.float32)
    hv = np.zeros(n, np.float32)
    tp = torch.nn.Parameter(p.clone())
    opt = torch.optim.AdamW([tp], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"], foreach=False, fused=False)
    g = torch.empty(n, device="cuda")
    for step in range(1, steps + 1):
        W.device_normal_(g, gen, 1e-3)
        asr.asr_adamw_sr_step(p, g, m, v, step=step, seed=0, **HP)
        tp.grad = g.clone()
        opt.step()
        orc.adamw_step(hp_, host(g), hm, hv, step=step, seed=0, **HP)
        if step in (1, 2, 50, 100):
            assert_same_bits(host(p), hp_, f"f32 p step {step}")
            assert_same_bits(host(m), hm, f"f32 m step {step}")
            assert_same_bits(host(v), hv, f"f32 v step {step}")
    diff = float((p.double() - tp.detach().double()).abs().max())
    assert diff < 1e-4, f"max |p - torch AdamW| = {diff}"


@pytest.mark.parametrize("states", ["zero", "random"])
def test_shard_invariance_268m(asr, orc, states):
    """268,435,456 bf16 params ~U(-1,1), bf16 grads ~N(0,1e-2), seed 1234,
    step 7: the whole tensor and 8 contiguous shards with their base_index
    give bitwise-equal results; sampled windows match the oracle."""
    import torch
    n, shards = 268_435_456, 8
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    p0 = W.device_uniform_(torch.empty(n, dtype=torch.bfloat16, device="cuda"), gen, -1.0, 1.0)
    g = W.device_normal_(torch.empty(n, dtype=torch.bfloat16, device="cuda"), gen, 1e-2)
    if states == "zero":
        m0 = torch.zeros(n, device="cuda")
        v0 = torch.zeros(n, device="cuda")
    else:
        m0 = W.device_normal_(torch.empty(n, device="cuda"), gen, 1e-3)
        v0 = W.device_normal_(torch.empty(n, device="cuda"), gen, 1e-4).abs_()
    rng = np.random.default_rng(7)
    win = [(0, 4096), (n - 4096, 4096)] + [(int(s), 4096) for s in rng.integers(0, n - 4096, 14)]
    before = [(host(p0[s:s + L]), host(g[s:s + L]), host(m0[s:s + L]), host(v0[s:s + L])) for s, L in win]
    pw, mw, vw = p0.clone(), m0.clone(), v0.clone()
    asr.asr_adamw_sr_step(pw, g, mw, vw, step=7, seed=1234, **HP)
    ps, ms, vs = p0.clone(), m0.clone(), v0.clone()
    L = n // shards
    for k in range(shards):
        sl = slice(k * L, (k + 1) * L)
        asr.asr_adamw_sr_step(ps[sl], g[sl], ms[sl], vs[sl], base_index=k * L, step=7, seed=1234, **HP)
    torch.cuda.synchronize()
    assert torch.equal(pw.view(torch.int16), ps.view(torch.int16))
    assert torch.equal(mw.view(torch.int32), ms.view(torch.int32))
    assert torch.equal(vw.view(torch.int32), vs.view(torch.int32))
    for (s, Ln), (hp0, hg, hm, hv) in zip(win, before):
        orc.adamw_step(hp0, hg, hm, hv, step=7, seed=1234, base_index=s, **HP)
        assert_same_bits(host(pw[s:s + Ln]), hp0, f"window {s} p")
        assert_same_bits(host(mw[s:s + Ln]), hm, f"window {s} m")
        assert_same_bits(host(vw[s:s + Ln]), hv, f"window {s} v")


def test_no_device_error_after_steps(asr):
    """Ordinary steps never trip a pipeline wait limit."""
    rng = np.random.default_rng(16)
    h = _make(rng, 3 * 4096 * 152 + 5, "bf16", "bf16")
    d = [dev(a) for a in h]
    asr.asr_take_device_error()
    for step in (1, 2, 3):
        asr.asr_adamw_sr_step(d[0], d[1], d[2], d[3], step=step, seed=1, **HP)
    assert asr.asr_take_device_error() == 0


def test_bounded_wait_gives_up_with_a_status(asr):
    """A wait on a barrier nothing arrives on ends after its limit (1 ms) and
    reports bit 0; the context stays usable (a step still runs afterwards)."""
    import time
    asr.asr_take_device_error()
    t0 = time.perf_counter()
    asr.asr_selftest_wait_timeout(1_000_000)
    bits = asr.asr_take_device_error()
    assert bits == 1
    assert time.perf_counter() - t0 < 10.0
    assert asr.asr_take_device_error() == 0
    rng = np.random.default_rng(17)
    h = _make(rng, 5000, "bf16", "bf16")
    d = [dev(a) for a in h]
    asr.asr_adamw_sr_step(d[0], d[1], d[2], d[3], step=1, seed=1, **HP)
    assert asr.asr_take_device_error() == 0


def test_concurrent_blocking_takes_see_each_bit_once(asr):
    """Blocking takes from several host threads at once, each on its own
    stream: after one raised bit, exactly one of the takes of a round reports
    it and the others report 0 -- none reads another call's copy of the
    word.  Two hundred rounds of four threads released together."""
    import threading

    import torch
    asr.asr_take_device_error()
    threads_n, rounds = 4, 200
    streams = [torch.cuda.Stream() for _ in range(threads_n)]
    barrier = threading.Barrier(threads_n + 1)
    results = [[0] * rounds for _ in range(threads_n)]
    failures = []

    def worker(i):
        try:
            for r in range(rounds):
                barrier.wait()
                results[i][r] = asr.asr_take_device_error(stream=streams[i])
                barrier.wait()
        except Exception as exc:          # reported by the main thread
            failures.append(exc)
            barrier.abort()

    workers = [threading.Thread(target=worker, args=(i,)) for i in range(threads_n)]
    for w in workers:
        w.start()
    try:
        for r in range(rounds):
            asr.asr_selftest_wait_timeout(20_000)
            torch.cuda.synchronize()
            barrier.wait()
            barrier.wait()
    finally:
        for w in workers:
            w.join(timeout=60)
    assert not failures, failures
    for r in range(rounds):
        got = [results[i][r] for i in range(threads_n)]
        assert sorted(got) == [0] * (threads_n - 1) + [1], (r, got)
    assert asr.asr_take_device_error() == 0


def test_error_bits_taken_without_waiting(asr):
    """asr_take_device_error_async: after a wait that gave up (the self-test)
    the bits land in page-locked host memory, or in device memory, once the
    stream gets there, and the word is clear afterwards.  Memory the GPU
    cannot write (pageable host memory, NULL, misaligned) is refused before
    anything is launched."""
    import ctypes
    import torch
    from stochastic_rounding_gb300 import _lib
    asr.asr_take_device_error()
    for target in ("pinned", "cuda"):
        word = (torch.full((1,), -1, dtype=torch.int32, pin_memory=True) if target == "pinned"
                else torch.full((1,), -1, dtype=torch.int32, device="cuda"))
        asr.asr_selftest_wait_timeout(1_000_000)
        asr.asr_take_device_error_async(word)
        torch.cuda.synchronize()
        assert int(word.item()) == 1, target
        asr.asr_take_device_error_async(word)
        torch.cuda.synchronize()
        assert int(word.item()) == 0, target
    assert asr.asr_take_device_error() == 0
    L = _lib.lib()
    pageable = np.zeros(4, np.uint32)
    sh = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.asr_take_device_error_async(ctypes.c_void_p(pageable.ctypes.data), sh) == _lib.ASR_ERR_INVALID_VALUE
    assert L.asr_take_device_error_async(None, sh) == _lib.ASR_ERR_INVALID_VALUE
    pinned = torch.zeros(4, dtype=torch.int32, pin_memory=True)
    assert L.asr_take_device_error_async(ctypes.c_void_p(pinned.data_ptr() + 2), sh) == _lib.ASR_ERR_INVALID_VALUE
    with pytest.raises(ValueError):
        asr.asr_take_device_error_async(torch.zeros(1, dtype=torch.int32))
    torch.cuda.synchronize()


@pytest.mark.parametrize("pdt,gdt,n,steps", [("bf16", "bf16", 48_000_000 + 4096 * 3 + 8, 24),
                                             ("f32", "f32", 16_777_216, 40),
                                             ("bf16", "f32", 20_000_000, 16)])
def test_pipeline_matches_plain_path_every_step(asr, pdt, gdt, n, steps):
    """Race check for the bulk-copy pipeline: the same inputs updated through
    the pipelined kernel (16-byte-aligned buffers) and through the plain
    kernel (the same data with params and grads one element and the moments
    two elements off alignment: no element where all four buffers are
    aligned, so no part of it can take the pipelined kernel) with equal
    global indices must agree bit for bit after every step."""
    import torch
    gen = torch.Generator(device="cuda")
    gen.manual_seed(n + steps)
    pt = torch.bfloat16 if pdt == "bf16" else torch.float32
    gt = torch.bfloat16 if gdt == "bf16" else torch.float32

    def pair(dtype, fill, shift):
        a = torch.empty(n, dtype=dtype, device="cuda")
        fill(a)
        b_full = torch.empty(n + shift, dtype=dtype, device="cuda")
        b = b_full[shift:]
        b.copy_(a)
        return a, b

    pa, pb = pair(pt, lambda t: W.device_normal_(t, gen, 0.02), 1)
    ma, mb = pair(torch.float32, lambda t: W.device_normal_(t, gen, 1e-4), 2)
    va, vb = pair(torch.float32, lambda t: W.device_normal_(t, gen, 1e-6).abs_(), 2)
    ga, gb = pair(gt, lambda t: W.device_normal_(t, gen, 1e-3), 1)
    assert pa.data_ptr() % 16 == 0 and pb.data_ptr() % 16 != 0
    # no h < 8 puts all four of the shifted buffers on a 16-byte boundary
    sizes = [pb.element_size(), gb.element_size(), 4, 4]
    assert not any(all((t.data_ptr() + h * sz) % 16 == 0 for t, sz in zip((pb, gb, mb, vb), sizes))
                   for h in range(8))
    asr.asr_take_device_error()
    for step in range(1, steps + 1):
        W.device_normal_(ga, gen, 1e-3)
        gb.copy_(ga)
        asr.asr_adamw_sr_step(pa, ga, ma, va, base_index=4096, step=step, seed=11, **HP)
        asr.asr_adamw_sr_step(pb, gb, mb, vb, base_index=4096, step=step, seed=11, **HP)
        iv = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)  # noqa: E731
        assert torch.equal(iv(pa), iv(pb)), f"params differ at step {step}"
        assert torch.equal(ma.view(torch.int32), mb.view(torch.int32)), f"m differs at step {step}"
        assert torch.equal(va.view(torch.int32), vb.view(torch.int32)), f"v differs at step {step}"
    assert asr.asr_take_device_error() == 0


@pytest.mark.parametrize("case", [
    dict(lr=0.0, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, step=5, seed=1),
    dict(lr=1e-3, beta1=0.0, beta2=0.0, eps=1e-8, weight_decay=0.01, step=3, seed=2),
    dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step=1, seed=3),
    dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=2 ** 32 - 1, seed=4),
    dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=7, seed=2 ** 64 - 1),
], ids=["lr0", "betas0", "wd0", "step_max", "seed_max"])
def test_degenerate_hyperparameters(asr, orc, case):
    """The corners of the accepted hyperparameters, on every vector kernel
    (base 0 alone: the register kernel; base 0 in a large launch group and
    base 3: the pipelined kernel, two and three counters per unit) with a
    ragged length, bit-exact against the oracle.  With
    lr = 0 the update is p * 1 - 0, so bf16 parameters come back unchanged
    under stochastic rounding (an exactly representable value has no bits to
    round) while the moments still move."""
    rng = np.random.default_rng(21)
    n = 3 * 5120 + 13
    for base, via in ((0, "alone"), (0, "pipelined"), (3, "alone")):
        h = _make(rng, n, "bf16", "bf16")
        p0, m0 = h[0].copy(), h[2].copy()
        d = [dev(a) for a in h]
        _step_both(asr, orc, h, d, via=via, base_index=base, **case)
        _check(h, d, f"{case} base={base} {via}")
        if case["lr"] == 0.0:
            assert np.array_equal(host(d[0]), p0), "lr = 0 changed a bf16 parameter"
            assert not np.array_equal(host(d[2]), m0), "lr = 0 must still update the first moment"
