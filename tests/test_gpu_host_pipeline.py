"""GPU parity of asr_adamw_sr_multi_tensor_host: gradients copied in from
page-locked host memory, the multi-tensor step, parameters copied back out,
pipelined over chunks and streams in the library -- bitwise the oracle's
step on every element, on the device and in the host copies."""
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


def _pinned(a):
    """A page-locked CPU tensor holding numpy array a (bf16 patterns as int16)."""
    import torch
    src = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    t = torch.empty(src.shape, dtype=src.dtype, pin_memory=True)
    t.copy_(src)
    return t


def _set(seed, count=30):
    """Host arrays and device / host tensors of `count` tensors: mixed
    dtypes, sizes up to ~20k (one of 40k, above the chunk size the tests
    use), a few device buffers off a 16-byte boundary, a few tensors whose
    params stay on the device (param_host None), bases end to end."""
    rng = np.random.default_rng(seed)
    out, base = [], 3
    for i in range(count):
        n = 40_000 if i == 7 else int(rng.integers(0, 20_000))
        pdt = "bf16" if i % 3 else "f32"
        gdt = "bf16" if i % 4 else "f32"
        off = 1 if i % 6 == 5 else 0
        p = W.normal_f32(rng, n + off, 0.02)
        g = W.normal_f32(rng, n, 1e-3)
        p = W.to_bf16_bits(p) if pdt == "bf16" else p
        g = W.to_bf16_bits(g) if gdt == "bf16" else g
        m = W.normal_f32(rng, n + off, 1e-4)
        v = np.abs(W.normal_f32(rng, n + off, 1e-6))
        d = [dev(p)[off:], None, dev(m)[off:], dev(v)[off:]]
        d[1] = dev(np.zeros(n + off, g.dtype))[off:]            # device gradient buffer, filled by the copy
        keep = i % 5 != 4
        ph = _pinned(np.zeros(n, p.dtype)) if keep else None
        out.append(dict(h=[p[off:].copy(), g, m[off:].copy(), v[off:].copy()], d=d, base=base,
                        gh=_pinned(g), ph=ph))
        base += n
    return out


def _rows(ts):
    return [(t["d"][0], t["d"][1], t["d"][2], t["d"][3], t["base"], t["gh"], t["ph"]) for t in ts]


@pytest.mark.parametrize("streams,chunk", [("three", 7_000), ("one", 7_000), ("three", 1), ("three", 0)])
def test_host_step_matches_the_oracle(asr, orc, streams, chunk):
    """Chunks of ~7,000 params (one tensor is larger than that), of one
    tensor each (chunk_elems 1), and all in one (0: the default 2^28)."""
    import torch
    ts = _set(41)
    s = torch.cuda.Stream()
    cin, cout = (torch.cuda.Stream(), torch.cuda.Stream()) if streams == "three" else (None, None)
    table = asr.make_host_table(_rows(ts))
    for step in (1, 2):
        for t in ts:                                   # new grads in the host buffers
            rng = np.random.default_rng(step * 1000 + t["base"])
            g = W.normal_f32(rng, t["h"][1].size, 1e-3)
            g = W.to_bf16_bits(g) if t["h"][1].dtype == np.uint16 else g
            t["h"][1] = g
            t["gh"].copy_(torch.from_numpy(g.view(np.int16) if g.dtype == np.uint16 else g))
        asr.asr_adamw_sr_multi_tensor_host(table, step=step, seed=2**34 + 1, chunk_elems=chunk, stream=s,
                                           copy_in=cin, copy_out=cout, device="cuda", **HP)
        torch.cuda.synchronize()                       # the copies out complete on copy_out
        for t in ts:
            p, g, m, v = t["h"]
            orc.adamw_step(p, g, m, v, step=step, seed=2**34 + 1, base_index=t["base"], **HP)
        for i, t in enumerate(ts):
            for k, name in ((0, "p"), (2, "m"), (3, "v")):
                assert_same_bits(host(t["d"][k]), t["h"][k], f"tensor {i} {name} step {step}")
            if t["ph"] is not None:
                got = t["ph"].numpy()
                assert_same_bits(got.view(np.uint16) if got.dtype == np.int16 else got, t["h"][0],
                                 f"tensor {i} host params step {step}")
    assert asr.asr_take_device_error() == 0


def test_host_step_orders_against_the_stream(asr):
    """Work queued on `stream` before the call is seen by it (the device
    params it steps are set by a fill queued just before), work queued on
    `stream` after it sees the stepped params (a copy queued right after),
    and once copy_out has been waited on the host holds the same values.
    Two calls back to back on the same buffers (the second's steps follow
    the first's copies out) give the host the second step's params."""
    import torch
    n = 300_000
    s = torch.cuda.Stream()
    p = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    g = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    m, v = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    gh = torch.full((n,), 1e-3, dtype=torch.bfloat16, pin_memory=True)
    ph = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    after = torch.empty_like(p)
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s):
        p.fill_(0.5)
        asr.asr_adamw_sr_multi_tensor_host([(p, g, m, v, 0, gh, ph)], step=1, seed=5, chunk_elems=50_000,
                                           stream=s, copy_in=cin, copy_out=cout, **HP)
        after.copy_(p)
    s.synchronize()
    assert float(after.float().mean()) < 0.5              # the step moved the params down from 0.5
    assert torch.equal(g.cpu().view(torch.int16), gh.view(torch.int16))
    cout.synchronize()
    assert torch.equal(ph.view(torch.int16), after.cpu().view(torch.int16))
    table = asr.make_host_table([(p, g, m, v, 0, gh, ph)])
    for step in (2, 3):
        asr.asr_adamw_sr_multi_tensor_host(table, step=step, seed=5, chunk_elems=50_000, stream=s, copy_in=cin,
                                           copy_out=cout, device="cuda", **HP)
    with torch.cuda.stream(s):
        after.copy_(p)
    torch.cuda.synchronize()
    assert torch.equal(ph.view(torch.int16), after.cpu().view(torch.int16))


def test_host_step_refuses_pageable_memory(asr):
    """Pageable host memory is refused before anything is queued: no kernel
    launched, the device buffers untouched."""
    import torch
    from stochastic_rounding_gb300 import _lib
    n = 4096
    p = torch.full((n,), 0.25, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    m, v = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    gh = torch.zeros(n, dtype=torch.bfloat16)                 # pageable
    before = asr.asr_kernel_launches()
    with pytest.raises(_lib.AsrError) as e:
        asr.asr_adamw_sr_multi_tensor_host([(p, g, m, v, 0, gh, None)], step=1, seed=0, **HP)
    assert e.value.status == _lib.ASR_ERR_INVALID_VALUE
    assert asr.asr_kernel_launches() == before
    torch.cuda.synchronize()
    assert bool((p.float() == 0.25).all())


def test_host_step_on_flat_buffers(asr, orc):
    """Tensors laid end to end in flat host and device buffers (copies of a
    run of them go out together), with one gap on the device side only and
    one on the host side only (where a run must break), bf16 params and
    grads: bitwise the oracle after two steps, on the device and in the host
    copies, and the gap words untouched on both sides."""
    import torch
    rng = np.random.default_rng(77)
    sizes = [4096, 1000, 333, 70_000, 8, 12_345, 4096, 2048, 999, 50_000, 16, 3]
    dev_gap_after, host_gap_after = 4, 7          # tensor index followed by a 64-element gap
    d_off, h_off, d, h = [], [], 0, 0
    for i, n in enumerate(sizes):
        d_off.append(d)
        h_off.append(h)
        d += n + (64 if i == dev_gap_after else 0)
        h += n + (64 if i == host_gap_after else 0)
    p = W.to_bf16_bits(W.normal_f32(rng, d, 0.02))
    m = W.normal_f32(rng, d, 1e-4)
    v = np.abs(W.normal_f32(rng, d, 1e-6))
    p_d, m_d, v_d = dev(p), dev(m), dev(v)
    g_d = dev(np.full(d, 0x7E7E, np.uint16))
    g_h = torch.empty(h, dtype=torch.int16, pin_memory=True)
    p_h = torch.full((h,), 0x5A5A, dtype=torch.int16, pin_memory=True)
    rows, base = [], 0
    for n, a, b in zip(sizes, d_off, h_off):
        rows.append((p_d[a:a + n], g_d[a:a + n], m_d[a:a + n], v_d[a:a + n], base, g_h[b:b + n], p_h[b:b + n]))
        base += n
    table = asr.make_host_table(rows)
    s, cin, cout = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    hp = [p.copy(), None, m.copy(), v.copy()]
    for step in (1, 2):
        g = W.to_bf16_bits(W.normal_f32(rng, h, 1e-3))
        g_h.copy_(torch.from_numpy(g.view(np.int16)))
        asr.asr_adamw_sr_multi_tensor_host(table, step=step, seed=9, chunk_elems=60_000, stream=s, copy_in=cin,
                                           copy_out=cout, device="cuda", **HP)
        torch.cuda.synchronize()
        base = 0
        for n, a, b in zip(sizes, d_off, h_off):
            pp, mm, vv = hp[0][a:a + n].copy(), hp[2][a:a + n].copy(), hp[3][a:a + n].copy()
            orc.adamw_step(pp, g[b:b + n].copy(), mm, vv, step=step, seed=9, base_index=base, **HP)
            hp[0][a:a + n], hp[2][a:a + n], hp[3][a:a + n] = pp, mm, vv
            base += n
        got_p = host(p_d)
        for i, (n, a, b) in enumerate(zip(sizes, d_off, h_off)):
            assert_same_bits(got_p[a:a + n], hp[0][a:a + n], f"tensor {i} p step {step}")
            assert_same_bits(host(m_d)[a:a + n], hp[2][a:a + n], f"tensor {i} m step {step}")
            assert_same_bits(host(v_d)[a:a + n], hp[3][a:a + n], f"tensor {i} v step {step}")
            assert np.array_equal(p_h.numpy()[b:b + n].view(np.uint16), hp[0][a:a + n]), f"tensor {i} host p"
    gap_d = d_off[dev_gap_after] + sizes[dev_gap_after]
    gap_h = h_off[host_gap_after] + sizes[host_gap_after]
    assert np.all(host(g_d)[gap_d:gap_d + 64] == 0x7E7E), "device gap written"
    assert np.all(p_h.numpy()[gap_h:gap_h + 64].view(np.uint16) == 0x5A5A), "host gap written"


def test_host_step_with_more_chunks_than_the_event_pool_keeps(asr, orc):
    """2,100 tensors of 1-9 params, one chunk each (4,202 events in one call,
    above the 4,096 the pool keeps): bitwise the oracle after two calls."""
    import torch
    rng = np.random.default_rng(5)
    rows, hosts, base = [], [], 0
    for i in range(2100):
        n = int(rng.integers(1, 10))
        p = W.to_bf16_bits(W.normal_f32(rng, n, 0.02))
        m = W.normal_f32(rng, n, 1e-4)
        v = np.abs(W.normal_f32(rng, n, 1e-6))
        d = (dev(p), dev(np.zeros(n, np.uint16)), dev(m), dev(v))
        gh = torch.empty(n, dtype=torch.int16, pin_memory=True)
        ph = torch.empty(n, dtype=torch.int16, pin_memory=True)
        rows.append((*d, base, gh, ph))
        hosts.append([p.copy(), None, m.copy(), v.copy(), base])
        base += n
    table = asr.make_host_table(rows)
    s, cin, cout = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    for step in (1, 2):
        for r, h in zip(rows, hosts):
            g = W.to_bf16_bits(W.normal_f32(rng, h[0].size, 1e-3))
            h[1] = g
            r[5].copy_(torch.from_numpy(g.view(np.int16)))
        asr.asr_adamw_sr_multi_tensor_host(table, step=step, seed=3, chunk_elems=1, stream=s, copy_in=cin,
                                           copy_out=cout, device="cuda", **HP)
        torch.cuda.synchronize()
        for h in hosts:
            orc.adamw_step(h[0], h[1], h[2], h[3], step=step, seed=3, base_index=h[4], **HP)
    for i, (r, h) in enumerate(zip(rows, hosts)):
        assert np.array_equal(host(r[0]), h[0]), f"tensor {i} p"
        assert np.array_equal(r[6].numpy().view(np.uint16), h[0]), f"tensor {i} host p"
        assert np.array_equal(host(r[2]).view(np.uint32), h[2].view(np.uint32)), f"tensor {i} m"
    assert asr.asr_take_device_error() == 0
