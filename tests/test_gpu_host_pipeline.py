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


@pytest.mark.parametrize("streams", ["three", "one"])
def test_host_step_matches_the_oracle(asr, orc, streams):
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
        asr.asr_adamw_sr_multi_tensor_host(table, step=step, seed=2**34 + 1, chunk_elems=7_000, stream=s,
                                           copy_in=cin, copy_out=cout, device="cuda", **HP)
        s.synchronize()
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
    params it steps are set by a fill queued just before), and work queued
    after it sees its results (a copy of the params queued right after on
    `stream` holds the stepped values, equal to what went to the host)."""
    import torch
    n = 300_000
    s = torch.cuda.Stream()
    p = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    g = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    m, v = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    gh = torch.full((n,), 1e-3, dtype=torch.bfloat16, pin_memory=True)
    ph = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    after = torch.empty_like(p)
    with torch.cuda.stream(s):
        p.fill_(0.5)
        asr.asr_adamw_sr_multi_tensor_host([(p, g, m, v, 0, gh, ph)], step=1, seed=5, chunk_elems=50_000,
                                           stream=s, copy_in=torch.cuda.Stream(), copy_out=torch.cuda.Stream(),
                                           **HP)
        after.copy_(p)
    s.synchronize()
    assert torch.equal(after.view(torch.int16), p.view(torch.int16))
    assert torch.equal(ph.view(torch.int16), after.cpu().view(torch.int16))
    assert float(after.float().mean()) < 0.5              # the step moved the params down from 0.5
    assert torch.equal(g.cpu().view(torch.int16), gh.view(torch.int16))


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
