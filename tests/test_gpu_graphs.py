"""The entry points captured into a CUDA graph (after one ordinary call has
set up their per-device caches) and replayed give the same bits as direct
calls: the multi-tensor step on all three of its kernel paths, the
stand-alone rounding and Philox ops, and the tensor-core GEMM.  Nothing on
these paths allocates, synchronises the host or keeps state between
launches, so a captured launch is the launch."""
import numpy as np
import pytest

from gpu_util import dev, torch_cuda
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


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype in (torch.bfloat16, torch.int16) else t.view(torch.int32)


def _tensor_set(seed, large=False):
    """Mixed tensors: aligned with bases that are multiples of 4 (the
    register kernel's vector units while their launch group is small, the
    pipelined kernel with `large`, which adds an 8M-param tensor to each such
    group), aligned with other bases (pipelined, three counters per unit),
    one element off a 16-byte boundary (scalar head, then vector units)."""
    rng = np.random.default_rng(seed)
    out, base = [], 0
    if large:
        for pdt in ("bf16", "f32"):
            n = 8_000_000
            p = np.zeros(n, np.uint16 if pdt == "bf16" else np.float32)
            out.append(([p, np.zeros(n, np.uint16), np.zeros(n, np.float32), np.zeros(n, np.float32)], 0, base))
            base += n
    for i in range(24):
        n = int(rng.integers(1, 30000))
        off = 1 if i % 5 == 4 else 0
        pdt = "bf16" if i % 3 else "f32"
        p = W.normal_f32(rng, n + off, 0.02)
        p = W.to_bf16_bits(p) if pdt == "bf16" else p
        g = W.to_bf16_bits(W.normal_f32(rng, n + off, 1e-3))
        m = W.normal_f32(rng, n + off, 1e-4)
        v = np.abs(W.normal_f32(rng, n + off, 1e-6))
        out.append(([p, g, m, v], off, base))
        base += n + int(rng.integers(0, 3))
    return out


def _device(hs):
    return [tuple(dev(a)[off:] for a in arrs) + (base,) for arrs, off, base in hs]


@pytest.mark.parametrize("large", [False, True], ids=["small-groups", "large-groups"])
def test_multi_tensor_step_in_a_graph(asr, large):
    import torch
    hs = _tensor_set(3, large)
    a, b = _device(hs), _device(hs)
    assert any(base % 4 for *_, base in a) and any(t[0].data_ptr() % 16 for t in a)
    for ts in (a, b):                          # first, ordinary call: sets up the caches
        asr.asr_adamw_sr_multi_tensor(ts, step=1, seed=7, **HP)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        asr.asr_adamw_sr_multi_tensor(a, step=2, seed=7, **HP)
        asr.asr_adamw_sr_multi_tensor(a, step=3, seed=7, **HP)
    graph.replay()
    for step in (2, 3):
        asr.asr_adamw_sr_multi_tensor(b, step=step, seed=7, **HP)
    torch.cuda.synchronize()
    for i, (x, y) in enumerate(zip(a, b)):
        for k in (0, 2, 3):
            assert torch.equal(_bits(x[k]), _bits(y[k])), f"tensor {i} buffer {k}"
    assert asr.asr_take_device_error() == 0


def test_rounding_philox_and_gemm_in_a_graph(asr):
    import torch
    n = (1 << 20) + 5
    x = torch.randn(n, device="cuda")
    out_g, out_d = (torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(2))
    w_g, w_d = (torch.empty(4 * 4097, dtype=torch.int32, device="cuda") for _ in range(2))
    a = torch.randn(512, 256, device="cuda").to(torch.bfloat16)
    bm = torch.randn(384, 256, device="cuda").to(torch.bfloat16)
    c_g, c_d = (torch.empty(512, 384, dtype=torch.bfloat16, device="cuda") for _ in range(2))
    calls = [lambda o: asr.asr_stochastic_round_bf16(x, o, base_index=6, step=3, seed=5),
             lambda o: asr.asr_philox4x32(o, 4097, 2 ** 32 - 9, 4, 1, 77),
             lambda o: asr.asr_gemm_bf16_sr(a, bm, o, step=2, seed=9)]
    for f, o in zip(calls, (out_d, w_d, c_d)):
        f(o)                                   # ordinary calls: set-up and the reference results
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for f, o in zip(calls, (out_g, w_g, c_g)):
            f(o)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_d)
    assert torch.equal(w_g, w_d)
    assert torch.equal(_bits(c_g), _bits(c_d))
    assert asr.asr_take_device_error() == 0


_FIRST_USE = r"""
import sys, torch
sys.path.insert(0, ".")
import stochastic_rounding_gb300 as asr
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
dev = torch.device("cuda", 0)
def mk(n, pdt, gdt):
    g = torch.Generator(device=dev); g.manual_seed(n)
    return ((torch.randn(n, device=dev, generator=g) * 0.02).to(pdt), (torch.randn(n, device=dev, generator=g) * 1e-3).to(gdt),
            torch.zeros(n, device=dev), torch.zeros(n, device=dev))
small = mk(5000, torch.bfloat16, torch.bfloat16)
asr.asr_adamw_sr_step(*small, step=1, seed=3, **HP)          # the only call before the capture
big = [mk(7_000_000, torch.float32, torch.float32), mk(6_000_000, torch.bfloat16, torch.float32)]
twin = [tuple(t.clone() for t in b) for b in big]
s = torch.cuda.Stream(); s.wait_stream(torch.cuda.current_stream())
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph, stream=s):
    asr.asr_adamw_sr_step(*big[0], step=2, seed=3, **HP)
    asr.asr_adamw_sr_multi_tensor([(*big[1], 5)], step=2, seed=3, **HP)
graph.replay()
asr.asr_adamw_sr_step(*twin[0], step=2, seed=3, **HP)
asr.asr_adamw_sr_multi_tensor([(*twin[1], 5)], step=2, seed=3, **HP)
torch.cuda.synchronize()
bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)
for b, w in zip(big, twin):
    for k in (0, 2, 3):
        assert torch.equal(bits(b[k]), bits(w[k]))
assert asr.asr_take_device_error() == 0
print("FIRST_USE_OK")
"""


def test_capture_of_kernels_not_used_before(asr):
    """In a fresh process, after one small bf16 step only, a capture holds
    steps that take kernels no earlier call used (the f32 pipelined kernel,
    the bf16/f32 kernel drawing three counters per unit): the first step on
    a device sets up every AdamW kernel, so nothing is set up inside the
    capture, and the replay gives the bits of direct calls."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_USE], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0 and "FIRST_USE_OK" in r.stdout, r.stderr[-3000:]
