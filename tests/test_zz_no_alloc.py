"""The allocation-free multi-tensor entry point.

Some callers cannot allocate device memory themselves: their framework's
allocator owns the device (a raw cudaMalloc would fail in a memory-capped job
or escape the allocator's accounting), or they must not pay for an
allocation inside a step.  asr_adamw_sr_multi_tensor_static serves them: its
scratch, the tensor descriptor table the kernel walks, sits in a
library-owned static device array.  These tests check, through the C ABI
and through the Python wrapper, that two calls in a row give bit for bit the
results of the regular multi-tensor entry point and of the oracle -- also
with a table of exactly the maximum size, every dtype group present -- and
that a table above the maximum is refused.

Kept in a file of its own that is collected last, so a failure here cannot
stop a run with -x before the other tests have run.
"""
import ctypes

import numpy as np
import pytest

from gpu_util import assert_same_bits, dev, host, torch_cuda
from stochastic_rounding_gb300 import workloads as W

pytestmark = pytest.mark.gpu
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@pytest.fixture(scope="module")
def L():
    torch_cuda()
    from stochastic_rounding_gb300 import build
    build.build()
    from stochastic_rounding_gb300 import _lib
    return _lib.lib()


def _tensor_set(seed):
    """About 700 tensors, more than one launch's parameter table holds:
    mixed dtypes, sizes from 1 to ~2M elements, a few starting off a
    16-byte boundary.  Returns (p, g, m, v, base) tuples of CUDA tensors."""
    import torch
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    out, base = [], 0
    sizes = [int(x) for x in rng.integers(1, 3000, 690)] + [2_000_003, 1 << 20, 65536 + 5, 4096, 7]
    for i, n in enumerate(sizes):
        pdt = torch.bfloat16 if rng.random() < 0.7 else torch.float32
        gdt = torch.bfloat16 if rng.random() < 0.6 else torch.float32
        off = 1 if i % 97 == 5 else 0

        def mk(dtype, std):
            return torch.randn(n + off, device="cuda", generator=gen).mul_(std).to(dtype)[off:]
        out.append((mk(pdt, 0.02), mk(gdt, 1e-3), mk(torch.float32, 1e-4),
                    mk(torch.float32, 1e-6).abs_(), base))
        base += n + int(rng.integers(0, 3))
    return out


def _clone(tensors):
    """Copies of params and moments at the same 16-byte alignment offset."""
    import torch

    def cp(t):
        off = (t.data_ptr() % 16) // t.element_size()
        full = torch.empty(t.numel() + off, dtype=t.dtype, device=t.device)
        full[off:].copy_(t)
        return full[off:]
    return [(cp(p), g, cp(m), cp(v), base) for p, g, m, v, base in tensors]


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_no_alloc_entry_matches_multi_tensor_entry(L):
    import torch
    from stochastic_rounding_gb300 import _lib
    a = _tensor_set(1234)
    b = _clone(a)
    ta = _lib.make_table(a)
    tb = _lib.make_table(b)
    sh = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for step in (1, 2):                      # two calls in a row
        hp = _lib.make_hparams(step=step, seed=2**33 + 7, **HP)
        assert L.asr_adamw_sr_multi_tensor(ta, len(ta), ctypes.byref(hp), sh) == _lib.ASR_OK
        assert L.asr_adamw_sr_multi_tensor_static(tb, len(tb), ctypes.byref(hp), sh) == _lib.ASR_OK
        torch.cuda.synchronize()
        for i, (x, y) in enumerate(zip(a, b)):
            for k in (0, 2, 3):
                assert torch.equal(_bits(x[k]), _bits(y[k])), f"step {step}: tensor {i} buffer {k} differs"
    bits = ctypes.c_uint32(0)
    assert L.asr_take_device_error(ctypes.byref(bits), sh) == _lib.ASR_OK and bits.value == 0


def test_no_alloc_entry_rejects_oversized_tables(L):
    from stochastic_rounding_gb300 import _lib
    hp = _lib.make_hparams(step=1, seed=0, **HP)
    big = (_lib.TensorDesc * (_lib.ASR_STATIC_TABLE_MAX + 1))()
    for d in big:
        d.param_dtype = d.grad_dtype = 1
    assert L.asr_adamw_sr_multi_tensor_static(big, len(big), ctypes.byref(hp), None) \
        == _lib.ASR_ERR_INVALID_VALUE


def _host_set(rng, count, max_n, unaligned_every=0, vector_bases=False):
    """Flat host buffers (params and grads of both dtypes, f32 moments) and,
    per tensor, (pdt, gdt, offset, n, base): slices at 8-element boundaries
    (16-byte aligned), every ``unaligned_every``-th tensor shifted by one
    element.  Base indices are cumulative with gaps of 0..2, so most are not
    multiples of 4 and take the plain kernel -- or, with ``vector_bases``,
    rounded up to multiples of 4, so every aligned tensor takes the
    pipelined kernel and its descriptor goes to the static array."""
    specs, off, base = [], 0, 0 if vector_bases else 3
    for i in range(count):
        n = int(rng.integers(1, max_n + 1))
        pdt, gdt = ("bf16", "f32")[i % 2], ("bf16", "f32")[(i // 2) % 2]
        shift = 1 if unaligned_every and i % unaligned_every == unaligned_every - 1 else 0
        specs.append((pdt, gdt, off + shift, n, base))
        off += (n + shift + 7) // 8 * 8
        base += n + int(rng.integers(0, 3))
        if vector_bases:
            base = (base + 3) // 4 * 4
    total = off
    bufs = {"p_bf16": W.to_bf16_bits(W.normal_f32(rng, total, 0.02)),
            "p_f32": W.normal_f32(rng, total, 0.02),
            "m": W.normal_f32(rng, total, 1e-4),
            "v": np.abs(W.normal_f32(rng, total, 1e-6))}
    return bufs, specs


def _grads(rng, total):
    return {"g_bf16": W.to_bf16_bits(W.normal_f32(rng, total, 1e-3)), "g_f32": W.normal_f32(rng, total, 1e-3)}


def _device_tuples(dbufs, specs):
    return [(dbufs["p_" + pdt][o:o + n], dbufs["g_" + gdt][o:o + n], dbufs["m"][o:o + n], dbufs["v"][o:o + n], base)
            for pdt, gdt, o, n, base in specs]


def _oracle_step(orc, bufs, grads, specs, step, seed):
    for pdt, gdt, o, n, base in specs:
        orc.adamw_step(bufs["p_" + pdt][o:o + n], grads["g_" + gdt][o:o + n], bufs["m"][o:o + n],
                       bufs["v"][o:o + n], step=step, seed=seed, base_index=base, **HP)


def _run_three_ways(orc, count, max_n, unaligned_every, seed, vector_bases=False):
    """The same tensor set updated by the allocation-free wrapper, by the
    regular multi-tensor wrapper and by the oracle, two steps in a row; the
    three must agree bit for bit after each step."""
    import torch
    import stochastic_rounding_gb300 as asr
    rng = np.random.default_rng(seed)
    bufs, specs = _host_set(rng, count, max_n, unaligned_every, vector_bases)
    a = {k: dev(v) for k, v in bufs.items()}
    b = {k: dev(v) for k, v in bufs.items()}
    total = bufs["m"].size
    for step in (1, 2):
        grads = _grads(rng, total)
        dg = {k: dev(v) for k, v in grads.items()}
        asr.asr_adamw_sr_multi_tensor_static(_device_tuples({**a, **dg}, specs), step=step, seed=seed, **HP)
        asr.asr_adamw_sr_multi_tensor(_device_tuples({**b, **dg}, specs), step=step, seed=seed, **HP)
        _oracle_step(orc, bufs, grads, specs, step, seed)
        torch.cuda.synchronize()
        for k in bufs:
            got_static, got_regular = host(a[k]), host(b[k])
            assert np.array_equal(got_static.view(np.uint8), got_regular.view(np.uint8)), \
                f"step {step}: buffer {k}: allocation-free entry differs from the regular one"
            assert_same_bits(got_static, bufs[k], f"step {step}: buffer {k} vs oracle")
    assert asr.asr_take_device_error() == 0


def test_no_alloc_wrapper_matches_regular_entry_and_oracle(L, orc):
    """Through the Python wrapper: 300 tensors of up to 20,000 elements, all
    four dtype groups, some off a 16-byte boundary."""
    _run_three_ways(orc, 300, 20000, 23, 77)


def test_no_alloc_full_table(L, orc):
    """Exactly ASR_STATIC_TABLE_MAX descriptors in one call, a quarter in
    each dtype group, every one aligned with a base that is a multiple of 4:
    the four groups' blocks fill the static array to its last entry, the last
    block starting three quarters of the way in."""
    from stochastic_rounding_gb300 import _lib
    _run_three_ways(orc, _lib.ASR_STATIC_TABLE_MAX, 40, 0, 78, vector_bases=True)
