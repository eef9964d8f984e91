"""Edge cases at the largest sizes the entry points take: one tensor longer
than 2^32 elements (offsets inside a single tensor past 32 bits, on both
forms of the pipelined kernel and on the plain kernel) and a GEMM with
M = 2^24 rows, the limit.
Windows and rows are checked against the oracle bit for bit."""
import numpy as np
import pytest

from gpu_util import assert_same_bits, host, torch_cuda

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


def test_single_tensor_longer_than_2_32(asr, orc):
    """n = 2^32 + 37 bf16 params with bf16 grads and f32 moments (51.5 GB):
    step 1 at base_index 8 (16-byte-aligned, base % 4 == 0: the pipelined
    kernel), step 2 from that state at base_index 5 (the pipelined kernel
    drawing three counters per unit), step 3 on the same buffers seen one
    element later (not 16-byte aligned: the plain kernel).  The first
    elements, the 4,096 around element 2^32 and the ragged end match the
    oracle run on the same windows with their base indices."""
    import torch
    n = 2 ** 32 + 37
    P = torch.empty(n + 1, dtype=torch.bfloat16, device="cuda")
    G = torch.empty(n + 1, dtype=torch.bfloat16, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    P.normal_(0.0, 0.02, generator=gen)
    G.normal_(0.0, 1e-3, generator=gen)
    M = torch.zeros(n + 1, dtype=torch.float32, device="cuda")
    V = torch.zeros(n + 1, dtype=torch.float32, device="cuda")
    windows = [(0, 4096), (2 ** 32 - 2048, 2 ** 32 + 2048), (n - 4133, n)]
    try:
        for step, base, shift in ((1, 8, 0), (2, 5, 0), (3, 8, 1)):
            p, g, m, v = (t[shift:shift + n] for t in (P, G, M, V))
            before = [(host(p[lo:hi]), host(g[lo:hi]), host(m[lo:hi]), host(v[lo:hi])) for lo, hi in windows]
            asr.asr_adamw_sr_step(p, g, m, v, step=step, seed=2 ** 40 + 3, base_index=base, **HP)
            torch.cuda.synchronize()
            for (lo, hi), (ph, gh, mh, vh) in zip(windows, before):
                orc.adamw_step(ph, gh, mh, vh, step=step, seed=2 ** 40 + 3, base_index=base + lo, **HP)
                assert_same_bits(host(p[lo:hi]), ph, f"step {step} p[{lo}:{hi}]")
                assert_same_bits(host(m[lo:hi]), mh, f"step {step} m[{lo}:{hi}]")
                assert_same_bits(host(v[lo:hi]), vh, f"step {step} v[{lo}:{hi}]")
        assert asr.asr_take_device_error() == 0
    finally:
        del P, G, M, V
        torch.cuda.empty_cache()


def test_gemm_at_the_row_limit(asr, orc):
    """M = 2^24 (the largest M accepted), N = 16, K = 8 with operands in
    {-8..8}: every sum is exact in binary32, so the sampled rows -- the first,
    the middle and the last -- equal the oracle GEMM's accumulator and bf16
    output bit for bit (element indices reach 2^28)."""
    import torch
    m, n, k = 2 ** 24, 16, 8
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    a = torch.randint(-8, 9, (m, k), device="cuda", generator=gen).to(torch.bfloat16)
    b = torch.randint(-8, 9, (n, k), device="cuda", generator=gen).to(torch.bfloat16)
    c = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
    try:
        asr.asr_gemm_bf16_sr(a, b, c, acc, rounding="sr", step=9, seed=123)
        torch.cuda.synchronize()
        bh = host(b)
        for lo, hi in ((0, 256), (2 ** 23 - 128, 2 ** 23 + 128), (m - 256, m)):
            want, want_acc = orc.gemm_bf16(host(a[lo:hi]), bh, row0=lo, step=9, seed=123)
            assert np.array_equal(host(acc[lo:hi]).view(np.uint32), want_acc.view(np.uint32)), f"acc rows {lo}"
            assert_same_bits(host(c[lo:hi]), want, f"rows {lo}:{hi}", nan_equal=False)
        assert asr.asr_take_device_error() == 0
    finally:
        del a, b, c, acc
        torch.cuda.empty_cache()
