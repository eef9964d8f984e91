"""GPU parity of the tcgen05 bf16 GEMM with a stochastic-rounding epilogue
("Add stochastic rounding and philox RNG helpers", Consumer).

The tensor cores' summation order is not a CPU's, so the f32 accumulator is
checked against a binary64 product within the error bound of an f32 sum of K
products; the bf16 output is then checked bit for bit against the oracle's
rounding of that very accumulator (element (i, j) at global index i*N + j),
which pins the epilogue exactly."""
import os

import numpy as np
import pytest

from gpu_util import assert_same_bits, host, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def asr():
    torch_cuda()
    from stochastic_rounding_gb300 import build
    build.build()
    import stochastic_rounding_gb300 as m
    m.lib()
    return m


def _operands(m, n, k, seed, scale=1.0):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    a = (torch.randn(m, k, device="cuda", generator=g) * scale).to(torch.bfloat16)
    b = (torch.randn(n, k, device="cuda", generator=g) * scale).to(torch.bfloat16)
    return a, b


def _check_accumulator(a, b, acc):
    """|acc - A.B^T| <= 2 K u sum_k |a_ik b_jk| with u = 2^-24 (an f32 sum of
    K exact products, allowing the tensor cores' own rounding)."""
    import torch
    ad, bd = a.double(), b.double()
    exact = ad @ bd.t()
    mag = ad.abs() @ bd.abs().t()
    k = a.shape[1]
    err = (acc.double() - exact).abs()
    bound = 2 * k * 2.0 ** -24 * mag + 1e-30
    worst = float((err / bound).max())
    assert worst <= 1.0, f"accumulator off the binary64 product by {worst:.3g} x the bound"


@pytest.mark.parametrize("m,n,k", [(128, 128, 64), (256, 384, 512), (128, 256, 64 * 13), (1, 16, 8),
                                   (200, 272, 520), (333, 1040, 72),
                                   (333, 1040, 1032), (1800, 1296, 136)])
@pytest.mark.parametrize("rounding", ["sr", "rne"])
def test_gemm_matches_oracle_rounding_of_accumulator(asr, orc, m, n, k, rounding):
    import torch
    a, b = _operands(m, n, k, seed=m + n + k)
    c = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
    asr.asr_gemm_bf16_sr(a, b, c, acc, rounding=rounding, step=3, seed=2**40 + 9)
    torch.cuda.synchronize()
    _check_accumulator(a, b, acc)
    acc_h = host(acc).reshape(-1)
    want = orc.sr_fill(acc_h, 0, 3, 2**40 + 9) if rounding == "sr" else orc.rne_fill(acc_h)
    assert_same_bits(host(c).reshape(-1), want, f"gemm {m}x{n}x{k} {rounding}", nan_equal=False)


def test_gemm_large_equals_standalone_rounding(asr, orc):
    """2048 x 2048 x 4096: the epilogue equals the library's stand-alone
    rounding op (itself bit-exact with the oracle) on the accumulator, the
    accumulator is within the bound, and sampled rows match the oracle."""
    import torch
    m, n, k = 2048, 2048, 4096
    a, b = _operands(m, n, k, seed=7, scale=0.5)
    c = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
    asr.asr_gemm_bf16_sr(a, b, c, acc, step=11, seed=5)
    ref = torch.empty(m * n, dtype=torch.int16, device="cuda")
    asr.asr_stochastic_round_bf16(acc.view(-1), ref, base_index=0, step=11, seed=5)
    torch.cuda.synchronize()
    assert torch.equal(c.view(torch.int16).view(-1), ref)
    _check_accumulator(a, b, acc)
    rng = np.random.default_rng(3)
    for i in rng.integers(0, m, 8):
        row = host(acc[int(i)])
        want = orc.sr_fill(row, int(i) * n, 11, 5)
        assert_same_bits(host(c[int(i)]), want, f"row {int(i)}", nan_equal=False)
    assert asr.asr_take_device_error() == 0


def test_gemm_seed_keying_and_unbiasedness(asr):
    """Same (seed, step) -> identical output; a new seed changes it; over 64
    seeds the mean of the bf16 outputs approaches the accumulator."""
    import torch
    m, n, k = 256, 256, 256
    a, b = _operands(m, n, k, seed=1)
    acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
    outs = []
    for seed in range(64):
        c = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        asr.asr_gemm_bf16_sr(a, b, c, acc if seed == 0 else None, step=1, seed=seed)
        outs.append(c.float())
    c0 = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    asr.asr_gemm_bf16_sr(a, b, c0, None, step=1, seed=0)
    torch.cuda.synchronize()
    assert torch.equal(c0.float(), outs[0])
    assert not torch.equal(outs[0], outs[1])
    mean = torch.stack(outs).mean(0)
    rn = acc.to(torch.bfloat16).float()
    # the SR mean is far closer to the accumulator than round-to-nearest is
    assert float((mean - acc).abs().mean()) < 0.25 * float((rn - acc).abs().mean())


def test_gemm_rejects_unsupported_shapes(asr):
    import torch
    from stochastic_rounding_gb300 import _lib
    a = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")
    L = _lib.lib()
    for m, n, k in ((128, 100, 64), (128, 128, 60), (128, 128, 0)):
        assert L.asr_gemm_bf16_sr(a.data_ptr(), b.data_ptr(), c.data_ptr(), None, m, n, k, 0, 1, 0, None) \
            == _lib.ASR_ERR_INVALID_VALUE


def test_gemm_many_tiles_per_cta(asr, orc):
    """4096 x 4224 x 256: 544 tiles (half tiles at the N edge) on 152 SMs, so
    every CTA reuses both accumulators several times; the epilogue equals the
    stand-alone rounding of the accumulator, which is within the bound, and
    sampled rows match the oracle."""
    import torch
    m, n, k = 4096, 4224, 256
    a, b = _operands(m, n, k, seed=12)
    c = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
    asr.asr_gemm_bf16_sr(a, b, c, acc, step=2, seed=77)
    ref = torch.empty(m * n, dtype=torch.int16, device="cuda")
    asr.asr_stochastic_round_bf16(acc.view(-1), ref, base_index=0, step=2, seed=77)
    torch.cuda.synchronize()
    assert torch.equal(c.view(torch.int16).view(-1), ref)
    _check_accumulator(a, b, acc)
    rng = np.random.default_rng(4)
    for i in rng.integers(0, m, 6):
        want = orc.sr_fill(host(acc[int(i)]), int(i) * n, 2, 77)
        assert_same_bits(host(c[int(i)]), want, f"row {int(i)}", nan_equal=False)
    assert asr.asr_take_device_error() == 0


@pytest.mark.parametrize("m,n,k,epilogue", [(2560, 2560, 768, 8), (2560, 2560, 1088, 4), (2816, 2560, 520, 8),
                                             (2304, 2816, 136, 16), (2048, 2048, 2048, 16)])
@pytest.mark.parametrize("rounding", ["sr", "rne"])
def test_gemm_epilogue_widths(asr, orc, m, n, k, epilogue, rounding):
    """Each epilogue width on the shapes that pick it: more pair tiles than
    resident pairs (76 on GB300) take 8 warps for 512 < K <= 1024 and 4 above,
    16 at K <= 512; every tile in one round (2048^2: 64 tiles) takes 16 at any
    K.  The output equals the stand-alone rounding of the accumulator (itself
    bit-exact with the oracle), the accumulator is within the bound, and
    sampled rows match the oracle."""
    import torch
    a, b = _operands(m, n, k, seed=m + k)
    c = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
    asr.asr_gemm_bf16_sr(a, b, c, acc, rounding=rounding, step=6, seed=31)
    ref = torch.empty(m * n, dtype=torch.int16, device="cuda")
    if rounding == "sr":
        asr.asr_stochastic_round_bf16(acc.view(-1), ref, base_index=0, step=6, seed=31)
    else:
        ref.copy_(acc.view(-1).to(torch.bfloat16).view(torch.int16))
    torch.cuda.synchronize()
    assert torch.equal(c.view(torch.int16).view(-1), ref), f"{m}x{n}x{k} ({epilogue} epilogue warps)"
    _check_accumulator(a, b, acc)
    rng = np.random.default_rng(m + n)
    for i in rng.integers(0, m, 4):
        row = host(acc[int(i)])
        want = orc.sr_fill(row, int(i) * n, 6, 31) if rounding == "sr" else orc.rne_fill(row)
        assert_same_bits(host(c[int(i)]), want, f"row {int(i)}", nan_equal=False)
    assert asr.asr_take_device_error() == 0


def test_one_sm_kernel_variant(asr, orc, tmp_path):
    """The one-SM 128 x 256 kernel, which the library falls back to where no
    CTA pair fits, built alone (-DASR_GEMM_PAIR=0) into a separate library:
    same bits as the oracle's rounding of its accumulator, ragged edges and
    K tails included, and no device error."""
    import ctypes
    import subprocess
    import torch
    from stochastic_rounding_gb300 import build as B
    so = str(tmp_path / "libasr_one_sm.so")
    subprocess.run([B.nvcc(), *B.NVCC_FLAGS, "-DASR_GEMM_PAIR=0", "-I", os.path.join(B.ROOT, "include"),
                    "-o", so, B.SRC], check=True)
    L = ctypes.CDLL(so)
    vp, u64, u32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32
    L.asr_gemm_bf16_sr.argtypes = [vp, vp, vp, vp, u64, u64, u64, u32, u32, u64, vp]
    L.asr_gemm_bf16_sr.restype = ctypes.c_int
    L.asr_take_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
    L.asr_take_device_error.restype = ctypes.c_int
    stream = torch.cuda.current_stream().cuda_stream
    for (m, n, k) in [(128, 256, 64), (200, 272, 520), (1, 16, 8), (333, 1040, 72), (640, 768, 256)]:
        a, b = _operands(m, n, k, seed=7 * m + n + k)
        c = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
        st = L.asr_gemm_bf16_sr(a.data_ptr(), b.data_ptr(), c.data_ptr(), acc.data_ptr(), m, n, k,
                                0, 5, 2**33 + 1, stream)
        assert st == 0, f"status {st}"
        torch.cuda.synchronize()
        _check_accumulator(a, b, acc)
        want = orc.sr_fill(host(acc).reshape(-1), 0, 5, 2**33 + 1)
        assert_same_bits(host(c).reshape(-1), want, f"one-SM gemm {m}x{n}x{k}", nan_equal=False)
    bits = ctypes.c_uint32(0)
    assert L.asr_take_device_error(ctypes.byref(bits), stream) == 0
    assert bits.value == 0


def test_output_only_16_byte_aligned(asr, orc):
    """An output that starts 16 bytes past a 32-byte boundary takes the
    128-bit store path (the 256-bit one needs 32-byte alignment): same bits,
    and the words around the output stay untouched."""
    import torch
    m, n, k = 200, 272, 1032
    a, b = _operands(m, n, k, seed=31)
    buf = torch.full((m * n + 32,), 0x1234, dtype=torch.int16, device="cuda")
    assert buf.data_ptr() % 32 == 0
    c = buf[8:8 + m * n].view(torch.bfloat16).view(m, n)
    acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
    asr.asr_gemm_bf16_sr(a, b, c, acc, rounding="sr", step=2, seed=99)
    torch.cuda.synchronize()
    want = orc.sr_fill(host(acc).reshape(-1), 0, 2, 99)
    assert_same_bits(host(c).reshape(-1), want, "16-byte-aligned output", nan_equal=False)
    h = host(buf)
    assert (h[:8] == 0x1234).all() and (h[8 + m * n:] == 0x1234).all()


@pytest.mark.parametrize("m,n,k", [(200, 272, 520), (333, 1040, 1032), (1, 16, 8), (512, 1024, 64),
                                   (1800, 1296, 136), (4096, 4096, 64)])
@pytest.mark.parametrize("rounding", ["sr", "rne"])
def test_gemm_equals_oracle_gemm_on_integer_operands(asr, orc, m, n, k, rounding):
    """Entries in {-8..8}: every partial sum is an integer below 2^24, exact in
    binary32 whatever the summation order, so the kernel's accumulator must
    equal the oracle GEMM's bit for bit, and so must the whole bf16 output
    (sums above 256 are not bf16 values: the rounding draws real bits)."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(m * 7 + k)
    a = torch.randint(-8, 9, (m, k), device="cuda", generator=g).to(torch.bfloat16)
    b = torch.randint(-8, 9, (n, k), device="cuda", generator=g).to(torch.bfloat16)
    c = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
    asr.asr_gemm_bf16_sr(a, b, c, acc, rounding=rounding, step=4, seed=1234)
    torch.cuda.synchronize()
    want, want_acc = orc.gemm_bf16(host(a), host(b), rounding=0 if rounding == "sr" else 1, step=4, seed=1234)
    assert np.array_equal(host(acc).view(np.uint32), want_acc.view(np.uint32)), "accumulators differ"
    assert_same_bits(host(c), want, f"gemm {m}x{n}x{k} {rounding} vs oracle GEMM", nan_equal=False)


def test_gemm_against_oracle_gemm(asr, orc):
    """Normal operands: the accumulators differ only by summation order
    (within the bound), and wherever they are equal the bf16 outputs are
    identical (same keying)."""
    import torch
    m, n, k = 200, 272, 520
    a, b = _operands(m, n, k, seed=41)
    c = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
    asr.asr_gemm_bf16_sr(a, b, c, acc, rounding="sr", step=4, seed=1234)
    torch.cuda.synchronize()
    want, want_acc = orc.gemm_bf16(host(a), host(b), step=4, seed=1234)
    _check_accumulator(a, b, acc)
    same = host(acc).view(np.uint32) == want_acc.view(np.uint32)
    assert same.sum() >= 100, f"only {same.sum()} accumulators agree bitwise"
    assert np.array_equal(host(c)[same], want[same]), "same accumulator, different rounding"


def test_gemm_special_values_in_the_epilogue(asr, orc):
    """Inf and NaN entries in A (and products that overflow binary32) give
    Inf / NaN accumulators; the epilogue's hardware rounding has a NaN
    fallback, so every output -- NaN patterns included -- equals the oracle's
    rounding of the kernel's own accumulator bit for bit (NaN: sign and top
    payload kept, quiet bit set), SR and RNE."""
    import torch
    m, n, k = 200, 272, 520
    a, b = _operands(m, n, k, seed=51)
    a[3, 7] = float("inf")
    a[10, 0] = float("-inf")
    a[20, 5] = float("nan")
    a[30, :] = 3.0e38            # row 30: products and sums overflow to +-Inf or Inf - Inf = NaN
    a[40, 100] = float("inf")
    b[50, 100] = 0.0             # inf * 0 = NaN in (40, 50)
    for rounding in ("sr", "rne"):
        c = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        acc = torch.empty(m, n, dtype=torch.float32, device="cuda")
        asr.asr_gemm_bf16_sr(a, b, c, acc, rounding=rounding, step=2, seed=77)
        torch.cuda.synchronize()
        acc_h = host(acc).reshape(-1)
        assert np.isnan(acc_h).sum() > 0 and np.isinf(acc_h).sum() > 0
        want = orc.sr_fill(acc_h, 0, 2, 77) if rounding == "sr" else orc.rne_fill(acc_h)
        assert_same_bits(host(c).reshape(-1), want, f"special values {rounding}", nan_equal=False)
