"""GPU parity: Philox words and stochastic rounding through the C ABI vs the
oracle (bit-exact), and Philox vs cuRAND's Philox4_32_10."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import pins
from gpu_util import assert_same_bits, dev, host, torch_cuda
from stochastic_rounding_gb300 import workloads as W

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def asr():
    torch_cuda()
    from stochastic_rounding_gb300 import build
    build.build()
    import stochastic_rounding_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("n_ctr,base,c2,c3,seed", [
    (1, 0, 0, 0, 0),
    (37, 5, 1, 0, 1),
    ((1 << 20) + 37, 2**32 - 1000, 7, 0, 1234),
    (4099, (5 << 32) + 3, 2**32 - 1, 2**31 + 5, 2**64 - 1),
])
def test_philox_words_match_oracle(asr, orc, n_ctr, base, c2, c3, seed):
    import torch
    out = torch.empty(4 * n_ctr, dtype=torch.int32, device="cuda")
    asr.asr_philox4x32(out, n_ctr, base, c2, c3, seed)
    assert_same_bits(host(out), orc.philox_fill(n_ctr, base, c2, c3, seed).reshape(-1), "philox")


def test_philox_unaligned_output(asr, orc):
    import torch
    buf = torch.zeros(4 * 1001 + 1, dtype=torch.int32, device="cuda")
    out = buf[1:]
    assert out.data_ptr() % 16 != 0
    asr.asr_philox4x32(out, 1001, 77, 3, 0, 99)
    assert_same_bits(host(out), orc.philox_fill(1001, 77, 3, 0, 99).reshape(-1), "philox unaligned")
    assert host(buf)[0] == 0


def _curand_lib(tmpdir):
    so = os.path.join(tmpdir, "curand_ref.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", "-o", so, os.path.join(HERE, "curand_ref.cu")], check=True)
    L = ctypes.CDLL(so)
    L.curand_ref_words.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_ulonglong,
                                   ctypes.c_uint, ctypes.c_ulonglong]
    L.curand_ref_words.restype = ctypes.c_int
    return L


def test_philox_matches_curand(asr, orc, tmp_path):
    """cuRAND's Philox4_32_10 with subsequence = step and offset = 4*q gives
    the words of our counter (q lo, q hi, step, 0) under key (seed lo, hi)."""
    import torch
    L = _curand_lib(str(tmp_path))
    for q0, step, seed, n in ((0, 1, 0, 4096), (2**32 - 7, 7, 1234, 100000), (123456789, 2**31 + 9, 2**63 + 11, 5000)):
        ref = torch.empty(4 * n, dtype=torch.int32, device="cuda")
        assert L.curand_ref_words(ref.data_ptr(), n, q0, step, seed) == 0
        ours = torch.empty(4 * n, dtype=torch.int32, device="cuda")
        asr.asr_philox4x32(ours, n, q0, step, 0, seed)
        torch.cuda.synchronize()
        assert_same_bits(host(ours), host(ref), f"philox vs cuRAND q0={q0}")
        # and so the oracle agrees with cuRAND too
        assert_same_bits(orc.philox_fill(64, q0, step, 0, seed).reshape(-1), host(ref)[:256], "oracle vs cuRAND")


def test_philox_large_no_repeats(asr, orc):
    """2^26 consecutive counters: no repeated 64-bit (w0, w1) prefix (the
    birthday expectation is ~1e-4), sampled rows match the oracle."""
    import torch
    n = 1 << 26
    out = torch.empty(4 * n, dtype=torch.int32, device="cuda")
    asr.asr_philox4x32(out, n, 0, 11, 0, 2024)
    w = out.view(n, 4).to(torch.int64) & 0xFFFFFFFF
    key = (w[:, 0] << 32) | w[:, 1]
    s, _ = torch.sort(key)
    assert int((s[1:] == s[:-1]).sum()) == 0
    del s, key, w
    rng = np.random.default_rng(1)
    rows = rng.integers(0, n, 2000)
    h = host(out).reshape(n, 4)
    for r in rows[:2000]:
        assert np.array_equal(h[r], orc.philox_fill(1, int(r), 11, 0, 2024)[0])


def _sr_inputs(rng, n):
    pats = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    # mostly ordinary magnitudes, plus edge patterns, Inf and NaNs
    x = rng.standard_normal(n).astype(np.float32)
    sel = rng.random(n) < 0.05
    x[sel] = pats[sel].view(np.float32)
    edge = np.concatenate([pins.sr_edge_patterns(),
                           np.array([0x7F800000, 0xFF800000, 0x7FC00000, 0xFF800001, 0x7FFFFFFF,
                                     0x7F7FFFFF, 0xFF7FFFFF], np.uint32)]).view(np.float32)
    x[:edge.size] = edge
    return x


@pytest.mark.parametrize("n,base", [(3 * (1 << 20) + 5, 0), (3 * (1 << 20) + 5, 1), (100003, 2),
                                    (100003, 3), (65536, 2**40 + 2), (4096 * 9 + 7, 2**33 + 1)])
def test_sr_matches_oracle(asr, orc, n, base):
    import torch
    rng = np.random.default_rng(n + base)
    x = _sr_inputs(rng, n)
    out = torch.empty(n, dtype=torch.int16, device="cuda")
    asr.asr_stochastic_round_bf16(dev(x), out, base_index=base, step=7, seed=1234)
    assert_same_bits(host(out), orc.sr_fill(x, base, 7, 1234), f"sr n={n} base={base}", nan_equal=False)


def test_sr_exhaustive_random_bits(asr, orc):
    """All 65,536 low random halves for 48 inputs via the rbits hook."""
    import torch
    rng = np.random.default_rng(3)
    xs = np.concatenate([pins.sr_edge_patterns(),
                         rng.integers(0, 2**32, 26, dtype=np.uint64).astype(np.uint32)]).view(np.float32)
    x = np.repeat(xs, 65536)
    r = np.tile(np.arange(65536, dtype=np.uint32), xs.size) | (
        rng.integers(0, 2**16, x.size, dtype=np.uint64).astype(np.uint32) << 16)
    out = torch.empty(x.size, dtype=torch.int16, device="cuda")
    asr.asr_stochastic_round_bf16(dev(x), out, rbits=dev(r))
    assert_same_bits(host(out), orc.sr_fill(x, 0, 0, 0, rbits=r), "sr rbits sweep", nan_equal=False)


def test_sr_unaligned_and_small(asr, orc):
    import torch
    rng = np.random.default_rng(4)
    for n in list(range(0, 34)) + [4095, 4097]:
        for off in (0, 1, 3):
            x = _sr_inputs(rng, n + off) if n + off > 40 else rng.standard_normal(n + off).astype(np.float32)
            xd = dev(x)[off:]
            buf = torch.full((n + off + 1,), 0x5A5A, dtype=torch.int16, device="cuda")
            out = buf[off:off + n]
            base = 2 + n
            asr.asr_stochastic_round_bf16(xd, out, base_index=base, step=2, seed=9)
            assert_same_bits(host(out), orc.sr_fill(x[off:], base, 2, 9), f"sr n={n} off={off}",
                             nan_equal=False)
            h = host(buf)
            assert np.all(h[:off] == 0x5A5A) and h[off + n] == 0x5A5A, "wrote outside the output"


def test_sr_large_unbiased(asr, orc):
    """2^28 copies of one value: the mean of the bf16 outputs equals x within
    5 sigma, outputs only on the two neighbours; sampled elements match."""
    import torch
    n = 1 << 28
    xv = np.float32(1.0 + 3e-4)
    x = torch.full((n,), float(xv), dtype=torch.float32, device="cuda")
    out = torch.empty(n, dtype=torch.int16, device="cuda")
    asr.asr_stochastic_round_bf16(x, out, base_index=0, step=1, seed=77)
    u = int(np.array([xv], np.float32).view(np.uint32)[0])
    lo = u >> 16
    up = (out.view(torch.int16).to(torch.int32) & 0xFFFF) == lo + 1
    dn = (out.view(torch.int16).to(torch.int32) & 0xFFFF) == lo
    assert bool((up | dn).all())
    p = (u & 0xFFFF) / 65536
    frac = float(up.double().mean())
    assert abs(frac - p) < 5 * np.sqrt(p * (1 - p) / n)
    rng = np.random.default_rng(5)
    idx = np.sort(rng.integers(0, n, 4000))
    got = host(out[torch.from_numpy(idx).cuda()])
    want = np.array([orc.sr_bf16(xv, orc.element_word(int(i), 1, 77)) for i in idx], np.uint16)
    assert_same_bits(got, want, "sampled", nan_equal=False)


def test_hardware_sr_conversion_equals_add_and_truncate(tmp_path):
    """cvt.rs.bf16x2.f32, which the stand-alone rounding op uses for non-NaN
    pairs, gives the add-and-truncate result in both lanes for every non-NaN
    binary32 pattern, with every 1024th random value and the two values at
    each input's round-up threshold (the full 2^16 sweep: `cvt_rs_sweep 1`)."""
    torch_cuda()
    exe = os.path.join(str(tmp_path), "cvt_rs_sweep")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-o", exe,
                    os.path.join(HERE, "cvt_rs_sweep.cu")], check=True)
    r = subprocess.run([exe, "1024"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert " 0 mismatches" in r.stdout
