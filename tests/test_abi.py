"""The C ABI library loads, exports every declared symbol, and rejects bad
arguments before launching anything (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import stochastic_rounding_gb300 as asr
from stochastic_rounding_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from stochastic_rounding_gb300 import build
    build.build()
    return asr.lib()


def header_functions():
    with open(os.path.join(ROOT, "include", "asr.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(asr_\w+)\s*\(", text, re.M)))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_header_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), f"{name} missing from libasr.so"


def test_status_strings(L):
    for s in range(4):
        assert asr.asr_status_string(s).startswith("ASR_")
    assert "unknown" in asr.asr_status_string(99)


def test_prepare_matches_oracle_scalars_bitwise(L, orc):
    """The library's per-step scalars equal the oracle's, formed independently
    from the same definition."""
    cases = [(1e-3, 0.9, 0.999, 1e-8, 0.01, 1), (1e-3, 0.9, 0.999, 1e-8, 0.01, 100),
             (3e-4, 0.95, 0.98, 1e-6, 0.1, 12345), (1e-4, 0.9, 0.999, 1e-8, 0.0, 6000),
             (1e-2, 0.0, 0.5, 0.0, 0.0, 7), (1e-3, 0.9, 0.999, 1e-8, 0.01, 4_000_000_000)]
    for lr, b1, b2, eps, wd, t in cases:
        got = asr.asr_adamw_prepare(lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=wd, step=t, seed=0)
        want = orc.adamw_scalars(lr, b1, b2, eps, wd, t)
        got = np.array([got[k] for k in ("b1", "b2", "eps", "decay", "omb1", "omb2", "step_size", "bc2s")],
                       dtype=np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (lr, b1, b2, eps, wd, t)


def _hp(**kw):
    base = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1, seed=0)
    base.update(kw)
    return _lib.make_hparams(**base)


@pytest.mark.parametrize("kw", [dict(step=0), dict(lr=-1.0), dict(lr=float("nan")), dict(eps=float("inf")),
                                dict(beta1=1.0), dict(beta2=-0.1), dict(weight_decay=-1e-3),
                                dict(beta1=float("nan"))])
def test_bad_hyperparameters_rejected(L, kw):
    h = _hp(**kw)
    assert L.asr_adamw_sr_step(ctypes.c_void_p(16), 1, ctypes.c_void_p(16), 1, ctypes.c_void_p(16),
                               ctypes.c_void_p(16), 8, 0, ctypes.byref(h), None) == _lib.ASR_ERR_INVALID_VALUE
    s = _lib.AdamwScalars()
    assert L.asr_adamw_prepare(ctypes.byref(h), ctypes.byref(s)) == _lib.ASR_ERR_INVALID_VALUE


def test_bad_rounding_and_dtype_rejected(L):
    h = _hp()
    h.rounding = 7
    assert L.asr_adamw_sr_step(None, 1, None, 1, None, None, 0, 0, ctypes.byref(h), None) \
        == _lib.ASR_ERR_UNSUPPORTED_DTYPE
    h = _hp()
    for pdt, gdt in ((2, 1), (1, -1)):
        assert L.asr_adamw_sr_step(ctypes.c_void_p(16), pdt, ctypes.c_void_p(16), gdt, ctypes.c_void_p(16),
                                   ctypes.c_void_p(16), 8, 0, ctypes.byref(h), None) \
            == _lib.ASR_ERR_UNSUPPORTED_DTYPE


def test_null_pointers_and_bad_sizes_rejected(L):
    h = _hp()
    p = ctypes.c_void_p(4096)
    for args in ((None, p, p, p), (p, None, p, p), (p, p, None, p), (p, p, p, None)):
        assert L.asr_adamw_sr_step(args[0], 1, args[1], 1, args[2], args[3], 8, 0, ctypes.byref(h), None) \
            == _lib.ASR_ERR_INVALID_VALUE
    # misaligned element pointers
    assert L.asr_adamw_sr_step(ctypes.c_void_p(4097), 1, p, 1, p, p, 8, 0, ctypes.byref(h), None) \
        == _lib.ASR_ERR_INVALID_VALUE
    assert L.asr_adamw_sr_step(p, 1, p, 1, ctypes.c_void_p(4098), p, 8, 0, ctypes.byref(h), None) \
        == _lib.ASR_ERR_INVALID_VALUE
    # base_index + n overflowing 64 bits
    assert L.asr_adamw_sr_step(p, 1, p, 1, p, p, 8, 2**64 - 4, ctypes.byref(h), None) \
        == _lib.ASR_ERR_INVALID_VALUE
    assert L.asr_philox4x32(None, 4, 0, 0, 0, 0, None) == _lib.ASR_ERR_INVALID_VALUE
    assert L.asr_stochastic_round_bf16(None, None, p, 4, 0, 0, 0, None) == _lib.ASR_ERR_INVALID_VALUE
    assert L.asr_stochastic_round_bf16(p, None, None, 4, 0, 0, 0, None) == _lib.ASR_ERR_INVALID_VALUE
    assert L.asr_adamw_sr_multi_tensor(None, 3, ctypes.byref(h), None) == _lib.ASR_ERR_INVALID_VALUE
    assert L.asr_adamw_sr_multi_tensor(None, -1, ctypes.byref(h), None) == _lib.ASR_ERR_INVALID_VALUE
    assert L.asr_adamw_sr_step(p, 1, p, 1, p, p, 8, 0, None, None) == _lib.ASR_ERR_INVALID_VALUE


def test_empty_work_is_a_noop(L):
    h = _hp()
    assert L.asr_adamw_sr_step(None, 1, None, 1, None, None, 0, 0, ctypes.byref(h), None) == _lib.ASR_OK
    assert L.asr_adamw_sr_multi_tensor(None, 0, ctypes.byref(h), None) == _lib.ASR_OK
    table = (_lib.TensorDesc * 2)()
    table[0].param_dtype = table[1].param_dtype = 1
    table[0].grad_dtype = table[1].grad_dtype = 1
    assert L.asr_adamw_sr_multi_tensor(table, 2, ctypes.byref(h), None) == _lib.ASR_OK
    assert L.asr_philox4x32(None, 0, 0, 0, 0, 0, None) == _lib.ASR_OK
    assert L.asr_stochastic_round_bf16(None, None, None, 0, 0, 0, 0, None) == _lib.ASR_OK


def test_multi_tensor_checks_every_descriptor_before_launching(L):
    """A bad descriptor anywhere in the table rejects the whole call."""
    h = _hp()
    table = (_lib.TensorDesc * 3)()
    for i in range(3):
        table[i] = _lib.TensorDesc(4096, 4096, 4096, 4096, 8, 8 * i, 1, 1)
    table[2].exp_avg = None
    assert L.asr_adamw_sr_multi_tensor(table, 3, ctypes.byref(h), None) == _lib.ASR_ERR_INVALID_VALUE
    table[2].exp_avg = 4096
    table[1].grad_dtype = 5
    assert L.asr_adamw_sr_multi_tensor(table, 3, ctypes.byref(h), None) == _lib.ASR_ERR_UNSUPPORTED_DTYPE


def test_binding_refuses_cpu_tensors(L):
    import torch
    p = torch.zeros(8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        asr.asr_adamw_sr_step(p, p, torch.zeros(8), torch.zeros(8), lr=1e-3, step=1)


def test_oracle_is_not_imported_by_the_product():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "stochastic_rounding_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".h", ".cuh", ".cpp")):
                with open(os.path.join(dirpath, fn)) as f:
                    text = f.read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "asr_oracle" not in text, fn


def test_gemm_rejects_bad_shapes_before_launching(L):
    """Shape, pointer and alignment checks of the GEMM run before any CUDA
    call (no GPU needed)."""
    p = ctypes.c_void_p(4096)
    g = L.asr_gemm_bf16_sr
    for m, n, k in ((128, 100, 64), (128, 136, 64 + 4), (128, 128, 0), (1 << 25, 128, 64), (128, 1 << 25, 64),
                    (1 << 24, 1 << 24, 64)):     # the last: within each limit, but 2^32 output tiles
        assert g(p, p, p, None, m, n, k, 0, 1, 0, None) == _lib.ASR_ERR_INVALID_VALUE, (m, n, k)
    assert g(None, p, p, None, 128, 128, 64, 0, 1, 0, None) == _lib.ASR_ERR_INVALID_VALUE
    assert g(ctypes.c_void_p(4097), p, p, None, 128, 128, 64, 0, 1, 0, None) == _lib.ASR_ERR_INVALID_VALUE
    assert g(p, p, p, None, 128, 128, 64, 7, 1, 0, None) == _lib.ASR_ERR_UNSUPPORTED_DTYPE
    assert g(None, None, None, None, 0, 128, 64, 0, 1, 0, None) == _lib.ASR_OK


def test_launch_counters_read_without_a_gpu(L):
    """asr_kernel_launches makes no CUDA call: it answers here, one counter
    per asr_kernel_kind (none has moved: nothing is launched without a GPU),
    fills at most ASR_KERNEL_KINDS entries and refuses a negative count."""
    counts = asr.asr_kernel_launches()
    assert list(counts) == list(_lib.KERNEL_KINDS) and all(v >= 0 for v in counts.values())
    with open(os.path.join(ROOT, "include", "asr.h")) as f:
        text = f.read()
    kinds = re.search(r"ASR_KERNEL_KINDS\s*=\s*(\d+)", text)
    assert kinds and int(kinds.group(1)) == len(_lib.KERNEL_KINDS)
    buf = (ctypes.c_uint64 * 12)(*([7] * 12))
    assert L.asr_kernel_launches(buf, 12) == _lib.ASR_OK
    assert list(buf)[len(_lib.KERNEL_KINDS):] == [7] * (12 - len(_lib.KERNEL_KINDS))
    assert L.asr_kernel_launches(None, 0) == _lib.ASR_OK
    assert L.asr_kernel_launches(buf, -1) == _lib.ASR_ERR_INVALID_VALUE
    assert L.asr_kernel_launches(None, 3) == _lib.ASR_ERR_INVALID_VALUE


def test_host_step_rejects_bad_arguments_before_any_cuda_call(L):
    """asr_adamw_sr_multi_tensor_host: an empty table is a no-op, and a
    missing or misaligned host gradient, a NULL table or bad hyperparameters
    are refused before anything is queued (no GPU here)."""
    h = _hp()
    assert L.asr_adamw_sr_multi_tensor_host(None, 0, ctypes.byref(h), 0, None, None, None) == _lib.ASR_OK
    assert L.asr_adamw_sr_multi_tensor_host(None, 2, ctypes.byref(h), 0, None, None, None) == \
        _lib.ASR_ERR_INVALID_VALUE

    def one(grad_host, param_host=None, n=8, gdt=_lib.ASR_BF16):
        d = _lib.TensorDesc(16, 16, 16, 16, n, 0, _lib.ASR_BF16, gdt)
        return (_lib.HostTensorDesc * 1)(_lib.HostTensorDesc(d, grad_host, param_host))

    for t in (one(None), one(18, gdt=_lib.ASR_F32), one(16, 17)):
        assert L.asr_adamw_sr_multi_tensor_host(t, 1, ctypes.byref(h), 0, None, None, None) == \
            _lib.ASR_ERR_INVALID_VALUE
    assert L.asr_adamw_sr_multi_tensor_host(one(None, n=0), 1, ctypes.byref(h), 0, None, None, None) == _lib.ASR_OK
    bad = _hp(step=0)
    assert L.asr_adamw_sr_multi_tensor_host(one(16), 1, ctypes.byref(bad), 0, None, None, None) == \
        _lib.ASR_ERR_INVALID_VALUE


def test_header_compiles_as_c99_and_cxx(tmp_path):
    """include/asr.h is a plain C header: a C99 translation unit (pedantic,
    all warnings as errors) and a C++17 one that use its types compile."""
    import shutil
    import subprocess
    src = tmp_path / "use_header.c"
    src.write_text('#include "asr.h"\n'
                   "int main(void) {\n"
                   "    asr_tensor_desc t; asr_host_tensor_desc h; asr_adamw_hparams hp; asr_adamw_scalars s;\n"
                   "    (void)t; (void)h; (void)hp; (void)s;\n"
                   "    return (int)ASR_KERNEL_KINDS + (int)ASR_STATIC_TABLE_MAX + (int)ASR_OK;\n"
                   "}\n")
    inc = os.path.join(ROOT, "include")
    for cc, flags in (("gcc", ["-std=c99", "-pedantic"]), ("g++", ["-std=c++17", "-x", "c++"])):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not found")
        r = subprocess.run([cc, *flags, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I", inc, str(src)],
                           capture_output=True, text=True)
        assert r.returncode == 0, f"{cc}: {r.stderr}"
