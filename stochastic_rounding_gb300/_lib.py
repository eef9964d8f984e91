"""ctypes binding of ``libasr.so`` with the C ABI's names.

Argument marshalling only: tensors are checked (device, dtype, contiguity,
size) and turned into device pointers, hyperparameters into the C struct, the
current torch stream into a cudaStream_t.  Every step of the computation runs
in the library's CUDA kernels.  There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import struct
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libasr.so")

ASR_OK, ASR_ERR_INVALID_VALUE, ASR_ERR_UNSUPPORTED_DTYPE, ASR_ERR_CUDA = 0, 1, 2, 3
ASR_F32, ASR_BF16 = 0, 1
ASR_ROUND_SR, ASR_ROUND_RNE = 0, 1

# Every function the header declares.
EXPORTS = ("asr_philox4x32", "asr_stochastic_round_bf16", "asr_adamw_prepare",
           "asr_adamw_sr_step", "asr_adamw_sr_multi_tensor", "asr_status_string",
           "asr_last_cuda_error", "asr_take_device_error", "asr_selftest_wait_timeout",
           "asr_adamw_sr_multi_tensor_static", "asr_gemm_bf16_sr", "asr_take_device_error_async",
           "asr_kernel_launches", "asr_adamw_sr_multi_tensor_host")
# asr_kernel_kind, in order
KERNEL_KINDS = ("adamw_scalar", "adamw_vector", "adamw_pipelined", "adamw_pipelined_any_base", "adamw_static",
                "round", "philox", "gemm")
ASR_STATIC_TABLE_MAX = 4096


class AdamwHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double), ("step", ctypes.c_uint32),
                ("rounding", ctypes.c_uint32), ("seed", ctypes.c_uint64)]


class AdamwScalars(ctypes.Structure):
    _fields_ = [(k, ctypes.c_float) for k in
                ("b1", "b2", "eps", "decay", "omb1", "omb2", "step_size", "bc2s")]


class TensorDesc(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p),
                ("exp_avg", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p),
                ("n", ctypes.c_uint64), ("base_index", ctypes.c_uint64),
                ("param_dtype", ctypes.c_int32), ("grad_dtype", ctypes.c_int32)]


class HostTensorDesc(ctypes.Structure):
    _fields_ = [("dev", TensorDesc), ("grad_host", ctypes.c_void_p), ("param_host", ctypes.c_void_p)]


class AsrError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = f"{what}: {status_string(status)}"
        if status == ASR_ERR_CUDA:
            msg += f" (cudaError {lib().asr_last_cuda_error()})"
        super().__init__(msg)
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with stochastic_rounding_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, u64, u32, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32
        L.asr_philox4x32.argtypes = [vp, u64, u64, u32, u32, u64, vp]
        L.asr_stochastic_round_bf16.argtypes = [vp, vp, vp, u64, u64, u32, u64, vp]
        L.asr_adamw_prepare.argtypes = [ctypes.POINTER(AdamwHparams), ctypes.POINTER(AdamwScalars)]
        L.asr_adamw_sr_step.argtypes = [vp, i32, vp, i32, vp, vp, u64, u64,
                                        ctypes.POINTER(AdamwHparams), vp]
        L.asr_adamw_sr_multi_tensor.argtypes = [ctypes.POINTER(TensorDesc), i32,
                                                ctypes.POINTER(AdamwHparams), vp]
        L.asr_adamw_sr_multi_tensor_static.argtypes = [ctypes.POINTER(TensorDesc), i32,
                                                       ctypes.POINTER(AdamwHparams), vp]
        L.asr_adamw_sr_multi_tensor_host.argtypes = [ctypes.POINTER(HostTensorDesc), i32,
                                                     ctypes.POINTER(AdamwHparams), u64, vp, vp, vp]
        L.asr_adamw_sr_multi_tensor_host.restype = ctypes.c_int
        L.asr_gemm_bf16_sr.argtypes = [vp, vp, vp, vp, u64, u64, u64, u32, u32, u64, vp]
        L.asr_gemm_bf16_sr.restype = ctypes.c_int
        for f in ("asr_philox4x32", "asr_stochastic_round_bf16", "asr_adamw_prepare",
                  "asr_adamw_sr_step", "asr_adamw_sr_multi_tensor",
                  "asr_adamw_sr_multi_tensor_static"):
            getattr(L, f).restype = ctypes.c_int
        L.asr_status_string.argtypes = [ctypes.c_int]
        L.asr_status_string.restype = ctypes.c_char_p
        L.asr_selftest_wait_timeout.argtypes = [u64, vp]
        L.asr_selftest_wait_timeout.restype = ctypes.c_int
        L.asr_take_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
        L.asr_take_device_error.restype = ctypes.c_int
        L.asr_take_device_error_async.argtypes = [vp, vp]
        L.asr_take_device_error_async.restype = ctypes.c_int
        L.asr_kernel_launches.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int32]
        L.asr_kernel_launches.restype = ctypes.c_int
        L.asr_last_cuda_error.argtypes = []
        L.asr_last_cuda_error.restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().asr_status_string(int(status)).decode()


asr_status_string = status_string


def asr_last_cuda_error() -> int:
    return int(lib().asr_last_cuda_error())


def asr_kernel_launches() -> dict:
    """Kernels the library has launched in this process, per kind (see
    ``KERNEL_KINDS``): counted on the host when queued, on every device and
    stream.  Makes no CUDA call."""
    counts = (ctypes.c_uint64 * len(KERNEL_KINDS))()
    _check(lib().asr_kernel_launches(counts, len(KERNEL_KINDS)), "asr_kernel_launches")
    return dict(zip(KERNEL_KINDS, (int(c) for c in counts)))


def asr_take_device_error(stream=None, device=None) -> int:
    """Read and clear the device-side error bits (0 = none); waits for the stream."""
    torch = _torch()
    dev = torch.device(device if device is not None else "cuda")
    bits = ctypes.c_uint32(0)
    with _on_device(dev):
        _check(lib().asr_take_device_error(ctypes.byref(bits), _stream_handle(dev, stream)),
               "asr_take_device_error")
    return int(bits.value)


def asr_take_device_error_async(out, stream=None, device=None):
    """Enqueue a read-and-clear of the device error bits into ``out`` (a
    one-element int32 tensor: page-locked CPU memory, or on the CUDA device)
    without waiting; ``out`` holds the bits once the stream gets there."""
    torch = _torch()
    if not isinstance(out, torch.Tensor) or out.dtype != torch.int32 or out.numel() != 1:
        raise TypeError("out must be a one-element int32 tensor")
    if out.is_cuda:
        dev = out.device
    else:
        if not out.is_pinned():
            raise ValueError("out must be page-locked (pin_memory=True) or a CUDA tensor")
        dev = torch.device(device if device is not None else "cuda")
    with _on_device(dev):
        _check(lib().asr_take_device_error_async(ctypes.c_void_p(out.data_ptr()), _stream_handle(dev, stream)),
               "asr_take_device_error_async")
    return out


def asr_selftest_wait_timeout(limit_ns: int = 1_000_000, stream=None, device=None):
    """Launch the bounded-wait self-test (a wait that must give up)."""
    torch = _torch()
    dev = torch.device(device if device is not None else "cuda")
    with _on_device(dev):
        _check(lib().asr_selftest_wait_timeout(int(limit_ns), _stream_handle(dev, stream)),
               "asr_selftest_wait_timeout")


def _check(status: int, what: str):
    if status != ASR_OK:
        raise AsrError(status, what)


_ROUNDING = {"sr": ASR_ROUND_SR, "rne": ASR_ROUND_RNE, ASR_ROUND_SR: ASR_ROUND_SR, ASR_ROUND_RNE: ASR_ROUND_RNE}


# AdamwHparams packed in one call (its fields in order, native alignment):
# one struct.pack is a fraction of the cost of eight ctypes field stores.
_HP_PACK = struct.Struct("=5dIIQ")
assert _HP_PACK.size == ctypes.sizeof(AdamwHparams)


def make_hparams(lr, beta1, beta2, eps, weight_decay, step, seed, rounding="sr") -> AdamwHparams:
    r = _ROUNDING.get(rounding)
    if r is None:
        raise ValueError(f"rounding must be 'sr' or 'rne', not {rounding!r}")
    h = AdamwHparams()
    try:
        _HP_PACK.pack_into(h, 0, lr, beta1, beta2, eps, weight_decay, step, r, int(seed) & (2**64 - 1))
    except struct.error as exc:
        raise ValueError(f"hyperparameters out of range (step must fit in 32 bits): {exc}") from None
    return h


# ------------------------------------------------------------ tensor helpers

def _torch():
    import torch
    return torch


def _dev_ptr(t, name, dtypes, numel=None, device=None):
    """Device pointer of ``t`` after the checks the C ABI cannot make: a
    contiguous CUDA tensor of one of ``dtypes`` (and ``numel`` elements),
    on CUDA device index ``device`` when given -- a kernel runs on one
    device, and a pointer into another device's memory would be
    dereferenced there."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if device is not None and t.get_device() != device:
        raise ValueError(f"{name} is on cuda:{t.get_device()}; the call's other tensors are on cuda:{device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements; expected {numel}")
    return t.data_ptr()


_NULL_CONTEXT = contextlib.nullcontext()


def _on_device(device):
    """Make ``device`` current for the call: a no-op (no device switch and
    back) when it already is, which is the common case."""
    torch = _torch()
    if not isinstance(device, torch.device):
        device = torch.device(device)
    if device.index is None or device.index == torch.cuda.current_device():
        return _NULL_CONTEXT
    return torch.cuda.device(device)


def _stream_handle(device, stream):
    """The cudaStream_t of ``stream``, or of the device's current stream."""
    torch = _torch()
    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            if not isinstance(device, torch.device):
                device = torch.device(device)
            idx = device.index if device.index is not None else torch.cuda.current_device()
            return ctypes.c_void_p(raw(idx))
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


_DTYPES = {}


def _dtype_codes():
    """torch dtype -> asr_dtype code (bf16 patterns may come as int16)."""
    if not _DTYPES:
        torch = _torch()
        _DTYPES.update({torch.float32: ASR_F32, torch.bfloat16: ASR_BF16, torch.int16: ASR_BF16})
    return _DTYPES


def _dt(t):
    code = _dtype_codes().get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return code


# ------------------------------------------------------------- entry points

def asr_philox4x32(out, n_ctr: int, ctr_base: int, ctr2: int, ctr3: int, seed: int, stream=None):
    """Philox4x32-10 words of ``n_ctr`` counters into ``out`` (int32/uint32
    CUDA tensor of 4*n_ctr elements)."""
    torch = _torch()
    dts = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())
    p = _dev_ptr(out, "out", dts, 4 * int(n_ctr))
    with _on_device(out.device):
        _check(lib().asr_philox4x32(p, int(n_ctr), int(ctr_base) & (2**64 - 1), int(ctr2) & 0xFFFFFFFF,
                                    int(ctr3) & 0xFFFFFFFF, int(seed) & (2**64 - 1),
                                    _stream_handle(out.device, stream)), "asr_philox4x32")
    return out


def asr_stochastic_round_bf16(x, out, *, base_index: int = 0, step: int = 0, seed: int = 0,
                              rbits=None, stream=None):
    """Stochastically round float32 ``x`` into ``out`` (bfloat16 or int16
    CUDA tensor holding bf16 patterns)."""
    torch = _torch()
    n = x.numel()
    px = _dev_ptr(x, "x", (torch.float32,))
    xd = x.get_device()
    po = _dev_ptr(out, "out", (torch.bfloat16, torch.int16), n, xd)
    pr = None
    if rbits is not None:
        dts = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())
        pr = _dev_ptr(rbits, "rbits", dts, n, xd)
    with _on_device(x.device):
        _check(lib().asr_stochastic_round_bf16(px, pr, po, n, int(base_index), int(step) & 0xFFFFFFFF,
                                               int(seed) & (2**64 - 1), _stream_handle(x.device, stream)),
               "asr_stochastic_round_bf16")
    return out


def asr_adamw_prepare(**hp) -> dict:
    """The binary32 per-step scalars the library uses (host only)."""
    h = make_hparams(**hp)
    s = AdamwScalars()
    _check(lib().asr_adamw_prepare(ctypes.byref(h), ctypes.byref(s)), "asr_adamw_prepare")
    return {k: getattr(s, k) for k, _ in AdamwScalars._fields_}


def asr_adamw_sr_step(param, grad, exp_avg, exp_avg_sq, *, lr, beta1=0.9, beta2=0.999, eps=1e-8,
                      weight_decay=0.0, step, seed=0, base_index: int = 0, rounding="sr", stream=None):
    """One fused AdamW step in place on one tensor or shard."""
    torch = _torch()
    n = param.numel()
    pp = _dev_ptr(param, "param", (torch.float32, torch.bfloat16, torch.int16))
    dev = param.device
    di = param.get_device()
    pg = _dev_ptr(grad, "grad", (torch.float32, torch.bfloat16, torch.int16), n, di)
    pm = _dev_ptr(exp_avg, "exp_avg", (torch.float32,), n, di)
    pv = _dev_ptr(exp_avg_sq, "exp_avg_sq", (torch.float32,), n, di)
    h = make_hparams(lr, beta1, beta2, eps, weight_decay, step, seed, rounding)
    with _on_device(dev):
        _check(lib().asr_adamw_sr_step(pp, _dt(param), pg, _dt(grad), pm, pv, n, int(base_index),
                                       ctypes.byref(h), _stream_handle(dev, stream)),
               "asr_adamw_sr_step")


def make_table(tensors: Sequence[Sequence]) -> ctypes.Array:
    """Descriptor array from (param, grad, exp_avg, exp_avg_sq, base_index)
    tuples, all on one CUDA device (the first parameter's)."""
    torch = _torch()
    arr = (TensorDesc * len(tensors))()
    dev = None
    for i, (p, g, m, v, base) in enumerate(tensors):
        n = p.numel()
        pp = _dev_ptr(p, f"param[{i}]", (torch.float32, torch.bfloat16, torch.int16), None, dev)
        dev = p.get_device()
        arr[i] = TensorDesc(
            pp,
            _dev_ptr(g, f"grad[{i}]", (torch.float32, torch.bfloat16, torch.int16), n, dev),
            _dev_ptr(m, f"exp_avg[{i}]", (torch.float32,), n, dev),
            _dev_ptr(v, f"exp_avg_sq[{i}]", (torch.float32,), n, dev),
            n, int(base), _dt(p), _dt(g))
    return arr


# TensorDesc packed in one call (four 64-bit pointers, n, base_index, two
# dtype codes; native alignment, no padding on the 64-bit hosts this runs on)
_DESC_PACK = struct.Struct("=6Q2i")
assert _DESC_PACK.size == ctypes.sizeof(TensorDesc)


def _pack_table(entries) -> ctypes.Array:
    """Descriptor array from (param, grad, exp_avg, exp_avg_sq, base_index)
    tuples whose tensors the caller has already checked as ``make_table``
    would (contiguous CUDA tensors on one device, matching sizes, supported
    dtypes): the descriptors are packed without repeating the checks."""
    arr = (TensorDesc * len(entries))()
    codes = _dtype_codes()
    off = 0
    for p, g, m, v, base in entries:
        _DESC_PACK.pack_into(arr, off, p.data_ptr(), g.data_ptr(), m.data_ptr(), v.data_ptr(), p.numel(), base,
                             codes[p.dtype], codes[g.dtype])
        off += _DESC_PACK.size
    return arr


def asr_adamw_sr_multi_tensor(tensors, *, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                              step, seed=0, rounding="sr", stream=None, device=None):
    """One fused AdamW step over many tensors.  ``tensors`` is a sequence of
    (param, grad, exp_avg, exp_avg_sq, base_index) tuples, or a descriptor
    array made by ``make_table`` (then ``device`` names the CUDA device)."""
    torch = _torch()
    if isinstance(tensors, ctypes.Array):
        table = tensors
        dev = torch.device(device if device is not None else "cuda")
    else:
        table = make_table(tensors)
        dev = tensors[0][0].device if len(tensors) else torch.device("cuda")
    h = make_hparams(lr, beta1, beta2, eps, weight_decay, step, seed, rounding)
    with _on_device(dev):
        _check(lib().asr_adamw_sr_multi_tensor(table, len(table), ctypes.byref(h),
                                               _stream_handle(dev, stream)),
               "asr_adamw_sr_multi_tensor")


def _host_ptr(t, name, dtypes, numel):
    """Address of a contiguous CPU tensor (page-locked memory: the library
    checks that and refuses anything else)."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor in page-locked memory")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
    if not t.is_contiguous() or t.numel() != numel:
        raise ValueError(f"{name} must be contiguous with {numel} elements")
    return t.data_ptr()


def make_host_table(tensors: Sequence[Sequence]) -> ctypes.Array:
    """Descriptor array for ``asr_adamw_sr_multi_tensor_host`` from
    (param, grad, exp_avg, exp_avg_sq, base_index, grad_host, param_host)
    tuples: the first five as for ``make_table`` (CUDA tensors, one device),
    grad_host a page-locked CPU tensor of grad's dtype and size, param_host one
    of param's dtype and size or None."""
    torch = _torch()
    dev_table = make_table([t[:5] for t in tensors])
    arr = (HostTensorDesc * len(tensors))()
    for i, t in enumerate(tensors):
        p, g, host_g, host_p = t[0], t[1], t[5], t[6]
        same = lambda x: (torch.bfloat16, torch.int16) if x.dtype in (torch.bfloat16, torch.int16) else (x.dtype,)  # noqa: E731
        gh = _host_ptr(host_g, f"grad_host[{i}]", same(g), g.numel())
        ph = _host_ptr(host_p, f"param_host[{i}]", same(p), p.numel()) if host_p is not None else None
        arr[i] = HostTensorDesc(dev_table[i], gh, ph)
    return arr


def asr_adamw_sr_multi_tensor_host(tensors, *, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step,
                                   seed=0, rounding="sr", chunk_elems=0, stream=None, copy_in=None,
                                   copy_out=None, device=None):
    """The multi-tensor step with gradients copied in from page-locked host
    memory and the updated parameters copied back to it, pipelined in the
    library over chunks of consecutive tensors: copies in on ``copy_in``,
    steps on ``stream``, copies out on ``copy_out`` (each defaulting to
    ``stream``, which gives no overlap; pass two other streams for it).
    Later work on ``stream`` follows the steps; the host parameters are
    ready once ``copy_out`` has reached the call's copies (wait on it).
    ``tensors``: a table made by ``make_host_table`` (then ``device`` names the
    CUDA device) or the tuples it takes."""
    torch = _torch()
    if isinstance(tensors, ctypes.Array):
        table = tensors
        dev = torch.device(device if device is not None else "cuda")
    else:
        table = make_host_table(tensors)
        dev = tensors[0][0].device if len(tensors) else torch.device("cuda")
    h = make_hparams(lr, beta1, beta2, eps, weight_decay, step, seed, rounding)
    with _on_device(dev):
        s = _stream_handle(dev, stream)
        cin = _stream_handle(dev, copy_in) if copy_in is not None else s
        cout = _stream_handle(dev, copy_out) if copy_out is not None else s
        _check(lib().asr_adamw_sr_multi_tensor_host(table, len(table), ctypes.byref(h), int(chunk_elems), s, cin,
                                                    cout), "asr_adamw_sr_multi_tensor_host")


def asr_adamw_sr_multi_tensor_static(tensors, *, lr, beta1=0.9, beta2=0.999, eps=1e-8,
                                     weight_decay=0.0, step, seed=0, rounding="sr", stream=None,
                                     device=None):
    """Allocation-free variant of ``asr_adamw_sr_multi_tensor`` for callers
    that may not allocate device memory: the descriptor table is staged in a
    library-owned device array (at most ASR_STATIC_TABLE_MAX tensors), and
    calls must not overlap on the GPU.  Same arguments, same results."""
    torch = _torch()
    if isinstance(tensors, ctypes.Array):
        table = tensors
        dev = torch.device(device if device is not None else "cuda")
    else:
        table = make_table(tensors)
        dev = tensors[0][0].device if len(tensors) else torch.device("cuda")
    h = make_hparams(lr, beta1, beta2, eps, weight_decay, step, seed, rounding)
    with _on_device(dev):
        _check(lib().asr_adamw_sr_multi_tensor_static(table, len(table), ctypes.byref(h),
                                                      _stream_handle(dev, stream)),
               "asr_adamw_sr_multi_tensor_static")


def asr_gemm_bf16_sr(a, b, c, c_f32=None, *, rounding="sr", step=0, seed=0, stream=None):
    """C = A . B^T on the tensor cores with a stochastic-rounding (or RNE)
    bf16 epilogue.  a: (m, k), b: (n, k), c: (m, n) contiguous bfloat16 CUDA
    tensors; c_f32: optional (m, n) float32 tensor receiving the accumulator."""
    torch = _torch()
    if a.dim() != 2 or b.dim() != 2 or c.dim() != 2:
        raise ValueError("a, b and c must be 2-D")
    m, k = a.shape
    n = b.shape[0]
    if b.shape[1] != k or tuple(c.shape) != (m, n):
        raise ValueError(f"shapes do not chain: a {tuple(a.shape)}, b {tuple(b.shape)}, c {tuple(c.shape)}")
    pa = _dev_ptr(a, "a", (torch.bfloat16,))
    ad = a.get_device()
    pb = _dev_ptr(b, "b", (torch.bfloat16,), None, ad)
    pc = _dev_ptr(c, "c", (torch.bfloat16,), None, ad)
    pf = _dev_ptr(c_f32, "c_f32", (torch.float32,), m * n, ad) if c_f32 is not None else None
    r = _ROUNDING.get(rounding)
    if r is None:
        raise ValueError(f"rounding must be 'sr' or 'rne', not {rounding!r}")
    with _on_device(a.device):
        _check(lib().asr_gemm_bf16_sr(pa, pb, pc, pf, m, n, k, r, int(step) & 0xFFFFFFFF,
                                      int(seed) & (2**64 - 1), _stream_handle(a.device, stream)),
               "asr_gemm_bf16_sr")
    return c
