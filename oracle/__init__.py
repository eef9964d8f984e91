"""CPU oracle for the fused AdamW step with Philox-keyed stochastic rounding.

TEST INFRASTRUCTURE ONLY: the plain single-threaded C checker (``asr_oracle.c``)
and a ctypes loader for it.  The tests, the smoke check and the benchmark's
CPU-baseline leg are its only users; the product library never imports it.

Every method below marshals numpy arrays into the C code and back; no
arithmetic of the method happens in Python.
"""
import ctypes

import numpy as np

from . import build as _build

U16P = ctypes.POINTER(ctypes.c_uint16)
U32P = ctypes.POINTER(ctypes.c_uint32)
F32P = ctypes.POINTER(ctypes.c_float)

F32, BF16 = 0, 1          # dtype codes
ROUND_SR, ROUND_RNE = 0, 1


def _ptr(a, ct):
    return a.ctypes.data_as(ct)


def _need(a, dtype):
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags["C_CONTIGUOUS"]:
        raise TypeError(f"expected a C-contiguous numpy array of {np.dtype(dtype)}")
    if not a.flags["WRITEABLE"]:
        raise TypeError("array must be writeable")


class Oracle:
    """ctypes view of one build of ``asr_oracle.c``."""

    def __init__(self, path):
        L = ctypes.CDLL(path)
        L.oracle_philox4x32_10.argtypes = [U32P, U32P, U32P]
        L.oracle_philox4x32_10.restype = None
        L.oracle_element_word.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64]
        L.oracle_element_word.restype = ctypes.c_uint32
        L.oracle_philox_fill.argtypes = [U32P, ctypes.c_uint64, ctypes.c_uint64,
                                         ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint64]
        L.oracle_philox_fill.restype = None
        L.oracle_sr_bf16.argtypes = [ctypes.c_float, ctypes.c_uint32]
        L.oracle_sr_bf16.restype = ctypes.c_uint16
        L.oracle_rne_bf16.argtypes = [ctypes.c_float]
        L.oracle_rne_bf16.restype = ctypes.c_uint16
        L.oracle_rne_fill.argtypes = [F32P, U16P, ctypes.c_uint64]
        L.oracle_rne_fill.restype = None
        L.oracle_sr_fill.argtypes = [F32P, U32P, U16P, ctypes.c_uint64, ctypes.c_uint64,
                                     ctypes.c_uint32, ctypes.c_uint64]
        L.oracle_sr_fill.restype = None
        L.oracle_gemm_bf16.argtypes = [U16P, U16P, F32P, U16P, ctypes.c_uint64, ctypes.c_uint64,
                                       ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int,
                                       ctypes.c_uint32, ctypes.c_uint64]
        L.oracle_gemm_bf16.restype = None
        L.oracle_adamw_scalars.argtypes = [ctypes.c_double] * 5 + [ctypes.c_uint32, F32P]
        L.oracle_adamw_scalars.restype = None
        L.oracle_adamw_step.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_int, F32P, F32P, ctypes.c_uint64,
                                        ctypes.c_uint64, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int]
        L.oracle_adamw_step.restype = None
        L.oracle_mul_add.argtypes = [ctypes.c_float] * 3
        L.oracle_mul_add.restype = ctypes.c_float
        self.lib = L
        self.path = path

    # -- Philox ---------------------------------------------------------------
    def philox4x32_10(self, ctr, key):
        """Philox4x32-10 of one 4-word counter under a 2-word key -> 4 uint32."""
        c = np.array(ctr, dtype=np.uint32)
        k = np.array(key, dtype=np.uint32)
        out = np.zeros(4, dtype=np.uint32)
        self.lib.oracle_philox4x32_10(_ptr(c, U32P), _ptr(k, U32P), _ptr(out, U32P))
        return out

    def element_word(self, i, step, seed):
        """The 32-bit Philox word global element ``i`` draws at (seed, step)."""
        return int(self.lib.oracle_element_word(int(i), int(step), int(seed)))

    def philox_fill(self, n_ctr, ctr_base, ctr2, ctr3, seed):
        """Words of ``n_ctr`` consecutive counters, shape (n_ctr, 4) uint32."""
        out = np.zeros((int(n_ctr), 4), dtype=np.uint32)
        self.lib.oracle_philox_fill(_ptr(out, U32P), int(n_ctr), int(ctr_base), int(ctr2),
                                    int(ctr3), int(seed))
        return out

    # -- rounding -------------------------------------------------------------
    def sr_bf16(self, x, r):
        """One stochastic rounding f32 -> bf16 bit pattern."""
        return int(self.lib.oracle_sr_bf16(float(np.float32(x)), int(r)))

    def rne_bf16(self, x):
        """One round-to-nearest-even f32 -> bf16 bit pattern."""
        return int(self.lib.oracle_rne_bf16(float(np.float32(x))))

    def rne_fill(self, x):
        """Round a float32 array to nearest-even bf16 patterns (uint16)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.zeros(x.shape, dtype=np.uint16)
        self.lib.oracle_rne_fill(_ptr(x, F32P), _ptr(out, U16P), x.size)
        return out

    def sr_fill(self, x, base_index, step, seed, rbits=None):
        """Stochastically round a float32 array to bf16 patterns (uint16)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.zeros(x.shape, dtype=np.uint16)
        rb = None
        if rbits is not None:
            rb = np.ascontiguousarray(rbits, dtype=np.uint32)
            if rb.shape != x.shape:
                raise ValueError("rbits must match x")
        self.lib.oracle_sr_fill(_ptr(x, F32P), _ptr(rb, U32P) if rb is not None else None,
                                _ptr(out, U16P), x.size, int(base_index), int(step), int(seed))
        return out

    # -- GEMM -----------------------------------------------------------------
    def gemm_bf16(self, a, b, *, row0=0, rounding=ROUND_SR, step=0, seed=0):
        """Rows row0 .. row0+m-1 of C = A.B^T rounded to bf16, and their
        binary32 accumulators: ``a`` (m x k) and ``b`` (n x k) uint16 arrays of
        bf16 patterns.  Returns (out uint16 (m, n), acc float32 (m, n))."""
        a = np.ascontiguousarray(a, dtype=np.uint16)
        b = np.ascontiguousarray(b, dtype=np.uint16)
        if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
            raise ValueError("a is m x k and b is n x k")
        m, k = a.shape
        n = b.shape[0]
        out = np.zeros((m, n), dtype=np.uint16)
        acc = np.zeros((m, n), dtype=np.float32)
        self.lib.oracle_gemm_bf16(_ptr(a, U16P), _ptr(b, U16P), _ptr(acc, F32P), _ptr(out, U16P),
                                  m, n, k, int(row0), int(rounding), int(step), int(seed))
        return out, acc

    # -- AdamW ----------------------------------------------------------------
    def adamw_scalars(self, lr, beta1, beta2, eps, weight_decay, step):
        """The eight binary32 per-step scalars (b1, b2, eps, decay, omb1, omb2,
        step_size, bc2s)."""
        out = np.zeros(8, dtype=np.float32)
        self.lib.oracle_adamw_scalars(float(lr), float(beta1), float(beta2), float(eps),
                                      float(weight_decay), int(step), _ptr(out, F32P))
        return out

    def adamw_step(self, param, grad, exp_avg, exp_avg_sq, *, lr, beta1, beta2, eps,
                   weight_decay, step, seed, base_index=0, rounding=ROUND_SR):
        """One AdamW-SR step, in place.

        ``param``: float32 array, or uint16 array of bf16 patterns.
        ``grad``: float32 array, or uint16 array of bf16 patterns.
        ``exp_avg``/``exp_avg_sq``: float32.  All of one length.
        """
        n = param.size
        for a in (grad, exp_avg, exp_avg_sq):
            if a.size != n:
                raise ValueError("all arrays must have the same number of elements")
        pdt = BF16 if param.dtype == np.uint16 else F32
        gdt = BF16 if grad.dtype == np.uint16 else F32
        _need(param, np.uint16 if pdt == BF16 else np.float32)
        _need(exp_avg, np.float32)
        _need(exp_avg_sq, np.float32)
        grad = np.ascontiguousarray(grad)
        if grad.dtype != (np.uint16 if gdt == BF16 else np.float32):
            raise TypeError("grad must be float32 or uint16 (bf16 patterns)")
        self.lib.oracle_adamw_step(param.ctypes.data, pdt, grad.ctypes.data, gdt,
                                   _ptr(exp_avg, F32P), _ptr(exp_avg_sq, F32P), n,
                                   int(base_index), float(lr), float(beta1), float(beta2),
                                   float(eps), float(weight_decay), int(step), int(seed),
                                   int(rounding))

    def mul_add(self, a, b, c):
        """(a*b)+c with two binary32 roundings, as the oracle build evaluates it."""
        return float(self.lib.oracle_mul_add(float(a), float(b), float(c)))


_default = None


def get():
    """The oracle built from ``asr_oracle.c`` (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def compile_variant(source_text, out_path):
    """Compile a (test-modified) copy of the oracle source with the oracle's
    own flags and load it; used by tests that plant a mistake in the oracle
    to show the pins catch it."""
    import os
    import subprocess
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", *_build.CFLAGS, "-o", out_path, src, "-lm"], check=True)
    os.remove(src)
    return Oracle(out_path)


def source_text():
    """The oracle's C source."""
    with open(_build.SRC) as f:
        return f.read()
