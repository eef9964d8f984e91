"""Independent Philox4x32-10 reference for the oracle's pins.

Runs Triton's library Philox (``tl.philox``, the generator behind ``tl.rand``)
in Triton's CPU interpreter -- no GPU involved -- over counters and keys read
from an .npz file, and writes the four output words per counter back.  It is
run in a child process because the interpreter must be selected before Triton
is imported.  Test infrastructure only.

usage: python philox_triton_ref.py IN.npz OUT.npy
  IN.npz holds uint32 arrays c0, c1, c2, c3 (the counter words) and uint64
  array seed (the key is (seed lo32, seed hi32)), all of one length.
"""
import os
import sys

os.environ["TRITON_INTERPRET"] = "1"

import numpy as np  # noqa: E402
import torch  # noqa: E402
import triton  # noqa: E402
import triton.language as tl  # noqa: E402


@triton.jit
def _philox_kernel(out_ptr, c0_ptr, c1_ptr, c2_ptr, c3_ptr, seed_ptr, N: tl.constexpr):
    offs = tl.arange(0, N)
    c0 = tl.load(c0_ptr + offs)
    c1 = tl.load(c1_ptr + offs)
    c2 = tl.load(c2_ptr + offs)
    c3 = tl.load(c3_ptr + offs)
    seed = tl.load(seed_ptr + offs)
    w0, w1, w2, w3 = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out_ptr + offs * 4 + 0, w0)
    tl.store(out_ptr + offs * 4 + 1, w1)
    tl.store(out_ptr + offs * 4 + 2, w2)
    tl.store(out_ptr + offs * 4 + 3, w3)


def main(inp, outp):
    d = np.load(inp)
    n = d["c0"].size
    N = 1
    while N < n:
        N *= 2
    pad = lambda a: np.concatenate([a, np.zeros(N - n, dtype=a.dtype)])  # noqa: E731
    as_t = lambda a: torch.from_numpy(pad(a).view(np.int32))  # noqa: E731
    seeds = torch.from_numpy(pad(d["seed"].astype(np.uint64)).view(np.int64))
    out = torch.zeros(4 * N, dtype=torch.int32)
    _philox_kernel[(1,)](out, as_t(d["c0"]), as_t(d["c1"]), as_t(d["c2"]), as_t(d["c3"]),
                         seeds, N=N)
    np.save(outp, out.numpy().view(np.uint32).reshape(N, 4)[:n])


if __name__ == "__main__":
    main(sys.argv[1], sys.argv[2])
