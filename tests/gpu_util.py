"""Helpers for the GPU parity tests: host<->device copies of bf16 patterns
and float32 arrays, bit comparisons, and sampled windows for large runs."""
import numpy as np
import pytest


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def dev(a, device="cuda"):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(device)
    return torch.from_numpy(a).to(device)


def host(t):
    import torch
    a = t.detach().cpu()
    if a.dtype in (torch.int16, torch.bfloat16):
        return a.view(torch.int16).numpy().view(np.uint16).copy()
    if a.dtype == torch.int32:
        return a.numpy().view(np.uint32).copy()
    return a.numpy().copy()


def _nan_mask(a):
    if a.dtype == np.uint16:
        a32 = a.astype(np.uint32)
        return ((a32 & 0x7F80) == 0x7F80) & ((a32 & 0x7F) != 0)
    return np.isnan(a.view(np.float32))


def assert_same_bits(got, want, what="", nan_equal=True):
    """Bitwise equality; with nan_equal, any NaN matches any NaN (CPU and GPU
    arithmetic produce different NaN payloads)."""
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    gb = got.view(np.uint16 if got.dtype == np.uint16 else np.uint32)
    wb = want.view(np.uint16 if want.dtype == np.uint16 else np.uint32)
    diff = gb != wb
    if nan_equal:
        both_nan = _nan_mask(got) & _nan_mask(want)
        diff &= ~both_nan
    if diff.any():
        idx = np.nonzero(diff.reshape(-1))[0]
        i = idx[0]
        raise AssertionError(f"{what}: {idx.size} of {diff.size} elements differ; first at {i}: "
                             f"got {gb.reshape(-1)[i]:#x} want {wb.reshape(-1)[i]:#x}")


def pick_windows(rng, sizes, per_tensor=2, length=4096, whole_below=8192):
    """(tensor, start, length) windows: small tensors whole; for the others
    the head, the tail and random unaligned windows."""
    out = []
    for t, n in enumerate(sizes):
        if n <= whole_below:
            out.append((t, 0, n))
            continue
        out.append((t, 0, min(length, n)))
        out.append((t, n - min(length, n), min(length, n)))
        for _ in range(per_tensor):
            s = int(rng.integers(0, n - length))
            out.append((t, s, length))
    return out
