"""Shared test set-up: markers, import path, and the Philox reference batch."""
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.get()


@pytest.fixture(scope="session")
def philox_ref():
    """(cases, words): random Philox cases and the words Triton's library
    Philox gives for them, computed in its CPU interpreter (child process)."""
    pytest.importorskip("triton")
    import pins
    cases = pins.make_philox_cases()
    with tempfile.TemporaryDirectory() as td:
        inp = os.path.join(td, "in.npz")
        out = os.path.join(td, "out.npy")
        np.savez(inp, **cases["inputs"])
        env = dict(os.environ, TRITON_INTERPRET="1", CUDA_VISIBLE_DEVICES="")
        r = subprocess.run([sys.executable, os.path.join(HERE, "philox_triton_ref.py"), inp, out],
                           env=env, capture_output=True, text=True, timeout=600)
        if r.returncode != 0:
            pytest.skip("Triton interpreter unavailable: " + r.stderr.strip().splitlines()[-1]
                        if r.stderr.strip() else "Triton interpreter unavailable")
        words = np.load(out)
    return cases, words
