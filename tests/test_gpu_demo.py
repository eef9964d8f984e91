"""The pages' sub-ULP demonstration ("adamw-sr", introduction) through the
CUDA path: AdamW on the loss (w - 1.5)^2 from w = 1.0 with bf16 weights and
no fp32 master copy, lr 1e-4 (about a fortieth of the bf16 spacing below
1.0), 6,000 steps.  Every step is bit-exact against the oracle run in
lockstep; with nearest rounding the mean weight stays exactly 1.0; with
stochastic rounding it climbs with the unrounded binary64 trajectory toward
the 1.5 target; a rerun gives the same bits."""
import numpy as np
import pytest

import pins
from gpu_util import host, torch_cuda
from stochastic_rounding_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def asr():
    torch_cuda()
    from stochastic_rounding_gb300 import build
    build.build()
    import stochastic_rounding_gb300 as m
    m.lib()
    return m


def _run(asr, orc, rounding, n, check_every=500):
    """The demo on the GPU, the oracle in lockstep (compared every
    check_every steps); returns the final bf16 weights and the mean at each
    thousandth step."""
    import torch
    d = pins.load_demo()
    hp = dict(lr=d["update"], beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    w = torch.full((n,), d["start"], dtype=torch.bfloat16, device="cuda")
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    wo = np.full(n, W.to_bf16_bits(np.array([d["start"]], np.float32))[0], np.uint16)
    mo = np.zeros(n, np.float32)
    vo = np.zeros(n, np.float32)
    target = np.float32(d["sr_target"])
    means = {}
    for k in range(1, d["steps"] + 1):
        g = 2.0 * (w.float() - d["sr_target"])          # exact in binary32 for w in [1, 2)
        asr.asr_adamw_sr_step(w, g, m, v, step=k, seed=7, rounding=rounding, **hp)
        if orc is not None:
            go = (np.float32(2.0) * (W.bf16_bits_to_f32(wo) - target)).astype(np.float32)
            orc.adamw_step(wo, go, mo, vo, step=k, seed=7, rounding=0 if rounding == "sr" else 1, **hp)
            if k % check_every == 0:
                assert np.array_equal(host(w), wo), f"{rounding} weights differ from the oracle at step {k}"
                assert np.array_equal(host(m).view(np.uint32), mo.view(np.uint32)), f"m at step {k}"
                assert np.array_equal(host(v).view(np.uint32), vo.view(np.uint32)), f"v at step {k}"
        if k % 1000 == 0:
            means[k] = float(w.float().mean())
    return host(w), means


def _unrounded(d, steps):
    """The same optimisation in binary64 with no rounding at all."""
    w, m, v, out = d["start"], 0.0, 0.0, {}
    for k in range(1, steps + 1):
        g = 2.0 * (w - d["sr_target"])
        m = 0.9 * m + 0.1 * g
        v = 0.999 * v + 0.001 * g * g
        w -= d["update"] * (m / (1 - 0.9 ** k)) / (np.sqrt(v / (1 - 0.999 ** k)) + 1e-8)
        out[k] = w
    return out


def test_subulp_demo_through_the_kernels(asr, orc):
    d = pins.load_demo()
    n = 4096
    w_rn, means_rn = _run(asr, orc, "rne", n)
    assert all(mean == d["rn_final_mean"] for mean in means_rn.values()), means_rn
    assert np.all(W.bf16_bits_to_f32(w_rn) == d["start"])
    w_sr, means_sr = _run(asr, orc, "sr", n)
    ref = _unrounded(d, d["steps"])
    prev = d["start"]
    for k in sorted(means_sr):
        # the SR mean follows the unrounded run (the oracle pin's bound) and keeps rising toward 1.5
        assert abs(means_sr[k] - ref[k]) < 0.01, (k, means_sr[k], ref[k])
        assert prev < means_sr[k] < d["sr_target"], (k, means_sr[k])
        prev = means_sr[k]
    again, _ = _run(asr, None, "sr", n)
    assert np.array_equal(again, w_sr), "a rerun of the SR demo gave different bits"
