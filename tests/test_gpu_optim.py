"""The AdamWSR optimizer class ("adamw-sr", Usage) and the bf16-only
training claim ("adamw-sr", Correctness: a layer kept only in bf16, with no
fp32 master copy, still learns under SR and ends with a lower loss than under
nearest rounding)."""
import io

import numpy as np
import pytest

from gpu_util import torch_cuda

pytestmark = pytest.mark.gpu
HP = dict(lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
SHAPES = [(64, 33), (7,), (128, 128), (1000,), (3, 5, 7)]


@pytest.fixture(scope="module")
def asr():
    torch_cuda()
    from stochastic_rounding_gb300 import build
    build.build()
    import stochastic_rounding_gb300 as m
    m.lib()
    return m


def _params(dtype, seed=0):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return [torch.nn.Parameter((torch.randn(s, device="cuda", generator=g) * 0.02).to(dtype)) for s in SHAPES]


def _grads(params, step, dtype=None):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 + step)
    return [(torch.randn(p.shape, device="cuda", generator=g) * 1e-3).to(dtype or p.dtype) for p in params]


def _bits(t):
    import torch
    return t.detach().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).clone()


def test_fp32_tracks_torch_adamw(asr):
    import torch
    ours = _params(torch.float32)
    ref = [torch.nn.Parameter(p.detach().clone()) for p in ours]
    opt = asr.AdamWSR(ours, **HP, seed=3)
    topt = torch.optim.AdamW(ref, **HP, foreach=False, fused=False)
    for step in range(1, 101):
        for p, r, g in zip(ours, ref, _grads(ours, step)):
            p.grad = g
            r.grad = g.clone()
        opt.step()
        topt.step()
    d = max(float((p.detach().double() - r.detach().double()).abs().max()) for p, r in zip(ours, ref))
    assert d < 1e-4


def test_bf16_equals_direct_calls_with_global_positions(asr):
    import torch
    ours = _params(torch.bfloat16, 1)
    copies = [p.detach().clone() for p in ours]
    ms = [torch.zeros(p.shape, device="cuda") for p in ours]
    vs = [torch.zeros(p.shape, device="cuda") for p in ours]
    opt = asr.AdamWSR(ours, **HP, seed=2**40 + 1)
    base, bases = 0, []
    for p in ours:
        bases.append(base)
        base += p.numel()
    assert [opt.base_index(p) for p in ours] == bases
    for step in range(1, 4):
        grads = _grads(ours, step)
        for p, g in zip(ours, grads):
            p.grad = g
        opt.step()
        for c, g, m, v, b in zip(copies, grads, ms, vs, bases):
            asr.asr_adamw_sr_step(c, g, m, v, lr=HP["lr"], beta1=0.9, beta2=0.999, eps=HP["eps"],
                                  weight_decay=HP["weight_decay"], step=step, seed=2**40 + 1, base_index=b)
    for p, c, m, v in zip(ours, copies, ms, vs):
        assert torch.equal(_bits(p), _bits(c))
        assert torch.equal(_bits(opt.state[p]["exp_avg"]), _bits(m))
        assert torch.equal(_bits(opt.state[p]["exp_avg_sq"]), _bits(v))
        assert opt.state[p]["exp_avg"].dtype == torch.float32


def test_state_dict_resume_is_bitwise(asr):
    import torch
    a = _params(torch.bfloat16, 2)
    b = [torch.nn.Parameter(p.detach().clone()) for p in a]
    oa = asr.AdamWSR(a, **HP, seed=9)
    for step in range(1, 11):
        for p, g in zip(a, _grads(a, step)):
            p.grad = g
        oa.step()
    ob = asr.AdamWSR(b, **HP, seed=9)
    for step in range(1, 6):
        for p, g in zip(b, _grads(b, step)):
            p.grad = g
        ob.step()
    buf = io.BytesIO()
    torch.save({"opt": ob.state_dict(), "params": [p.detach().cpu() for p in b]}, buf)
    buf.seek(0)
    saved = torch.load(buf, weights_only=False)
    c = [torch.nn.Parameter(t.to("cuda")) for t in saved["params"]]
    oc = asr.AdamWSR(c, **HP, seed=0)
    oc.load_state_dict(saved["opt"])
    assert oc.param_groups[0]["seed"] == 9
    for p in c:
        assert oc.state[p]["exp_avg"].dtype == torch.float32
    for step in range(6, 11):
        for p, g in zip(c, _grads(c, step)):
            p.grad = g
        oc.step()
    for p, q in zip(a, c):
        assert torch.equal(_bits(p), _bits(q))
        assert torch.equal(_bits(oa.state[p]["exp_avg_sq"]), _bits(oc.state[q]["exp_avg_sq"]))


def test_param_groups_and_missing_grads(asr):
    import torch
    ps = _params(torch.bfloat16, 3)
    copies = [p.detach().clone() for p in ps]
    opt = asr.AdamWSR([{"params": ps[:2], "lr": 3e-3, "weight_decay": 0.1},
                       {"params": ps[2:], "rounding": "rne"}], **HP, seed=5)
    bases = [opt.base_index(p) for p in ps]
    grads = _grads(ps, 1)
    for i, (p, g) in enumerate(zip(ps, grads)):
        p.grad = None if i == 3 else g
    opt.step()
    for i, (p, c, g, b) in enumerate(zip(ps, copies, grads, bases)):
        if i == 3:
            assert torch.equal(_bits(p), _bits(c)) and p not in opt.state
            continue
        lr, wd, rnd = (3e-3, 0.1, "sr") if i < 2 else (HP["lr"], HP["weight_decay"], "rne")
        m = torch.zeros(p.shape, device="cuda")
        v = torch.zeros(p.shape, device="cuda")
        asr.asr_adamw_sr_step(c, g, m, v, lr=lr, beta1=0.9, beta2=0.999, eps=HP["eps"], weight_decay=wd,
                              step=1, seed=5, base_index=b, rounding=rnd)
        assert torch.equal(_bits(p), _bits(c)), f"param {i}"


def test_seed_keys_the_rounding(asr):
    import torch
    outs = []
    for seed in (1, 1, 2):
        ps = _params(torch.bfloat16, 4)
        opt = asr.AdamWSR(ps, **HP, seed=seed)
        for p, g in zip(ps, _grads(ps, 1)):
            p.grad = g
        opt.step()
        outs.append(torch.cat([_bits(p).view(-1) for p in ps]))
    assert torch.equal(outs[0], outs[1]) and not torch.equal(outs[0], outs[2])


def _regression(asr, rounding, steps=1500, seed=0):
    """Least squares y = X W*, W (512 x 16) kept only in bf16 (no fp32
    master), AdamW lr 2e-3, full-batch gradient computed in fp32 and handed
    to the optimizer in bf16 (torch keeps .grad in the parameter's dtype).
    Returns the loss history."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    n, d, o = 4096, 512, 16
    X = torch.randn(n, d, device="cuda", generator=g) / d ** 0.5
    W_true = torch.randn(d, o, device="cuda", generator=g)
    y = X @ W_true
    W = torch.nn.Parameter(torch.zeros(d, o, device="cuda", dtype=torch.bfloat16))
    opt = asr.AdamWSR([W], lr=2e-3, weight_decay=0.0, seed=seed, rounding=rounding)
    hist = []
    for _ in range(steps):
        r = X @ W.float() - y
        hist.append(float((r * r).mean()))
        W.grad = ((2.0 / n) * (X.t() @ r)).to(torch.bfloat16)
        opt.step()
    return hist


def test_bf16_only_layer_sr_out_trains_round_to_nearest(asr):
    sr = _regression(asr, "sr")
    rn = _regression(asr, "rne")
    assert sr[-1] < 0.05 * sr[0], "SR did not converge"
    assert sr[-1] < 0.5 * rn[-1], f"SR final loss {sr[-1]:.4g} does not beat RNE {rn[-1]:.4g}"
    # RNE stalls: over the last third its loss hardly moves
    assert rn[-1] > 0.9 * rn[len(rn) * 2 // 3]
    assert sr == _regression(asr, "sr"), "SR training is not reproducible"
