"""The AdamWSR optimizer class ("adamw-sr", Usage) and the bf16-only
training claim ("adamw-sr", Correctness: a layer kept only in bf16, with no
fp32 master copy, still learns under SR and ends with a lower loss than under
nearest rounding)."""
import io

import numpy as np
import pytest

from gpu_util import assert_same_bits, host, torch_cuda
from stochastic_rounding_gb300 import workloads as W

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


def _regression(asr, rounding, steps=1500, seed=0, orc=None, oracle_steps=0):
    """Least squares y = X W*, W (512 x 16) kept only in bf16 (no fp32
    master), AdamW lr 2e-3, full-batch gradient computed in fp32 and handed
    to the optimizer in bf16 (torch keeps .grad in the parameter's dtype).
    Returns the loss history.  With ``orc``, the first ``oracle_steps``
    steps are also taken by the oracle on host copies of W and its moments,
    fed the very bf16 gradients the optimizer got, and W, m and v must match
    it bit for bit after each of them."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    n, d, o = 4096, 512, 16
    X = torch.randn(n, d, device="cuda", generator=g) / d ** 0.5
    W_true = torch.randn(d, o, device="cuda", generator=g)
    y = X @ W_true
    W = torch.nn.Parameter(torch.zeros(d, o, device="cuda", dtype=torch.bfloat16))
    opt = asr.AdamWSR([W], lr=2e-3, weight_decay=0.0, seed=seed, rounding=rounding)
    hw = host(W)
    hm = np.zeros(d * o, np.float32)
    hv = np.zeros(d * o, np.float32)
    hist = []
    for k in range(steps):
        r = X @ W.detach().float() - y
        hist.append(float((r * r).mean()))
        W.grad = ((2.0 / n) * (X.t() @ r)).to(torch.bfloat16)
        opt.step()
        if orc is not None and k < oracle_steps:
            hw = hw.reshape(-1)
            orc.adamw_step(hw, host(W.grad).reshape(-1), hm, hv, lr=2e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                           weight_decay=0.0, step=k + 1, seed=seed, base_index=0,
                           rounding=0 if rounding == "sr" else 1)
            assert_same_bits(host(W).reshape(-1), hw, f"{rounding} step {k + 1}: W")
            assert_same_bits(host(opt.state[W]["exp_avg"]).reshape(-1), hm, f"{rounding} step {k + 1}: m")
            assert_same_bits(host(opt.state[W]["exp_avg_sq"]).reshape(-1), hv, f"{rounding} step {k + 1}: v")
    return hist


def test_bf16_only_layer_sr_out_trains_round_to_nearest(asr, orc):
    sr = _regression(asr, "sr", orc=orc, oracle_steps=20)
    rn = _regression(asr, "rne", orc=orc, oracle_steps=20)
    assert sr[-1] < 0.05 * sr[0], "SR did not converge"
    assert sr[-1] < 0.5 * rn[-1], f"SR final loss {sr[-1]:.4g} does not beat RNE {rn[-1]:.4g}"
    # RNE stalls: over the last third its loss hardly moves
    assert rn[-1] > 0.9 * rn[len(rn) * 2 // 3]
    assert sr == _regression(asr, "sr"), "SR training is not reproducible"


def _host_param(rng, shape, dtype):
    x = W.normal_f32(rng, int(np.prod(shape)), 0.02)
    return W.to_bf16_bits(x) if dtype == "bf16" else x


def _to_dev(a, shape):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).to("cuda").view(torch.bfloat16).view(shape)
    return torch.from_numpy(a.copy()).to("cuda").view(shape)


def test_optimizer_equals_oracle_mixed_groups(asr, orc):
    """AdamWSR against the oracle element by element after every one of 5
    steps: bf16 and f32 parameters (torch keeps each .grad in its parameter's
    dtype), two groups with different lr / weight decay / rounding, a third
    group placed by its own base_index, a global offset for the optimizer,
    one parameter that skips step 2 and one that first gets a gradient at
    step 3 (so a group holds parameters at different step counts)."""
    import torch
    rng = np.random.default_rng(5)
    shapes = [(64, 33), (7,), (128, 128), (1000,), (3, 5, 7), (4099,), (33,)]
    dts = ["bf16", "f32", "bf16", "f32", "bf16", "bf16", "f32"]
    hp = [_host_param(rng, sh, dt) for sh, dt in zip(shapes, dts)]
    ps = [torch.nn.Parameter(_to_dev(a, sh)) for a, sh in zip(hp, shapes)]
    groups = [{"params": ps[:3], "lr": 3e-3, "weight_decay": 0.1},
              {"params": ps[3:6], "rounding": "rne"},
              {"params": ps[6:], "base_index": 2**36 + 2}]
    opt = asr.AdamWSR(groups, **HP, seed=2**63 + 5, base_offset=2**33 + 3)
    cfg = [(3e-3, 0.1, 0)] * 3 + [(HP["lr"], HP["weight_decay"], 1)] * 3 + [(HP["lr"], HP["weight_decay"], 0)]
    hm = [np.zeros(a.size, np.float32) for a in hp]
    hv = [np.zeros(a.size, np.float32) for a in hp]
    steps = [0] * len(ps)
    bases = [opt.base_index(p) for p in ps]
    assert bases[0] == 2**33 + 3 and bases[6] == 2**36 + 2
    for k in range(1, 6):
        has_grad = [not (i == 4 and k == 2) and not (i == 5 and k < 3) for i in range(len(ps))]
        for i, (p, sh, dt) in enumerate(zip(ps, shapes, dts)):
            if not has_grad[i]:
                p.grad = None
                continue
            g = W.normal_f32(rng, int(np.prod(sh)), 1e-3)
            g = W.to_bf16_bits(g) if dt == "bf16" else g
            p.grad = _to_dev(g, sh)
            steps[i] += 1
            lr, wd, rnd = cfg[i]
            orc.adamw_step(hp[i], g, hm[i], hv[i], lr=lr, beta1=0.9, beta2=0.999, eps=HP["eps"],
                           weight_decay=wd, step=steps[i], seed=2**63 + 5, base_index=bases[i], rounding=rnd)
        opt.step()
        torch.cuda.synchronize()
        for i, p in enumerate(ps):
            assert_same_bits(host(p).reshape(-1), hp[i], f"step {k}: param {i}")
            if steps[i]:
                assert opt.state[p]["step"] == steps[i]
                assert_same_bits(host(opt.state[p]["exp_avg"]).reshape(-1), hm[i], f"step {k}: exp_avg {i}")
                assert_same_bits(host(opt.state[p]["exp_avg_sq"]).reshape(-1), hv[i], f"step {k}: exp_avg_sq {i}")
            else:
                assert p not in opt.state


def test_rank_local_optimizers_equal_the_whole(asr, orc):
    """Two AdamWSR instances that own the two halves of a model's flat
    parameter vector, cut inside a tensor at an odd position, each given its
    half's start as base_offset: after 3 steps their pieces equal, bit for
    bit, one AdamWSR over the whole model, and the oracle ("adamw-sr",
    Method: identical whether updated whole or split across ranks)."""
    import torch
    from stochastic_rounding_gb300 import sharding
    rng = np.random.default_rng(6)
    sizes = [1000, 3001, 517, 2048]
    dts = ["bf16", "bf16", "f32", "bf16"]
    total = sum(sizes)
    hp = [_host_param(rng, (n,), dt) for n, dt in zip(sizes, dts)]
    whole = [torch.nn.Parameter(_to_dev(a, (a.size,))) for a in hp]
    opt_whole = asr.AdamWSR(whole, **HP, seed=11)
    ranks = []
    for r in range(2):
        start, end = sharding.shard_bounds(total, 2, r, align=1)
        pieces = sharding.shard_pieces(sizes, start, end)
        params = [torch.nn.Parameter(_to_dev(hp[t][off:off + n], (n,))) for t, off, n, _ in pieces]
        opt = asr.AdamWSR(params, **HP, seed=11, base_offset=start)
        assert [opt.base_index(p) for p in params] == [b for _, _, _, b in pieces]
        ranks.append((pieces, params, opt))
    cut = ranks[1][0][0][3]
    assert cut % 4 != 0 and ranks[1][0][0][1] > 0, "the cut must fall inside a tensor, off a multiple of 4"
    hm = [np.zeros(n, np.float32) for n in sizes]
    hv = [np.zeros(n, np.float32) for n in sizes]
    for step in range(1, 4):
        grads = [W.normal_f32(rng, n, 1e-3) for n in sizes]
        grads = [W.to_bf16_bits(g) if dt == "bf16" else g for g, dt in zip(grads, dts)]
        for p, g in zip(whole, grads):
            p.grad = _to_dev(g, (g.size,))
        for pieces, params, _ in ranks:
            for (t, off, n, _), p in zip(pieces, params):
                p.grad = _to_dev(grads[t][off:off + n], (n,))
        opt_whole.step()
        for _, _, opt in ranks:
            opt.step()
        for t in range(len(sizes)):
            orc.adamw_step(hp[t], grads[t], hm[t], hv[t], step=step, seed=11, base_index=sum(sizes[:t]),
                           lr=HP["lr"], beta1=0.9, beta2=0.999, eps=HP["eps"], weight_decay=HP["weight_decay"])
    torch.cuda.synchronize()
    for t, p in enumerate(whole):
        assert_same_bits(host(p), hp[t], f"whole: tensor {t}")
        assert_same_bits(host(opt_whole.state[p]["exp_avg_sq"]), hv[t], f"whole: exp_avg_sq {t}")
    for r, (pieces, params, opt) in enumerate(ranks):
        for (t, off, n, _), p in zip(pieces, params):
            assert np.array_equal(host(p).view(np.uint8), host(whole[t])[off:off + n].view(np.uint8)), \
                f"rank {r}: piece of tensor {t} differs from the whole-model update"
            assert_same_bits(host(opt.state[p]["exp_avg"]), hm[t][off:off + n], f"rank {r}: exp_avg of {t}")


def test_step_raises_after_a_device_error(asr):
    """A kernel's wait that gave up (the bounded-wait self-test raises the
    same bit) makes the next checked step raise instead of returning as if
    all were well; the bit is cleared by the read, so the step after that
    runs normally."""
    import torch
    ps = _params(torch.bfloat16, 7)
    opt = asr.AdamWSR(ps, **HP, seed=1)
    for p, g in zip(ps, _grads(ps, 1)):
        p.grad = g
    asr.asr_take_device_error()
    asr.asr_selftest_wait_timeout(1_000_000)
    with pytest.raises(asr.DeviceError):
        opt.step(check_errors=True)
    opt.step()
    asr.asr_selftest_wait_timeout(1_000_000)
    opt.step(check_errors=False)               # not read here ...
    assert asr.asr_take_device_error() == 1    # ... so it is still set


def test_deferred_error_check(asr):
    """check_errors="deferred": steps do not wait for the GPU; a device error
    raised during one step is reported by a later step() or by
    poll_errors(wait=True), and clean steps report nothing.  The parameters
    end as with the blocking check."""
    import torch
    a = _params(torch.bfloat16, 8)
    b = [torch.nn.Parameter(p.detach().clone()) for p in a]
    oa = asr.AdamWSR(a, **HP, seed=3, check_errors="deferred")
    ob = asr.AdamWSR(b, **HP, seed=3)
    asr.asr_take_device_error()
    for step in range(1, 7):
        for p, q, g in zip(a, b, _grads(a, step)):
            p.grad = g
            q.grad = g.clone()
        oa.step()
        ob.step()
    oa.poll_errors(wait=True)
    for p, q in zip(a, b):
        assert torch.equal(_bits(p), _bits(q))
    asr.asr_selftest_wait_timeout(1_000_000)
    oa.step()                                   # the bit is taken behind this step
    with pytest.raises(asr.DeviceError):
        oa.poll_errors(wait=True)
    oa.step()
    oa.poll_errors(wait=True)                   # clean again
    assert asr.asr_take_device_error() == 0
