"""AdamWSR argument checking (no GPU)."""
import pytest
import torch

from stochastic_rounding_gb300.optim import AdamWSR


@pytest.mark.parametrize("kw", [dict(lr=-1.0), dict(eps=-1e-8), dict(betas=(1.0, 0.999)),
                                dict(betas=(0.9, -0.1)), dict(weight_decay=-0.1), dict(rounding="up"),
                                dict(seed=2**64), dict(check_errors="later"), dict(check_errors=2)])
def test_rejects_bad_arguments(kw):
    p = torch.nn.Parameter(torch.zeros(4))
    with pytest.raises(ValueError):
        AdamWSR([p], **kw)


def test_positions_follow_parameter_order():
    ps = [torch.nn.Parameter(torch.zeros(s)) for s in (3, 5, 7)]
    opt = AdamWSR([{"params": ps[:1]}, {"params": ps[1:]}])
    assert [opt.base_index(p) for p in ps] == [0, 3, 8]


def test_cpu_parameters_are_refused():
    p = torch.nn.Parameter(torch.zeros(4, dtype=torch.bfloat16))
    p.grad = torch.zeros(4, dtype=torch.bfloat16)
    opt = AdamWSR([p])
    with pytest.raises(ValueError, match="CUDA"):
        opt.step()


def test_base_offset_and_group_base_index():
    ps = [torch.nn.Parameter(torch.zeros(s)) for s in (3, 5, 7, 2)]
    opt = AdamWSR([{"params": ps[:2]}, {"params": ps[2:3], "base_index": 1000}, {"params": ps[3:]}],
                  base_offset=2**40 + 1)
    assert [opt.base_index(p) for p in ps] == [2**40 + 1, 2**40 + 4, 1000, 1007]
    opt.add_param_group({"params": [torch.nn.Parameter(torch.zeros(4))], "base_index": 5})
    assert opt.base_index(opt.param_groups[-1]["params"][0]) == 5
    with pytest.raises(ValueError):
        AdamWSR(ps, base_offset=-1)
    with pytest.raises(ValueError):
        AdamWSR([torch.nn.Parameter(torch.zeros(8))], base_offset=2**64 - 4)


def test_positions_survive_a_state_dict_round_trip():
    ps = [torch.nn.Parameter(torch.zeros(s)) for s in (3, 5)]
    a = AdamWSR([{"params": ps[:1]}, {"params": ps[1:], "base_index": 77}], base_offset=9)
    qs = [torch.nn.Parameter(torch.zeros(s)) for s in (3, 5)]
    b = AdamWSR([{"params": qs[:1]}, {"params": qs[1:]}], base_offset=9)
    assert b.base_index(qs[1]) == 12
    b.load_state_dict(a.state_dict())
    assert [b.base_index(q) for q in qs] == [a.base_index(p) for p in ps] == [9, 77]


class _FakeLib:
    """Stands in for the binding: records launches, reports set error bits."""

    def __init__(self, bits):
        self.bits = bits
        self.calls = []
        self.reads = 0

    def make_table(self, entries):
        return [e[4] for e in entries]

    _pack_table = make_table

    def asr_adamw_sr_multi_tensor(self, table, **kw):
        self.calls.append((list(table), kw["step"]))

    def asr_take_device_error(self, device=None):
        self.reads += 1
        return self.bits


def _fake_step(monkeypatch, bits, **kw):
    from stochastic_rounding_gb300 import optim
    fake = _FakeLib(bits)
    monkeypatch.setattr(optim, "_lib", fake)
    monkeypatch.setattr(AdamWSR, "_check", staticmethod(lambda p: None))
    ps = [torch.nn.Parameter(torch.zeros(s)) for s in (4, 6)]
    for p in ps:
        p.grad = torch.zeros_like(p)
    opt = AdamWSR(ps, base_offset=100, **kw)
    return opt, fake


def test_step_raises_when_a_kernel_reported_a_device_error(monkeypatch):
    from stochastic_rounding_gb300.optim import DeviceError
    opt, fake = _fake_step(monkeypatch, 1)
    with pytest.raises(DeviceError, match="0x1"):
        opt.step()
    assert fake.calls == [([100, 104], 1)] and fake.reads == 1
    opt.step(check_errors=False)              # per-call override: no read
    assert fake.reads == 1


def test_step_without_error_checks_reads_nothing(monkeypatch):
    opt, fake = _fake_step(monkeypatch, 1, check_errors=False)
    opt.step()
    opt.step()
    assert fake.reads == 0 and [s for _, s in fake.calls] == [1, 2]
    fake.bits = 0
    opt.step(check_errors=True)               # clean word: no exception
    assert fake.reads == 1


def test_a_refused_parameter_leaves_every_group_unstepped(monkeypatch):
    """A parameter the optimizer refuses in the second group raises before
    the first group is launched, and no step count moves."""
    from stochastic_rounding_gb300 import optim
    fake = _FakeLib(0)
    refused = set()

    def check(p):
        if id(p) in refused:
            raise ValueError("refused parameter")

    monkeypatch.setattr(optim, "_lib", fake)
    monkeypatch.setattr(AdamWSR, "_check", staticmethod(check))
    a, b = torch.nn.Parameter(torch.zeros(4)), torch.nn.Parameter(torch.zeros(6))
    a.grad, b.grad = torch.zeros(4), torch.zeros(6)
    opt = AdamWSR([{"params": [a]}, {"params": [b]}])
    refused.add(id(b))
    with pytest.raises(ValueError, match="refused"):
        opt.step()
    assert fake.calls == [] and len(opt.state) == 0
    refused.clear()
    opt.step()
    assert [s for _, s in fake.calls] == [1, 1] and opt.state[a]["step"] == 1


def test_takes_torch_adamw_keywords():
    """The keywords of torch.optim.AdamW are accepted where they change
    nothing and refused where the fused step cannot honour them."""
    p = torch.nn.Parameter(torch.zeros(4))
    AdamWSR([p], 1e-3, (0.9, 0.999), 1e-8, 1e-2, False, maximize=False, foreach=True, capturable=True,
            differentiable=False, fused=True)
    for kw in (dict(amsgrad=True), dict(maximize=True), dict(differentiable=True)):
        with pytest.raises(ValueError, match="does not support"):
            AdamWSR([p], **kw)
