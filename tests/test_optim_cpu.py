"""AdamWSR argument checking (no GPU)."""
import pytest
import torch

from stochastic_rounding_gb300.optim import AdamWSR


@pytest.mark.parametrize("kw", [dict(lr=-1.0), dict(eps=-1e-8), dict(betas=(1.0, 0.999)),
                                dict(betas=(0.9, -0.1)), dict(weight_decay=-0.1), dict(rounding="up"),
                                dict(seed=2**64)])
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
