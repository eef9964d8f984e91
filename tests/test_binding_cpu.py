"""The multi-tensor wrappers of the binding against a stand-in library (no
GPU): one C call per wrapper call, None on success, AsrError carrying the
status otherwise -- never an exception after a call that succeeded, which
would invite a caller to retry and apply the step twice."""
import contextlib
import ctypes

import pytest

from stochastic_rounding_gb300 import _lib

NAMES = ("asr_adamw_sr_multi_tensor", "asr_adamw_sr_multi_tensor_static")


class _StubLib:
    def __init__(self, status):
        self.status = status
        self.calls = {n: 0 for n in NAMES}

    def __getattr__(self, name):
        if name in NAMES:
            def call(table, n, hp, stream):
                self.calls[name] += 1
                assert n == len(table) and hp._obj.step == 3
                return self.status
            return call
        raise AttributeError(name)

    @staticmethod
    def asr_status_string(s):
        return b"ASR_STATUS_%d" % s

    @staticmethod
    def asr_last_cuda_error():
        return 0


@pytest.fixture
def stub(monkeypatch):
    def make(status):
        s = _StubLib(status)
        monkeypatch.setattr(_lib, "_lib", s)
        monkeypatch.setattr(_lib, "_on_device", lambda d: contextlib.nullcontext())
        monkeypatch.setattr(_lib, "_stream_handle", lambda d, s: ctypes.c_void_p(None))
        return s
    return make


@pytest.mark.parametrize("name", NAMES)
def test_wrapper_returns_once_on_success(stub, name):
    s = stub(_lib.ASR_OK)
    table = (_lib.TensorDesc * 3)()
    assert getattr(_lib, name)(table, lr=1e-3, step=3, device="cpu") is None
    assert s.calls[name] == 1


@pytest.mark.parametrize("name", NAMES)
def test_wrapper_raises_the_status(stub, name):
    s = stub(_lib.ASR_ERR_INVALID_VALUE)
    table = (_lib.TensorDesc * 2)()
    with pytest.raises(_lib.AsrError) as e:
        getattr(_lib, name)(table, lr=1e-3, step=3, device="cpu")
    assert e.value.status == _lib.ASR_ERR_INVALID_VALUE and name in str(e.value)
    assert s.calls[name] == 1


def test_package_exports_both_wrappers():
    import stochastic_rounding_gb300 as asr
    for name in NAMES:
        assert getattr(asr, name) is getattr(_lib, name)


class _OnDevice(__import__("torch").Tensor):
    """A CPU tensor that reports itself as living on cuda:<idx>, so the
    binding's device checks can be exercised without a GPU (no pointer of
    it ever reaches the library here)."""

    @property
    def is_cuda(self):
        return True

    @property
    def device(self):
        import torch
        return torch.device("cuda", self._idx)

    def get_device(self):
        return self._idx


def _on(idx, *shape, dtype=None):
    import torch
    t = torch.Tensor._make_subclass(_OnDevice, torch.zeros(*shape, dtype=dtype or torch.float32))
    t._idx = idx
    return t


def test_tensors_on_another_device_are_refused_before_any_call(stub):
    """A kernel runs on one device: a grad, moment, output or operand on
    another device is refused by the binding instead of being handed to the
    kernel as a foreign pointer."""
    import torch
    fake = stub(_lib.ASR_OK)
    p, g, m, v = _on(0, 8, dtype=torch.bfloat16), _on(0, 8, dtype=torch.bfloat16), _on(0, 8), _on(0, 8)
    _lib.make_table([(p, g, m, v, 0)])                       # one device: accepted
    with pytest.raises(ValueError, match="cuda:1"):
        _lib.make_table([(p, g, m, v, 0), (_on(1, 8), _on(1, 8), _on(1, 8), _on(1, 8), 8)])
    with pytest.raises(ValueError, match="exp_avg_sq"):
        _lib.make_table([(p, g, m, _on(1, 8), 0)])
    with pytest.raises(ValueError, match="grad"):
        _lib.asr_adamw_sr_step(p, _on(1, 8, dtype=torch.bfloat16), m, v, lr=1e-3, step=1)
    with pytest.raises(ValueError, match="out"):
        _lib.asr_stochastic_round_bf16(_on(0, 8), _on(1, 8, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="b is on"):
        _lib.asr_gemm_bf16_sr(_on(0, 4, 8, dtype=torch.bfloat16), _on(1, 4, 8, dtype=torch.bfloat16),
                              _on(0, 4, 4, dtype=torch.bfloat16))
    assert sum(fake.calls.values()) == 0


def test_host_table_checks_its_host_tensors():
    """make_host_table: the device parts as make_table checks them, the host
    gradient of the gradient's dtype and size, the host params of the
    params' dtype and size or None; CPU tensors only (page-locking is the
    library's check)."""
    import torch
    p, g = _on(0, 8, dtype=torch.bfloat16), _on(0, 8, dtype=torch.float32)
    m, v = _on(0, 8), _on(0, 8)
    gh, ph = torch.zeros(8, dtype=torch.float32), torch.zeros(8, dtype=torch.int16)
    t = _lib.make_host_table([(p, g, m, v, 3, gh, ph), (p, g, m, v, 11, gh, None)])
    assert t[0].dev.base_index == 3 and t[0].grad_host == gh.data_ptr() and t[0].param_host == ph.data_ptr()
    assert t[1].param_host is None
    for bad_gh, bad_ph, err in ((torch.zeros(8, dtype=torch.bfloat16), ph, TypeError),
                                (torch.zeros(7), ph, ValueError),
                                (gh, torch.zeros(8), TypeError),
                                (gh, torch.zeros(9, dtype=torch.bfloat16), ValueError),
                                (_on(0, 8), ph, ValueError)):
        with pytest.raises(err):
            _lib.make_host_table([(p, g, m, v, 0, bad_gh, bad_ph)])


def test_e2e_chunks_follow_the_library_rule():
    """bench.e2e_chunks groups consecutive tensors while they hold at most
    max_params (a larger tensor alone) -- the grouping the host-buffer step
    applies -- into contiguous [lo, hi) ranges covering every tensor once."""
    import bench

    class T:
        def __init__(self, n):
            self.n = n

        def numel(self):
            return self.n

    sizes = [5, 3, 9, 20, 1, 1, 6, 30, 2]
    tensors, base = [], 0
    for n in sizes:
        tensors.append((T(n), None, None, None, base))
        base += n + 2                            # a gap after each tensor
    chunks = bench.e2e_chunks(tensors, max_params=10)
    starts = [t[4] for t in tensors]
    assert chunks[0][0] == 0 and chunks[-1][1] == starts[-1] + sizes[-1]
    covered, i = [], 0
    for lo, hi in chunks:
        members = [k for k, s in enumerate(starts) if lo <= s < hi]
        assert members and members[0] == i
        total = sum(sizes[k] for k in members)
        assert total <= 10 or len(members) == 1
        if members[-1] + 1 < len(sizes):
            assert total + sizes[members[-1] + 1] > 10          # a chunk stops only when the next would not fit
        covered += members
        i = members[-1] + 1
    assert covered == list(range(len(sizes)))


def test_packed_table_equals_the_checked_one():
    """The optimizer's unchecked descriptor packing gives the same bytes as
    make_table on the same tensors."""
    import torch
    rows = [(_on(0, 8, dtype=torch.bfloat16), _on(0, 8, dtype=torch.float32), _on(0, 8), _on(0, 8), 2**40 + 3),
            (_on(0, 5), _on(0, 5, dtype=torch.bfloat16), _on(0, 5), _on(0, 5), 7)]
    assert bytes(_lib._pack_table(rows)) == bytes(_lib.make_table(rows))
