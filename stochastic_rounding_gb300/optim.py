"""``AdamWSR``: a torch optimizer over the fused AdamW-SR kernels.

"adamw-sr", section Usage: it takes the place of ``torch.optim.AdamW`` with
the same arguments plus a seed.  Moment buffers are kept in float32;
parameters are float32 or bfloat16, the bfloat16 ones updated in place by
stochastic rounding with no float32 copy kept; gradients are float32 or
bfloat16.  Section Method: the rounding bits are keyed by (seed, step) and
indexed by each element's global parameter position.

Global positions: the parameters, in the order the optimizer was given them
(all groups, in group order), are laid end to end from ``base_offset``; a
parameter's base index is ``base_offset`` plus the number of elements before
it.  A group may instead name the position of its first element with a
``base_index`` key (its later parameters follow on from there, and so does
the next group).  An optimizer that holds one rank's contiguous share of a
model's flat parameter vector therefore passes the share's start as
``base_offset`` and draws exactly the bits the whole-model update would
(section Method: identical whether a parameter is updated whole or split
across shards and ranks).  Every step of a group is one multi-tensor launch
(per device and per distinct step count).

Device errors: the kernels' pipeline waits give up after a time limit rather
than hang, leaving the step incomplete and raising a sticky device error bit.
``check_errors`` says when ``step()`` looks at it:
  - ``True`` (the default): once the step's launches are queued it reads the
    bit, which waits for the step to finish on the device (one host
    synchronisation per step), and raises ``DeviceError`` if it is set;
  - ``"deferred"``: it queues the read behind the step into page-locked host
    memory without waiting, and raises ``DeviceError`` at a later ``step()``
    (or ``poll_errors()``) once that read has landed -- the host keeps
    running ahead of the GPU, and an error is reported a step or two late;
  - ``False``: no read; the caller checks with
    ``stochastic_rounding_gb300.asr_take_device_error`` when it wants to.
"""
from __future__ import annotations

from typing import Dict, List

import torch

from . import _lib


class DeviceError(RuntimeError):
    """A kernel of the step reported a device error (a pipeline wait that
    gave up): the step was not completed on every element, so parameters
    and moments are partly updated and should be restored from a checkpoint."""


class AdamWSR(torch.optim.Optimizer):
    """AdamW with stochastic rounding of bf16 parameters.

    Arguments follow ``torch.optim.AdamW`` (``lr``, ``betas``, ``eps``,
    ``weight_decay``) plus ``seed`` (64-bit key of the rounding stream) and
    ``rounding`` (``"sr"``, or ``"rne"`` for round-to-nearest-even, the
    biased baseline), ``base_offset`` (global position of the first
    parameter's element 0) and ``check_errors`` (when to read the device
    error bit: ``True``, ``"deferred"`` or ``False``; see the module notes).
    Parameters must be contiguous CUDA tensors of float32 or bfloat16;
    gradients dense float32 or bfloat16.

    ``torch.optim.AdamW``'s other keywords are taken so that code written for
    it runs unchanged: ``foreach``, ``fused`` and ``capturable`` are accepted
    and have no effect (every step is one fused launch per group);
    ``amsgrad``, ``maximize`` and ``differentiable`` are accepted when False
    and refused otherwise (the fused step implements neither variant).
    """

    def __init__(self, params, lr: float = 1e-3, betas=(0.9, 0.999), eps: float = 1e-8,
                 weight_decay: float = 1e-2, amsgrad: bool = False, *, maximize: bool = False,
                 foreach=None, capturable: bool = False, differentiable: bool = False, fused=None,
                 seed: int = 0, rounding: str = "sr", base_offset: int = 0, check_errors=True):
        for name, value in (("amsgrad", amsgrad), ("maximize", maximize), ("differentiable", differentiable)):
            if value:
                raise ValueError(f"AdamWSR does not support {name}=True")
        if not 0.0 <= lr:
            raise ValueError(f"Invalid learning rate: {lr}")
        if not 0.0 <= eps:
            raise ValueError(f"Invalid epsilon value: {eps}")
        if not 0.0 <= betas[0] < 1.0:
            raise ValueError(f"Invalid beta parameter at index 0: {betas[0]}")
        if not 0.0 <= betas[1] < 1.0:
            raise ValueError(f"Invalid beta parameter at index 1: {betas[1]}")
        if not 0.0 <= weight_decay:
            raise ValueError(f"Invalid weight_decay value: {weight_decay}")
        if rounding not in ("sr", "rne"):
            raise ValueError(f"rounding must be 'sr' or 'rne', not {rounding!r}")
        if not 0 <= int(seed) < 2**64:
            raise ValueError("seed must fit in 64 bits")
        if not 0 <= int(base_offset) < 2**64:
            raise ValueError("base_offset must fit in 64 bits")
        self.base_offset = int(base_offset)
        self.check_errors = self._error_mode(check_errors)
        self._pending: Dict[torch.device, List[tuple]] = {}
        defaults = dict(lr=lr, betas=tuple(betas), eps=eps, weight_decay=weight_decay,
                        seed=int(seed), rounding=rounding, base_index=None)
        super().__init__(params, defaults)
        self._assign_positions()

    def _assign_positions(self):
        pos = self.base_offset
        self._base: Dict[int, int] = {}
        for group in self.param_groups:
            if group.get("base_index") is not None:
                if not 0 <= int(group["base_index"]) < 2**64:
                    raise ValueError("a group's base_index must fit in 64 bits")
                pos = int(group["base_index"])
            for p in group["params"]:
                if id(p) in self._base:
                    continue
                if pos + p.numel() > 2**64:
                    raise ValueError("global positions run past 2^64")
                self._base[id(p)] = pos
                pos += p.numel()

    def add_param_group(self, param_group):
        super().add_param_group(param_group)
        if hasattr(self, "_base"):
            self._assign_positions()

    @staticmethod
    def _error_mode(mode):
        if mode is True or mode is False or mode == "deferred":
            return mode
        raise ValueError(f"check_errors must be True, False or 'deferred', not {mode!r}")

    # Reads of the error word queued by "deferred" steps: per device a list of
    # (event, page-locked one-word tensor), oldest first, at most this many.
    _MAX_PENDING = 4

    def poll_errors(self, wait: bool = False):
        """Look at the error reads queued by earlier "deferred" steps: those
        already landed (all of them, waiting, with ``wait``).  Raises
        ``DeviceError`` if any found a bit set."""
        bad = []
        for device, queue in self._pending.items():
            while queue and (wait or queue[0][0].query()):
                event, word = queue.pop(0)
                event.synchronize()
                if int(word.item()):
                    bad.append((device, int(word.item())))
        if bad:
            device, bits = bad[0]
            raise DeviceError(f"AdamWSR: device error bits {bits:#x} on {device} from an earlier step "
                              "(a pipeline wait gave up; that step is incomplete)")

    def _queue_error_read(self, device):
        queue = self._pending.setdefault(device, [])
        if len(queue) >= self._MAX_PENDING:
            queue[0][0].synchronize()
            self.poll_errors()
        word = torch.zeros(1, dtype=torch.int32, pin_memory=True)
        _lib.asr_take_device_error_async(word, device=device)
        event = torch.cuda.Event()
        event.record(torch.cuda.current_stream(device))
        queue.append((event, word))

    def base_index(self, p: torch.Tensor) -> int:
        """Global parameter position of element 0 of ``p``."""
        return self._base[id(p)]

    _DTYPES = frozenset((torch.float32, torch.bfloat16))

    @staticmethod
    def _check(p: torch.Tensor):
        if not p.is_cuda:
            raise ValueError("AdamWSR parameters must live on a CUDA device")
        if p.dtype not in AdamWSR._DTYPES:
            raise TypeError(f"AdamWSR supports float32 and bfloat16 parameters, not {p.dtype}")
        if not p.is_contiguous():
            raise ValueError("AdamWSR parameters must be contiguous")
        g = p.grad
        if g.is_sparse:
            raise RuntimeError("AdamWSR does not support sparse gradients")
        if g.dtype not in AdamWSR._DTYPES:
            raise TypeError(f"AdamWSR supports float32 and bfloat16 gradients, not {g.dtype}")
        if not g.is_contiguous() or g.shape != p.shape or g.get_device() != p.get_device():
            raise ValueError("gradient must be contiguous, on the parameter's device and of its shape")

    @torch.no_grad()
    def step(self, closure=None, *, check_errors=None):
        """One AdamW-SR step of every parameter that has a gradient.
        ``check_errors`` overrides the optimizer's setting for this call."""
        mode = self.check_errors if check_errors is None else self._error_mode(check_errors)
        if self._pending:
            self.poll_errors()
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        # every parameter is checked before anything is launched or counted,
        # so a refused parameter leaves the whole model as it was
        for group in self.param_groups:
            for p in group["params"]:
                if p.grad is not None:
                    self._check(p)
        devices = set()
        for group in self.param_groups:
            beta1, beta2 = group["betas"]
            # (device, step) -> list of (p, g, m, v, base)
            batches: Dict[tuple, List[tuple]] = {}
            for p in group["params"]:
                if p.grad is None:
                    continue
                state = self.state[p]
                if len(state) == 0:
                    state["step"] = 0
                    state["exp_avg"] = torch.zeros_like(p, dtype=torch.float32,
                                                        memory_format=torch.contiguous_format)
                    state["exp_avg_sq"] = torch.zeros_like(p, dtype=torch.float32,
                                                           memory_format=torch.contiguous_format)
                state["step"] = int(state["step"]) + 1
                key = (p.device, state["step"])
                batches.setdefault(key, []).append(
                    (p, p.grad, state["exp_avg"], state["exp_avg_sq"], self._base[id(p)]))
            for (device, step), entries in batches.items():
                table = _lib._pack_table(entries)
                _lib.asr_adamw_sr_multi_tensor(
                    table, lr=group["lr"], beta1=beta1, beta2=beta2, eps=group["eps"],
                    weight_decay=group["weight_decay"], step=step, seed=group["seed"],
                    rounding=group["rounding"], device=device)
                devices.add(device)
        if mode == "deferred":
            for device in devices:
                self._queue_error_read(device)
        elif mode:
            for device in devices:
                bits = _lib.asr_take_device_error(device=device)
                if bits:
                    raise DeviceError(f"AdamWSR.step: device error bits {bits:#x} on {device} "
                                      "(a pipeline wait gave up; the step is incomplete)")
        return loss

    def load_state_dict(self, state_dict):
        """Like torch's, but the moments stay float32: torch's loader casts
        floating-point state to the parameter's dtype, which for a bf16
        parameter would round the moments to bf16."""
        from itertools import chain
        super().load_state_dict(state_dict)
        saved_ids = chain.from_iterable(g["params"] for g in state_dict["param_groups"])
        params = chain.from_iterable(g["params"] for g in self.param_groups)
        id_map = dict(zip(saved_ids, params))
        for pid, st in state_dict["state"].items():
            p = id_map[pid]
            for k in ("exp_avg", "exp_avg_sq"):
                if k in st:
                    self.state[p][k] = st[k].to(device=p.device, dtype=torch.float32, copy=True)
            if "step" in self.state[p]:
                self.state[p]["step"] = int(self.state[p]["step"])
        for group in self.param_groups:
            group.setdefault("base_index", None)
        self._assign_positions()
