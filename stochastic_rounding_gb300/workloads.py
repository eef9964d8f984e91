"""Synthetic workloads: parameter-set shapes and seeded input generators.

This module holds no arithmetic of the optimizer step or of the rounding; it
only lays out parameter sets and draws random inputs (numpy PCG64 on the host,
torch's generator on the device) so that the CUDA path and its checker can be
fed the very same bytes.  bf16 inputs are produced by the framework's own
float32 -> bfloat16 conversion.

Parameter sets follow a Llama-style decoder: per layer the attention
projections q, k, v, o, the SwiGLU feed-forward gate/up/down, two RMSNorm
weights; plus untied token embedding and output head and a final RMSNorm.
"""
from __future__ import annotations

import dataclasses
from typing import List, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class DecoderShape:
    name: str
    layers: int
    hidden: int
    ffn: int
    q_heads: int
    kv_heads: int
    head_dim: int
    vocab: int


# 16 layers, hidden 2048, FFN 8192, 32 q / 8 kv heads of 64, vocab 128,256,
# untied embed / lm_head: 1,498,482,688 parameters in 147 tensors.
LLAMA_1B = DecoderShape("llama-16L-h2048", 16, 2048, 8192, 32, 8, 64, 128256)
# Llama-3-8B shapes: 32 layers, hidden 4096, FFN 14,336, 32 q / 8 kv heads of
# 128, vocab 128,256: 8,030,261,248 parameters in 291 tensors.
LLAMA_8B = DecoderShape("llama3-8b", 32, 4096, 14336, 32, 8, 128, 128256)


def param_table(shape: DecoderShape) -> List[Tuple[str, int, bool]]:
    """(name, numel, is_norm) for every parameter tensor, in model order."""
    h, f = shape.hidden, shape.ffn
    q = shape.q_heads * shape.head_dim
    kv = shape.kv_heads * shape.head_dim
    out = [("embed_tokens", shape.vocab * h, False)]
    for layer in range(shape.layers):
        pre = f"layers.{layer}."
        out += [
            (pre + "input_layernorm", h, True),
            (pre + "q_proj", q * h, False),
            (pre + "k_proj", kv * h, False),
            (pre + "v_proj", kv * h, False),
            (pre + "o_proj", h * q, False),
            (pre + "post_attention_layernorm", h, True),
            (pre + "gate_proj", f * h, False),
            (pre + "up_proj", f * h, False),
            (pre + "down_proj", h * f, False),
        ]
    out += [("norm", h, True), ("lm_head", shape.vocab * h, False)]
    return out


def offsets(table) -> Tuple[np.ndarray, int]:
    """Cumulative element offset of each tensor (its global base index) and
    the total element count."""
    sizes = np.array([n for _, n, _ in table], dtype=np.int64)
    starts = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)
    return starts, int(sizes.sum())


# ----------------------------------------------------------------- host side

def host_rng(seed: int, step: int = 0) -> np.random.Generator:
    """A PCG64 stream for (seed, step)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(step)])))


def normal_f32(rng: np.random.Generator, n: int, std: float, mean: float = 0.0) -> np.ndarray:
    return (rng.standard_normal(n, dtype=np.float32) * np.float32(std)
            + np.float32(mean)).astype(np.float32)


def uniform_f32(rng: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    return rng.uniform(lo, hi, n).astype(np.float32)


def to_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """bf16 patterns (uint16) of a float32 array via torch's own conversion."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """float32 values of bf16 patterns via torch's own conversion."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float32).numpy().copy()


# -------------------------------------------------------------- device side

def device_normal_(t, gen, std: float, mean: float = 0.0, chunk: int = 1 << 27):
    """Fill a CUDA tensor (bf16 or f32) with N(mean, std) from generator
    ``gen`` in chunks (bounded temporary memory)."""
    import torch
    flat = t.view(-1)
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        tmp = torch.randn(e - s, device=t.device, dtype=torch.float32, generator=gen)
        tmp.mul_(std).add_(mean)
        flat[s:e].copy_(tmp)
    return t


def device_uniform_(t, gen, lo: float, hi: float, chunk: int = 1 << 27):
    import torch
    flat = t.view(-1)
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        tmp = torch.rand(e - s, device=t.device, dtype=torch.float32, generator=gen)
        tmp.mul_(hi - lo).add_(lo)
        flat[s:e].copy_(tmp)
    return t


class DeviceParamSet:
    """A decoder's parameter set laid out for one fused multi-tensor step.

    Four flat device buffers -- bf16 params, bf16 grads, f32 first and second
    moments -- hold every tensor back to back in model order, so tensor t is
    the slice [start_t, start_t + n_t) of each buffer and its global parameter
    position (base index) is start_t.  Every start is a multiple of 2048
    elements, so every slice is 16-byte aligned.

    Initial values: params ~N(0, 0.02) except RMSNorm weights = 1.0; grads
    ~N(0, 1e-3); moments zero.  Drawn from torch's CUDA generator seeded with
    ``seed``.
    """

    def __init__(self, shape: DecoderShape, device="cuda", seed: int = 0,
                 p_std: float = 0.02, g_std: float = 1e-3, max_params: int = 0):
        import torch
        self.shape = shape
        self.table = param_table(shape)
        if max_params:
            # the leading tensors of the layout, at most max_params in total
            kept, total = [], 0
            for entry in self.table:
                if total + entry[1] > max_params:
                    continue
                kept.append(entry)
                total += entry[1]
            self.table = kept
        starts, total = offsets(self.table)
        self.starts = [int(s) for s in starts]
        self.sizes = [n for _, n, _ in self.table]
        self.numel = total
        self.device = torch.device(device)
        self.gen = torch.Generator(device=self.device)
        self.gen.manual_seed(int(seed))
        self.p = torch.empty(total, dtype=torch.bfloat16, device=self.device)
        self.g = torch.empty(total, dtype=torch.bfloat16, device=self.device)
        self.m = torch.zeros(total, dtype=torch.float32, device=self.device)
        self.v = torch.zeros(total, dtype=torch.float32, device=self.device)
        for (name, n, is_norm), s in zip(self.table, self.starts):
            if is_norm:
                self.p[s:s + n].fill_(1.0)
            else:
                device_normal_(self.p[s:s + n], self.gen, p_std)
        self.g_std = g_std
        self.new_grads()

    def new_grads(self):
        device_normal_(self.g, self.gen, self.g_std)

    def tensors(self):
        """(param, grad, exp_avg, exp_avg_sq, base_index) per tensor."""
        out = []
        for s, n in zip(self.starts, self.sizes):
            out.append((self.p[s:s + n], self.g[s:s + n], self.m[s:s + n], self.v[s:s + n], s))
        return out

    def nbytes(self) -> int:
        return self.numel * (2 + 2 + 4 + 4)
