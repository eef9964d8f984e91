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
