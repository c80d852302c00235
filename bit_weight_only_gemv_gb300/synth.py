"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no part of the method's arithmetic: it only draws random
packed words, steps, activations, token ids and expert-routing traces, and
names the workload shapes.  Both the CUDA path and the CPU oracle consume what
it produces; the oracle always reads back the exact bytes the GPU used.

Recipe (the shapes and distributions of the decode workloads):

* packed code words: uniform 32-bit words, so every nibble (code) is uniform
  on 0..15;
* steps: bf16 of |z| * 0.02 / 8 with z ~ N(0, 1);
* activations: bf16 of N(0, 1);
* token ids: uniform on [0, vocab);
* routed experts: per layer a seeded permutation maps Zipf ranks to expert
  ids; step 0 draws 8 distinct experts by Zipf(s) over the ranks; every later
  step keeps each previous expert with probability 0.7 and fills up to 8
  distinct experts with fresh Zipf draws.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

GROUP = 32


# --------------------------------------------------------------------------
# host (NumPy) draws, for CPU tests and small GPU cases
# --------------------------------------------------------------------------
def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def np_words(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.integers(0, 1 << 32, size=shape, dtype=np.uint64).astype(np.uint32)


def np_steps(rng: np.random.Generator, shape, scale: float = 0.02 / 8) -> np.ndarray:
    return _to_bf16_bits(np.abs(rng.standard_normal(shape)) * scale)


def np_x(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    return _to_bf16_bits(rng.standard_normal(shape) * scale)


def np_ids(rng: np.random.Generator, n: int, vocab: int) -> np.ndarray:
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def np_codes(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.integers(0, 16, size=shape, dtype=np.int64).astype(np.uint8)


# --------------------------------------------------------------------------
# device (torch) draws, for the large benchmark workloads
# --------------------------------------------------------------------------
def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def torch_words(shape, seed: int, device) -> torch.Tensor:
    """int32 tensor of uniform 32-bit words (the bit patterns matter, not the sign)."""
    return torch.randint(-(1 << 31), 1 << 31, tuple(shape), dtype=torch.int32,
                         device=device, generator=_gen(seed, device))


def torch_steps(shape, seed: int, device, scale: float = 0.02 / 8) -> torch.Tensor:
    z = torch.randn(tuple(shape), dtype=torch.float32, device=device, generator=_gen(seed, device))
    return (z.abs_() * scale).to(torch.bfloat16)


def torch_x(shape, seed: int, device) -> torch.Tensor:
    z = torch.randn(tuple(shape), dtype=torch.float32, device=device, generator=_gen(seed, device))
    return z.to(torch.bfloat16)


def torch_ids(n: int, vocab: int, seed: int, device) -> torch.Tensor:
    return torch.randint(0, vocab, (n,), dtype=torch.int32, device=device,
                         generator=_gen(seed, device))


def seed_of(*parts: int) -> int:
    """Stable 63-bit seed from small integers (workload, layer, projection ...)."""
    h = 0x9E3779B97F4A7C15
    for p in parts:
        h ^= (int(p) + 0x632BE59BD9B4E019 + ((h << 6) & 0xFFFFFFFFFFFFFFFF) + (h >> 2))
        h &= 0xFFFFFFFFFFFFFFFF
    return h & 0x7FFFFFFFFFFFFFFF


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Proj:
    name: str
    n: int          # output rows
    k: int          # reduction length
    x_key: str      # projections with the same key read the same activation


@dataclasses.dataclass(frozen=True)
class DenseDecoder:
    name: str
    layers: int
    hidden: int
    projs: tuple
    vocab: int
    per_layer_width: int   # 0 = no per-layer table


def dense_2048() -> DenseDecoder:
    """35-layer decoder, hidden 2048, 4-bit tied table 262144 x 2048 and a
    per-layer table 262144 x (35 * 256)."""
    h = 2048
    projs = (Proj("q", 2048, h, "attn"), Proj("k", 512, h, "attn"), Proj("v", 512, h, "attn"),
             Proj("o", 2048, h, "o"), Proj("gate", 8192, h, "mlp"), Proj("up", 8192, h, "mlp"),
             Proj("down", h, 8192, "down"))
    return DenseDecoder("dense-35L-h2048", 35, h, projs, 262144, 35 * 256)


def dense_5376() -> DenseDecoder:
    """60-layer decoder, hidden 5376, 4-bit tied table 262144 x 5376."""
    h = 5376
    projs = (Proj("q", 5376, h, "attn"), Proj("k", 2048, h, "attn"), Proj("v", 2048, h, "attn"),
             Proj("o", 5376, h, "o"), Proj("gate", 21504, h, "mlp"), Proj("up", 21504, h, "mlp"),
             Proj("down", h, 21504, "down"))
    return DenseDecoder("dense-60L-h5376", 60, h, projs, 262144, 0)


@dataclasses.dataclass(frozen=True)
class MoEDecoder:
    name: str
    layers: int
    hidden: int
    experts: int
    top_k: int
    expert_inter: int
    slots: int
    zipf_s: float
    repeat_p: float


def moe_2816() -> MoEDecoder:
    """30 MoE layers, hidden 2816, 128 experts of gate/up 704 x 2816 and down
    2816 x 704, top-8 routing, 32-slot pool per layer."""
    return MoEDecoder("moe-30L-h2816-128e", 30, 2816, 128, 8, 704, 32, 1.1, 0.7)


SWEEP_BATCHES = (1, 2, 4, 8, 16, 32)


# --------------------------------------------------------------------------
# routed-expert traces
# --------------------------------------------------------------------------
def moe_trace(num_experts: int, top_k: int, steps: int, zipf_s: float, repeat_p: float,
              seed: int) -> np.ndarray:
    """int32 [steps, top_k] of distinct expert ids per step (one layer)."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_experts)
    ranks = np.arange(1, num_experts + 1, dtype=np.float64)
    p = ranks ** (-zipf_s)
    p /= p.sum()
    out = np.empty((steps, top_k), dtype=np.int32)
    prev: list = []
    for t in range(steps):
        cur = [e for e in prev if rng.random() < repeat_p]
        while len(cur) < top_k:
            e = int(perm[rng.choice(num_experts, p=p)])
            if e not in cur:
                cur.append(e)
        out[t] = cur
        prev = cur
    return out
