"""Seeded synthetic inputs for the codec's workloads.

This module only draws random numbers and lays them out; it holds none of the codec's
arithmetic, so both the CUDA path and the CPU oracle may consume what it makes.  Every draw
goes through a ``torch.Generator`` seeded explicitly, on the device the caller names, so a
workload is reproducible on that device; the GPU tests copy the exact bytes to the host before
handing them to the oracle.

Workloads (sizes and distributions follow the pages' setting: a 72.7B-parameter decoder with
width 8192, 64 query heads and 8 KV heads, per "Covenant-72B: Largest Decentralized GPU
Model", "Technical Deep Dive"; the value distributions are synthetic stand-ins for real
pseudo-gradients, which need trained weights):

- ``tiny``: 1,048,576 fp32 values, N(0, 1e-3), beta 1.0, 3 rounds; 4 peers.
- ``heavy_tail_bf16``: 134,217,728 bf16 values, 1e-4 * Student-t(3) with 0.1 % of positions
  multiplied by 100; beta 0.95, 5 rounds; 8 peers.
- ``decoder_layer``: one 72B-class decoder layer's tensors, each N(0, 2e-4) times a per-row
  scale drawn log-uniform in [0.1, 10]; beta 1.0, 3 rounds.
- ``large_flat``: 2^30 fp32 values, Laplace(0, 1e-4); beta 0.95, 10 rounds.
- ``receive``: 24 peers, each the payload of one round from zero error feedback on its own
  2^30-value Laplace(0, 1e-4) draw; theta ~ N(0, 0.02); outer learning rate 0.7.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n: int                      # total elements (sum over tensors for multi-tensor workloads)
    dtype: str                  # "f32" or "bf16" for the pseudo-gradient
    beta: float
    rounds: int
    peers: int
    shapes: tuple = field(default=())   # per-tensor shapes for multi-tensor workloads
    lr: float = 0.0


DECODER_LAYER_SHAPES = (
    ("q_proj", (8192, 8192)),
    ("k_proj", (1024, 8192)),
    ("v_proj", (1024, 8192)),
    ("o_proj", (8192, 8192)),
    ("gate_proj", (28672, 8192)),
    ("up_proj", (28672, 8192)),
    ("down_proj", (8192, 28672)),
    ("input_norm", (8192,)),
    ("post_attn_norm", (8192,)),
)

WORKLOADS = {
    "tiny": Workload("tiny", 1 << 20, "f32", 1.0, 3, 4),
    "heavy_tail_bf16": Workload("heavy_tail_bf16", 1 << 27, "bf16", 0.95, 5, 8),
    "decoder_layer": Workload(
        "decoder_layer", sum(math.prod(s) for _, s in DECODER_LAYER_SHAPES), "f32", 1.0, 3, 1,
        shapes=DECODER_LAYER_SHAPES),
    "large_flat": Workload("large_flat", 1 << 30, "f32", 0.95, 10, 1),
    "receive": Workload("receive", 1 << 30, "f32", 0.95, 1, 24, lr=0.7),
}


def generator(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(int(seed))


def normal(n: int, std: float, gen: torch.Generator, device) -> torch.Tensor:
    """fp32 draws from N(0, std^2)."""
    return torch.randn(n, generator=gen, device=device, dtype=torch.float32).mul_(std)


def laplace(n: int, b: float, gen: torch.Generator, device) -> torch.Tensor:
    """fp32 draws from Laplace(0, b), as b times the difference of two Exp(1) draws."""
    x = torch.empty(n, device=device, dtype=torch.float32).exponential_(1.0, generator=gen)
    y = torch.empty(n, device=device, dtype=torch.float32).exponential_(1.0, generator=gen)
    return x.sub_(y).mul_(b)


def student_t3(n: int, gen: torch.Generator, device) -> torch.Tensor:
    """fp32 draws from Student-t with 3 degrees of freedom: z / sqrt(chi2_3 / 3)."""
    z = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    chi2 = torch.zeros(n, device=device, dtype=torch.float32)
    for _ in range(3):
        w = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        chi2.addcmul_(w, w)
    return z.div_(chi2.div_(3.0).sqrt_())


def heavy_tail_bf16(n: int, gen: torch.Generator, device) -> torch.Tensor:
    """bf16 of 1e-4 * t_3, with round(0.001 n) uniformly chosen positions multiplied by 100."""
    x = student_t3(n, gen, device).mul_(1e-4)
    k = int(round(0.001 * n))
    if k:
        pos = torch.randperm(n, generator=gen, device=device)[:k]
        x[pos] *= 100.0
    return x.to(torch.bfloat16)


def row_scaled_normal(shape, std: float, gen: torch.Generator, device) -> torch.Tensor:
    """N(0, std^2) times a per-row scale drawn log-uniform in [0.1, 10] (one scale for 1-D)."""
    rows = shape[0] if len(shape) == 2 else 1
    cols = math.prod(shape) // rows
    u = torch.rand(rows, 1, generator=gen, device=device, dtype=torch.float32)
    sigma = torch.exp(math.log(0.1) + u * (math.log(10.0) - math.log(0.1)))
    x = torch.randn(rows, cols, generator=gen, device=device, dtype=torch.float32)
    return x.mul_(std).mul_(sigma).reshape(-1)


def delta_round(wl: Workload, gen: torch.Generator, device, n: int | None = None):
    """One round's pseudo-gradient for flat workloads (n overrides the size for small cases)."""
    n = wl.n if n is None else n
    if wl.name == "tiny":
        return normal(n, 1e-3, gen, device)
    if wl.name == "heavy_tail_bf16":
        return heavy_tail_bf16(n, gen, device)
    if wl.name in ("large_flat", "receive"):
        return laplace(n, 1e-4, gen, device)
    raise ValueError(f"{wl.name} is not a flat workload")


def decoder_layer_round(gen: torch.Generator, device, shapes=DECODER_LAYER_SHAPES):
    """One round's per-tensor pseudo-gradients of a 72B-class decoder layer (list of flat fp32)."""
    return [row_scaled_normal(s, 2e-4, gen, device) for _, s in shapes]


def theta(n: int, gen: torch.Generator, device) -> torch.Tensor:
    """Outer parameters for the fused outer step: N(0, 0.02^2)."""
    return normal(n, 0.02, gen, device)
