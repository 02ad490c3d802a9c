"""Seeded synthetic K/V workloads for the codec's tests and benchmark.

Random inputs only: nothing here touches the codec's arithmetic. Each
workload fixes the shapes, dtype, bit widths and value distribution of one
benchmark configuration; tensors come from a torch generator seeded per
workload, on the CPU (the bytes both the oracle and the GPU path read) or on a
GPU (fast bulk generation for timing runs).

Workloads (K uses 8-bit signed codes everywhere; each also runs other key
widths in the tests):
  tiny            [1, 2, 16, 64]  fp32 iid N(0,1), seed 0; K[0,0,0,0:32] = +0.5
                  (a constant group), V 3 bits
  llama3_8b_layer [1, 8, 4096, 128] bf16 N(0,1), 1% of elements x10
                  (Bernoulli(0.01) from the same stream), seed 1, V 3 bits
  hd256           [4, 4, 8192, 256] bf16 Student-t(5) scaled to unit
                  variance, seed 2, V 4 bits
  hd512           [2, 2, 16384, 512] bf16 N(0,1), seed 3, V 2 and 5 bits
  long_context    [32, 8, 8192, 128] bf16 N(0, 0.5^2), seed 4, cache capacity
                  8192 + 64, then 64 decode-step appends of [32, 8, 1, 128]
                  (seed 5), V 8 and 3 bits
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    D: int
    dtype: torch.dtype
    v_bits: tuple
    seed: int
    dist: str
    k_bits: int = 8
    k_signed: bool = True
    t_cap: int | None = None
    append_steps: int = 0
    append_seed: int | None = None

    @property
    def rows(self) -> int:
        return self.B * self.H * self.T

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 16, 64, torch.float32, (3,), 0, "normal_const_group"),
    "llama3_8b_layer": Workload("llama3_8b_layer", 1, 8, 4096, 128, torch.bfloat16, (3,), 1, "normal_outliers"),
    "hd256": Workload("hd256", 4, 4, 8192, 256, torch.bfloat16, (4,), 2, "student_t5"),
    "hd512": Workload("hd512", 2, 2, 16384, 512, torch.bfloat16, (2, 5), 3, "normal"),
    "long_context": Workload("long_context", 32, 8, 8192, 128, torch.bfloat16, (8, 3), 4, "normal_half",
                             t_cap=8192 + 64, append_steps=64, append_seed=5),
}


def _draw(shape, dist: str, gen: torch.Generator, device) -> torch.Tensor:
    if dist in ("normal", "normal_const_group"):
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if dist == "normal_half":
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * 0.5
    if dist == "normal_outliers":
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        out = torch.rand(shape, generator=gen, device=device, dtype=torch.float32) < 0.01
        return torch.where(out, x * 10.0, x)
    if dist == "student_t5":
        # t_5 = Z / sqrt(chi2_5 / 5), chi2_5 = sum of 5 squared normals; scaled by
        # sqrt(3/5) to unit variance (Var t_5 = 5/3)
        z = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
        for _ in range(5):
            chi2 += torch.randn(shape, generator=gen, device=device, dtype=torch.float32) ** 2
        return z / torch.sqrt(chi2 / 5.0) * math.sqrt(3.0 / 5.0)
    raise ValueError(dist)


def make_kv(w: Workload, device="cpu", B=None, H=None, T=None, seed=None, dist=None):
    """K, V [B,H,T,D] of the workload's dtype (shape overridable for reduced runs)."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    dist = w.dist if dist is None else dist
    k = _draw((B, H, T, w.D), dist, gen, device)
    v = _draw((B, H, T, w.D), dist, gen, device)
    if dist == "normal_const_group" and T > 0 and B > 0 and H > 0:
        k[0, 0, 0, 0:32] = 0.5
    return k.to(w.dtype).contiguous(), v.to(w.dtype).contiguous()


def make_append_steps(w: Workload, device="cpu"):
    """The decode-step appends of a workload: a list of (K, V) [B,H,1,D]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.append_seed)
    steps = []
    for _ in range(w.append_steps):
        k = _draw((w.B, w.H, 1, w.D), w.dist, gen, device).to(w.dtype).contiguous()
        v = _draw((w.B, w.H, 1, w.D), w.dist, gen, device).to(w.dtype).contiguous()
        steps.append((k, v))
    return steps


def to_oracle(x: torch.Tensor):
    """A CPU tensor as the oracle's numpy input: fp32 as-is, bf16 as raw bits."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.float32:
        return x.numpy()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view("uint16")
    raise ValueError(x.dtype)
