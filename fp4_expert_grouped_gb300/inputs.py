"""Seeded synthetic inputs for the MoE layer forward.

This module only draws random numbers; it holds none of the layer's arithmetic
(no quantisation, gating or GEMM).  Both the CUDA path and the CPU oracle are
fed from it, so that they see identical inputs.

Recipe (per workload, one ``torch.Generator`` seeded with the workload seed):
  x        [T, d]        standard normal, rounded to bf16 (returned as bf16)
  gate_w   [d, E]        standard normal * 1/sqrt(d), fp32
  W13[e]   [2*inter, d]  standard normal * 1/sqrt(d), fp32; rows 0..inter-1
                         are the gate projection, inter..2*inter-1 the up one
  W2[e]    [d, inter]    standard normal * 1/sqrt(inter), fp32
x and gate_w come from the workload generator in that order; expert e's weights
come from a generator of their own seeded with ``expert_seed(seed, e)`` so that
one expert can be regenerated without drawing all the others (the largest
workload's fp32 weights are ~45 GB, far more than fits at once).

The skewed workload adds a per-expert logit bias b[e] = fp32(2*ln p(e+1)),
p(r) = r^-1.2 / sum_{r'=1..E} r'^-1.2 (Zipf, s = 1.2, expert e has rank e+1).
"""
import math
from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    inter: int
    E: int
    k: int
    seed: int
    zipf_bias: bool = False

    @property
    def P(self) -> int:
        return self.T * self.k


# The five synthetic workloads: a tiny one, small-batch decode, mid batch,
# skewed routing and large prefill.
WORKLOADS = {
    "tiny": Workload("tiny", T=32, d=256, inter=128, E=8, k=2, seed=0),
    "decode": Workload("decode", T=128, d=4096, inter=2048, E=256, k=8, seed=1),
    "mid": Workload("mid", T=4096, d=4096, inter=2048, E=256, k=8, seed=2),
    "skew": Workload("skew", T=8192, d=4096, inter=2048, E=256, k=8, seed=3, zipf_bias=True),
    "prefill": Workload("prefill", T=16384, d=7168, inter=2048, E=256, k=8, seed=4),
}


def expert_seed(seed: int, e: int) -> int:
    return (seed + 1) * 1_000_003 + e


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_x_gate(w: Workload, device="cpu", T: Optional[int] = None):
    """Return (x bf16 [T, d], gate_w fp32 [d, E], bias fp32 [E] or None) on `device`."""
    T = w.T if T is None else T
    g = _gen(device, w.seed)
    x = torch.randn((T, w.d), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    gate_w = torch.randn((w.d, w.E), generator=g, device=device, dtype=torch.float32) * (1.0 / math.sqrt(w.d))
    bias = zipf_bias(w.E).to(device) if w.zipf_bias else None
    return x, gate_w, bias


def make_expert(w: Workload, e: int, device="cpu"):
    """Return (W13 fp32 [2*inter, d], W2 fp32 [d, inter]) of expert e on `device`."""
    g = _gen(device, expert_seed(w.seed, e))
    w13 = torch.randn((2 * w.inter, w.d), generator=g, device=device, dtype=torch.float32) * (1.0 / math.sqrt(w.d))
    w2 = torch.randn((w.d, w.inter), generator=g, device=device, dtype=torch.float32) * (1.0 / math.sqrt(w.inter))
    return w13, w2


def make_all_experts(w: Workload, device="cpu"):
    """All experts stacked: (W13 [E, 2*inter, d], W2 [E, d, inter]); small workloads only."""
    w13 = torch.empty((w.E, 2 * w.inter, w.d), dtype=torch.float32, device=device)
    w2 = torch.empty((w.E, w.d, w.inter), dtype=torch.float32, device=device)
    for e in range(w.E):
        a, b = make_expert(w, e, device)
        w13[e].copy_(a)
        w2[e].copy_(b)
    return w13, w2


def zipf_bias(E: int, s: float = 1.2) -> torch.Tensor:
    ranks = [r ** (-s) for r in range(1, E + 1)]
    tot = math.fsum(ranks)
    return torch.tensor([2.0 * math.log(p / tot) for p in ranks], dtype=torch.float64).to(torch.float32)


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


def from_bf16_bits(a) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor (CPU)."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
