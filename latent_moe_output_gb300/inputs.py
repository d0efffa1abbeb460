"""Seeded synthetic inputs for the latent-MoE output tail.

This module draws random tensors and nothing else: it holds none of the tail's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Recipe (same for every workload; the pages measure end-to-end Kimi-K3 serving,
and these tensors stand in for the tail's operands at those shapes):

* draw order: [stress only: the outlier-row permutation], routed, shared, g, W;
* routed[p] and shared[p] ~ N(0, 1) drawn per partial p in FP32, cast to bf16
  (round to nearest even);
* g = 1 + 0.1 * N(0, 1), kept in FP32;
* W ~ N(0, 1/L), i.e. randn / sqrt(L), cast to bf16;
* stress only: a randperm(T) picks 1% of the token rows (the first T//100) to
  scale by 100 and the next T//100 to scale by 1e-3; the factor multiplies that
  token's row in every routed and every shared partial, in FP32 before the cast.

The values depend on the generator's device: the same seed gives different
numbers on the CPU and on CUDA. Every consumer receives the same tensors, so
parity does not depend on it.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

EPS = 1e-6


@dataclass(frozen=True)
class Workload:
    name: str
    P: int
    T: int
    L: int
    H: int
    seed: int
    outlier_rows: bool = False

    @property
    def tokens(self) -> int:
        return self.T


TINY = Workload("tiny", P=2, T=5, L=64, H=128, seed=0)
DECODE = Workload("decode", P=8, T=16, L=2048, H=7168, seed=1)
DECODE_SWEEP = tuple(
    Workload(f"decode_T{t}", P=8, T=t, L=2048, H=7168, seed=1000 + t)
    for t in (1, 2, 4, 8, 32, 64, 128)
)
PREFILL = Workload("prefill", P=8, T=8192, L=2048, H=7168, seed=2)
STRESS = Workload("stress", P=16, T=16384, L=2048, H=7168, seed=3, outlier_rows=True)
# One routed and one shared partial: the per-rank work after the reference's
# all-reduce (tensor-core bound rather than bandwidth bound).
PREFILL_P1 = Workload("prefill_p1", P=1, T=8192, L=2048, H=7168, seed=4)

WORKLOADS = {w.name: w for w in (TINY, DECODE, *DECODE_SWEEP, PREFILL, STRESS, PREFILL_P1)}

# Column shards of the stress workload: 16 equal ranges of H.
STRESS_SHARDS = 16


@dataclass
class Inputs:
    routed: torch.Tensor   # [P, T, L] bf16
    shared: torch.Tensor   # [P, T, H] bf16
    g: torch.Tensor        # [L] fp32
    W: torch.Tensor        # [H, L] bf16
    eps: float
    scaled_up: torch.Tensor    # token indices scaled by 100 (empty unless stress)
    scaled_down: torch.Tensor  # token indices scaled by 1e-3


def outlier_rows(T: int, gen: torch.Generator, device) -> tuple[torch.Tensor, torch.Tensor]:
    n = T // 100
    perm = torch.randperm(T, generator=gen, device=device)
    return perm[:n].sort().values, perm[n:2 * n].sort().values


def make(P: int, T: int, L: int, H: int, seed: int, device="cpu",
         outliers: bool = False, eps: float = EPS) -> Inputs:
    """Draw one seeded set of tail operands on ``device``."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    bf16 = torch.bfloat16
    if outliers:
        up, down = outlier_rows(T, gen, device)
        scale = torch.ones(T, 1, dtype=torch.float32, device=device)
        scale[up] = 100.0
        scale[down] = 1e-3
    else:
        up = down = torch.empty(0, dtype=torch.long, device=device)
        scale = None

    def partials(cols: int) -> torch.Tensor:
        out = torch.empty(P, T, cols, dtype=bf16, device=device)
        for p in range(P):
            v = torch.randn(T, cols, generator=gen, device=device, dtype=torch.float32)
            if scale is not None:
                v.mul_(scale)
            out[p].copy_(v)  # FP32 -> bf16, round to nearest even
            del v
        return out

    routed = partials(L)
    shared = partials(H)
    g = 1.0 + 0.1 * torch.randn(L, generator=gen, device=device, dtype=torch.float32)
    W = (torch.randn(H, L, generator=gen, device=device, dtype=torch.float32)
         / math.sqrt(L)).to(bf16)
    return Inputs(routed, shared, g, W, float(eps), up, down)


def make_workload(w: Workload, device="cpu") -> Inputs:
    return make(w.P, w.T, w.L, w.H, w.seed, device=device, outliers=w.outlier_rows)

