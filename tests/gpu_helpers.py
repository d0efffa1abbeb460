"""Shared helpers for the GPU parity tests (CUDA path through the C ABI versus
the CPU oracle, element by element)."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from latent_moe_output_gb300 import binding, inputs

ATOL, RTOL = 8e-2, 3e-2  # bf16 tolerance of the pages' shard tests


def library():
    from latent_moe_output_gb300 import build

    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return binding.load_library()


def to_dev(x: inputs.Inputs, dev="cuda") -> inputs.Inputs:
    return inputs.Inputs(x.routed.to(dev), x.shared.to(dev), x.g.to(dev), x.W.to(dev), x.eps,
                         x.scaled_up, x.scaled_down)


def run(x: inputs.Inputs, c0=0, c1=None, out=None, stream=None):
    """CUDA tail through the C ABI; inputs on the device."""
    out = binding.forward(x.routed, x.shared, x.g, x.W, x.eps, c0, c1, out=out, stream=stream)
    binding.latent_tail_check(stream)
    return out


def oracle_rows(x: inputs.Inputs, rows, c0=0, c1=None) -> np.ndarray:
    """FP32 oracle on the given token rows (inputs may live on the device)."""
    idx = torch.as_tensor(rows, dtype=torch.long, device=x.routed.device)
    r = x.routed.index_select(1, idx).cpu()
    s = x.shared.index_select(1, idx).cpu()
    return oracle.forward(r, s, x.g.cpu(), x.W.cpu(), x.eps, c0, c1)


def assert_parity(got: torch.Tensor, want: np.ndarray, what: str = ""):
    g = got.float().cpu()
    w = torch.from_numpy(np.asarray(want, dtype=np.float32))
    torch.testing.assert_close(g, w, atol=ATOL, rtol=RTOL, msg=lambda m: f"{what}: {m}")
