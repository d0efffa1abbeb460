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


def oracle_all_rows(x: inputs.Inputs, c0=0, c1=None, chunk=64, workers=None) -> np.ndarray:
    """FP32 oracle on every token row, [T, c1 - c0].

    Rows of the tail never interact, so the token range is cut into chunks and
    each chunk is one ordinary single-threaded oracle call; the chunks run
    concurrently on the host's cores (ctypes releases the GIL during the call).
    The result is exactly that of one call over all rows."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    lib = oracle.load()

    def bits(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    r, s, w = bits(x.routed), bits(x.shared), bits(x.W)
    g = None if x.g is None else x.g.detach().cpu().float().numpy()
    T, H = r.shape[1], w.shape[0]
    c1 = H if c1 is None else c1
    out = np.empty((T, c1 - c0), dtype=np.float32)

    def one(t0):
        t1 = min(T, t0 + chunk)
        out[t0:t1] = oracle.forward(np.ascontiguousarray(r[:, t0:t1]),
                                    np.ascontiguousarray(s[:, t0:t1]), g, w, x.eps, c0, c1,
                                    lib=lib)

    with ThreadPoolExecutor(max_workers=workers or os.cpu_count() or 4) as ex:
        list(ex.map(one, range(0, T, chunk)))
    return out


def assert_parity(got: torch.Tensor, want: np.ndarray, what: str = ""):
    g = got.float().cpu()
    w = torch.from_numpy(np.asarray(want, dtype=np.float32))
    torch.testing.assert_close(g, w, atol=ATOL, rtol=RTOL, msg=lambda m: f"{what}: {m}")
