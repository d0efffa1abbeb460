"""CPU oracle for the latent-MoE output tail (test infrastructure only).

    out[t, h] = sum_l rms_norm(sum_p routed[p, t, :], g, eps)[l] * W[h, l]
                + sum_p shared[p, t, h]        for h in [col_start, col_end)

The arithmetic lives in ``latent_tail_oracle.cpp`` (plain single-threaded
loops, see its header for the page citations). This module only compiles it
with g++ and marshals arrays through ctypes.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never does, and this
package imports nothing from it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "latent_tail_oracle.cpp"
BUILD_DIR = _HERE / "_build"
LIB_PATH = BUILD_DIR / "liblt_oracle.so"

# No fast-math and no FMA contraction: gcc contracts a*b+c by default on Arm,
# which would make the two hosts disagree in the last bit.
CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC"]

_lib = None


def build(out_path: Path | None = None, source: Path | None = None,
          force: bool = False) -> Path:
    """Compile the oracle and return the .so path. ``source`` replaces the
    oracle's own source file (the mutation test compiles patched copies)."""
    out = Path(out_path) if out_path is not None else LIB_PATH
    src = Path(source) if source is not None else SOURCE
    if source is None and out_path is None and out.exists() and not force:
        if out.stat().st_mtime >= SOURCE.stat().st_mtime:
            return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_name(out.name + f".tmp{os.getpid()}")
    cmd = ["g++", *CXXFLAGS, str(src), "-o", str(tmp)]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, lg, dbl = ctypes.c_void_p, ctypes.c_long, ctypes.c_double
    for name in ("lt_oracle_forward_f32", "lt_oracle_forward_f64"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, vp, vp, vp, lg, lg, lg, lg, dbl, lg, lg, vp]
        fn.restype = ctypes.c_int
    for name in ("lt_oracle_latent_f32", "lt_oracle_latent_f64"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, vp, lg, lg, lg, dbl, vp]
        fn.restype = ctypes.c_int
    return lib


def load(path: Path | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(str(path)))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(str(build())))
    return _lib


def _bf16_bits(a) -> np.ndarray:
    """bf16 tensor/array -> contiguous uint16 numpy array of its bit patterns."""
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint16:
            raise TypeError("numpy inputs must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(a)
    import torch  # local import: the oracle itself needs only numpy

    if a.dtype != torch.bfloat16:
        raise TypeError(f"expected bfloat16, got {a.dtype}")
    return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _f32(a) -> np.ndarray | None:
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return np.ascontiguousarray(a, dtype=np.float32)
    return a.detach().cpu().contiguous().float().numpy()


def _ptr(a: np.ndarray | None) -> int | None:
    return None if a is None else a.ctypes.data


def forward(routed, shared, g, W, eps: float, col_start: int = 0,
            col_end: int | None = None, precision: str = "f32", lib=None) -> np.ndarray:
    """Oracle output [T, col_end-col_start] for routed [P,T,L], shared [P,T,H], W [H,L].
    g=None selects the no-norm branch (the latent is the routed partial sum)."""
    lib = lib or load()
    r, s, w, gg = _bf16_bits(routed), _bf16_bits(shared), _bf16_bits(W), _f32(g)
    P, T, L = r.shape
    H = w.shape[0]
    if s.shape != (P, T, H) or w.shape != (H, L) or (gg is not None and gg.shape != (L,)):
        raise ValueError("shape mismatch between routed, shared, W and g")
    c1 = H if col_end is None else int(col_end)
    c0 = int(col_start)
    dt = np.float32 if precision == "f32" else np.float64
    out = np.empty((T, max(c1 - c0, 0)), dtype=dt)
    fn = lib.lt_oracle_forward_f32 if precision == "f32" else lib.lt_oracle_forward_f64
    rc = fn(_ptr(r), _ptr(s), _ptr(gg), _ptr(w), P, T, L, H,
            float(np.float32(eps)), c0, c1, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out


def latent(routed, g, eps: float, precision: str = "f32", lib=None) -> np.ndarray:
    """Normalized latent y [T, L] (steps 1 and 2 only)."""
    lib = lib or load()
    r, gg = _bf16_bits(routed), _f32(g)
    P, T, L = r.shape
    dt = np.float32 if precision == "f32" else np.float64
    y = np.empty((T, L), dtype=dt)
    fn = lib.lt_oracle_latent_f32 if precision == "f32" else lib.lt_oracle_latent_f64
    rc = fn(_ptr(r), _ptr(gg), P, T, L, float(np.float32(eps)), _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return y
