"""ctypes binding over the C ABI in ``include/latent_tail.h``.

Argument marshalling only: shapes are read from the tensors, pointers and the
current CUDA stream are passed through, and a non-OK status raises
``LatentTailError``. Every step of the computation runs in the CUDA library;
if that library is missing, the first call raises instead of falling back.
"""

from __future__ import annotations

import ctypes
import enum
import os
from pathlib import Path

_PKG = Path(__file__).resolve().parent
LIB_NAME = "liblatent_tail.so"


def library_path() -> Path:
    return _PKG / "_lib" / LIB_NAME


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    ALIGNMENT = 2
    UNSUPPORTED = 3
    WORKSPACE = 4
    CUDA = 5
    TIMEOUT = 6


class LatentTailError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status)
        super().__init__(f"{where}: {latent_tail_status_string(status)}")


_lib = None

_SIGNATURES = {
    "latent_tail_workspace_size": (ctypes.c_size_t, [ctypes.c_int] * 4),
    "latent_tail_forward": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4
                            + [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t,
                               ctypes.c_void_p]),
    "latent_tail_forward_cols": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4
                                 + [ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "latent_tail_norm": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3
                         + [ctypes.c_float, ctypes.c_void_p]),
    "latent_tail_project_cols": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int] * 6
                                 + [ctypes.c_void_p]),
    "latent_tail_check": (ctypes.c_int, [ctypes.c_void_p]),
    "latent_tail_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint, ctypes.c_void_p]),
    "latent_tail_forward_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4
                                    + [ctypes.c_float, ctypes.c_void_p]),
    "latent_tail_host_workspace_size": (ctypes.c_size_t, [ctypes.c_int] * 4),
    "latent_tail_forward_host": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4
                                 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t,
                                    ctypes.c_void_p]),
    "latent_tail_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}


def load_library(path: str | os.PathLike | None = None) -> ctypes.CDLL:
    """Load the CUDA library (built in-tree by ``build.py``); raise if absent."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    p = Path(path) if path is not None else library_path()
    if not p.exists():
        raise FileNotFoundError(
            f"CUDA library {p} is not built; run `python -c \"import __graft_entry__ as g;"
            f" g.build()\"` first (there is no CPU fallback)")
    lib = ctypes.CDLL(str(p))
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def latent_tail_status_string(status: int) -> str:
    try:
        return load_library().latent_tail_status_string(int(status)).decode()
    except FileNotFoundError:
        return Status(status).name


def _check(status: int, where: str) -> None:
    if status != 0:
        raise LatentTailError(status, where)


def _stream_handle(stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t, name: str, dtype, ndim: int, optional: bool = False):
    import torch

    if t is None and optional:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or t.dim() != ndim:
        raise TypeError(f"{name}: expected {ndim}-d {dtype}, got {t.dim()}-d {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def latent_tail_workspace_size(P: int, T: int, L: int, H: int) -> int:
    return int(load_library().latent_tail_workspace_size(P, T, L, H))


def latent_tail_forward(routed, shared, norm_weight, W, out, eps: float, workspace,
                        stream=None) -> None:
    latent_tail_forward_cols(routed, shared, norm_weight, W, out, eps, 0, W.shape[0],
                             workspace, stream)


def latent_tail_forward_cols(routed, shared, norm_weight, W, out, eps: float,
                             col_start: int, col_end: int, workspace, stream=None) -> None:
    import torch

    bf = torch.bfloat16
    r = _dev(routed, "routed", bf, 3)
    s = _dev(shared, "shared", bf, 3)
    g = _dev(norm_weight, "norm_weight", torch.float32, 1, optional=True)
    w = _dev(W, "W", bf, 2)
    o = _dev(out, "out", bf, 2)
    ws = _dev(workspace, "workspace", workspace.dtype, workspace.dim())
    P, T, L = routed.shape
    H = W.shape[0]
    if tuple(shared.shape) != (P, T, H) or tuple(W.shape) != (H, L) \
            or tuple(out.shape) != (T, H) \
            or (norm_weight is not None and tuple(norm_weight.shape) != (L,)):
        raise ValueError("inconsistent shapes: routed [P,T,L], shared [P,T,H], W [H,L], "
                         "out [T,H], norm_weight [L]")
    nbytes = workspace.numel() * workspace.element_size()
    lib = load_library()
    if col_start == 0 and col_end == H:
        st = lib.latent_tail_forward(r, s, g, w, o, P, T, L, H, float(eps), ws, nbytes,
                                     _stream_handle(stream))
    else:
        st = lib.latent_tail_forward_cols(r, s, g, w, o, P, T, L, H, float(eps),
                                          int(col_start), int(col_end), ws, nbytes,
                                          _stream_handle(stream))
    _check(st, "latent_tail_forward_cols")


def latent_tail_norm(routed, norm_weight, latent, eps: float, stream=None) -> None:
    import torch

    r = _dev(routed, "routed", torch.bfloat16, 3)
    g = _dev(norm_weight, "norm_weight", torch.float32, 1, optional=True)
    y = _dev(latent, "latent", torch.bfloat16, 2)
    P, T, L = routed.shape
    if tuple(latent.shape) != (T, L) or (norm_weight is not None
                                         and tuple(norm_weight.shape) != (L,)):
        raise ValueError("inconsistent shapes: routed [P,T,L], latent [T,L], norm_weight [L]")
    _check(load_library().latent_tail_norm(r, g, y, P, T, L, float(eps),
                                           _stream_handle(stream)), "latent_tail_norm")


def latent_tail_project_cols(latent, shared, W, out, col_start: int, col_end: int,
                             stream=None) -> None:
    import torch

    bf = torch.bfloat16
    y = _dev(latent, "latent", bf, 2)
    s = _dev(shared, "shared", bf, 3)
    w = _dev(W, "W", bf, 2)
    o = _dev(out, "out", bf, 2)
    T, L = latent.shape
    P = shared.shape[0]
    H = W.shape[0]
    if tuple(shared.shape) != (P, T, H) or tuple(W.shape) != (H, L) \
            or tuple(out.shape) != (T, H):
        raise ValueError("inconsistent shapes: latent [T,L], shared [P,T,H], W [H,L], out [T,H]")
    _check(load_library().latent_tail_project_cols(y, s, w, o, P, T, L, H, int(col_start),
                                                   int(col_end), _stream_handle(stream)),
           "latent_tail_project_cols")


def latent_tail_forward_noalloc(routed, shared, norm_weight, W, out, eps: float,
                                stream=None) -> None:
    """Whole tail with the library's fixed 8 MiB device scratch instead of a
    caller workspace (for callers that cannot allocate); T * L * 2 must fit."""
    import torch

    bf = torch.bfloat16
    r = _dev(routed, "routed", bf, 3)
    s = _dev(shared, "shared", bf, 3)
    g = _dev(norm_weight, "norm_weight", torch.float32, 1, optional=True)
    w = _dev(W, "W", bf, 2)
    o = _dev(out, "out", bf, 2)
    P, T, L = routed.shape
    H = W.shape[0]
    if tuple(shared.shape) != (P, T, H) or tuple(W.shape) != (H, L) \
            or tuple(out.shape) != (T, H) \
            or (norm_weight is not None and tuple(norm_weight.shape) != (L,)):
        raise ValueError("inconsistent shapes: routed [P,T,L], shared [P,T,H], W [H,L], "
                         "out [T,H], norm_weight [L]")
    _check(load_library().latent_tail_forward_noalloc(r, s, g, w, o, P, T, L, H, float(eps),
                                                      _stream_handle(stream)),
           "latent_tail_forward_noalloc")


def latent_tail_check(stream=None) -> None:
    _check(load_library().latent_tail_check(_stream_handle(stream)), "latent_tail_check")


def forward(routed, shared, norm_weight, W, eps: float, col_start: int = 0,
            col_end: int | None = None, out=None, workspace=None, stream=None):
    """Allocate ``out`` (and the workspace) with torch and run the tail."""
    import torch

    P, T, L = routed.shape
    H = W.shape[0]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=routed.device)
    if workspace is None:
        n = latent_tail_workspace_size(P, T, L, H)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=routed.device)
    latent_tail_forward_cols(routed, shared, norm_weight, W, out, eps, col_start,
                             H if col_end is None else col_end, workspace, stream)
    return out


def _host(t, name: str, dtype, ndim: int):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or t.dim() != ndim:
        raise TypeError(f"{name}: expected {ndim}-d {dtype}, got {t.dim()}-d {t.dtype}")
    if t.is_cuda:
        raise ValueError(f"{name} must be in host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def latent_tail_host_workspace_size(P: int, T: int, L: int, H: int) -> int:
    return int(load_library().latent_tail_host_workspace_size(P, T, L, H))


def latent_tail_forward_host(routed_host, shared_host, norm_weight, W, out_host, eps: float,
                             workspace, stream=None) -> None:
    """Whole tail with routed/shared/out in page-locked host memory (the library
    checks that they are; pageable memory is rejected) and W, g, workspace on the
    device."""
    import torch

    bf = torch.bfloat16
    r = _host(routed_host, "routed_host", bf, 3)
    s = _host(shared_host, "shared_host", bf, 3)
    o = _host(out_host, "out_host", bf, 2)
    g = _dev(norm_weight, "norm_weight", torch.float32, 1, optional=True)
    w = _dev(W, "W", bf, 2)
    ws = _dev(workspace, "workspace", workspace.dtype, workspace.dim())
    P, T, L = routed_host.shape
    H = W.shape[0]
    if tuple(shared_host.shape) != (P, T, H) or tuple(W.shape) != (H, L) \
            or tuple(out_host.shape) != (T, H) \
            or (norm_weight is not None and tuple(norm_weight.shape) != (L,)):
        raise ValueError("inconsistent shapes: routed [P,T,L], shared [P,T,H], W [H,L], "
                         "out [T,H], norm_weight [L]")
    nbytes = workspace.numel() * workspace.element_size()
    _check(load_library().latent_tail_forward_host(r, s, g, w, o, P, T, L, H, float(eps), ws,
                                                   nbytes, _stream_handle(stream)),
           "latent_tail_forward_host")


def forward_host(routed_host, shared_host, norm_weight, W, eps: float, out_host=None,
                 workspace=None, stream=None):
    """End-to-end call on page-locked host tensors: allocate ``out_host``
    (pinned) and the device workspace with torch when not given, run the tail
    through latent_tail_forward_host and return ``out_host`` (valid once the
    stream is synchronized)."""
    import torch

    P, T, L = routed_host.shape
    H = W.shape[0]
    if out_host is None:
        out_host = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    if workspace is None:
        n = latent_tail_host_workspace_size(P, T, L, H)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=W.device)
    latent_tail_forward_host(routed_host, shared_host, norm_weight, W, out_host, eps,
                             workspace, stream)
    return out_host
