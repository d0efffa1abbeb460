"""The C-ABI library: builds, loads, exports every declared symbol, and rejects
bad arguments on the host before touching a GPU (no compute call here)."""

import ctypes
import re
import subprocess
from pathlib import Path

import pytest

from latent_moe_output_gb300 import binding
from latent_moe_output_gb300.binding import Status

ROOT = Path(__file__).resolve().parents[1]
HEADERS = sorted((ROOT / "include").glob("*.h"))


@pytest.fixture(scope="module")
def lib():
    from latent_moe_output_gb300 import build

    build.build()
    return binding.load_library()


def declared_symbols():
    names = set()
    for h in HEADERS:
        text = h.read_text()
        for m in re.finditer(r"LT_API\s+[\w\s\*]+?\b(\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("latent_tail_forward", "latent_tail_forward_cols",
                     "latent_tail_workspace_size", "latent_tail_status_string",
                     "latent_tail_norm", "latent_tail_project_cols", "latent_tail_check"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    so = binding.library_path()
    out = subprocess.run(["nm", "-D", "--defined-only", str(so)], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_symbols():
        assert getattr(lib, n) is not None


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "latent_tail.h"\nint main(void){return (int)LT_OK;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", f"-I{ROOT / 'include'}", "-c",
                    str(src), "-o", str(tmp_path / "use.o")], check=True)


def test_status_strings(lib):
    for s in Status:
        text = lib.latent_tail_status_string(int(s)).decode()
        assert text.startswith("LT_") and s.name.replace("_", "") in text.replace("_", "").upper()
    assert lib.latent_tail_status_string(99).decode() == "unknown lt_status"


def test_workspace_size(lib):
    assert lib.latent_tail_workspace_size(8, 16, 2048, 7168) == 16 * 2048 * 2
    assert lib.latent_tail_workspace_size(8, 8192, 2048, 7168) == 8192 * 2048 * 2
    assert lib.latent_tail_workspace_size(2, 5, 64, 128) == 768  # 640 rounded up to 256
    assert lib.latent_tail_workspace_size(8, 0, 2048, 7168) == 0
    assert lib.latent_tail_workspace_size(8, 16, 2047, 7168) == 0
    assert lib.latent_tail_workspace_size(0, 16, 2048, 7168) == 0


# Fake, never-dereferenced addresses: validation fails before any CUDA call.
A = 0x10000
B = 0x20000000
C = 0x40000000
D = 0x60000000
E = 0x80000000
WS = 0xA0000000


def fwd(lib, routed=A, shared=B, g=C, W=D, out=E, P=2, T=4, L=64, H=128, eps=1e-6,
        c0=0, c1=128, ws=WS, wsb=1 << 20):
    return lib.latent_tail_forward_cols(routed, shared, g, W, out, P, T, L, H, eps, c0, c1,
                                        ws, wsb, None)


@pytest.mark.parametrize("kwargs,expect", [
    (dict(P=0), Status.INVALID_ARG),
    (dict(P=65), Status.INVALID_ARG),
    (dict(T=-1), Status.INVALID_ARG),
    (dict(L=4), Status.INVALID_ARG),
    (dict(L=60), Status.ALIGNMENT),
    (dict(H=120, c1=120), Status.OK),  # valid shape: reaches the pointer checks below
    (dict(H=124, c1=124), Status.ALIGNMENT),
    (dict(c0=8, c1=8), Status.INVALID_ARG),
    (dict(c0=-8), Status.INVALID_ARG),
    (dict(c1=136), Status.INVALID_ARG),
    (dict(c0=4), Status.ALIGNMENT),
    (dict(c1=100), Status.ALIGNMENT),
    (dict(eps=0.0), Status.INVALID_ARG),
    (dict(eps=-1e-6), Status.INVALID_ARG),
    (dict(eps=float("nan")), Status.INVALID_ARG),
    (dict(eps=float("inf")), Status.INVALID_ARG),
    (dict(routed=None), Status.INVALID_ARG),
    (dict(g=None, routed=None), Status.INVALID_ARG),  # no-norm: other checks still apply
    (dict(g=None, eps=0.0, out=E + 8), Status.ALIGNMENT),  # eps unused without a norm
    (dict(W=None), Status.INVALID_ARG),
    (dict(out=E + 8), Status.ALIGNMENT),
    (dict(g=C + 4), Status.ALIGNMENT),
    (dict(ws=None), Status.WORKSPACE),
    (dict(wsb=100), Status.WORKSPACE),
    (dict(ws=WS + 8), Status.ALIGNMENT),
    (dict(out=A + 64), Status.INVALID_ARG),      # out overlaps routed
    (dict(ws=B + 256), Status.INVALID_ARG),      # workspace overlaps shared
    (dict(ws=E + 256), Status.INVALID_ARG),      # workspace overlaps out
])
def test_forward_validation(lib, kwargs, expect):
    st = fwd(lib, **kwargs)
    if expect == Status.OK:
        # shape accepted; make it fail at the first pointer check instead
        st = fwd(lib, **{**kwargs, "routed": None})
        assert st == Status.INVALID_ARG
    else:
        assert st == expect


def test_zero_tokens_is_a_noop(lib):
    # T == 0 returns OK without looking at pointers (torch gives null for empty tensors)
    assert fwd(lib, routed=None, shared=None, out=None, ws=None, T=0) == Status.OK
    assert lib.latent_tail_norm(None, None, None, 2, 0, 64, 1e-6, None) == Status.OK
    assert lib.latent_tail_project_cols(None, None, None, None, 2, 0, 64, 128, 0, 128,
                                        None) == Status.OK


def test_norm_and_project_validation(lib):
    assert lib.latent_tail_norm(A, C, E, 2, 4, 60, 1e-6, None) == Status.ALIGNMENT
    assert lib.latent_tail_norm(A, C, E, 2, 4, 64, 0.0, None) == Status.INVALID_ARG
    assert lib.latent_tail_norm(A, C, A + 16, 2, 4, 64, 1e-6, None) == Status.INVALID_ARG
    pc = lib.latent_tail_project_cols
    assert pc(A, B, D, E, 2, 4, 64, 128, 0, 136, None) == Status.INVALID_ARG
    assert pc(A, B, D, B + 32, 2, 4, 64, 128, 0, 128, None) == Status.INVALID_ARG
    assert pc(A, B, None, E, 2, 4, 64, 128, 0, 128, None) == Status.INVALID_ARG
    assert pc(A, B, D, E + 8, 2, 4, 64, 128, 0, 128, None) == Status.ALIGNMENT


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(FileNotFoundError):
        binding.load_library(tmp_path / "missing.so")


def test_selftest_limit_validation(lib):
    assert lib.latent_tail_selftest_wait_timeout(0, None) == Status.INVALID_ARG
    assert lib.latent_tail_selftest_wait_timeout(1000001, None) == Status.INVALID_ARG


def test_host_workspace_size(lib):
    hws = lib.latent_tail_host_workspace_size
    # decode sizes: the latent only (the kernels reach the host buffers directly)
    assert hws(8, 16, 2048, 7168) == lib.latent_tail_workspace_size(8, 16, 2048, 7168)
    assert hws(8, 128, 2048, 7168) == 128 * 2048 * 2
    assert hws(8, 224, 2048, 7168) == 224 * 2048 * 2  # the decode kernel's largest call
    # the persistent kernel (above 224 tokens, or 224 tokens at a latent too
    # narrow for the decode kernel's buffers): latent + staging for routed,
    # shared and out, each 256-rounded
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    for P, T, L, H in [(2, 225, 64, 128), (2, 224, 64, 128)]:
        assert hws(P, T, L, H) == r256(T * L * 2) + r256(P * T * L * 2) + \
            r256(P * T * H * 2) + r256(T * H * 2)
    assert hws(2, 129, 64, 128) == 129 * 64 * 2 + 128  # decode kernel: latent only
    assert hws(8, 0, 2048, 7168) == 0
    assert hws(8, 16, 2047, 7168) == 0


def fwd_host(lib, routed=A, shared=B, g=C, W=D, out=E, P=2, T=4, L=64, H=128, eps=1e-6,
             ws=WS, wsb=1 << 20):
    return lib.latent_tail_forward_host(routed, shared, g, W, out, P, T, L, H, eps, ws, wsb,
                                        None)


@pytest.mark.parametrize("kwargs,expect", [
    (dict(P=0), Status.INVALID_ARG),
    (dict(L=60), Status.ALIGNMENT),
    (dict(eps=0.0), Status.INVALID_ARG),
    (dict(routed=None), Status.INVALID_ARG),
    (dict(out=None), Status.INVALID_ARG),
    (dict(W=None), Status.INVALID_ARG),
    (dict(routed=A + 8), Status.ALIGNMENT),
    (dict(ws=None), Status.WORKSPACE),
    (dict(wsb=100), Status.WORKSPACE),
    (dict(T=300, wsb=300 * 64 * 2 + 256), Status.WORKSPACE),  # staging not included
    (dict(ws=WS + 8), Status.ALIGNMENT),
    (dict(g=C + 4), Status.ALIGNMENT),
    (dict(out=A + 64), Status.INVALID_ARG),   # out overlaps routed
    (dict(out=B + 32), Status.INVALID_ARG),   # out straddles the shared partials
    (dict(ws=D + 256), Status.INVALID_ARG),   # workspace overlaps W
])
def test_forward_host_validation(lib, kwargs, expect):
    assert fwd_host(lib, **kwargs) == expect


def test_forward_host_zero_tokens(lib):
    assert fwd_host(lib, routed=None, shared=None, out=None, ws=None, T=0) == Status.OK
