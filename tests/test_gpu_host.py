"""GPU tests of the host-buffer entry point (latent_tail_forward_host): results
bit-identical to the device entry point on the same values, in-place into a
host shared partial, the no-norm branch, graph capture, and rejection of
memory that is not page-locked host memory."""

import ctypes

import pytest
import torch

from latent_moe_output_gb300 import binding, inputs
from latent_moe_output_gb300.binding import LatentTailError, Status

pytestmark = pytest.mark.gpu


def _device_result(x, g):
    out = torch.empty(x.routed.shape[1], x.W.shape[0], dtype=torch.bfloat16, device="cuda")
    binding.forward(x.routed, x.shared, g, x.W, x.eps, out=out)
    return out.cpu()


def _host_result(x, g, ws=None, out_host=None, hr=None, hs=None):
    hr = x.routed.cpu().pin_memory() if hr is None else hr
    hs = x.shared.cpu().pin_memory() if hs is None else hs
    out = binding.forward_host(hr, hs, g, x.W, x.eps, out_host=out_host, workspace=ws)
    torch.cuda.synchronize()
    binding.latent_tail_check()
    return out


@pytest.mark.parametrize("P,T,L,H", [(8, 16, 2048, 7168), (8, 1, 2048, 7168), (8, 4, 2048, 7168),
                                     (3, 2, 512, 1032), (3, 5, 512, 1032),
                                     (8, 128, 2048, 7168), (2, 200, 1024, 1024),
                                     (2, 300, 1024, 1024)])
def test_host_matches_device_bitwise(P, T, L, H):
    x = inputs.make(P, T, L, H, seed=7000 + T, device="cuda")
    assert torch.equal(_host_result(x, x.g), _device_result(x, x.g))


@pytest.mark.parametrize("T", [2, 16, 200, 300])
def test_host_no_norm(T):
    x = inputs.make(4, T, 1024, 2048, seed=7100 + T, device="cuda")
    assert torch.equal(_host_result(x, None), _device_result(x, None))


@pytest.mark.parametrize("T", [2, 16, 200, 300])
def test_host_in_place_into_shared_partial(T):
    P, L, H = 4, 1024, 2048
    x = inputs.make(P, T, L, H, seed=7200 + T, device="cuda")
    expect = _device_result(x, x.g)
    hs = x.shared.cpu().pin_memory()
    out_view = hs[2]
    _host_result(x, x.g, out_host=out_view, hs=hs)
    assert torch.equal(hs[2], expect)
    assert torch.equal(hs[1], x.shared[1].cpu())


def test_host_graph_capture_replay():
    P, T, L, H = 8, 16, 2048, 7168
    xs = [inputs.make(P, T, L, H, seed=7300 + i, device="cuda") for i in range(2)]
    hr = [x.routed.cpu().pin_memory() for x in xs]
    hs = [x.shared.cpu().pin_memory() for x in xs]
    outs = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in xs]
    ws = torch.empty(binding.latent_tail_host_workspace_size(P, T, L, H), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # warm-up (first call sets the device up)
        for i in range(2):
            binding.latent_tail_forward_host(hr[i], hs[i], xs[i].g, xs[i].W, outs[i],
                                             xs[i].eps, ws, s)
    s.synchronize()
    for o in outs:
        o.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(2):
            binding.latent_tail_forward_host(hr[i], hs[i], xs[i].g, xs[i].W, outs[i],
                                             xs[i].eps, ws, s)
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    binding.latent_tail_check(s)
    for i, x in enumerate(xs):
        assert torch.equal(outs[i], _device_result(x, x.g))


def _raw_call(routed_ptr, shared_ptr, x, out_ptr, ws, nbytes=None):
    P, T, L = x.routed.shape
    H = x.W.shape[0]
    lib = binding.load_library()
    return lib.latent_tail_forward_host(
        routed_ptr, shared_ptr, x.g.data_ptr(), x.W.data_ptr(), out_ptr, P, T, L, H,
        ctypes.c_float(x.eps), ws.data_ptr(),
        ws.numel() if nbytes is None else nbytes, torch.cuda.current_stream().cuda_stream)


def test_host_rejects_pageable_and_device_memory():
    P, T, L, H = 2, 8, 256, 512
    x = inputs.make(P, T, L, H, seed=7400, device="cuda")
    ws = torch.empty(binding.latent_tail_host_workspace_size(P, T, L, H), dtype=torch.uint8,
                     device="cuda")
    hr, hs = x.routed.cpu().pin_memory(), x.shared.cpu().pin_memory()
    out = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    pageable_r, pageable_o = x.routed.cpu(), torch.empty(T, H, dtype=torch.bfloat16)
    assert not pageable_r.is_pinned()
    d_out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    out.fill_(1.0)
    cases = [(pageable_r.data_ptr(), hs.data_ptr(), out.data_ptr()),
             (hr.data_ptr(), hs.data_ptr(), pageable_o.data_ptr()),
             (x.routed.data_ptr(), hs.data_ptr(), out.data_ptr()),
             (hr.data_ptr(), hs.data_ptr(), d_out.data_ptr())]
    for r, s, o in cases:
        assert _raw_call(r, s, x, o, ws) == Status.INVALID_ARG
    # a range running past the end of its pinned allocation (2 MiB, a power of
    # two, so the host caching allocator does not round it up)
    big = torch.empty(1 << 20, dtype=torch.bfloat16).pin_memory()
    tail = big[(1 << 20) - (P * T * L) // 2:]
    assert _raw_call(tail.data_ptr(), hs.data_ptr(), x, out.data_ptr(), ws) == Status.INVALID_ARG
    # small workspace
    assert _raw_call(hr.data_ptr(), hs.data_ptr(), x, out.data_ptr(), ws,
                     nbytes=ws.numel() - 256) == Status.WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out.float() == 1.0)  # nothing was written by the rejected calls
    with pytest.raises(ValueError):
        binding.latent_tail_forward_host(x.routed, hs, x.g, x.W, out, x.eps, ws)
    with pytest.raises(LatentTailError):
        binding.latent_tail_forward_host(x.routed.cpu(), hs, x.g, x.W, out, x.eps, ws)


def test_host_memory_registered_with_cuda_host_register():
    """Ordinary host buffers registered (mapped) with cudaHostRegister, not allocated
    pinned, are accepted and give the device call's bits."""
    import numpy as np

    cudart = torch.cuda.cudart()
    if not hasattr(cudart, "cudaHostRegister"):
        pytest.skip("this torch build does not expose cudaHostRegister")
    P, T, L, H = 4, 16, 1024, 2048
    x = inputs.make(P, T, L, H, seed=7500, device="cuda")
    keep, registered = [], []

    def registered_like(shape, src=None):
        n = int(np.prod(shape)) * 2
        raw = np.empty(n + 8192, dtype=np.uint8)
        off = (-raw.ctypes.data) % 4096
        t = torch.from_numpy(raw[off:off + n]).view(torch.bfloat16).view(*shape)
        if src is not None:
            t.copy_(src.cpu())
        rc = cudart.cudaHostRegister(t.data_ptr(), n, 2)  # cudaHostRegisterMapped
        assert int(rc) == 0, f"cudaHostRegister failed: {rc}"
        keep.append(raw)
        registered.append(t.data_ptr())
        return t

    try:
        hr = registered_like((P, T, L), x.routed)
        hs = registered_like((P, T, H), x.shared)
        out = registered_like((T, H))
        ws = torch.empty(binding.latent_tail_host_workspace_size(P, T, L, H), dtype=torch.uint8,
                         device="cuda")
        binding.latent_tail_forward_host(hr, hs, x.g, x.W, out, x.eps, ws)
        torch.cuda.synchronize()
        binding.latent_tail_check()
        assert torch.equal(out, _device_result(x, x.g))
    finally:
        torch.cuda.synchronize()
        for ptr in registered:
            cudart.cudaHostUnregister(ptr)
