"""Boundary behaviour on the GPU: errors leave outputs untouched, the call is
capturable in a CUDA graph, and works on a side stream."""

import pytest
import torch

from latent_moe_output_gb300 import binding, inputs
from latent_moe_output_gb300.binding import LatentTailError, Status

import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return gh.library()


def test_small_workspace_is_rejected_and_nothing_runs():
    x = gh.to_dev(inputs.make(2, 16, 256, 256, seed=1))
    out = torch.zeros(16, 256, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(LatentTailError) as e:
        binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, out, x.eps, ws)
    assert e.value.status == Status.WORKSPACE
    binding.latent_tail_check()
    assert (out == 0).all()


def test_overlapping_output_is_rejected():
    x = gh.to_dev(inputs.make(2, 16, 256, 256, seed=2))
    ws = torch.empty(16 * 256 * 2, dtype=torch.uint8, device="cuda")
    flat = x.shared.view(-1)
    straddle = flat[8 * 256: 8 * 256 + 16 * 256].view(16, 256)  # half in each partial
    with pytest.raises(LatentTailError) as e:
        binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, straddle, x.eps, ws)
    assert e.value.status == Status.INVALID_ARG
    with pytest.raises(LatentTailError) as e:  # out overlapping W
        binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, x.W[:16], x.eps, ws)
    assert e.value.status == Status.INVALID_ARG


@pytest.mark.parametrize("T,c0,c1", [(16, 0, 1024), (16, 256, 512), (300, 0, 1024),
                                     (300, 128, 896), (200, 0, 1024), (200, 128, 896)])
def test_in_place_into_a_shared_partial(T, c0, c1):
    """out aliasing shared[p] (the pages' in-place addmm_ into the shared
    output): same values as the out-of-place call; columns outside the range
    keep the partial's own values."""
    x = gh.to_dev(inputs.make(3, T, 512, 1024, seed=T + c0))
    ref = torch.full((T, 1024), float("nan"), dtype=torch.bfloat16, device="cuda")
    gh.run(x, c0, c1, out=ref)
    for p in (0, 2):
        shared = x.shared.clone()
        before = shared[p].clone()
        ws = torch.empty(binding.latent_tail_workspace_size(3, T, 512, 1024),
                         dtype=torch.uint8, device="cuda")
        binding.latent_tail_forward_cols(x.routed, shared, x.g, x.W, shared[p], x.eps, c0, c1,
                                         ws)
        binding.latent_tail_check()
        assert torch.equal(shared[p][:, c0:c1].view(torch.int16), ref[:, c0:c1].view(torch.int16))
        assert torch.equal(shared[p][:, :c0], before[:, :c0])
        assert torch.equal(shared[p][:, c1:], before[:, c1:])


@pytest.mark.parametrize("T", [16, 512])
def test_graph_capture_replay(T):
    x = gh.to_dev(inputs.make(8, T, 2048, 2048, seed=T))
    ref = gh.run(x)
    out = torch.empty_like(ref)
    ws = torch.empty(binding.latent_tail_workspace_size(8, T, 2048, 2048), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, out, x.eps, ws)  # warm
        torch.cuda.current_stream().synchronize()
        with torch.cuda.graph(g, stream=s):
            binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, out, x.eps, ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    binding.latent_tail_check()
    assert torch.equal(out, ref)


def test_side_stream_and_repeat_determinism():
    x = gh.to_dev(inputs.make(8, 64, 2048, 1024, seed=3))
    a = gh.run(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = gh.run(x, stream=s)
    s.synchronize()
    assert torch.equal(a, b)
    for _ in range(3):
        assert torch.equal(gh.run(x), a)
