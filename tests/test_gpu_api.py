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
    x = gh.to_dev(inputs.make(1, 16, 256, 256, seed=2))
    ws = torch.empty(16 * 256 * 2, dtype=torch.uint8, device="cuda")
    alias = x.shared[0]  # out aliasing shared[0] (the pages' in-place addmm_) is not allowed
    with pytest.raises(LatentTailError) as e:
        binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, alias, x.eps, ws)
    assert e.value.status == Status.INVALID_ARG


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
