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
    ws = torch.empty(binding.latent_tail_workspace_size(2, 16, 256, 256), dtype=torch.uint8,
                     device="cuda")
    flat = x.shared.view(-1)
    straddle = flat[8 * 256: 8 * 256 + 16 * 256].view(16, 256)  # half in each partial
    with pytest.raises(LatentTailError) as e:
        binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, straddle, x.eps, ws)
    assert e.value.status == Status.INVALID_ARG
    with pytest.raises(LatentTailError) as e:  # out overlapping W
        binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, x.W[:16], x.eps, ws)
    assert e.value.status == Status.INVALID_ARG


@pytest.mark.parametrize("P,T,L,H,c0,c1", [
    (3, 2, 2048, 7168, 0, 7168), (3, 2, 2048, 7168, 1000, 5000),   # one-launch kernel
    (3, 16, 512, 1024, 0, 1024), (3, 16, 512, 1024, 256, 512),     # decode kernel
    (3, 300, 512, 1024, 0, 1024), (3, 300, 512, 1024, 128, 896),   # prefill, 192-col tiles
    (3, 3328, 256, 1024, 0, 1024), (3, 3328, 256, 1024, 128, 896),  # prefill, 256-col tiles
    (3, 200, 512, 1024, 0, 1024), (3, 200, 512, 1024, 128, 896),   # decode above 128 tokens
    (3, 240, 512, 1024, 0, 1024), (3, 240, 512, 1024, 128, 896),   # prefill, 128-col tiles
    (8, 1000, 2048, 7168, 0, 7168),                                # production widths
    (1, 4096, 256, 1544, 0, 1544), (1, 4096, 256, 1544, 136, 648),  # P = 1, 512-col tiles
])
def test_in_place_into_a_shared_partial(P, T, L, H, c0, c1):
    """out aliasing shared[p] (the pages' in-place addmm_ into the shared output)
    matches the FP32 oracle on the original partials, leaves the columns outside
    the range at the partial's own values, and equals the out-of-place call bit
    for bit. T is not a multiple of 128 on the prefill path, so the shared-partial
    boxes of one plane run into the next plane (and past the last one)."""
    x = inputs.make(P, T, L, H, seed=T + c0)
    xd = gh.to_dev(x)
    want = gh.oracle_all_rows(x, c0, c1)
    ref = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    gh.run(xd, c0, c1, out=ref)
    for p in (0, P - 1):
        shared = xd.shared.clone()
        before = shared[p].clone()
        ws = torch.empty(binding.latent_tail_workspace_size(P, T, L, H),
                         dtype=torch.uint8, device="cuda")
        binding.latent_tail_forward_cols(xd.routed, shared, xd.g, xd.W, shared[p], x.eps, c0, c1,
                                         ws)
        binding.latent_tail_check()
        gh.assert_parity(shared[p][:, c0:c1], want, f"in place into shared[{p}]")
        assert torch.equal(shared[p][:, :c0], before[:, :c0])
        assert torch.equal(shared[p][:, c1:], before[:, c1:])
        assert torch.equal(shared[p][:, c0:c1].view(torch.int16), ref[:, c0:c1].view(torch.int16))


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


@pytest.mark.parametrize("T", [16, 64, 128, 200, 256])
def test_back_to_back_calls_read_what_the_previous_call_wrote(T):
    """Each call's output is every input of the next one (P = 1, T = H = L: the
    output [T, H] doubles as latent/routed [T, L], shared [1, T, H] and W [H, L]).
    Issued back to back on one stream, the chain must give the same bits as the
    same calls with a device synchronize between them: a call that started early
    (programmatic dependent launch) must still read only after the previous call
    has finished writing."""
    torch.manual_seed(T)
    H = L = T
    eps = inputs.EPS
    a0 = (torch.randn(T, H, device="cuda") / 8).to(torch.bfloat16)
    g = (1.0 + 0.1 * torch.randn(L, device="cuda")).float()

    def project_chain(sync):
        bufs = [a0.clone()] + [torch.empty_like(a0) for _ in range(4)]
        for i in range(4):
            a = bufs[i]
            binding.latent_tail_project_cols(a, a.view(1, T, H), a, bufs[i + 1], 0, H)
            if sync:
                torch.cuda.synchronize()
        binding.latent_tail_check()
        return bufs[1:]

    def forward_chain(sync):
        bufs = [a0.clone()] + [torch.empty_like(a0) for _ in range(4)]
        ws = torch.empty(binding.latent_tail_workspace_size(1, T, L, H), dtype=torch.uint8,
                         device="cuda")
        for i in range(4):
            a = bufs[i]
            binding.latent_tail_forward(a.view(1, T, L), a.view(1, T, H), g, a, bufs[i + 1], eps,
                                        ws)
            if sync:
                torch.cuda.synchronize()
        binding.latent_tail_check()
        return bufs[1:]

    for chain in (project_chain, forward_chain):
        free, synced = chain(False), chain(True)
        for i, (u, v) in enumerate(zip(free, synced)):
            assert torch.equal(u.view(torch.int16), v.view(torch.int16)), f"{chain.__name__} step {i}"
    # and the first projection step against a float64 evaluation of its inputs
    first = project_chain(True)[0]
    a = a0.double()
    want = a @ a.t() + a
    torch.testing.assert_close(first.double(), want, atol=gh.ATOL, rtol=gh.RTOL)


@pytest.mark.parametrize("T", [1, 2])
def test_back_to_back_one_launch_calls_read_what_the_previous_call_wrote(T):
    """The same property at T <= 2 (the one-launch kernel, which starts before
    the previous kernel on the stream has finished): with H = L, each call writes
    its [T, H] output into the first T rows of the next call's W, and that block
    is also the next call's latent/routed and shared partial."""
    torch.manual_seed(60 + T)
    H = L = 1024
    eps = inputs.EPS
    w0 = (torch.randn(H, L, device="cuda") / 32).to(torch.bfloat16)
    g = (1.0 + 0.1 * torch.randn(L, device="cuda")).float()

    def chain(forward, sync):
        Ws = [w0.clone() for _ in range(5)]
        ws = torch.empty(binding.latent_tail_workspace_size(1, T, L, H), dtype=torch.uint8,
                         device="cuda")
        for i in range(4):
            a, out = Ws[i][:T], Ws[i + 1][:T]
            if forward:
                binding.latent_tail_forward(a.view(1, T, L), a.view(1, T, H), g, Ws[i], out, eps,
                                            ws)
            else:
                binding.latent_tail_project_cols(a, a.view(1, T, H), Ws[i], out, 0, H)
            if sync:
                torch.cuda.synchronize()
        binding.latent_tail_check()
        return [w[:T] for w in Ws[1:]]

    for forward in (False, True):
        free, synced = chain(forward, False), chain(forward, True)
        for i, (u, v) in enumerate(zip(free, synced)):
            assert torch.equal(u.view(torch.int16), v.view(torch.int16)), f"forward={forward} step {i}"
    first = chain(False, True)[0].double()
    a, w = w0[:T].double(), w0.double()
    torch.testing.assert_close(first, a @ w.t() + a, atol=gh.ATOL, rtol=gh.RTOL)
