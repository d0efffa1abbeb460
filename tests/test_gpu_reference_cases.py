"""The two checks of the page's runner test, restated for one GPU.

PR #51253 report, key source (test source), `_check_matches_replicated`: with the
routed and shared outputs of tp ranks drawn per rank (seed 100*it + rank + 1) for
the token counts (1, 5, 8, 16, 5), the sharded tail equals F.linear(F.rms_norm(sum of
routed), W) + sum of shared within atol 8e-2 / rtol 3e-2. Here the tp ranks'
partials are the stacked P = tp partials of one call, and the expectation is the
FP32 oracle.

Same test, `_check_writes_only_its_own_shard`: each rank adds latent . W[start:end]^T
into its own shared output in place, over its column shard [rank*H/tp,
(rank+1)*H/tp) only; every other column stays bit-identical. Here that is
latent_tail_project_cols with P = 1, out aliasing the single shared partial, and
the expectation is the FP32 oracle given the all-reduced routed partials and that
rank's shared output as its only shared partial."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_parity
from latent_moe_output_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

L, H = 2048, 7168
TOKENS = (1, 5, 8, 16, 5)


def rank_partials(tp, it, T):
    """Per-rank routed [T, L] and shared [T, H] partials, rank r drawn with seed
    100*it + r + 1 (the page test's seeding), stacked to [tp, T, *]."""
    routed, shared = [], []
    for r in range(tp):
        x = inputs.make(1, T, L, H, seed=100 * it + r + 1, device="cpu")
        routed.append(x.routed[0])
        shared.append(x.shared[0])
    return torch.stack(routed), torch.stack(shared)


@pytest.fixture(scope="module")
def weights():
    x = inputs.make(1, 1, L, H, seed=4242, device="cpu")  # g and W shared by all ranks
    return x.g, x.W


@pytest.mark.parametrize("tp", [4, 8])
def test_matches_replicated(tp, weights):
    g, W = weights
    gd, Wd = g.cuda(), W.cuda()
    for it, T in enumerate(TOKENS):
        routed, shared = rank_partials(tp, it, T)
        out = binding.forward(routed.cuda(), shared.cuda(), gd, Wd, inputs.EPS)
        binding.latent_tail_check()
        want = oracle.forward(routed, shared, g, W, inputs.EPS)
        assert_parity(out, want, f"tp{tp} it{it} T{T}")


@pytest.mark.parametrize("tp", [4, 8])
def test_writes_only_its_own_shard(tp, weights):
    g, W = weights
    gd, Wd = g.cuda(), W.cuda()
    shard = H // tp
    for it, T in enumerate(TOKENS):
        routed, shared = rank_partials(tp, it, T)
        latent = torch.empty(T, L, dtype=torch.bfloat16, device="cuda")
        binding.latent_tail_norm(routed.cuda(), gd, latent, inputs.EPS)
        for rank in range(tp):
            start, end = rank * shard, (rank + 1) * shard
            before = shared[rank].cuda()
            local = before.clone()
            # in place: the rank's own shared output is both the partial and out
            binding.latent_tail_project_cols(latent, local.view(1, T, H), Wd, local, start, end)
            binding.latent_tail_check()
            bits, bbits = local.view(torch.int16), before.view(torch.int16)
            assert torch.equal(bits[:, :start], bbits[:, :start]), f"rank {rank}: wrote below start"
            assert torch.equal(bits[:, end:], bbits[:, end:]), f"rank {rank}: wrote past end"
            # the FP32 oracle with this rank's shared output as the only partial:
            # before[:, start:end] + F.linear(latent, W[start:end])
            # (zero partials next to it keep the partial count equal to routed's)
            only = torch.zeros_like(shared)
            only[0] = shared[rank]
            want = oracle.forward(routed, only, g, W, inputs.EPS, start, end)
            assert_parity(local[:, start:end], want, f"tp{tp} it{it} T{T} rank{rank}")
