"""The column-parallel tail across tensor-parallel ranks (latent_moe_output_gb300.tp),
on CPU gloo ranks, no GPU.

Restates the two checks of the PR #51253 runner test for this module:
`_check_matches_replicated` (with per-rank partials drawn with seed
100 * iteration + rank + 1 for the token counts 1, 5, 8, 16, 5, the stitched result
equals the replicated expectation within atol 8e-2 / rtol 3e-2; here the
expectation is the FP32 oracle on the stacked partials) and
`_check_writes_only_its_own_shard` (before the final collective each rank has
changed only its own column shard, by the projection of the all-reduced latent).
The per-rank projection here is a float64 torch expression written in this test
(the CUDA kernels need a GPU); what is under test is the partition, the
collectives and their order."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from latent_moe_output_gb300 import inputs, tp

L, H = 64, 256
TOKENS = (1, 5, 8, 16, 5)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _project_f64(routed_stack, g, eps, W, shared_rank, start, end):
    """Steps 2-3 in float64 on the CPU: rms_norm of the summed latent, then the
    rank's columns of its shared partial += latent . W[start:end]^T."""
    x = routed_stack.double().sum(0)
    if g is not None:
        x = x * torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + eps) * g.double()
    cols = shared_rank[:, start:end].double() + x @ W[start:end].double().t()
    shared_rank[:, start:end] = cols.to(torch.bfloat16)


def _weights():
    x = inputs.make(1, 1, L, H, seed=4242)  # g and W shared by every rank
    return x.g, x.W


def _rank_partials(it, rank, T):
    x = inputs.make(1, T, L, H, seed=100 * it + rank + 1)
    return x.routed[0], x.shared[0]


def _worker(rank, world, port, exchange, with_norm, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        g, W = _weights()
        g = g if with_norm else None
        report = []
        for it, T in enumerate(TOKENS):
            routed, shared = _rank_partials(it, rank, T)
            before = shared.clone()
            # writes only its own shard, before the final collective
            local = tp.shard_up_proj_partial(routed, shared.clone(), g, W, inputs.EPS,
                                             routed_exchange=exchange, project=_project_f64)
            start, end = tp.shard_range(H, rank, world)
            outside_ok = (torch.equal(local[:, :start], before[:, :start])
                          and torch.equal(local[:, end:], before[:, end:]))
            # the whole tail, stitched by the final all-reduce
            out = tp.column_parallel_tail(routed, shared.clone(), g, W, inputs.EPS,
                                          routed_exchange=exchange, project=_project_f64)
            report.append((it, T, start, end, outside_ok, local[:, start:end].float().numpy(),
                           before[:, start:end].float().numpy(), out.float().numpy()))
        q.put((rank, report))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,exchange,with_norm", [
    (2, "all_reduce", True), (2, "all_gather", True), (4, "all_reduce", True),
    (2, "all_reduce", False),
])
def test_column_parallel_tail_on_gloo_ranks(world, exchange, with_norm):
    import oracle

    ctx = mp.get_context("spawn")
    q = ctx.Manager().Queue()
    mp.start_processes(_worker, args=(world, _free_port(), exchange, with_norm, q), nprocs=world,
                       join=True, start_method="spawn")
    reports = dict(q.get() for _ in range(world))
    g, W = _weights()
    g = g if with_norm else None
    for it, T in enumerate(TOKENS):
        parts = [_rank_partials(it, r, T) for r in range(world)]
        routed = torch.stack([p[0] for p in parts])
        shared = torch.stack([p[1] for p in parts])
        want = oracle.forward(routed, shared, g, W, inputs.EPS)  # replicated expectation
        # the rank's own columns before the final collective: its shared partial
        # plus the projection of the all-reduced latent (no other rank's shared)
        only = torch.zeros_like(shared)
        covered = []
        for r in range(world):
            _, T_r, start, end, outside_ok, local, before, out = reports[r][it]
            assert T_r == T and outside_ok, f"rank {r} wrote outside [{start},{end}) it {it}"
            only.zero_()
            only[0] = parts[r][1]
            own = oracle.forward(routed, only, g, W, inputs.EPS, start, end)
            np.testing.assert_allclose(local, own, atol=8e-2, rtol=3e-2)
            # every rank ends with the whole stitched output
            np.testing.assert_allclose(out, want, atol=8e-2, rtol=3e-2)
            covered.append((start, end))
        assert covered[0][0] == 0 and covered[-1][1] == H
        assert all(covered[i][1] == covered[i + 1][0] for i in range(world - 1))


@pytest.mark.parametrize("H_,world", [(7168, 2), (7168, 8), (7168, 16), (1000, 3), (8, 1), (64, 8)])
def test_shard_ranges_tile_the_columns(H_, world):
    ranges = [tp.shard_range(H_, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == H_
    for (a0, a1), (b0, _) in zip(ranges, ranges[1:]):
        assert a1 == b0
    assert all(s % 8 == 0 and e % 8 == 0 and e > s for s, e in ranges)
    if H_ % (8 * world) == 0:  # the pages' equal H / tp slices
        assert all(e - s == H_ // world for s, e in ranges)


def test_shard_range_rejects_bad_arguments():
    with pytest.raises(ValueError):
        tp.shard_range(1001, 0, 2)
    with pytest.raises(ValueError):
        tp.shard_range(1024, 2, 2)
