"""The column-parallel tail's product path on one GPU: a one-rank NCCL group
runs latent_moe_output_gb300.tp with the CUDA kernels (norm, then the in-place
narrowed projection over the rank's shard, which is every column) and the
collectives, checked against the FP32 oracle. The multi-rank partition and
collectives are covered on CPU gloo ranks (test_tp_cpu.py)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist

from latent_moe_output_gb300 import inputs, tp

import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("exchange", ["all_reduce", "all_gather"])
@pytest.mark.parametrize("T", [16, 200, 300])
def test_one_rank_nccl_group_matches_oracle(exchange, T):
    gh.library()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        x = inputs.make(1, T, 2048, 7168, seed=900 + T)
        xd = gh.to_dev(x)
        out = tp.column_parallel_tail(xd.routed[0], xd.shared[0].clone(), xd.g, xd.W, x.eps,
                                      routed_exchange=exchange)
        torch.cuda.synchronize()
        gh.assert_parity(out, gh.oracle_all_rows(x), f"one-rank tp T{T} {exchange}")
    finally:
        dist.destroy_process_group()
