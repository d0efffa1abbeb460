"""Column-parallel form (`_check_writes_only_its_own_shard` in the PR #51253
test): a call for [c0,c1) writes exactly those columns, leaves every other
byte of `out` bit-identical, and shards that tile [0,H) reproduce the full
call bit for bit."""

import pytest
import torch

from latent_moe_output_gb300 import binding, inputs

import gpu_helpers as gh

pytestmark = pytest.mark.gpu

SENTINEL = 0x7FC1  # a bf16 NaN payload the kernels never produce


@pytest.fixture(scope="module", autouse=True)
def lib():
    return gh.library()


def sentinel_out(T, H):
    return torch.full((T, H), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)


@pytest.mark.parametrize("P,T,L,H,shards", [
    (8, 16, 2048, 7168, 16),     # decode, 448-column shards
    (4, 5, 64, 128, 16),         # tiny, 8-column shards
    (8, 300, 512, 1792, 16),     # prefill path, 112-column shards (not tile aligned)
    (16, 1024, 2048, 7168, 16),  # stress-like partial count, prefill path
])
def test_shards_concatenate_bitwise(P, T, L, H, shards):
    x = gh.to_dev(inputs.make(P, T, L, H, seed=T + H))
    full = gh.run(x)
    step = H // shards
    stitched = sentinel_out(T, H)
    for k in range(shards):
        c0, c1 = k * step, (k + 1) * step
        out = sentinel_out(T, H)
        gh.run(x, c0, c1, out=out)
        bits = out.view(torch.int16)
        assert (bits[:, :c0] == SENTINEL).all() and (bits[:, c1:] == SENTINEL).all(), \
            f"shard [{c0},{c1}) wrote outside its range"
        stitched[:, c0:c1] = out[:, c0:c1]
    assert torch.equal(stitched.view(torch.int16), full.view(torch.int16))


@pytest.mark.parametrize("T", [9, 200])
@pytest.mark.parametrize("c0,c1", [(8, 16), (120, 136), (248, 520), (0, 1000), (992, 1000)])
def test_odd_ranges(T, c0, c1):
    H = 1000
    x = inputs.make(3, T, 328, H, seed=c0 + c1 + T)
    xd = gh.to_dev(x)
    out = sentinel_out(T, H)
    gh.run(xd, c0, c1, out=out)
    bits = out.view(torch.int16)
    assert (bits[:, :c0] == SENTINEL).all() and (bits[:, c1:] == SENTINEL).all()
    want = gh.oracle_all_rows(x, c0, c1)
    gh.assert_parity(out[:, c0:c1], want, f"cols [{c0},{c1}) T{T}")


def test_stress_sixteen_shards_full_size():
    """The stress workload (P=16, T=16384) as 16 column-shard calls of 448
    columns: every shard stays in its range and the stitched result equals the
    full call bit for bit."""
    w = inputs.STRESS
    x = inputs.make_workload(w, device="cuda")
    full = gh.run(x)
    stitched = sentinel_out(w.T, w.H)
    step = w.H // inputs.STRESS_SHARDS
    ws = torch.empty(binding.latent_tail_workspace_size(w.P, w.T, w.L, w.H),
                     dtype=torch.uint8, device="cuda")
    for k in range(inputs.STRESS_SHARDS):
        c0, c1 = k * step, (k + 1) * step
        binding.latent_tail_forward_cols(x.routed, x.shared, x.g, x.W, stitched, x.eps, c0, c1,
                                         ws)
    binding.latent_tail_check()
    assert torch.equal(stitched.view(torch.int16), full.view(torch.int16))


def test_single_tile_and_multi_tile_epilogues_agree_bitwise():
    """T = 600, H = 7168 (192-column tiles): the full call has 114 tiles for 76 CTA
    pairs (two tiles for some pairs: accumulators double-buffered), each 1792-column
    shard has 30 (one per pair: the shared sums are parked in the idle accumulator's
    TMEM columns while the mainloop runs; shards cut tiles, which start at absolute
    multiples of 192). Both must give the same bits."""
    P, T, L, H = 8, 600, 2048, 7168
    x = gh.to_dev(inputs.make(P, T, L, H, seed=6007))
    full = gh.run(x)
    stitched = sentinel_out(T, H)
    for k in range(4):
        c0, c1 = k * 1792, (k + 1) * 1792
        gh.run(x, c0, c1, out=stitched)
    assert torch.equal(stitched.view(torch.int16), full.view(torch.int16))
