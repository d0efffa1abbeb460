"""CUDA path versus the CPU oracle, element by element, at the pages' bf16
tolerance (atol 8e-2, rtol 3e-2). Every config of the benchmark list plus
ragged shapes that span several tiles and leave partial tails."""

import numpy as np
import pytest
import torch

from latent_moe_output_gb300 import binding, inputs

import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return gh.library()


def check_full(x, c0=0, c1=None, what=""):
    xd = gh.to_dev(x)
    got = gh.run(xd, c0, c1)
    H = x.W.shape[0]
    c1 = H if c1 is None else c1
    want = gh.oracle_all_rows(x, c0, c1)
    gh.assert_parity(got[:, c0:c1], want, what)
    return got


def test_tiny():
    check_full(inputs.make_workload(inputs.TINY), what="tiny")


def test_decode():
    check_full(inputs.make_workload(inputs.DECODE), what="decode P8 T16")


@pytest.mark.parametrize("w", inputs.DECODE_SWEEP, ids=lambda w: w.name)
def test_decode_sweep(w):
    check_full(inputs.make_workload(w), what=w.name)


@pytest.mark.parametrize("P,T,L,H", [
    (1, 1, 64, 128),       # single token, single partial, one tile
    (3, 7, 328, 1000),     # ragged K-block (328 = 5*64 + 8) and ragged 128-row tile
    (5, 17, 2048, 520),    # tokens not a multiple of 16
    (3, 13, 2248, 392),    # eight K slices (T <= 16), the last one a single ragged K-block
    (2, 128, 512, 384),    # decode, 128 tokens
    (2, 224, 512, 384),    # largest decode token count (two K slices)
    (3, 129, 328, 1000),   # decode above 128 tokens with one K slice, ragged everywhere
    (3, 225, 328, 1000),   # smallest prefill token count, ragged everywhere
    (2, 300, 192, 776),    # several 128-token tiles plus a tail; ragged 192-col tile
    (2, 4100, 192, 776),   # the same with 256-col tiles (17 token groups)
    (4, 520, 2048, 512),   # several token tiles at the production latent width
    (1, 1000, 64, 2056),   # many tiles, one K-block, P = 1 (pre-reduced latent)
    (16, 200, 256, 264),   # P = 16 partials
    (64, 4, 256, 256),     # P = 64, the largest partial count accepted (decode)
    (64, 2, 256, 256),     # P = 64 on the one-launch kernel
    (64, 240, 128, 256),   # P = 64 on the prefill path
    (2, 8, 16384, 256),    # L = 16384, the largest latent width accepted (decode)
    (2, 2, 4096, 256),     # T = 2 at L = 4096: the widest latent the one-launch kernel takes
    (2, 2, 8192, 256),     # T = 2 at L = 8192: too wide for it, the two-kernel path runs
    (3, 2, 2048, 19464),   # T = 2, one SM's W slice too large: the two-kernel path runs
    (3, 2, 328, 1000),     # one-launch kernel, ragged latent (328 = 256 + 72)
    (1, 1, 8, 8),          # L = H = 8 on the one-launch kernel: one CTA, one 8-row chunk
    (7, 1, 2056, 7176),    # one-launch: 257 latent pieces (two for thread 0), P = 7, last CTA 24 rows
    (9, 2, 4096, 1024),    # one-launch: the widest latent (two pieces per thread), P = 9 (two batches)
    (2, 260, 16384, 128),  # L = 16384 on the prefill path
    (2, 200, 16384, 136),  # L = 16384 on the decode kernel above 128 tokens (two K slices)
    (64, 160, 256, 256),   # P = 64 on the decode kernel above 128 tokens (one K slice)
    (1, 200, 64, 2056),    # P = 1, one K-block, 200 tokens on the decode kernel
    (1, 3, 8, 8),          # L = H = 8, the smallest accepted: boxes wider than the tensor
    (2, 130, 8, 16),       # the same above 128 tokens (decode kernel)
    (2, 230, 8, 16),       # the same on the prefill path
])
def test_ragged_shapes(P, T, L, H):
    x = inputs.make(P, T, L, H, seed=P * 1000 + T)
    check_full(x, what=f"P{P} T{T} L{L} H{H}")


@pytest.mark.parametrize("w", [inputs.PREFILL, inputs.STRESS, inputs.PREFILL_P1],
                         ids=lambda w: w.name)
def test_full_size_every_element(w):
    """Full benchmark sizes on the device, every output element against the FP32
    oracle (token ranges of the oracle run concurrently on the host cores). The
    stress workload includes its x100 and x1e-3 outlier rows."""
    x = inputs.make_workload(w, device="cuda")
    got = gh.run(x)
    want = gh.oracle_all_rows(x)
    gh.assert_parity(got, want, w.name)
    if w.outlier_rows:  # the outlier rows are among the rows compared above
        assert len(x.scaled_up) == len(x.scaled_down) == w.T // 100


@pytest.mark.parametrize("T", [129, 160, 224, 225])
def test_decode_tier_above_128_tokens(T):
    """The decode kernel's range above 128 tokens at the production widths (P = 8,
    L = 2048, H = 7168: two K slices, one CTA per SM, the K-slice partials in the
    stage ring), every element; T = 225 is the first token count of the prefill
    kernel."""
    check_full(inputs.make(8, T, 2048, 7168, seed=1300 + T), what=f"T{T}")


@pytest.mark.parametrize("T", [72, 96, 97, 112])
def test_decode_tier_around_the_slice_switch(T):
    """The decode kernel keeps four K slices (two CTAs per SM) up to 96 tokens and
    two slices (one CTA per SM) above: both sides of the switch, every element at
    the production widths."""
    check_full(inputs.make(8, T, 2048, 7168, seed=1500 + T), what=f"T{T}")


@pytest.mark.parametrize("P,T,L,H", [
    (2, 65, 64, 264),      # one K-block, one slice; the last 128-row tile has 8 rows
    (3, 100, 328, 392),    # ragged K-block, one slice, last tile 8 rows
    (2, 97, 512, 136),     # two slices just above the switch, last tile 8 rows
    (5, 224, 1024, 520),   # the largest decode token count, five tiles
])
def test_decode_tier_ragged(P, T, L, H):
    check_full(inputs.make(P, T, L, H, seed=P * 1000 + T + 7), what=f"P{P} T{T} L{L} H{H}")


@pytest.mark.parametrize("T", [104, 160, 224])
def test_decode_tier_column_ranges_tile_the_full_call(T):
    """Column ranges of the decode kernel with two K slices (tiles cut by the
    range, partial first and last tiles) reproduce the full call bit for bit."""
    x = gh.to_dev(inputs.make(8, T, 2048, 7168, seed=1400 + T))
    full = gh.run(x)
    pieces = torch.full_like(full, float("nan"))
    for c0, c1 in ((0, 1000), (1000, 4104), (4104, 7160), (7160, 7168)):
        gh.run(x, c0, c1, out=pieces)
    assert torch.equal(pieces.view(torch.int16), full.view(torch.int16))


@pytest.mark.parametrize("T,L,H", [
    (4096, 2048, 7168),    # the first token count of the 512-column tiles, production widths
    (4100, 328, 1416),     # ragged token group and K-block; the last tile ends inside its
                           # fourth 128-column block (tile columns 384..391 of 512)
    (4100, 64, 1032),      # one K-block; the last tile holds 8 columns, 4 tokens in the last group
])
def test_wide_tiles_single_partial(T, L, H):
    """With one shared partial, T >= 4096 and at most half the waves of 256-column
    tiles, the prefill kernel uses 512-column tiles
    (two N = 256 instructions per K-step whose accumulator blocks hold tile columns
    0, 256, 128, 384): every element against the oracle."""
    check_full(inputs.make(1, T, L, H, seed=2600 + T), what=f"P1 T{T} L{L} H{H}")


def test_wide_tiles_column_ranges_tile_the_full_call():
    """Column ranges that cut 512-column tiles inside every 128-column block
    reproduce the full call bit for bit, and write nothing outside their range."""
    x = gh.to_dev(inputs.make(1, 4096, 256, 1544, seed=2700))
    full = gh.run(x)
    pieces = torch.full_like(full, float("nan"))
    for c0, c1 in ((0, 136), (136, 648), (648, 1160), (1160, 1544)):
        gh.run(x, c0, c1, out=pieces)
    assert torch.equal(pieces.view(torch.int16), full.view(torch.int16))


@pytest.mark.parametrize("T", [1, 2, 3])
def test_one_launch_token_counts(T):
    """T <= 2 at the production widths (P = 8, L = 2048, H = 7168): the CUDA-core
    kernel that does the whole tail in one launch, every element; T = 3 is the
    first token count of the two-kernel path."""
    check_full(inputs.make(8, T, 2048, 7168, seed=900 + T), what=f"one-launch T{T}")


@pytest.mark.parametrize("T", [1, 2])
def test_one_launch_column_ranges_tile_the_full_call(T):
    """Column ranges that tile [0, H) reproduce the full call bit for bit: each
    output element is formed by one warp in the same order whatever the range,
    and every CTA builds the same FP32 latent. The ranges have different widths,
    so each gives its CTAs a different number of W rows."""
    assert T <= 2  # the one-launch kernel
    x = gh.to_dev(inputs.make(8, T, 2048, 7168, seed=950 + T))
    full = gh.run(x)
    pieces = torch.full_like(full, float("nan"))
    for c0, c1 in ((0, 1000), (1000, 4104), (4104, 7160), (7160, 7168)):
        gh.run(x, c0, c1, out=pieces)
    assert torch.equal(pieces.view(torch.int16), full.view(torch.int16))


def test_norm_stage_matches_oracle_latent():
    import oracle

    x = inputs.make(8, 37, 2048, 128, seed=9)
    xd = gh.to_dev(x)
    y = torch.empty(37, 2048, dtype=torch.bfloat16, device="cuda")
    binding.latent_tail_norm(xd.routed, xd.g, y, x.eps)
    binding.latent_tail_check()
    want = oracle.latent(x.routed, x.g, x.eps)
    # one bf16 rounding of an FP32 value: relative error <= 2^-8
    err = np.abs(y.float().cpu().numpy() - want)
    assert np.all(err <= 2.0 ** -8 * np.abs(want) + 1e-6)


@pytest.mark.parametrize("T", [16, 600])
def test_forward_equals_norm_then_project(T):
    x = gh.to_dev(inputs.make(8, T, 2048, 1024, seed=T))
    full = gh.run(x)
    y = torch.empty(T, 2048, dtype=torch.bfloat16, device="cuda")
    binding.latent_tail_norm(x.routed, x.g, y, x.eps)
    out = torch.empty_like(full)
    binding.latent_tail_project_cols(y, x.shared, x.W, out, 0, 1024)
    binding.latent_tail_check()
    assert torch.equal(out, full)


def test_zero_tokens():
    x = gh.to_dev(inputs.make(2, 0, 64, 128, seed=0))
    out = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.latent_tail_forward(x.routed, x.shared, x.g, x.W, out, x.eps, ws)
    binding.latent_tail_check()


@pytest.mark.parametrize("P,T,L,H", [(2, 5, 64, 128), (8, 2, 2048, 7168), (8, 16, 2048, 7168), (3, 300, 328, 1000),
                                     (2, 200, 256, 1000)])
def test_no_norm_branch(P, T, L, H):
    """norm_weight = None: the latent is the routed partial sum itself (the
    `transform.norm is None` branch of `_shard_up_proj_tail`)."""
    import oracle

    x = inputs.make(P, T, L, H, seed=77 + T)
    xd = gh.to_dev(x)
    got = binding.forward(xd.routed, xd.shared, None, xd.W, x.eps)
    binding.latent_tail_check()
    want = oracle.forward(x.routed, x.shared, None, x.W, x.eps)
    gh.assert_parity(got, want, f"no-norm P{P} T{T} L{L} H{H}")
    y = torch.empty(T, L, dtype=torch.bfloat16, device="cuda")
    binding.latent_tail_norm(xd.routed, None, y, x.eps)
    binding.latent_tail_check()
    ywant = oracle.latent(x.routed, None, x.eps)
    err = np.abs(y.float().cpu().numpy() - ywant)
    assert np.all(err <= 2.0 ** -8 * np.abs(ywant) + 1e-6)
