"""The CPU oracle against its pins (no GPU)."""

import numpy as np
import pytest
import torch

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_lib, pin):
    pin(oracle_lib)


def test_oracle_rejects_bad_arguments(oracle_lib):
    r = torch.zeros(1, 2, 8, dtype=torch.bfloat16)
    s = torch.zeros(1, 2, 16, dtype=torch.bfloat16)
    w = torch.zeros(16, 8, dtype=torch.bfloat16)
    g = np.ones(8, np.float32)
    for c0, c1 in ((8, 8), (-8, 8), (0, 24), (16, 8)):
        with pytest.raises(ValueError):
            oracle.forward(r, s, g, w, 1e-6, c0, c1, lib=oracle_lib)


def test_oracle_zero_tokens(oracle_lib):
    r = torch.zeros(2, 0, 8, dtype=torch.bfloat16)
    s = torch.zeros(2, 0, 16, dtype=torch.bfloat16)
    w = torch.zeros(16, 8, dtype=torch.bfloat16)
    out = oracle.forward(r, s, np.ones(8, np.float32), w, 1e-6, lib=oracle_lib)
    assert out.shape == (0, 16)


def test_fp32_oracle_within_fp32_rounding_of_double_at_production_width(oracle_lib):
    """One decode-shaped token (P=8, L=2048, H=7168): the FP32 oracle differs
    from the double one only by FP32 rounding, far inside the bf16 tolerance."""
    from latent_moe_output_gb300 import inputs

    x = inputs.make(8, 2, 2048, 7168, seed=5)
    a = oracle.forward(x.routed, x.shared, x.g, x.W, x.eps, precision="f32", lib=oracle_lib)
    b = oracle.forward(x.routed, x.shared, x.g, x.W, x.eps, precision="f64", lib=oracle_lib)
    assert np.max(np.abs(a - b)) < 1e-4
    y32 = oracle.latent(x.routed, x.g, x.eps, precision="f32", lib=oracle_lib)
    y64 = oracle.latent(x.routed, x.g, x.eps, precision="f64", lib=oracle_lib)
    assert np.max(np.abs(y32 - y64)) < 1e-5
    # the normalized latent has unit RMS up to the weight g and eps
    rms = np.sqrt(np.mean((y64 / x.g.double().numpy()) ** 2, axis=1))
    assert np.allclose(rms, 1.0, atol=1e-5)


def test_chunked_concurrent_oracle_equals_one_call(oracle_lib):
    """The GPU parity tests run the oracle over token ranges concurrently (rows
    are independent); the stitched result is bit for bit the one-call result."""
    import gpu_helpers as gh
    from latent_moe_output_gb300 import inputs

    x = inputs.make(3, 37, 64, 96, seed=8)
    one = oracle.forward(x.routed, x.shared, x.g, x.W, x.eps, 8, 88, lib=oracle_lib)
    many = gh.oracle_all_rows(x, 8, 88, chunk=5, workers=4)
    assert np.array_equal(one, many)
