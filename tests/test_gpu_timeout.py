"""Bounded device waits: a wait made to run out (a barrier nothing completes)
reports LT_ERR_TIMEOUT through latent_tail_check, and the context stays usable."""

import pytest
import torch

from latent_moe_output_gb300 import binding, inputs
from latent_moe_output_gb300.binding import LatentTailError, Status

import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives():
    lib = gh.library()
    x = gh.to_dev(inputs.make(2, 16, 256, 256, seed=8))
    before = gh.run(x)
    stream = torch.cuda.current_stream()
    assert lib.latent_tail_selftest_wait_timeout(2000, stream.cuda_stream) == Status.OK
    with pytest.raises(LatentTailError) as e:
        binding.latent_tail_check()
    assert e.value.status == Status.TIMEOUT
    binding.latent_tail_check()  # the error word was cleared
    after = gh.run(x)
    assert torch.equal(before, after)


def test_selftest_rejects_bad_limits():
    lib = gh.library()
    assert lib.latent_tail_selftest_wait_timeout(0, None) == Status.INVALID_ARG
    assert lib.latent_tail_selftest_wait_timeout(2000000, None) == Status.INVALID_ARG
