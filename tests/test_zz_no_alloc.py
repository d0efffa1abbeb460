"""The allocation-free entry point, latent_tail_forward_noalloc.

It serves callers that cannot allocate device memory (a custom op that its
host runtime gives only input and output buffers, or code that must not
allocate while it runs): the path's scratch lives in a fixed 8 MiB device
array inside the library instead of a caller workspace. These tests
call it through the C ABI and compare it with latent_tail_forward on two calls
in a row, so the second call also shows that the first call's leftovers in the
shared array do not leak into the result. The file sorts last so that a run
stopping at the first failure has already run every other test.
"""

import ctypes

import pytest
import torch

from latent_moe_output_gb300 import binding, inputs
from latent_moe_output_gb300.binding import Status

import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, x, out, stream):
    P, T, L = x.routed.shape
    H = x.W.shape[0]
    return lib.latent_tail_forward_noalloc(_ptr(x.routed), _ptr(x.shared), _ptr(x.g), _ptr(x.W),
                                           _ptr(out), P, T, L, H, x.eps, stream.cuda_stream)


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    lib = gh.library()
    stream = torch.cuda.current_stream()
    cases = [inputs.make(8, 16, 2048, 7168, seed=41), inputs.make(8, 128, 2048, 7168, seed=42)]
    for x in cases:  # two different calls back to back on the same scratch
        xd = gh.to_dev(x)
        ref = gh.run(xd)
        out = torch.full_like(ref, float("nan"))
        st = _noalloc(lib, xd, out, stream)
        assert st == Status.OK, binding.latent_tail_status_string(st)
        binding.latent_tail_check()
        torch.testing.assert_close(out.float(), ref.float(), atol=gh.ATOL, rtol=gh.RTOL)
        T = x.routed.shape[1]
        want = gh.oracle_rows(x, [0, T // 2, T - 1])
        gh.assert_parity(out[[0, T // 2, T - 1]], want, "noalloc vs oracle")


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    lib = gh.library()
    # workspace 2049 * 2048 * 2 bytes > 8 MiB: rejected before any launch
    x = gh.to_dev(inputs.make(1, 2049, 2048, 128, seed=5))
    out = torch.zeros(2049, 128, dtype=torch.bfloat16, device="cuda")
    st = _noalloc(lib, x, out, torch.cuda.current_stream())
    assert st == Status.WORKSPACE
    binding.latent_tail_check()
    assert (out == 0).all()
