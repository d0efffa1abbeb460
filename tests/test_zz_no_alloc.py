"""The allocation-free entry point, latent_tail_forward_noalloc.

It serves callers that cannot allocate device memory (a custom op that its
host runtime gives only input and output buffers, or code that must not
allocate while it runs): the path's scratch lives in a fixed 8 MiB device
array inside the library instead of a caller workspace. These tests call it
through the C ABI and compare it with latent_tail_forward and with the FP32
oracle on calls in a row that share the array: first a prefill-sized call that
fills the array exactly, then smaller calls that leave its later rows stale,
so a result that picked up another call's leftovers would show. The file sorts
last so that a run stopping at the first failure has already run every other
test.
"""

import ctypes

import pytest
import torch

from latent_moe_output_gb300 import binding, inputs
from latent_moe_output_gb300.binding import Status

import gpu_helpers as gh

pytestmark = pytest.mark.gpu

MAX_SCRATCH = 8 << 20  # LT_NOALLOC_MAX_SCRATCH_BYTES


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, x, out, stream):
    P, T, L = x.routed.shape
    H = x.W.shape[0]
    return lib.latent_tail_forward_noalloc(_ptr(x.routed), _ptr(x.shared), _ptr(x.g), _ptr(x.W),
                                           _ptr(out), P, T, L, H, x.eps, stream.cuda_stream)


def test_noalloc_matches_forward_on_calls_in_a_row():
    lib = gh.library()
    stream = torch.cuda.current_stream()
    # T = 2048 at L = 2048 needs exactly the whole array (prefill kernel); the
    # decode-sized calls after it read only the first rows of what it left.
    shapes = [(8, 2048, 2048, 7168, 41), (8, 16, 2048, 7168, 42), (8, 128, 2048, 7168, 43),
              (8, 1, 2048, 7168, 44)]
    assert binding.latent_tail_workspace_size(8, 2048, 2048, 7168) == MAX_SCRATCH
    for P, T, L, H, seed in shapes:
        x = inputs.make(P, T, L, H, seed=seed)
        xd = gh.to_dev(x)
        ref = gh.run(xd)
        out = torch.full_like(ref, float("nan"))
        st = _noalloc(lib, xd, out, stream)
        assert st == Status.OK, binding.latent_tail_status_string(st)
        binding.latent_tail_check()
        torch.testing.assert_close(out.float(), ref.float(), atol=gh.ATOL, rtol=gh.RTOL)
        gh.assert_parity(out, gh.oracle_all_rows(x), f"noalloc T{T} vs oracle")


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    lib = gh.library()
    # workspace 2049 * 2048 * 2 bytes > 8 MiB: rejected before any launch
    x = gh.to_dev(inputs.make(1, 2049, 2048, 128, seed=5))
    out = torch.zeros(2049, 128, dtype=torch.bfloat16, device="cuda")
    st = _noalloc(lib, x, out, torch.cuda.current_stream())
    assert st == Status.WORKSPACE
    binding.latent_tail_check()
    assert (out == 0).all()
