"""Pins for the CPU oracle: checks against facts the pages and the mathematics
fix, none of which re-types the oracle's own loop.

Each pin takes a loaded oracle library, raises AssertionError on a mismatch,
and is chosen so that a specific plausible mistake fails it (the mutation
test builds the oracle with planted mistakes and checks each one is caught):

* g_zero            - closed form: zero norm weight leaves out = sum_p shared
* constant_row      - closed form: a token whose latent sum is the constant c
                      everywhere, W = I, gives out = c*g/sqrt(c^2+eps)
* selection_matrix  - W with one 1 per row at a permuted column, L != H:
                      out[t,h] = y[t, pi(h)], y from the textbook identity
                      rms(x) = ||x||_2 / sqrt(L) via numpy.linalg.norm
* shared_linearity  - out(shared + D) - out(shared) = sum_p D
* p_split           - re-splitting the same exact sums over P partials gives
                      bitwise-identical output
* column_concat     - 16 column ranges concatenate bitwise to the full range
* brute_force       - 40-digit mpmath evaluation of the definition on tiny
                      inputs; the double oracle agrees to 1e-12 and the FP32
                      oracle to FP32 rounding
* no_norm           - without a norm weight the latent is the plain partial
                      sum: W = I gives out = sum_p routed + sum_p shared exactly,
                      and a permuted selection matrix picks x[t, pi(h)]
* torch_formula     - the expectation the PR #51253 runner test prints,
                      F.linear(F.rms_norm(sum_p routed, (L,), g, eps), W) + sum_p
                      shared, evaluated by PyTorch's own CPU kernels in float64 on
                      the tiny configuration and on decode shapes (P = 8, L = 2048,
                      H = 7168, T = 1 and 16): the FP32 oracle agrees to FP32
                      rounding, the double oracle to double rounding
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle

BF16 = torch.bfloat16


def _bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(BF16)


def _rand(gen, *shape, scale=1.0) -> torch.Tensor:
    return (torch.randn(*shape, generator=gen) * scale).to(BF16)


def _f(t: torch.Tensor) -> np.ndarray:
    return t.float().numpy().astype(np.float64)


def g_zero(lib):
    gen = torch.Generator().manual_seed(11)
    P, T, L, H = 3, 4, 16, 24
    routed = _rand(gen, P, T, L)
    W = _rand(gen, H, L, scale=0.25)
    shared = _bf16(torch.randint(-8, 9, (P, T, H), generator=gen))
    g = np.zeros(L, np.float32)
    want = _f(shared).sum(0)
    for prec in ("f32", "f64"):
        got = oracle.forward(routed, shared, g, W, 1e-6, precision=prec, lib=lib)
        assert np.array_equal(got, want), f"g=0 closed form broken ({prec})"
        got = oracle.forward(routed, shared, g, W, 1e-6, 8, 16, precision=prec, lib=lib)
        assert np.array_equal(got, want[:, 8:16]), f"g=0 closed form, cols ({prec})"


def constant_row(lib):
    gen = torch.Generator().manual_seed(12)
    P, L = 2, 32
    H = L
    consts = np.array([2.0 ** -10, 0.75, 3.0, 192.0, -0.5])
    T = len(consts)
    halves = np.repeat((consts / 2)[:, None], L, axis=1)      # exact in bf16
    routed = _bf16(np.stack([halves, halves]))                  # [2, T, L]
    shared = torch.zeros(P, T, H, dtype=BF16)
    W = torch.eye(H, L, dtype=BF16)
    g = (1.0 + 0.1 * torch.randn(L, generator=gen)).numpy().astype(np.float32)
    eps = float(np.float32(1e-6))
    for prec, rtol in (("f32", 3e-6), ("f64", 1e-12)):
        got = oracle.forward(routed, shared, g, W, eps, precision=prec, lib=lib)
        c = consts[:, None]
        want = c * g.astype(np.float64)[None, :] / np.sqrt(c * c + eps)
        assert np.allclose(got, want, rtol=rtol, atol=0), f"constant-row closed form ({prec})"


def selection_matrix(lib):
    gen = torch.Generator().manual_seed(13)
    P, T, L, H = 2, 3, 48, 40
    pi = (7 * np.arange(H) + 3) % L
    Wn = np.zeros((H, L), np.float32)
    Wn[np.arange(H), pi] = 1.0
    W = _bf16(Wn)
    routed = _rand(gen, P, T, L)
    shared = torch.zeros(P, T, H, dtype=BF16)
    g = (1.0 + 0.1 * torch.randn(L, generator=gen)).numpy().astype(np.float32)
    eps = float(np.float32(1e-6))
    x = _f(routed).sum(0)
    rms = np.linalg.norm(x, axis=1, keepdims=True) / math.sqrt(L)
    y = x / np.sqrt(rms * rms + eps) * g.astype(np.float64)
    want = y[:, pi]
    for prec, rtol in (("f32", 2e-5), ("f64", 1e-12)):
        got = oracle.forward(routed, shared, g, W, eps, precision=prec, lib=lib)
        assert np.allclose(got, want, rtol=rtol, atol=rtol), f"selection matrix ({prec})"
        got = oracle.forward(routed, shared, g, W, eps, 8, 40, precision=prec, lib=lib)
        assert np.allclose(got, want[:, 8:40], rtol=rtol, atol=rtol), \
            f"selection matrix, cols ({prec})"


def shared_linearity(lib):
    gen = torch.Generator().manual_seed(14)
    P, T, L, H = 3, 4, 32, 24
    routed = _rand(gen, P, T, L)
    # shared on a 1/8 grid so that shared + delta is exact in bf16
    shared = _bf16(torch.randint(-32, 33, (P, T, H), generator=gen).float() / 8)
    W = _rand(gen, H, L, scale=1 / math.sqrt(L))
    g = (1.0 + 0.1 * torch.randn(L, generator=gen)).numpy().astype(np.float32)
    delta = torch.randint(-4, 5, (P, T, H), generator=gen).float()
    shifted = (shared.float() + delta).to(BF16)
    assert torch.equal(shifted.float() - shared.float(), delta), "delta must be exact"
    for prec, tol in (("f32", 2e-5), ("f64", 1e-12)):
        a = oracle.forward(routed, shared, g, W, 1e-6, precision=prec, lib=lib)
        b = oracle.forward(routed, shifted, g, W, 1e-6, precision=prec, lib=lib)
        want = delta.double().sum(0).numpy()
        assert np.allclose(b - a, want, rtol=0, atol=tol * 16), f"shared linearity ({prec})"


def p_split(lib):
    gen = torch.Generator().manual_seed(15)
    T, L, H = 3, 64, 40
    parts_r = [torch.randint(-40, 41, (T, L), generator=gen) for _ in range(3)]
    parts_s = [torch.randint(-40, 41, (T, H), generator=gen) for _ in range(3)]
    q = 2.0 ** -4
    W = _rand(gen, H, L, scale=1 / math.sqrt(L))
    g = (1.0 + 0.1 * torch.randn(L, generator=gen)).numpy().astype(np.float32)

    def stack(parts):
        return _bf16(torch.stack(parts).float() * q)

    def one(parts):
        return _bf16((sum(p.float() for p in parts) * q)[None])

    two_r = [parts_r[0] + parts_r[1], parts_r[2]]
    two_s = [parts_s[0], parts_s[1] + parts_s[2]]
    for prec in ("f32", "f64"):
        ref = oracle.forward(one(parts_r), one(parts_s), g, W, 1e-6, precision=prec, lib=lib)
        got3 = oracle.forward(stack(parts_r), stack(parts_s), g, W, 1e-6, precision=prec, lib=lib)
        got2 = oracle.forward(stack(two_r), stack(two_s), g, W, 1e-6, precision=prec, lib=lib)
        assert np.array_equal(ref, got3), f"P=3 split differs from P=1 ({prec})"
        assert np.array_equal(ref, got2), f"P=2 split differs from P=1 ({prec})"


def column_concat(lib):
    gen = torch.Generator().manual_seed(16)
    P, T, L, H = 2, 3, 32, 128
    routed = _rand(gen, P, T, L)
    shared = _rand(gen, P, T, H)
    W = _rand(gen, H, L, scale=1 / math.sqrt(L))
    g = (1.0 + 0.1 * torch.randn(L, generator=gen)).numpy().astype(np.float32)
    for prec in ("f32", "f64"):
        full = oracle.forward(routed, shared, g, W, 1e-6, precision=prec, lib=lib)
        step = H // 16
        parts = [oracle.forward(routed, shared, g, W, 1e-6, k * step, (k + 1) * step,
                                precision=prec, lib=lib) for k in range(16)]
        assert np.array_equal(np.concatenate(parts, axis=1), full), \
            f"column shards do not concatenate to the full output ({prec})"
        odd = oracle.forward(routed, shared, g, W, 1e-6, 40, 72, precision=prec, lib=lib)
        assert np.array_equal(odd, full[:, 40:72]), f"odd column range ({prec})"


def brute_force(lib):
    import mpmath

    mpmath.mp.dps = 40
    gen = torch.Generator().manual_seed(17)
    P, T, L, H = 2, 3, 8, 8
    routed = _rand(gen, P, T, L)
    shared = _rand(gen, P, T, H)
    W = _rand(gen, H, L, scale=0.5)
    g = (1.0 + 0.1 * torch.randn(L, generator=gen)).numpy().astype(np.float32)
    eps = float(np.float32(1e-6))
    R, S, Wf = routed.float().tolist(), shared.float().tolist(), W.float().tolist()
    want = np.zeros((T, H))
    scale = np.zeros((T, H))
    for t in range(T):
        x = [mpmath.fsum(mpmath.mpf(R[p][t][l]) for p in range(P)) for l in range(L)]
        ms = mpmath.fsum(v * v for v in x) / L
        inv = 1 / mpmath.sqrt(ms + mpmath.mpf(eps))
        y = [x[l] * inv * mpmath.mpf(float(g[l])) for l in range(L)]
        for h in range(H):
            terms = [y[l] * mpmath.mpf(Wf[h][l]) for l in range(L)]
            terms += [mpmath.mpf(S[p][t][h]) for p in range(P)]
            want[t, h] = float(mpmath.fsum(terms))
            scale[t, h] = float(mpmath.fsum(abs(v) for v in terms))
    got64 = oracle.forward(routed, shared, g, W, eps, precision="f64", lib=lib)
    assert np.all(np.abs(got64 - want) <= 1e-12 * (scale + 1)), "double oracle vs exact"
    got32 = oracle.forward(routed, shared, g, W, eps, precision="f32", lib=lib)
    # forward error of an (L+P)-term FP32 sum of products, with margin for the norm
    bound = (L + P + 8) * 2.0 ** -24 * (scale + 1)
    assert np.all(np.abs(got32 - want) <= bound), "FP32 oracle vs exact"


def no_norm(lib):
    gen = torch.Generator().manual_seed(18)
    P, T, L = 3, 4, 32
    # dyadic partials: every sum below is exact in FP32
    routed = _bf16(torch.randint(-16, 17, (P, T, L), generator=gen).float() / 4)
    shared = _bf16(torch.randint(-16, 17, (P, T, L), generator=gen).float() / 4)
    x = _f(routed).sum(0)
    s = _f(shared).sum(0)
    W = torch.eye(L, dtype=BF16)
    for prec in ("f32", "f64"):
        got = oracle.forward(routed, shared, None, W, 1e-6, precision=prec, lib=lib)
        assert np.array_equal(got, x + s), f"no-norm identity closed form ({prec})"
    H = 24
    pi = (5 * np.arange(H) + 1) % L
    Wn = np.zeros((H, L), np.float32)
    Wn[np.arange(H), pi] = 1.0
    zeros = torch.zeros(P, T, H, dtype=BF16)
    for prec in ("f32", "f64"):
        got = oracle.forward(routed, zeros, None, _bf16(Wn), 1e-6, precision=prec, lib=lib)
        assert np.array_equal(got, x[:, pi]), f"no-norm selection matrix ({prec})"
        y = oracle.latent(routed, None, 1e-6, precision=prec, lib=lib)
        assert np.array_equal(y, x), f"no-norm latent ({prec})"


def _formula(routed, shared, g, W, eps):
    """The page test's expectation in float64: F.linear(F.rms_norm(all-reduced
    routed, (L,), weight, eps), up_proj weight) plus the all-reduced shared
    output, the all-reduce over ranks being the sum over the stacked partials.
    Also returns sum_l |y W| + sum_p |shared|, the scale of the rounding error of
    any evaluation order."""
    import torch.nn.functional as F

    L = routed.shape[-1]
    x = routed.double().sum(0)
    y = F.rms_norm(x, (L,), torch.as_tensor(g).double(), eps)
    Wd = W.double()
    out = F.linear(y, Wd) + shared.double().sum(0)
    scale = F.linear(y.abs(), Wd.abs()) + shared.double().abs().sum(0)
    return out.numpy(), scale.numpy()


def torch_formula(lib):
    from latent_moe_output_gb300 import inputs

    cases = [inputs.make_workload(inputs.TINY),
             inputs.make(8, 1, 2048, 7168, seed=21),
             inputs.make(8, 16, 2048, 7168, seed=22)]
    for x in cases:
        eps = float(np.float32(x.eps))
        want, scale = _formula(x.routed, x.shared, x.g, x.W, eps)
        got64 = oracle.forward(x.routed, x.shared, x.g, x.W, eps, precision="f64", lib=lib)
        assert np.all(np.abs(got64 - want) <= 1e-12 * (scale + 1)), \
            "double oracle differs from F.linear(F.rms_norm(...)) + shared"
        got32 = oracle.forward(x.routed, x.shared, x.g, x.W, eps, lib=lib)
        # FP32 rounding of sums of ~L terms stays far below 1e-5 of their scale
        assert np.all(np.abs(got32 - want) <= 1e-5 * (scale + 1)), \
            "FP32 oracle differs from F.linear(F.rms_norm(...)) + shared"
        # a column range is the matching slice of the formula
        got = oracle.forward(x.routed, x.shared, x.g, x.W, eps, 64, 128, precision="f64",
                             lib=lib)
        assert np.all(np.abs(got - want[:, 64:128]) <= 1e-12 * (scale[:, 64:128] + 1)), \
            "column range differs from the formula's columns"


ALL_PINS = (g_zero, constant_row, selection_matrix, shared_linearity, p_split,
            column_concat, brute_force, no_norm, torch_formula)
