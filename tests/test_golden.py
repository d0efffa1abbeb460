"""The CPU oracle against its stored regression fixture (tests/golden/).

The fixture was written by tests/golden/make_golden.py from the oracle itself
(the pages print no worked example), so it pins the oracle against unintended
change, bit for bit, in FP32 and FP64, with and without the norm, for the full
column range and a sub-range. Its correctness is pinned by test_oracle.py."""

import struct
from pathlib import Path

import numpy as np
import pytest

import oracle

FIXTURE = Path(__file__).resolve().parent / "golden" / "oracle_small.txt"


def load():
    rows = {}
    for line in FIXTURE.read_text().splitlines():
        if line.startswith("#") or not line.strip():
            continue
        key, *vals = line.split()
        rows[key] = vals
    return rows


def shape_args():
    head = FIXTURE.read_text().splitlines()[0]
    kv = dict(item.split("=") for item in head.split(":")[1].split())
    return int(kv["P"]), int(kv["T"]), int(kv["L"]), int(kv["H"]), float(kv["eps"])


def u16(vals, shape):
    return np.array([int(v, 16) for v in vals], dtype=np.uint16).reshape(shape)


def f32(vals):
    return np.array([struct.unpack("<f", struct.pack("<I", int(v, 16)))[0] for v in vals],
                    dtype=np.float32)


@pytest.fixture(scope="module")
def fx():
    P, T, L, H, eps = shape_args()
    r = load()
    return dict(P=P, T=T, L=L, H=H, eps=eps, rows=r,
                routed=u16(r["routed_bf16"], (P, T, L)), shared=u16(r["shared_bf16"], (P, T, H)),
                g=f32(r["g_f32"]), W=u16(r["W_bf16"], (H, L)))


@pytest.mark.parametrize("name", ["norm", "nonorm"])
@pytest.mark.parametrize("cols", ["full", "range"])
def test_oracle_matches_stored_fixture(fx, name, cols):
    keys = [k for k in fx["rows"] if k.startswith(f"out_f32_{name}_")]
    key32 = sorted(keys)[0] if cols == "full" else sorted(keys)[-1]
    c0, c1 = (int(v) for v in key32.split("_")[-2:])
    g = fx["g"] if name == "norm" else None
    o32 = oracle.forward(fx["routed"], fx["shared"], g, fx["W"], fx["eps"], c0, c1,
                         precision="f32")
    o64 = oracle.forward(fx["routed"], fx["shared"], g, fx["W"], fx["eps"], c0, c1,
                         precision="f64")
    got32 = [f"{struct.unpack('<I', struct.pack('<f', float(v)))[0]:08x}" for v in o32.ravel()]
    got64 = [float(v).hex() for v in o64.ravel()]
    assert got32 == fx["rows"][key32], f"FP32 oracle output changed ({key32})"
    assert got64 == fx["rows"][key32.replace("f32", "f64")], f"FP64 oracle output changed"


def test_fixture_inputs_are_the_seeded_generator_output(fx):
    """The fixture's inputs are what the input generator draws for its seed (a change
    here means the generator, not the oracle, changed)."""
    import torch

    from latent_moe_output_gb300 import inputs

    head = FIXTURE.read_text().splitlines()[0]
    seed = int(head.split("seed=")[1])
    x = inputs.make(fx["P"], fx["T"], fx["L"], fx["H"], seed=seed, device="cpu")
    as16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    assert np.array_equal(as16(x.routed), fx["routed"])
    assert np.array_equal(as16(x.shared), fx["shared"])
    assert np.array_equal(as16(x.W), fx["W"])
    assert np.array_equal(x.g.numpy(), fx["g"])
