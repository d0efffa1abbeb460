"""Writes tests/golden/oracle_small.txt: a regression fixture of the CPU oracle.

The pages print no worked example of the tail, so no fixture here is the pages'
own numbers. This one records what the oracle (pinned separately against closed
forms, brute force and library special cases) computes on one small seeded
input, so that any later change to the oracle's arithmetic shows up as a
changed bit. It calls only `oracle` and the seeded input generator.

    python tests/golden/make_golden.py
"""

from __future__ import annotations

import struct
import sys
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
ROOT = HERE.parents[1]
sys.path.insert(0, str(ROOT))

import oracle  # noqa: E402
from latent_moe_output_gb300 import inputs  # noqa: E402

P, T, L, H, SEED = 2, 3, 16, 24, 11
COLS = (8, 24)  # a column range as well as the full call


def bits16(t) -> list[str]:
    a = t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16).ravel()
    return [f"{int(v):04x}" for v in a]


def f32hex(a) -> list[str]:
    return [f"{struct.unpack('<I', struct.pack('<f', float(v)))[0]:08x}" for v in np.ravel(a)]


def f64hex(a) -> list[str]:
    return [float(v).hex() for v in np.ravel(a)]


def main() -> None:
    x = inputs.make(P, T, L, H, seed=SEED, device="cpu")
    lines = [f"# oracle regression fixture: P={P} T={T} L={L} H={H} eps={x.eps!r} seed={SEED}",
             "# written by tests/golden/make_golden.py from the CPU oracle; not values from the pages",
             "routed_bf16 " + " ".join(bits16(x.routed)),
             "shared_bf16 " + " ".join(bits16(x.shared)),
             "g_f32 " + " ".join(f32hex(x.g.numpy())),
             "W_bf16 " + " ".join(bits16(x.W))]
    for name, g in (("norm", x.g), ("nonorm", None)):
        for c0, c1 in ((0, H), COLS):
            o32 = oracle.forward(x.routed, x.shared, g, x.W, x.eps, c0, c1, precision="f32")
            o64 = oracle.forward(x.routed, x.shared, g, x.W, x.eps, c0, c1, precision="f64")
            lines.append(f"out_f32_{name}_{c0}_{c1} " + " ".join(f32hex(o32)))
            lines.append(f"out_f64_{name}_{c0}_{c1} " + " ".join(f64hex(o64)))
    (HERE / "oracle_small.txt").write_text("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
