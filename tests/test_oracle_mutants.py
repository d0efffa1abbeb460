"""Mutation test of the oracle's pins: each planted mistake must fail at least
one pin. A mistake is planted by patching one line of a temporary copy of the
oracle's source (on the CPU); the oracle's own file holds only the definition."""

from pathlib import Path

import pytest

import oracle
import pins

ROUTED_SUM = "for (long p = 0; p < P; ++p) s += widen_bf16(routed[((p * T) + t) * L + l]);"
SHARED_SUM = ("for (long p = 0; p < P; ++p)\n"
              "        s += widen_bf16(shared[((p * T) + t) * H + h]);")
DOT = "for (long l = 0; l < L; ++l) acc += y[l] * widen_bf16(W[h * L + l]);"

# id: (what goes wrong, text in the oracle's source, text that replaces it)
MUTANTS = {
    1: ("eps added outside the square root",
        "const Acc r = static_cast<Acc>(1) / std::sqrt(ms + eps);",
        "const Acc r = static_cast<Acc>(1) / (std::sqrt(ms) + eps);"),
    2: ("sum of squares used instead of the mean",
        "const Acc ms = ss / static_cast<Acc>(L);",
        "const Acc ms = ss;"),
    3: ("W read transposed, as if it were [L, H]",
        DOT, DOT.replace("W[h * L + l]", "W[l * H + h]")),
    4: ("first shared partial dropped",
        SHARED_SUM, SHARED_SUM.replace("long p = 0", "long p = 1")),
    5: ("routed partials read as if laid out [T, P, L]",
        ROUTED_SUM, ROUTED_SUM.replace("((p * T) + t)", "((t * P) + p)")),
    6: ("norm weight dropped",
        "y[l] = x[l] * r * static_cast<Acc>(g[l]);",
        "y[l] = x[l] * r;"),
    7: ("shared partials read as if laid out [T, P, H]",
        SHARED_SUM, SHARED_SUM.replace("((p * T) + t)", "((t * P) + p)")),
    8: ("W row taken relative to the column range start",
        DOT, DOT.replace("W[h * L + l]", "W[(h - c0) * L + l]")),
    9: ("squares of the partials summed instead of the square of the sum",
        "for (long l = 0; l < L; ++l) ss += x[l] * x[l];",
        "for (long l = 0; l < L; ++l)\n"
        "    for (long p = 0; p < P; ++p) {\n"
        "      const Acc v = widen_bf16(routed[((p * T) + t) * L + l]);\n"
        "      ss += v * v;\n"
        "    }"),
    10: ("no-norm branch still normalizes (unit weight)",
         "for (long l = 0; l < L; ++l) y[l] = x[l];\n    return;",
         "Acc ss0 = 0;\n"
         "    for (long l = 0; l < L; ++l) ss0 += x[l] * x[l];\n"
         "    const Acc r0 = static_cast<Acc>(1) / std::sqrt(ss0 / static_cast<Acc>(L) + eps);\n"
         "    for (long l = 0; l < L; ++l) y[l] = x[l] * r0;\n    return;"),
    11: ("only the first four routed partials summed",
         ROUTED_SUM, ROUTED_SUM.replace("p < P;", "p < P && p < 4;")),
}


def planted(tmp_path: Path, mutant: int) -> Path:
    _, old, new = MUTANTS[mutant]
    text = oracle.SOURCE.read_text()
    assert text.count(old) == 1, f"mutant {mutant}: its target text must occur once"
    src = tmp_path / f"oracle_m{mutant}.cpp"
    src.write_text(text.replace(old, new))
    return src


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda k: f"m{k}")
def test_pins_catch_planted_mistake(tmp_path, mutant):
    so = oracle.build(tmp_path / f"liblt_oracle_m{mutant}.so", source=planted(tmp_path, mutant))
    lib = oracle.load(so)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {mutant}: {MUTANTS[mutant][0]}"


def test_unpatched_source_passes_every_pin(tmp_path):
    so = oracle.build(tmp_path / "liblt_oracle_copy.so", source=oracle.SOURCE)
    lib = oracle.load(so)
    for pin in pins.ALL_PINS:
        pin(lib)
