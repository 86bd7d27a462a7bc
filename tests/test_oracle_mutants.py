"""Planted mistakes in the oracle (on the CPU) must each fail some pin.

Every mutant is a copy of the oracle's C source with one plausible mistake
applied to both orders (so the order-equivalence pin alone cannot catch it),
built into a temporary directory and run through the full pin set.
"""
import os
import subprocess

import pytest

import oracle
from tests.oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "tw_oracle.c")

# (name, [(old, new), ...]); every `old` must occur in the source.
MUTANTS = [
    ("residual dropped", [("reduced[i * H + h] + residual[t * H + h]", "reduced[i * H + h]"),
                          ("row[h] + residual[t * H + h]", "row[h]")]),
    ("eps outside sqrt", [("sqrt(sum_sq / (double)H + eps)", "(sqrt(sum_sq / (double)H) + eps)")]),
    ("eps dropped", [("sqrt(sum_sq / (double)H + eps)", "sqrt(sum_sq / (double)H)")]),
    ("sum not mean", [("sqrt(sum_sq / (double)H + eps)", "sqrt(sum_sq + eps)")]),
    ("weight dropped", [("(x[h] / rms) * w[h]", "(x[h] / rms)")]),
    ("weight reversed", [("(x[h] / rms) * w[h]", "(x[h] / rms) * w[H - 1 - h]")]),
    ("rms not inverted", [("(x[h] / rms) * w[h]", "(x[h] * rms) * w[h]")]),
    ("sign of a partial", [("s += partials[r][t * H + h]", "s += (r ? -1.0 : 1.0) * partials[r][t * H + h]"),
                           ("s += partials[q][t * H + h]", "s += (q ? -1.0 : 1.0) * partials[q][t * H + h]")]),
    ("last partial dropped", [("for (int r = 0; r < n_parts; ++r)\n                s +=", "for (int r = 0; r < n_parts - 1; ++r)\n                s +="),
                              ("for (int q = 0; q < n_parts; ++q)", "for (int q = 0; q < n_parts - 1; ++q)")]),
    ("first partial twice", [("s += partials[r][t * H + h]", "s += partials[0][t * H + h]"),
                             ("s += partials[q][t * H + h]", "s += partials[0][t * H + h]")]),
    ("slice drops a token", [("*last = (n_tokens * (int64_t)(r + 1)) / n_ranks;",
                              "*last = (n_tokens * (int64_t)(r + 1)) / n_ranks - (r == 0 && n_tokens > n_ranks);")]),
    ("gather to one destination", [("for (int k = 0; k < n_out; ++k)\n            memcpy", "for (int k = 0; k < 1; ++k)\n            memcpy")]),
    ("residual_out holds y", [("memcpy(residual_out + t * H, x,", "memcpy(residual_out + t * H, out[k] + t * H,"),
                              ("memcpy(row, y, (size_t)H * sizeof(double));",
                               "memcpy(row, y, (size_t)H * sizeof(double));\n            memcpy(residual_out + t * H, y, (size_t)H * sizeof(double));")]),
]


def _build_mutant(tmp_path, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert old in src, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new)
    c_path = tmp_path / "tw_oracle_mut.c"
    c_path.write_text(src)
    inc = os.path.dirname(SRC)
    so = tmp_path / "libtw_oracle_mut.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-I", inc,
                    "-shared", "-fPIC", "-o", str(so), str(c_path), "-lm"],
                   check=True)
    return oracle.Oracle(str(so))


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, edits):
    orc = _build_mutant(tmp_path, edits)
    failed = []
    for pin in PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake: {name}"
