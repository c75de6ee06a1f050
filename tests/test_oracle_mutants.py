"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a temporary copy of
oracle/gsi_oracle.c (a dropped term, a wrong sign, a transposed index, a
wrong tie rule, ...), compiles it, and requires that at least one pin in
tests/oracle_pins.py rejects the broken copy.  The oracle itself is never
modified.
"""
import os

import pytest

import oracle as orc_pkg
import oracle_pins as pins
from oracle.oracle import OracleLib

MUTANTS = [
    ("residual sign", "double ri = x[i] - vg;", "double ri = x[i] + vg;"),
    ("residual drops V g", "double ri = x[i] - vg;", "double ri = x[i];"),
    ("projection transposed", "s += V[i * k + j] * x[i];", "s += V[j * d + i] * x[i];"),
    ("tie goes fast", "gate[t] = (p < eps) ? 0 : 1;", "gate[t] = (p <= eps) ? 0 : 1;"),
    ("branches swapped", "if (gate[t]) {", "if (!gate[t]) {"),
    ("norm without sqrt", "double nx = sqrt(xx);", "double nx = xx;"),
    ("zero token slow", "        return 0.0;\n    return nr / nx;", "        return 1.0;\n    return nr / nx;"),
    ("ratio inverted", "return nr / nx;", "return nr / (nx + nr);"),
    ("M transposed", "s += W[o * d + i] * V[i * k + j];", "s += W[o * d + i] * V[j * d + i];"),
    ("fast path M transposed", "s += M[o * k + j] * g[j];", "s += M[j * d_out + o] * g[j];"),
    ("slow path W transposed", "s += W[o * d + i] * x[i];", "s += W[i * d_out + o] * x[i];"),
    ("bf16 ties away", "double r = ldexp(rint(ldexp(v, -q)), q);",
     "double r = ldexp(round(ldexp(v, -q)), q);"),
    ("bf16 quantum", "int q = e - 8;", "int q = e - 7;"),
    ("spectral norm squared", "double est = sqrt(ww);", "double est = ww;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    with open(orc_pkg.SRC_PATH) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for '{name}' not unique"
    mpath = os.path.join(tmp_path, "mutant.c")
    with open(mpath, "w") as f:
        f.write(src.replace(old, new))
    so = orc_pkg.build(src=mpath, out=os.path.join(tmp_path, "libmutant.so"), force=True)
    mut = OracleLib(so)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            getattr(pins, pin)(mut)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin)
    assert caught, f"no pin caught the planted mistake '{name}'"
