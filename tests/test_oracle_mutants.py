"""Mutation checks for the oracle's pins: each test plants one plausible slip in a COPY of
the oracle's C source (on the CPU), builds it, and asserts that at least one pin fails.
The shipped oracle is never modified."""

import os

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mg_oracle.c")

# (name, text in the source, replacement). Every replacement keeps indices in bounds.
MUTANTS = [
    ("exp of the negated score", "E[n] = exp(A[n]);", "E[n] = exp(-A[n]);"),
    ("stray 1/sqrt(d) scale", "E[n] = exp(A[n]);", "E[n] = exp(A[n] / sqrt((double)d));"),
    ("normalisation dropped", "E[n] = E[n] / S;", "E[n] = E[n];"),
    ("first term dropped from the row sum",
     "for (int64_t n = 0; n < N; ++n)\n        S += E[n];", "for (int64_t n = 1; n < N; ++n)\n        S += E[n];"),
    ("last head-dim term dropped from Q.K", "for (int64_t k = 0; k < d; ++k) {", "for (int64_t k = 0; k < d - 1; ++k) {"),
    ("K read transposed", "A[n] += qk * H(krow[n]);", "A[n] += qk * H(Kb[n * d + k]);"),
    ("V read transposed", "out[c] += w * H(vrow[c]);", "out[c] += w * H(Vb[c * N + n]);"),
    ("V always from batch 0", "const uint16_t *Vb = V + b * N * d;", "const uint16_t *Vb = V;"),
    ("Q row index swapped", "const uint16_t *q = Q + (b * M + m) * d;", "const uint16_t *q = Q + (m * 0 + b * M) * d;"),
    ("exp replaced by 1 + x", "E[n] = exp(A[n]);", "E[n] = 1.0 + A[n];"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(text.replace(old, new))
    lib_path = oracle.compile_library(str(mutant_src), str(tmp_path / "libmutant.so"))
    lib = oracle.load_library(lib_path)

    def fn(q, k, v):
        return oracle.attention(q, k, v, threads=1, lib=lib)

    caught = []
    for pin in pins.PINS:
        try:
            pin(fn)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {name}"
