"""Mutation checks for the oracle's pins: each test plants one plausible slip in a COPY of
the oracle's C source (on the CPU), builds it, and asserts that at least one pin fails.
The shipped oracle is never modified."""

import os

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mg_oracle.c")


def mutate(text, start, end, old, new):
    """Replace `old` (unique between the markers `start` and `end`) inside that span only."""
    i = text.index(start)
    j = text.index(end, i)
    span = text[i:j]
    assert span.count(old) == 1, f"mutation anchor not unique in its function: {old!r}"
    return text[:i] + span.replace(old, new) + text[j:]

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
    text = mutate(open(SRC).read(), "static void oracle_row(", "static int bad_shape(", old, new)
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(text)
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


QK_MUTANTS = [
    ("key vectors normalised over N instead of d",
     "sk += H(Kb[k * N + n]) * H(Kb[k * N + n]);", "sk += H(Kb[n % d * N + (k * 7 + n) % N]) * H(Kb[n % d * N + (k * 7 + n) % N]);"),
    ("query not normalised", "qn[k] = H(q[k]) * rq;", "qn[k] = H(q[k]);"),
    ("key not normalised", "kn[k * N + n] = H(Kb[k * N + n]) * rk;", "kn[k * N + n] = H(Kb[k * N + n]);"),
    ("sum instead of mean of squares", "const double rq = 1.0 / sqrt(ss / (double)d + eps);",
     "const double rq = 1.0 / sqrt(ss + eps);"),
    ("eps dropped", "const double rk = 1.0 / sqrt(sk / (double)d + eps);", "const double rk = 1.0 / sqrt(sk / (double)d);"),
    ("multiplied by the rms instead of divided", "const double rk = 1.0 / sqrt(sk / (double)d + eps);",
     "const double rk = sqrt(sk / (double)d + eps);"),
]


@pytest.mark.parametrize("name,old,new", QK_MUTANTS, ids=[m[0] for m in QK_MUTANTS])
def test_qknorm_pins_catch_planted_mistake(tmp_path, name, old, new):
    text = mutate(open(SRC).read(), "static void oracle_row_qknorm(", "int mg_oracle_attention_qknorm_rows(", old, new)
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(text)
    lib = oracle.load_library(oracle.compile_library(str(mutant_src), str(tmp_path / "libmutant.so")))

    def fn(q, k, v, eps):
        return oracle.attention_qknorm(q, k, v, eps=eps, threads=1, lib=lib)

    caught = []
    for pin in pins.QK_PINS:
        try:
            pin(fn)
        except (AssertionError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {name}"


# Slips in the binary16 widening. The subnormal branch is reached only by the exhaustive decode
# pins (random draws almost never produce an fp16 subnormal).
DECODE_MUTANTS = [
    ("subnormal exponent -14 instead of -24", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -14);"),
    ("subnormals flushed to zero", "v = ldexp((double)f, -24);", "v = 0.0 * f;"),
    ("normal exponent bias off by one", "v = ldexp((double)(f | 0x400), e - 25);",
     "v = ldexp((double)(f | 0x400), e - 24);"),
    ("implicit leading bit dropped", "v = ldexp((double)(f | 0x400), e - 25);", "v = ldexp((double)f, e - 25);"),
    ("infinity and NaN swapped", "v = f ? NAN : INFINITY;", "v = f ? INFINITY : NAN;"),
    ("sign bit ignored", "return sign ? -v : v;", "return v + 0.0 * sign;"),
]


@pytest.mark.parametrize("name,old,new", DECODE_MUTANTS, ids=[m[0] for m in DECODE_MUTANTS])
def test_pins_catch_planted_decode_mistake(tmp_path, name, old, new):
    text = mutate(open(SRC).read(), "static double half_bits_to_double(", "static double g_half[", old, new)
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(text)
    lib = oracle.load_library(oracle.compile_library(str(mutant_src), str(tmp_path / "libmutant.so")))

    def fn(q, k, v):
        return oracle.attention(q, k, v, threads=1, lib=lib)

    caught = []
    for pin in (pins.pin_half_decode_exhaustive, pins.pin_half_decode_scores):
        try:
            pin(fn)
        except (AssertionError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no decode pin caught the planted mistake: {name}"
