"""Plant plausible mistakes in copies of the oracle (CPU only) and check that
the pins in test_oracle_pins catch every one of them."""
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "direction flipped":
        ("return (c->direction == ORC_MAX) ? (ab > 0) : (ab < 0);",
         "return (c->direction == ORC_MAX) ? (ab < 0) : (ab > 0);"),
    "tie rule swapped":
        ("if (c->output_order || c->tie != ORC_TIE_LARGER)\n    return a < b;\n  return a > b;",
         "if (c->output_order || c->tie != ORC_TIE_LARGER)\n    return a > b;\n  return a < b;"),
    "output order follows tie preference":
        ("c.output_order = 1;", "c.output_order = 0;"),
    "one item short":
        ("const int64_t m = n < (int64_t)k ? n : (int64_t)k;",
         "const int64_t m = n < (int64_t)k ? n : (int64_t)k - 1;"),
    "signed zeros ordered":
        ("  /* +0.0 == -0.0 under C's numeric comparison */\n",
         "  if (a->num == 0.0 && b->num == 0.0 && signbit(a->num) != signbit(b->num))\n"
         "    return signbit(a->num) ? -1 : 1;\n"),
    "f16 exponent bias off by one":
        ("v = ldexp((double)(1024 + f), e - 25);", "v = ldexp((double)(1024 + f), e - 24);"),
    "value taken from wrong position":
        ("out_values[s * (int64_t)k + j] = values[src];",
         "out_values[s * (int64_t)k + j] = values[begin + j];"),
}

CHECKS = [
    lambda: [P.test_worked_example(d) for d in P.DTYPES],
    lambda: [P.test_brute_force_rank_definition(d, dr, t) for d in ("f16", "f32", "u32")
             for dr in ("max", "min") for t in P.TIES],
    P.test_brute_force_signed_zero_ties,
    P.test_decode_f16_exhaustive,
    P.test_untouched_tail_and_empty_segments,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation anchor missing: %s" % name
    path = tmp_path / "mutant.c"
    path.write_text(text.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", str(so),
                           str(path), "-lm"])
    caught = False
    oracle.use_library(str(so))
    try:
        for check in CHECKS:
            try:
                check()
            except AssertionError:
                caught = True
                break
    finally:
        oracle.use_library(None)
    assert caught, "no pin caught the planted mistake: %s" % name
