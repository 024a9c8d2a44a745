"""Each plausible mistake planted in a copy of the oracle must break a pin.

The copies are made from the oracle's C source by one textual substitution,
compiled with the same flags and run on the CPU only, each in a child process
(a mutant that indexes out of bounds may crash, which also counts as caught).
"""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle_sgemm.c")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "B indexed transposed": ("B[k * ldb + j]", "B[j * ldb + k]"),
    "A indexed transposed": ("A[i * lda + k]", "A[k * lda + i]"),
    "beta term sign": ("v += (double)beta * c;", "v -= (double)beta * c;"),
    "beta term dropped": ("v += (double)beta * c;", "v += 0.0 * c;"),
    "last k term dropped": ("for (long k = 0; k < K; ++k)", "for (long k = 0; k < K - 1; ++k)"),
    "first k term dropped": ("for (long k = 0; k < K; ++k)", "for (long k = 1; k < K; ++k)"),
    "lda ignored": ("A[i * lda + k]", "A[i * K + k]"),
    "ldc confused with ldb": ("C[i * ldc + j]", "C[i * ldb + j]"),
    "alpha added": ("double v = (double)alpha * sum;", "double v = (double)alpha + sum;"),
    "alpha dropped": ("double v = (double)alpha * sum;", "double v = sum;"),
    "magnitude keeps signs": ("abs_sum += fabs(product);", "abs_sum += product;"),
    "C read when beta is zero": ("if (beta != 0.0f) {", "if (1) {"),
    "A and B read when alpha is zero": ("if (alpha != 0.0f) {", "if (1) {"),
    "single-precision accumulation": ("double sum = 0.0; ", "float sum = 0.0f; "),
    "product rounded to float": ("double product = (double)A[i * lda + k] * (double)B[k * ldb + j];",
                                 "double product = (float)(A[i * lda + k] * B[k * ldb + j]);"),
}

CHILD = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
fails = oracle_pins.run_all(oracle.load_library({lib!r}))
print(len(fails))
sys.exit(0 if fails else 3)
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not unique: {old!r}"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "mutant.c")
        with open(src, "w") as f:
            f.write(text.replace(old, new))
        lib = oracle.compile_library(src, os.path.join(d, "libmutant.so"))
        code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                           timeout=300)
    # exit 0: pins failed as they should; negative: the mutant crashed (caught);
    # 3: every pin passed on a broken oracle.
    assert r.returncode != 3, f"no pin caught the mutant '{name}'"
    assert r.returncode == 0 or r.returncode < 0, r.stderr[-2000:]
