"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Every mutant is a textual edit of oracle.c compiled with the oracle's own flags
into a temporary shared object, on the CPU.  The real oracle is never modified.
A mutant survives when every pin still passes; none may survive.
"""

import os

import pytest

import oracle
import oracle_pins

# (name, original text, replacement); each original must occur exactly once.
MUTANTS = [
    ("A transpose index swapped",
     "j->ta ? j->A[k * j->lda + i] : j->A[i * j->lda + k]",
     "j->ta ? j->A[i * j->lda + k] : j->A[i * j->lda + k]"),
    ("lda ignored", "j->A[i * j->lda + k])", "j->A[i * j->K + k])"),
    ("B transpose index swapped", "j->tb ? j->B[c * j->ldb + k]", "j->tb ? j->B[k * j->ldb + c]"),
    ("ldc ignored", "j->C0[i * j->ldc + c]", "j->C0[i * j->N + c]"),
    ("beta term dropped", "v += j->beta * c0;", "v += 0.0 * c0;"),
    ("beta term sign", "v += j->beta * c0;", "v -= j->beta * c0;"),
    ("alpha dropped", "products ? j->alpha * orow[c] : 0.0", "products ? orow[c] : 0.0"),
    ("bias dropped", "v += (double)j->bias[c];", "v += 0.0;"),
    ("relu dropped", "if (j->relu) v = (v > 0.0) ? v : 0.0;", "if (j->relu) v = v;"),
    ("relu inverted", "if (j->relu) v = (v > 0.0) ? v : 0.0;", "if (j->relu) v = (v < 0.0) ? v : 0.0;"),
    ("first k skipped (row-walk path)",
     "for (k = 0; k < K; ++k) {\n                const double a = arow[k];",
     "for (k = 1; k < K; ++k) {\n                const double a = arow[k];"),
    ("last k dropped (dot path)", "const double b = b_at(j, k, c);",
     "const double b = (k + 1 < K) ? b_at(j, k, c) : 0.0;"),
    ("float accumulation (dot path)", "double s = 0.0, m = 0.0;", "float s = 0.0f; double m = 0.0;"),
    ("mag beta term dropped", "m += fabs(j->beta) * fabs(c0);", "m += 0.0;"),
    ("mag bias term dropped", "m += fabs((double)j->bias[c]);", "m += 0.0;"),
    ("row bias dropped", "v += (double)j->row_bias[i];", "v += 0.0;"),
    ("row bias by column", "v += (double)j->row_bias[i];", "v += (double)j->row_bias[c < j->M ? c : 0];"),
    ("mag alpha dropped", "fabs(j->alpha) * mrow[c]", "mrow[c]"),
    ("selected rows ignored", "const int64_t i = j->rows ? j->rows[r] : r;", "const int64_t i = r;"),
    ("batch stride of B ignored", "B ? B + b * strideB : NULL", "B"),
]


def _survivors(tmp_path, name, old, new):
    src = open(oracle.SOURCE, encoding="utf-8").read()
    assert src.count(old) == 1, "mutation site for %r not found exactly once" % name
    path = os.path.join(tmp_path, "mut.c")
    with open(path, "w", encoding="utf-8") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, os.path.join(tmp_path, "libmut.so"))
    mutant = oracle.Oracle(lib)
    passed = []
    for pin in oracle_pins.PINS:
        try:
            pin(mutant)
            passed.append(pin.__name__)
        except (AssertionError, ValueError):
            pass
    return passed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    passed = _survivors(str(tmp_path), name, old, new)
    assert len(passed) < len(oracle_pins.PINS), "mutant %r passes every pin" % name
