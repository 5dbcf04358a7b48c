"""Plant mistakes in copies of the oracle source and check that a pin catches each.

The mutants are compiled from edited copies of ``oracle/oracle.c`` into a
temporary directory; the real oracle is never modified.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins as P
from oracle import build as obuild

SRC = os.path.join(os.path.dirname(obuild.__file__), "oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("scale_dropped", "lora *= scale[a];", "lora *= 1.0;"),
    ("shrink_transposed", "acc += (double)xrow[k] * (double)Aa[(int64_t)j * K + k];",
     "acc += (double)xrow[k] * (double)Aa[(int64_t)k * r + j];"),
    ("lora_sign", "y[i * N + n] = base + lora;", "y[i * N + n] = base - lora;"),
    ("dx_lora_missing", "dX[i * K + k] = base + scale[a] * lora;", "dX[i * K + k] = base;"),
    ("dB_uses_v", "acc += s * uu[i * ORACLE_MAX_RANK + j] * (double)dY[tok[i] * N + n];",
     "acc += s * vv[i * ORACLE_MAX_RANK + j] * (double)dY[tok[i] * N + n];"),
    ("dA_wrong_operand", "acc += s * vv[i * ORACLE_MAX_RANK + j] * (double)x[tok[i] * K + k];",
     "acc += s * uu[i * ORACLE_MAX_RANK + j] * (double)x[tok[i] * K + k];"),
    ("accumulate_ignored", "dAa[(int64_t)j * K + k] = (accumulate ? dAa[(int64_t)j * K + k] : 0.0) + acc;",
     "dAa[(int64_t)j * K + k] = acc;"),
    ("wrong_B_row", "lora += ut[j] * (double)Ba[(int64_t)j * N + n];",
     "lora += ut[j] * (double)Ba[(int64_t)(r - 1 - j) * N + n];"),
]


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, orig, bad):
    text = open(SRC).read()
    assert text.count(orig) == 1, "mutation anchor not unique: " + orig
    path = tmp_path / ("oracle_%s.c" % name)
    path.write_text(text.replace(orig, bad))
    lib_path = obuild.build(str(path), str(tmp_path / ("lib_%s.so" % name)))
    lib = oracle.load_library(lib_path)
    caught = []
    for pin in P.ALL_PINS:
        try:
            if pin is P.pin_finite_differences:
                pin(lib=lib, n_dx=16, every=False)
            else:
                pin(lib=lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "no pin caught mutant " + name
