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
    ("saved_u_ignored", "            if (u_saved) {", "            if (0) {"),
    ("saved_u_segment_offset_dropped", "uoff[p] = blk + (int64_t)i * r_q;", "uoff[p] = (int64_t)i * r_q;"),
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


# Mistakes planted in the sliced-projection layer of the oracle (``oracle/sliced.py``), loaded as a separate module
# from an edited copy; each must fail one of the sliced pins.
SLICED_SRC = os.path.join(os.path.dirname(obuild.__file__), "sliced.py")
SLICED_MUTANTS = [
    ("slice_down_factor_fixed", "[base + i * r:base + (i + 1) * r]", "[base:base + r]"),
    ("slice_up_columns_shifted", "reshape(-1, N)[brow:brow + r, c0:c1]", "reshape(-1, N)[brow:brow + r, 0:c1 - c0]"),
    ("dx_last_slice_only", "dX = dXi if dX is None else dX + dXi", "dX = dXi"),
    ("dA_into_slice_zero", "dA[base + i * r * K:base + (i + 1) * r * K] = dAi[ao[a]:ao[a] + r * K]",
     "dA[base:base + r * K] += dAi[ao[a]:ao[a] + r * K]"),
    ("saved_u_slice_zero_columns", "out.append(blk[:, i * r:(i + 1) * r].reshape(-1))",
     "out.append(blk[:, 0:r].reshape(-1))"),
]
SLICED_PINS = [P.pin_sliced_block_diagonal, P.pin_sliced_merged_weight, P.pin_sliced_finite_differences,
               P.pin_sliced_saved_u]


@pytest.mark.parametrize("name,orig,bad", SLICED_MUTANTS, ids=[m[0] for m in SLICED_MUTANTS])
def test_sliced_mutant_is_caught(tmp_path, monkeypatch, name, orig, bad):
    import importlib.util
    text = open(SLICED_SRC).read()
    assert text.count(orig) == 1, "mutation anchor not unique: " + orig
    path = tmp_path / "sliced_mutant.py"
    path.write_text(text.replace(orig, bad))
    spec = importlib.util.spec_from_file_location("oracle.sliced_mutant", str(path))
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    spec.loader.exec_module(mod)
    monkeypatch.setattr(P, "sliced", mod)
    caught = []
    for pin in SLICED_PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "no pin caught sliced mutant " + name
