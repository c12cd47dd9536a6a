"""Pins of the oracle's bias-gradient column sum and planted mistakes they catch.

The pins tie ``oracle.bias_grad`` to facts that do not come from it: sums of
small integers (exact in float64, computed here with Python integers), a
closed form, the correctly rounded sum of ``math.fsum``, invariance under a
row permutation and the two output conventions of the pages ("Phase 3
Kernel Optimization Implementation Plan", Tasks 2 and 3: add into db, or
overwrite grad_b). Each mutant is a one-line change to the oracle's C source,
compiled into a temporary library; at least one pin must fail on it.
"""
import math
import os

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "m2scan_oracle.c")


def pin_integer_matrix(lib):
    N, C = 37, 5
    vals = [[(7 * r + 3 * c) % 11 - 5 for c in range(C)] for r in range(N)]
    want = [sum(vals[r][c] for r in range(N)) for c in range(C)]
    got = oracle.bias_grad(np.array(vals, dtype=np.float32), lib=lib)
    assert list(got) == [float(w) for w in want], (list(got), want)


def pin_closed_form(lib):
    N, C = 1000, 3
    r = np.arange(N, dtype=np.float64)[:, None]
    c = np.arange(C, dtype=np.float64)[None, :]
    dy = (r + 10 * c).astype(np.float32)
    want = [N * (N - 1) / 2 + N * 10 * k for k in range(C)]
    got = oracle.bias_grad(dy, lib=lib)
    assert np.array_equal(got, np.array(want)), (got, want)


def pin_fsum(lib):
    rng = np.random.default_rng(5)
    dy = rng.standard_normal((4099, 7), dtype=np.float32)
    got = oracle.bias_grad(dy, lib=lib)
    for c in range(dy.shape[1]):
        col = [float(v) for v in dy[:, c]]
        want = math.fsum(col)
        bound = 1e-12 * sum(abs(v) for v in col)
        assert abs(got[c] - want) <= bound, (c, got[c], want)


def pin_row_permutation(lib):
    rng = np.random.default_rng(6)
    dy = rng.standard_normal((513, 4), dtype=np.float32)
    a = oracle.bias_grad(dy, lib=lib)
    b = oracle.bias_grad(dy[rng.permutation(dy.shape[0])], lib=lib)
    assert np.allclose(a, b, rtol=0, atol=1e-12 * np.abs(dy).sum(axis=0).max())
    # and the columns are not interchangeable
    assert not np.allclose(a, a[::-1])


def pin_conventions(lib):
    dy = np.array([[1.0, 2.0], [3.0, 4.0]], dtype=np.float32)
    db = np.array([10.0, 20.0])
    assert list(oracle.bias_grad(dy, lib=lib)) == [4.0, 6.0]
    assert list(oracle.bias_grad(dy, db, accumulate=True, lib=lib)) == [14.0, 26.0]
    empty = np.zeros((0, 2), dtype=np.float32)
    assert list(oracle.bias_grad(empty, lib=lib)) == [0.0, 0.0]
    assert list(oracle.bias_grad(empty, db, accumulate=True, lib=lib)) == [10.0, 20.0]
    one = np.array([[-2.5]], dtype=np.float32)
    assert list(oracle.bias_grad(one, lib=lib)) == [-2.5]


PINS = [pin_integer_matrix, pin_closed_form, pin_fsum, pin_row_permutation, pin_conventions]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(None)


MUTANTS = {
    "drop_last_row": ("for (int64_t r = 0; r < N; r++) acc += dy[r * C + c];",
                      "for (int64_t r = 0; r + 1 < N; r++) acc += dy[r * C + c];"),
    "row_stride_off_by_one": ("for (int64_t r = 0; r < N; r++) acc += dy[r * C + c];",
                              "for (int64_t r = 0; r < N; r++) acc += dy[r * (C - 1) + c];"),
    "sum_rows_not_columns": ("for (int64_t r = 0; r < N; r++) acc += dy[r * C + c];",
                             "for (int64_t r = 0; r < N; r++) acc += dy[(r % C) * C + (c % C) + 0 * r];"),
    "accumulate_ignored": ("db_out[c] = accumulate ? db_in[c] + acc : acc;", "db_out[c] = acc;"),
    "always_accumulate": ("db_out[c] = accumulate ? db_in[c] + acc : acc;",
                          "db_out[c] = (accumulate ? db_in[c] : 1.0) + acc;"),
    "float_accumulator": ("    double acc = 0.0;\n    for (int64_t r = 0; r < N; r++) acc += dy[r * C + c];",
                          "    float acc = 0.0f;\n    for (int64_t r = 0; r < N; r++) acc += (float)dy[r * C + c];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, "mutation site not unique/found: %s" % name
    path = tmp_path / ("mutant_%s.c" % name)
    path.write_text(src.replace(before, after))
    lib = oracle.open_library(oracle.compile_source(str(path), str(tmp_path / "lib.so")))
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError as e:
            caught.append("%s: %s" % (pin.__name__, str(e)[:80]))
    assert caught, "mutant %s passed every pin" % name
