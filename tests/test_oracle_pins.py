"""The CPU oracle against closed forms, invariants, a hand-worked example and an
independent matrix form; then planted mistakes in copies of the oracle, each of
which must be caught by at least one pin."""
import functools
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.scan)


def test_oracle_single_thread_equals_threaded():
    from state_space_model_ssm_gb300.workloads import workload
    import numpy as np
    inp = workload("tiny")
    y1, s1 = oracle.scan_inputs(inp, n_threads=1)
    y8, s8 = oracle.scan_inputs(inp, n_threads=8)
    assert np.array_equal(y1, y8, equal_nan=True) and np.array_equal(s1, s8)


def test_oracle_head_subset_matches_full():
    from state_space_model_ssm_gb300.workloads import workload
    import numpy as np
    inp = workload("tiny")
    y, s = oracle.scan_inputs(inp)
    ys, ss = oracle.scan_inputs(inp, heads=[1, 3])
    for h in (1, 3):
        assert np.array_equal(ys[:, h], y[:, h], equal_nan=True)
        assert np.array_equal(ss[:, h], s[:, h])
    assert np.all(np.isnan(ys[:, 0])) and np.all(np.isnan(ss[:, 2]))


def test_oracle_rejects_bad_arguments():
    import numpy as np
    x = np.zeros((2, 3, 1)); dt = np.zeros((2, 3)); A = np.zeros(3)
    B = np.zeros((2, 2, 1)); D = np.zeros(3); S = np.zeros((1, 3, 1, 1))
    with pytest.raises(ValueError):   # H % G != 0
        oracle.scan(x, dt, A, B, B, D, S, [0], [2], [0])
    B = np.zeros((2, 1, 1))
    with pytest.raises(ValueError):   # sequence runs past the token count
        oracle.scan(x, dt, A, B, B, D, S, [1], [2], [0])


# Planted mistakes: (name, text in ssm_oracle.c, replacement).
MUTANTS = [
    ("no_skip_term", "acc + J->D[h] * x_thp", "acc"),
    ("y_before_update", "Sp[n] = a * Sp[n] + xdt * Bt[n];\n                acc += Sp[n] * Ct[n];",
     "acc += Sp[n] * Ct[n];\n                Sp[n] = a * Sp[n] + xdt * Bt[n];"),
    ("decay_sign", "exp(dt_th * J->A[h])", "exp(-dt_th * J->A[h])"),
    ("decay_on_input", "a * Sp[n] + xdt * Bt[n]", "Sp[n] + a * xdt * Bt[n]"),
    ("interleaved_groups", "const int g = h / (H / G);", "const int g = h % G;"),
    ("b_c_swapped", "acc += Sp[n] * Ct[n];", "acc += Sp[n] * Bt[n];"),
    ("no_dt_on_input", "const double xdt = dt_th * x_thp;", "const double xdt = x_thp;"),
    ("resume_ignored", "J->resume[i] ? J->state_in[slot + e] : 0.0", "0.0"),
    ("row_index_transposed", "J->x[((size_t)t * H + h) * P + p]", "J->x[((size_t)t * P + p) * H + h]"),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path_c = tmp_path / f"{name}.c"
    path_c.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-ffp-contract=off", str(path_c), "-o", str(so), "-lm"], check=True)
    return oracle.load_library(str(so))


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    lib = _build_mutant(tmp_path, name, old, new)
    run = functools.partial(oracle.scan, lib=lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(run)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
