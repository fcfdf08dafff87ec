"""The float64 chunked matrix form (the decomposition the SSD kernels use)
against the token-by-token oracle, on the CPU.

In exact arithmetic the two are the same map, so in float64 they must agree to
rounding for every chunk length: 1 (the recurrence itself), lengths that cut
sequences mid-way with ragged tails, and one longer than every sequence (the
whole-sequence matrix form)."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_ssm_gb300.workloads import Geometry, make_inputs, workload

TIGHT = 1e-10


def _close(got, ref, what):
    ok = ~np.isnan(ref)
    assert np.array_equal(ok, ~np.isnan(got)), f"{what}: different coverage"
    err = np.abs(got[ok] - ref[ok])
    assert np.all(err <= TIGHT * (1.0 + np.abs(ref[ok]))), f"{what}: max err {err.max():.3e}"


def _chunked(inp, chunk):
    return oracle.chunked_form(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.state,
                               inp.seq_starts, inp.seq_lens, inp.resume, chunk)


@pytest.mark.parametrize("chunk", [1, 3, 8, 16, 64, 1000])
def test_chunked_form_equals_recurrence_tiny(chunk):
    inp = workload("tiny")
    y_ref, s_ref = oracle.scan_inputs(inp, n_threads=1)
    y, s = _chunked(inp, chunk)
    _close(y, y_ref, "y")
    _close(s, s_ref, "state")


def test_chunked_form_equals_recurrence_ragged():
    """Short, empty and multi-chunk sequences, fresh and resuming, with
    tokens owned by no sequence between them."""
    geom = Geometry(n_heads=4, head_dim=8, d_state=12, n_groups=2)
    lens = [1, 0, 5, 17, 40, 33]
    starts = [0, 3, 3, 10, 30, 75]
    inp = make_inputs(geom, lens, resume=[0, 1, 1, 0, 1, 0], seed=11, starts=starts, n_tokens=110)
    y_ref, s_ref = oracle.scan_inputs(inp, n_threads=1)
    for chunk in (4, 16, 32):
        y, s = _chunked(inp, chunk)
        _close(y, y_ref, f"y chunk {chunk}")
        _close(s, s_ref, f"state chunk {chunk}")


def test_chunked_form_single_chunk_is_matrix_form():
    inp = workload("tiny")
    y_m, s_m = oracle.matrix_form(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.state,
                                  inp.seq_starts, inp.seq_lens, inp.resume)
    y, s = _chunked(inp, 4096)
    _close(y, y_m, "y")
    _close(s, s_m, "state")


def test_chunked_form_strong_decay_has_no_overflow():
    """Steep decay inside a chunk: exp(a_t - a_s) is only taken for s <= t, so
    nothing overflows even where exp(-a_s) alone would."""
    geom = Geometry(n_heads=2, head_dim=4, d_state=8, n_groups=1)
    inp = make_inputs(geom, [96], resume=[1], seed=5)
    inp.dt.fill_(4.0)
    inp.A.fill_(-40.0)                   # a drops by 160 per token
    with np.errstate(over="raise", invalid="raise"):
        y, s = _chunked(inp, 64)
    y_ref, s_ref = oracle.scan_inputs(inp, n_threads=1)
    _close(y, y_ref, "y")
    _close(s, s_ref, "state")
