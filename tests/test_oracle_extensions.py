"""Pins of the oracle's steps around the scan (CPU only), each against values
fixed by the mathematics or by an independent evaluation."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import extensions as ext
from state_space_model_ssm_gb300.workloads import Geometry, make_inputs, workload


# ---- dt discretisation ----

def test_softplus_special_values():
    v = np.array([[0.0, 20.0, 20.5, -40.0, 1.0, -3.0]])
    got = ext.discretize_dt(v, softplus=True)[0]
    assert got[0] == pytest.approx(math.log(2.0), rel=1e-15)
    assert got[1] == pytest.approx(20.0 + math.log1p(math.exp(-20.0)), rel=1e-15)   # 20 itself: softplus
    assert got[2] == 20.5                                                            # above 20: identity
    assert got[3] == pytest.approx(math.exp(-40.0), rel=1e-12)
    assert got[4] == pytest.approx(math.log(1.0 + math.e), rel=1e-15)


def test_softplus_bias_per_head_elementwise():
    rng = np.random.default_rng(3)
    dt = rng.normal(-2.0, 3.0, size=(7, 5))
    bias = rng.uniform(-1.0, 25.0, size=5)
    got = ext.discretize_dt(dt, bias, softplus=True)
    for t in range(7):
        for h in range(5):
            v = dt[t, h] + bias[h]
            want = v if v > 20.0 else math.log1p(math.exp(v))
            assert got[t, h] == pytest.approx(want, rel=1e-14, abs=1e-300)
    assert np.array_equal(ext.discretize_dt(dt, bias), dt + bias[None, :])     # bias only
    assert np.array_equal(ext.discretize_dt(dt), dt)                           # nothing


def test_scan_with_dt_options_equals_scan_of_discretised_dt():
    """The oracle's fused path is the plain scan of the discretised step, and
    that scan matches the independent matrix form."""
    inp = workload("tiny")
    bias = torch.linspace(-0.5, 0.5, inp.geom.n_heads, dtype=torch.float64)
    raw = inp.dt.double().log()                   # some raw values, positive and negative steps
    y1, s1 = oracle.scan(inp.x, raw, inp.A, inp.B, inp.C, inp.D, inp.state, inp.seq_starts,
                         inp.seq_lens, inp.resume, dt_bias=bias, dt_softplus=True, n_threads=1)
    dt_eff = ext.discretize_dt(raw, bias, softplus=True)
    y2, s2 = oracle.matrix_form(inp.x, dt_eff, inp.A, inp.B, inp.C, inp.D, inp.state, inp.seq_starts,
                                inp.seq_lens, inp.resume)
    ok = ~np.isnan(y2)
    assert np.allclose(y1[ok], y2[ok], rtol=1e-10, atol=1e-12)
    assert np.allclose(s1, s2, rtol=1e-10, atol=1e-12)


# ---- gated RMSNorm ----

def test_gated_rmsnorm_special_cases():
    rng = np.random.default_rng(5)
    y = rng.normal(size=(4, 3, 16))
    z = rng.normal(size=(4, 3, 16))
    w = rng.uniform(0.5, 1.5, size=16)
    got = ext.gated_rmsnorm(y, z, w, 1e-6)
    # scale invariance of the normalisation (eps -> 0)
    assert np.allclose(ext.gated_rmsnorm(7.0 * y, z, w, 0.0), ext.gated_rmsnorm(y, z, w, 0.0), rtol=1e-12)
    # z = 0 gates everything off
    assert np.all(ext.gated_rmsnorm(y, np.zeros_like(z), w, 1e-6) == 0.0)
    # a constant row normalises to its sign
    c = np.full((1, 16), -2.5)
    assert np.allclose(ext.gated_rmsnorm(c, np.full((1, 16), 30.0), np.ones(16), 0.0), -30.0, rtol=1e-12)
    # elementwise against the definition written in plain Python
    for i in (0, 3):
        for h in (0, 2):
            row = y[i, h]
            rms = math.sqrt(sum(v * v for v in row) / 16 + 1e-6)
            for p in (0, 9, 15):
                zz = z[i, h, p]
                want = row[p] / rms * w[p] * (zz / (1.0 + math.exp(-zz)))
                assert got[i, h, p] == pytest.approx(want, rel=1e-13)


# ---- state snapshots ----

def test_snapshots_last_equals_final_state_and_y_equals_scan():
    inp = make_inputs(Geometry(2, 4, 8, 1), [5, 0, 3], [0, 1, 1], seed=9, starts=[0, 6, 6], n_tokens=10)
    y_ref, s_ref = oracle.scan_inputs(inp, n_threads=1)
    y, s, snaps = ext.scan_with_snapshots(oracle.scan, inp, n_threads=1)
    ok = ~np.isnan(y_ref)
    assert np.allclose(y[ok], y_ref[ok], rtol=1e-12, atol=1e-14)
    assert np.allclose(s, s_ref, rtol=1e-12, atol=1e-14)
    assert np.allclose(snaps[4], s_ref[0]) and np.allclose(snaps[8], s_ref[2])
    assert np.isnan(snaps[5]).all() and np.isnan(snaps[9]).all()      # rows owned by no sequence
    # one token from a zero state: the snapshot is dt * x (outer) B
    dt = ext.discretize_dt(inp.dt)
    want = dt[0][:, None, None] * inp.x[0].double().numpy()[:, :, None] * inp.B[0, 0].double().numpy()[None, None, :]
    assert np.allclose(snaps[0], want, rtol=1e-12)


# ---- conv1d + SiLU ----

def test_conv1d_identity_and_shift_taps():
    rng = np.random.default_rng(2)
    T, Cch, K = 9, 6, 4
    x = rng.normal(size=(T, Cch))
    st = rng.normal(size=(1, Cch, K - 1))
    w_id = np.zeros((Cch, K)); w_id[:, K - 1] = 1.0                     # current input only
    out, new_st, _ = ext.conv1d_silu(x, w_id, st, [0], [T], [1])
    assert np.allclose(out, x / (1.0 + np.exp(-x)), rtol=1e-14)
    assert np.allclose(new_st[0], x[T - 3:].T)                           # the last K-1 inputs, oldest first
    w_old = np.zeros((Cch, K)); w_old[:, 0] = 1.0                        # the input K-1 steps back
    out, _, _ = ext.conv1d_silu(x, w_old, st, [0], [T], [1])
    want = np.concatenate([st[0].T, x[:T - 3]], axis=0)                   # history first, then the inputs
    assert np.allclose(out, want / (1.0 + np.exp(-want)), rtol=1e-14)
    out_fresh, _, _ = ext.conv1d_silu(x, w_old, st, [0], [T], [0])       # fresh: zero history
    assert np.allclose(out_fresh[:K - 1], 0.0)


def test_conv1d_split_resume_and_snapshots():
    rng = np.random.default_rng(4)
    T, Cch, K = 11, 5, 4
    x = rng.normal(size=(T, Cch))
    w = rng.normal(size=(Cch, K))
    st = rng.normal(size=(1, Cch, K - 1))
    out, s_full, snaps = ext.conv1d_silu(x, w, st, [0], [T], [1])
    o1, s1, _ = ext.conv1d_silu(x[:4], w, st, [0], [4], [1])
    o2, s2, _ = ext.conv1d_silu(x[4:], w, s1, [0], [T - 4], [1])
    assert np.array_equal(np.concatenate([o1, o2]), out)
    assert np.array_equal(s2, s_full)
    assert np.array_equal(snaps[3], s1[0]) and np.array_equal(snaps[T - 1], s_full[0])
    # brute force: the convolution sum of one channel from the padded input
    c = 2
    seq = np.concatenate([st[0, c], x[:, c]])
    for t in range(T):
        acc = sum(seq[t + u] * w[c, u] for u in range(K))
        assert out[t, c] == pytest.approx(acc / (1.0 + math.exp(-acc)), rel=1e-13)
