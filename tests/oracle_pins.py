"""Checks that pin the CPU oracle to facts outside itself.

Each pin takes ``run``, a callable with the signature of ``oracle.scan``, so the
same checks run on the oracle and on planted-mistake copies of it (those must
fail at least one pin).  Nothing here re-types the oracle's loop: every
expected value comes from a closed form, an invariant, the independent matrix
form, a hand-worked fixture, or a brute-force product formula.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
from state_space_model_ssm_gb300.workloads import Geometry, make_inputs, workload

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _run_inp(run, inp, **kw):
    return run(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.state,
               inp.seq_starts, inp.seq_lens, inp.resume, **kw)


def _f64(t):
    return t.double().numpy()


def _close(a, b, tol):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape
    err = np.abs(a - b)
    bound = tol * (1.0 + np.abs(b))
    assert np.all(err <= bound), f"max err {np.nanmax(err):.3e}"


def pin_hand_worked(run):
    """The hand-worked two-sequence example in tests/golden."""
    with open(os.path.join(GOLDEN, "hand_worked_scalar_pair.json")) as f:
        g = json.load(f)
    T = len(g["x"])
    x = np.array(g["x"], dtype=np.float64).reshape(T, 1, 1)
    dt = np.array(g["dt"], dtype=np.float64).reshape(T, 1)
    A = np.array([-math.log(2.0)])
    B = np.array(g["B"], dtype=np.float64).reshape(T, 1, 2)
    C = np.array(g["C"], dtype=np.float64).reshape(T, 1, 2)
    D = np.array(g["D"], dtype=np.float64)
    S0 = np.array(g["state_in"], dtype=np.float64).reshape(2, 1, 1, 2)
    y, S = run(x, dt, A, B, C, D, S0, np.array(g["seq_starts"]),
               np.array(g["seq_lens"]), np.array(g["resume"]))
    _close(y.reshape(-1), g["expect_y"], 1e-14)
    _close(S.reshape(2, 2), g["expect_state"], 1e-14)


def pin_matrix_form(run):
    """Token-by-token loop == explicit-sum matrix form on the tiny workload."""
    inp = workload("tiny")
    y, S = _run_inp(run, inp)
    y2, S2 = oracle.matrix_form(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D,
                                inp.state, inp.seq_starts, inp.seq_lens, inp.resume)
    _close(y, y2, 1e-12)
    _close(S, S2, 1e-12)


def pin_a_zero_running_sums(run):
    """A = 0: no decay, the state is a running sum, S_t = S0 + sum dt x (outer) B."""
    inp = workload("tiny", a_zero=True)
    y, S = _run_inp(run, inp)
    H = inp.geom.n_heads
    hpg = H // inp.geom.n_groups
    x, dt, B, C, D = map(_f64, (inp.x, inp.dt, inp.B, inp.C, inp.D))
    gidx = np.arange(H) // hpg
    for i in range(inp.n_seqs):
        t0, L = int(inp.seq_starts[i]), int(inp.seq_lens[i])
        S0 = _f64(inp.state[i]) if int(inp.resume[i]) else np.zeros(inp.state.shape[1:])
        sl = slice(t0, t0 + L)
        # increments [L,H,P,N], then a cumulative sum over tokens
        inc = (dt[sl][:, :, None, None] * x[sl][:, :, :, None]
               * B[sl][:, gidx, None, :])
        St = S0[None] + np.cumsum(inc, axis=0)
        y_exp = np.einsum("thpn,thn->thp", St, C[sl][:, gidx, :]) + D[None, :, None] * x[sl]
        _close(y[sl], y_exp, 1e-12)
        _close(S[i], St[-1], 1e-12)


def pin_b_zero_pure_decay(run):
    """B = 0: pure decay, S_t = exp(A sum dt) S0 and y = exp(A sum dt) (S0 . C_t) + D x."""
    inp = workload("tiny", b_zero=True)
    y, S = _run_inp(run, inp)
    H = inp.geom.n_heads
    gidx = np.arange(H) // (H // inp.geom.n_groups)
    x, dt, A, C, D = map(_f64, (inp.x, inp.dt, inp.A, inp.C, inp.D))
    for i in range(inp.n_seqs):
        t0, L = int(inp.seq_starts[i]), int(inp.seq_lens[i])
        sl = slice(t0, t0 + L)
        S0 = _f64(inp.state[i]) if int(inp.resume[i]) else np.zeros(inp.state.shape[1:])
        decay = np.exp(np.cumsum(dt[sl] * A[None, :], axis=0))       # [L,H]
        y_exp = (decay[:, :, None] * np.einsum("hpn,thn->thp", S0, C[sl][:, gidx, :])
                 + D[None, :, None] * x[sl])
        _close(y[sl], y_exp, 1e-12)
        _close(S[i], decay[-1][:, None, None] * S0, 1e-12)


def pin_single_token_from_zero(run):
    """One token from a zero state: S = dt x B and y = dt x (B . C) + D x."""
    geom = Geometry(6, 5, 8, 3)
    inp = make_inputs(geom, [1, 1, 1], [0, 0, 0], seed=11)
    y, S = _run_inp(run, inp)
    gidx = np.arange(6) // 2
    x, dt, B, C, D = map(_f64, (inp.x, inp.dt, inp.B, inp.C, inp.D))
    for t in range(3):
        Bt, Ct = B[t][gidx], C[t][gidx]                     # [H,N]
        xdt = dt[t][:, None] * x[t]                          # [H,P]
        _close(S[t], xdt[:, :, None] * Bt[:, None, :], 1e-13)
        y_exp = xdt * np.sum(Bt * Ct, axis=1)[:, None] + D[:, None] * x[t]
        _close(y[t], y_exp, 1e-13)


def pin_d_path_exact(run):
    """B = 0 from a zero state: y = D x exactly and the state stays zero."""
    inp = workload("tiny", b_zero=True)
    inp.resume.zero_()
    y, S = _run_inp(run, inp)
    x, D = _f64(inp.x), _f64(inp.D)
    T = int(inp.seq_lens.sum())
    assert np.array_equal(y[:T], D[None, :, None] * x[:T])
    assert np.array_equal(S, np.zeros_like(S))


def pin_split_resume(run):
    """A sequence run as two calls (the second resuming) equals one call, bit for bit."""
    geom = Geometry(4, 8, 16, 2)
    inp = make_inputs(geom, [29], [1], seed=5)
    y_one, S_one = _run_inp(run, inp)
    k = 11
    a = make_inputs(geom, [29], [1], seed=5)
    y1, S1 = run(a.x[:k], a.dt[:k], a.A, a.B[:k], a.C[:k], a.D, a.state,
                 [0], [k], [1])
    y2, S2 = run(a.x[k:], a.dt[k:], a.A, a.B[k:], a.C[k:], a.D, S1,
                 [0], [29 - k], [1])
    assert np.array_equal(np.concatenate([y1, y2]), y_one)
    assert np.array_equal(S2, S_one)


def pin_linearity(run):
    """y and the final state are jointly linear in (x, S0): doubling both doubles
    them exactly (a power-of-two scaling is exact in binary floating point)."""
    inp = workload("tiny")
    inp.resume.fill_(1)
    inp.state = inp.state.nan_to_num(0.25)
    y, S = _run_inp(run, inp)
    y2, S2 = run(inp.x * 2, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.state * 2,
                 inp.seq_starts, inp.seq_lens, inp.resume)
    assert np.array_equal(y2, 2 * y)
    assert np.array_equal(S2, 2 * S)


def pin_group_map(run):
    """Zeroing group g's B and C changes exactly the heads g*H/G .. (g+1)*H/G-1,
    and turns their y into D x (heads of a group are contiguous)."""
    geom = Geometry(8, 4, 8, 4)
    inp = make_inputs(geom, [13, 7], [0, 1], seed=7)
    y, S = _run_inp(run, inp)
    for g in range(4):
        B, C = inp.B.clone(), inp.C.clone()
        B[:, g].zero_()
        C[:, g].zero_()
        yg, Sg = run(inp.x, inp.dt, inp.A, B, C, inp.D, inp.state,
                     inp.seq_starts, inp.seq_lens, inp.resume)
        for h in range(8):
            if h // 2 == g:
                assert not np.array_equal(yg[:, h], y[:, h])
                assert np.array_equal(yg[:, h], _f64(inp.D)[h] * _f64(inp.x)[:, h])
            else:
                assert np.array_equal(yg[:, h], y[:, h])
                assert np.array_equal(Sg[:, h], S[:, h])


def pin_scalar_brute_force(run):
    """H = P = N = G = 1: a first-order linear recurrence whose solution is the
    explicit sum of products S_t = prod_{r<=t} a_r S0 + sum_s prod_{s<r<=t} a_r dt_s x_s B_s,
    evaluated here term by term in Python floats for T <= 8."""
    rng = np.random.default_rng(3)
    for T in range(1, 9):
        x = rng.normal(size=T)
        dt = rng.uniform(0.05, 1.5, size=T)
        A = -rng.uniform(0.1, 3.0)
        Bv = rng.normal(size=T)
        Cv = rng.normal(size=T)
        D = rng.normal()
        S0 = rng.normal()
        a = [math.exp(dt[r] * A) for r in range(T)]
        y_exp, S_t = [], None
        for t in range(T):
            prod_all = 1.0
            for r in range(t + 1):
                prod_all *= a[r]
            S_t = prod_all * S0
            for s in range(t + 1):
                w = 1.0
                for r in range(s + 1, t + 1):
                    w *= a[r]
                S_t += w * dt[s] * x[s] * Bv[s]
            y_exp.append(S_t * Cv[t] + D * x[t])
        y, S = run(x.reshape(T, 1, 1), dt.reshape(T, 1), np.array([A]),
                   Bv.reshape(T, 1, 1), Cv.reshape(T, 1, 1), np.array([D]),
                   np.array([S0]).reshape(1, 1, 1, 1), [0], [T], [1])
        _close(y.reshape(-1), y_exp, 1e-13)
        _close(S.reshape(-1), [S_t], 1e-13)


def pin_zero_length_and_untouched(run):
    """A zero-length sequence writes no y; fresh slot -> 0, resumed slot unchanged;
    tokens outside every sequence are not written."""
    geom = Geometry(2, 3, 4, 1)
    inp = make_inputs(geom, [0, 0, 4], [0, 1, 0], seed=9,
                      starts=[0, 0, 2], n_tokens=8)
    y, S = _run_inp(run, inp)
    assert np.array_equal(S[0], np.zeros_like(S[0]))
    assert np.array_equal(S[1], _f64(inp.state[1]))
    assert np.all(np.isnan(y[:2])) and np.all(np.isnan(y[6:]))
    assert np.all(np.isfinite(y[2:6]))


ALL_PINS = [pin_hand_worked, pin_matrix_form, pin_a_zero_running_sums,
            pin_b_zero_pure_decay, pin_single_token_from_zero, pin_d_path_exact,
            pin_split_resume, pin_linearity, pin_group_map, pin_scalar_brute_force,
            pin_zero_length_and_untouched]
