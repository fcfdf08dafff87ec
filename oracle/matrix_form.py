"""Second, independent CPU form of the scan, for tiny inputs (test infrastructure).

Unrolling the recurrence of the Mamba2 scan ("The llama journey", Day 14
kernel body: S <- exp(dt*A) S + dt*x*B, y = S.C) over the tokens of one
sequence gives, for token t (s, r index tokens of the same sequence, both
counted from its first token):

    S_t = exp(A * sum_{r<=t} dt_r) * S_0
          + sum_{s<=t} exp(A * sum_{s<r<=t} dt_r) * dt_s * x_s (outer) B_s

    y_t = sum_{s<=t} (C_t . B_s) * exp(A * sum_{s<r<=t} dt_r) * dt_s * x_s
          + exp(A * sum_{r<=t} dt_r) * (S_0 . C_t) + D * x_t

This file evaluates those sums directly: a lower-triangular decay matrix
L[t, s] = exp(cum_t - cum_s), the per-group matrix C B^T, and two matrix
products, in float64.  It never steps through the recurrence, so agreement with
the token-by-token oracle pins both.  The skip term D*x and the per-sequence
slot follow the same readings as ``ssm_oracle.c``.
"""
from __future__ import annotations

import numpy as np


def _np64(a):
    a = a.detach().cpu().numpy() if hasattr(a, "detach") else np.asarray(a)
    return np.asarray(a, dtype=np.float64)


def matrix_form(x, dt, A, B, C, D, state, seq_starts, seq_lens, resume):
    x, dt, A, B, C, D, state = map(_np64, (x, dt, A, B, C, D, state))
    seq_starts = np.asarray(_np64(seq_starts), dtype=np.int64)
    seq_lens = np.asarray(_np64(seq_lens), dtype=np.int64)
    resume = np.asarray(_np64(resume), dtype=np.int64)
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    n = seq_lens.shape[0]
    y = np.full((T, H, P), np.nan)
    S_out = np.full((n, H, P, N), np.nan)
    heads_per_group = H // G
    for i in range(n):
        t0, L = int(seq_starts[i]), int(seq_lens[i])
        for h in range(H):
            g = h // heads_per_group
            S0 = state[i, h] if resume[i] else np.zeros((P, N))
            if L == 0:
                S_out[i, h] = S0
                continue
            sl = slice(t0, t0 + L)
            dth = dt[sl, h]                      # [L]
            cum = np.cumsum(dth * A[h])          # log-decay from the start, inclusive
            Bg, Cg = B[sl, g, :], C[sl, g, :]    # [L, N]
            X = x[sl, h, :]                      # [L, P]
            Ldec = np.tril(np.exp(cum[:, None] - cum[None, :]))   # [t, s], s <= t
            CB = Cg @ Bg.T                                         # [t, s]
            u = dth[:, None] * X                                   # dt_s * x_s
            y_seq = (Ldec * CB) @ u + np.exp(cum)[:, None] * (Cg @ S0.T) + D[h] * X
            y[sl, h, :] = y_seq
            w = np.exp(cum[-1] - cum)[:, None] * u                 # [L, P]
            S_out[i, h] = np.exp(cum[-1]) * S0 + w.T @ Bg
    return y, S_out
