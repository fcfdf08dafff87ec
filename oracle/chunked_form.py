"""The scan in chunked matrix form, in float64 (test infrastructure).

The gllm PR 90 page ("keep the Mamba2 scan state in registers, stage tokens by
chunk", "What changes" and "Not in this PR") names Mamba2's SSD
chunked-matmul algorithm as the way to run prefill in parallel over time and
gives no algorithm.  This file states the one derived from the recurrence of
"The llama journey", Day 14 (S <- exp(dt*A) S + dt*x*B, y = S.C + D*x), by
unrolling it over the tokens of one chunk of Q tokens of a sequence.  With
a_t = A * sum_{s<=t in the chunk} dt_s (inclusive) and S_in the state entering
the chunk:

  (1) CB[t, s]   = C_t . B_s                              (per group)
  (2) L[t, s]    = exp(a_t - a_s) for s <= t, else 0
  (3) Y_intra    = (L * CB) @ (dt * X)
  (4) dS         = sum_s exp(a_last - a_s) dt_s x_s (outer) B_s
  (5) S_out      = exp(a_last) S_in + dS                   (S_in of the next chunk)
  (6) Y_inter[t] = exp(a_t) * (S_in . C_t)
  (7) y          = Y_intra + Y_inter + D x

Every step is a plain NumPy expression in float64 with no blocking beyond the
chunking itself, so with exact arithmetic it reproduces the token-by-token
oracle; in float64 the two agree to rounding (about 1e-12 relative), which the
CPU tests check for several chunk lengths, including 1 (the recurrence itself)
and one longer than every sequence (the whole-sequence matrix form).  The CUDA
form evaluates the same seven steps with TF32 operands.
"""
from __future__ import annotations

import numpy as np


def _np64(a):
    a = a.detach().cpu().numpy() if hasattr(a, "detach") else np.asarray(a)
    return np.asarray(a, dtype=np.float64)


def chunk_step(Xc, dtc, Ah, Bc, Cc, Dh, S_in):
    """Steps (1)-(7) for one chunk of one head.

    Xc [L, P], dtc [L], Bc/Cc [L, N], S_in [P, N]; returns (y [L, P], S_out)."""
    a = np.cumsum(dtc * Ah)                                   # a_t, inclusive
    CB = Cc @ Bc.T                                            # (1)
    causal = np.tril(np.ones((len(a), len(a)), dtype=bool))
    diff = np.where(causal, a[:, None] - a[None, :], 0.0)
    Lmat = np.where(causal, np.exp(diff), 0.0)                # (2)
    y_intra = (Lmat * CB) @ (dtc[:, None] * Xc)               # (3)
    w = np.exp(a[-1] - a) * dtc
    dS = (w[:, None] * Xc).T @ Bc                             # (4)
    S_out = np.exp(a[-1]) * S_in + dS                         # (5)
    y_inter = np.exp(a)[:, None] * (Cc @ S_in.T)              # (6)
    return y_intra + y_inter + Dh * Xc, S_out                 # (7)


def chunked_form(x, dt, A, B, C, D, state, seq_starts, seq_lens, resume, chunk):
    """The scan of every (sequence, head) in chunks of `chunk` tokens.

    Same tensors and conventions as the oracle's ``scan``; returns
    (y [T, H, P], final state [n, H, P, N]) in float64, y NaN where no
    sequence owns the token."""
    if chunk < 1:
        raise ValueError("chunk must be >= 1")
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
            S = state[i, h].copy() if resume[i] else np.zeros((P, N))
            for c0 in range(0, L, chunk):
                sl = slice(t0 + c0, t0 + min(L, c0 + chunk))
                y[sl, h], S = chunk_step(x[sl, h], dt[sl, h], A[h], B[sl, g], C[sl, g], D[h], S)
            S_out[i, h] = S
    return y, S_out
