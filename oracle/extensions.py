"""Oracle of the steps around the scan (test infrastructure), NumPy float64.

* ``discretize_dt`` -- Mamba2's step size: v = dt + dt_bias[h], then softplus
  with the identity above 20.  "The llama journey", Day 14 kernel body (the
  scan applies log1p(exp(dt)) when dt <= 20 and uses dt as is above), and the
  decay-gate kernel of "ssm_gated_delta.cu" (v = alpha + dt; v > 20 ? v :
  log1p(exp(v))).
* ``gated_rmsnorm`` -- kernel 3 of "ssm_gated_delta.cu": per row of S values
  (here the head_dim values of one token and head), y / sqrt(mean(y^2) + eps)
  * w * silu(z), silu(z) = z / (1 + exp(-z)), the weight shared by all rows.
* ``scan_with_snapshots`` -- the state after every token, by running the loop
  oracle one token at a time with each call resuming from the previous
  call's state (the split-resume property of the scan, pinned separately).
* ``conv1d_silu`` -- the causal depthwise convolution with SiLU of
  "ssm_gated_delta.cu", kernel 2 and its batched variant: per channel c,
  out[t, c] = silu(sum_{u < k-1} hist[u] w[c, u] + x[t, c] w[c, k-1]) where
  hist holds the previous k-1 inputs (oldest first), taken from the channel's
  conv-state slot before the first token and shifted by one after each.

Each function is the definition written out with no blocking or reordering.
Only the tests, the package smoke check and the bench's CPU-baseline leg use
this module.
"""
from __future__ import annotations

import numpy as np

SOFTPLUS_THRESHOLD = 20.0


def _np64(a):
    a = a.detach().cpu().numpy() if hasattr(a, "detach") else np.asarray(a)
    return np.asarray(a, dtype=np.float64)


def discretize_dt(dt, dt_bias=None, softplus=False):
    """dt [T, H] -> the step size the recurrence uses, float64 [T, H]."""
    v = _np64(dt).copy()
    if dt_bias is not None:
        v = v + _np64(dt_bias)[None, :]
    if softplus:
        small = v <= SOFTPLUS_THRESHOLD
        v = np.where(small, np.log1p(np.exp(np.where(small, v, 0.0))), v)
    return v


def silu(z):
    z = _np64(z)
    return z / (1.0 + np.exp(-z))


def gated_rmsnorm(y, z, w, eps):
    """y, z [..., S]; w [S] -> y / sqrt(mean(y^2) + eps) * w * silu(z)."""
    y, z, w = _np64(y), _np64(z), _np64(w)
    ms = np.mean(y * y, axis=-1, keepdims=True)
    return y / np.sqrt(ms + eps) * w * silu(z)


def scan_with_snapshots(scan, inp, **kw):
    """Run ``scan`` (the loop oracle's entry point) token by token.

    Returns (y, final state, snapshots [T, H, P, N]) with snapshots[t] the
    state right after token t for every token owned by a sequence (NaN
    elsewhere).  ``kw`` goes to every call (e.g. dt_bias, dt_softplus)."""
    x, dt, B, C = inp.x, inp.dt, inp.B, inp.C
    T, H, P = x.shape
    N = B.shape[2]
    n = inp.n_seqs
    y = np.full((T, H, P), np.nan)
    snaps = np.full((T, H, P, N), np.nan)
    state = _np64(inp.state).copy()
    out_state = np.full_like(state, np.nan)
    starts, lens, resume = (np.asarray(v.tolist()) for v in (inp.seq_starts, inp.seq_lens, inp.resume))
    for i in range(n):
        s_i = state[i:i + 1].copy()
        res = int(resume[i])
        if lens[i] == 0:
            _, s_out = scan(x[:0], dt[:0], inp.A, B[:0], C[:0], inp.D, s_i, [0], [0], [res], **kw)
            out_state[i] = s_out[0]
            continue
        for j in range(int(lens[i])):
            t = int(starts[i]) + j
            sl = slice(t, t + 1)
            y_t, s_out = scan(x[sl], dt[sl], inp.A, B[sl], C[sl], inp.D, s_i, [0], [1], [res], **kw)
            y[t] = y_t[0]
            snaps[t] = s_out[0]
            s_i = s_out
            res = 1
        out_state[i] = s_i[0]
    return y, out_state, snaps


def conv1d_silu(x, weight, conv_state, seq_starts, seq_lens, resume, bias=None):
    """x [T, Cch] packed tokens, weight [Cch, K], conv_state [n, Cch, K-1]
    (read for resuming sequences; fresh ones start from zeros).

    Returns (out [T, Cch] (NaN on unowned rows), new conv_state [n, Cch, K-1],
    snapshots [T, Cch, K-1]: the history right after each owned token)."""
    x, w, cs = _np64(x), _np64(weight), _np64(conv_state)
    T, Cch = x.shape
    K = w.shape[1]
    out = np.full((T, Cch), np.nan)
    snaps = np.full((T, Cch, K - 1), np.nan)
    new_state = np.full_like(cs, np.nan)
    b = np.zeros(Cch) if bias is None else _np64(bias)
    for i, (s0, L, r) in enumerate(zip(seq_starts, seq_lens, resume)):
        hist = cs[i].copy() if int(r) else np.zeros((Cch, K - 1))
        for t in range(int(s0), int(s0) + int(L)):
            acc = b + x[t] * w[:, K - 1]
            for u in range(K - 1):
                acc = acc + hist[:, u] * w[:, u]
            out[t] = silu(acc)
            if K > 1:
                hist = np.concatenate([hist[:, 1:], x[t][:, None]], axis=1)
            snaps[t] = hist
        new_state[i] = hist
    return out, new_state, snaps
