"""Helpers for the GPU parity tests: run the CUDA scan with guard bands and
compare with the CPU oracle under the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

from state_space_model_ssm_gb300 import binding as bd

# Sequential fp32 kernels: max |gpu - ref| <= TOL * (1 + |ref|), elementwise.
TOL = 1e-4
GUARD = 64   # floats of NaN canary on each side of y and of the state slots


def _guarded(shape, fill, device):
    numel = int(np.prod(shape)) if len(shape) else 1
    buf = torch.full((numel + 2 * GUARD,), fill, dtype=torch.float32, device=device)
    return buf, buf[GUARD:GUARD + numel].view(*shape)


def _opt_tensors(device, kw):
    """Move tensor-valued scan options to the device."""
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}


def run_gpu(inp, tuning=None, device="cuda", stream=None, y_fill=float("nan"), workspace=False, **opts):
    """Run libssmscan on a ScanInputs bundle; returns (y, state) as float64
    numpy arrays.  Checks that the NaN guard bands around y and the state are
    intact afterwards.  workspace=True calls ssm_scan_ws with a workspace of
    the size the library asks for (NaN-filled, so stale reads show)."""
    d = inp.to(device)
    sbuf, state = _guarded(tuple(inp.state.shape), float("nan"), device)
    state.copy_(d.state)
    ybuf, y = _guarded(tuple(inp.x.shape), y_fill, device)
    ws = None
    if workspace:
        g = inp.geom
        nbytes = bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state,
                                    g.n_groups, tuning)
        ws = torch.full((max(nbytes, 256) // 4,), float("nan"), dtype=torch.float32, device=device)
    bd.ssm_scan(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume,
                y=y, tuning=tuning, stream=stream, workspace=ws, **_opt_tensors(device, opts))
    torch.cuda.synchronize()
    for buf in (sbuf, ybuf):
        head, tail = buf[:GUARD], buf[-GUARD:]
        assert torch.isnan(head).all() and torch.isnan(tail).all(), "guard band overwritten"
    return y.double().cpu().numpy(), state.double().cpu().numpy()


def covered_tokens(inp):
    mask = np.zeros(inp.n_tokens, dtype=bool)
    for s, L in zip(inp.seq_starts.tolist(), inp.seq_lens.tolist()):
        mask[s:s + L] = True
    return mask


def assert_parity(inp, y_gpu, s_gpu, y_ref, s_ref, heads=None, tol=TOL):
    """y minus its exact skip term D*x, and the final state, within
    tol * (1 + |ref|); tokens outside every sequence untouched (NaN)."""
    H = inp.geom.n_heads
    hsel = np.arange(H) if heads is None else np.asarray(sorted(heads))
    mask = covered_tokens(inp)
    x = inp.x.double().numpy()
    D = inp.D.double().numpy()
    dx = D[None, :, None] * x
    yg = (y_gpu - dx)[mask][:, hsel]
    yr = (y_ref - dx)[mask][:, hsel]
    assert np.isfinite(yg).all(), "non-finite y from the GPU"
    err = np.abs(yg - yr)
    bound = tol * (1.0 + np.abs(yr))
    worst = np.unravel_index(np.argmax(err / bound), err.shape) if err.size else None
    assert np.all(err <= bound), (
        f"y parity: max err {err.max():.3e}, worst at {worst}, ref {yr[worst]:.6e}, gpu {yg[worst]:.6e}")
    if (~mask).any():
        assert np.all(np.isnan(y_gpu[~mask])), "y written for a token owned by no sequence"
    sg, sr = s_gpu[:, hsel], s_ref[:, hsel]
    assert np.isfinite(sg).all(), "non-finite state from the GPU"
    serr = np.abs(sg - sr)
    sbound = tol * (1.0 + np.abs(sr))
    assert np.all(serr <= sbound), f"state parity: max err {serr.max():.3e}"
    return float(err.max() if err.size else 0.0), float(serr.max() if serr.size else 0.0)


# SSD chunked form with TF32 operands: max |gpu - ref| <= SSD_TOL * (1 + |ref|).
SSD_TOL = 5e-3


def run_gpu_ssd(inp, chunk=0, device="cuda", stream=None, y_fill=float("nan"), **opts):
    """ssm_scan_ssd on a ScanInputs bundle with NaN guard bands around y and the
    state and a NaN-filled workspace of exactly the size the library asks for
    (so a read of a word the call did not write shows up).  Returns (y, state)
    as float64 numpy arrays."""
    d = inp.to(device)
    g = inp.geom
    sbuf, state = _guarded(tuple(inp.state.shape), float("nan"), device)
    state.copy_(d.state)
    ybuf, y = _guarded(tuple(inp.x.shape), y_fill, device)
    need = bd.ssd_workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state,
                                  g.n_groups, chunk)
    assert need > 0
    ws = torch.full((need // 4,), float("nan"), dtype=torch.float32, device=device)
    bd.ssm_scan_ssd(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume,
                    y=y, chunk=chunk, workspace=ws, stream=stream, **_opt_tensors(device, opts))
    torch.cuda.synchronize()
    for buf in (sbuf, ybuf):
        head, tail = buf[:GUARD], buf[-GUARD:]
        assert torch.isnan(head).all() and torch.isnan(tail).all(), "guard band overwritten"
    return y.double().cpu().numpy(), state.double().cpu().numpy()


def run_gpu_gated(inp, eps=1e-5, seed=7, ssd_chunk=None, tuning=None, workspace=False, **opts):
    """The scan with the gated RMSNorm output (gate z ~ N(0,1), weight ~ U(0.5,1.5));
    returns (y, state, gated, z, w) as float64 numpy arrays (gated NaN where not written)."""
    g = torch.Generator().manual_seed(seed)
    T, H, P = inp.x.shape
    z = torch.randn((T, H, P), generator=g)
    w = torch.rand((P,), generator=g) + 0.5
    d = inp.to("cuda")
    state = d.state.clone()
    y = torch.full_like(d.x, float("nan"))
    gated = torch.full_like(d.x, float("nan"))
    zc, wc = z.cuda(), w.cuda()
    kw = dict(gate_z=zc, norm_weight=wc, norm_eps=eps, gated_y=gated, **_opt_tensors("cuda", opts))
    if ssd_chunk is not None:
        bd.ssm_scan_ssd(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume,
                        y=y, chunk=ssd_chunk, **kw)
    else:
        ws = None
        if workspace:
            gg = inp.geom
            nbytes = bd.workspace_bytes(inp.n_seqs, inp.n_tokens, gg.n_heads, gg.head_dim, gg.d_state,
                                        gg.n_groups, tuning)
            ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        bd.ssm_scan(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume,
                    y=y, tuning=tuning, workspace=ws, **kw)
    torch.cuda.synchronize()
    return (y.double().cpu().numpy(), state.double().cpu().numpy(), gated.double().cpu().numpy(),
            z.double().numpy(), w.double().numpy())


def gated_bound(inp, y_ref, z, w, eps, tol=TOL):
    """Elementwise bound on |gated_gpu - gated_ref| when gated_ref is the
    oracle's RMSNorm of the oracle's own y.

    The scan bound is |y_gpu - y_ref| <= e_p = tol*(1 + |y_p - D x_p|) on the
    state readout, plus the fp32 rounding of the skip term D x (bounded here by
    1e-6*|D x|).  Through ms = mean_p(y^2) + eps, inv = ms^-1/2 and
    gated_p = y_p * inv * w_p * silu(z_p), to first order:
        |d ms|  <= (2/P) sum_p |y_p| e_p + (1/P) sum_p e_p^2
        |d inv| <= inv * |d ms| / (2 ms)
        |d gated_p| <= |w_p silu(z_p)| * (e_p inv + (|y_p| + e_p) |d inv|)
    The neglected remainder is second order, a fraction of about tol of that
    bound, covered by a factor (1 + 20 tol); the epilogue's own fp32 rounding
    (a few ulp) adds 2e-6*|gated_p| + 1e-7."""
    x = inp.x.double().numpy()
    D = inp.D.double().numpy()
    dx = D[None, :, None] * x
    e = tol * (1.0 + np.abs(y_ref - dx)) + 1e-6 * np.abs(dx)
    P = y_ref.shape[-1]
    ms = np.mean(y_ref * y_ref, axis=-1, keepdims=True) + eps
    inv = 1.0 / np.sqrt(ms)
    dms = (2.0 / P) * np.sum(np.abs(y_ref) * e, axis=-1, keepdims=True) + np.mean(e * e, axis=-1, keepdims=True)
    dinv = inv * dms / (2.0 * ms)
    zs = z / (1.0 + np.exp(-z))
    ws = np.abs(w[None, None, :] * zs)
    gated_ref = y_ref * inv * w[None, None, :] * zs
    return (1.0 + 20.0 * tol) * ws * (e * inv + (np.abs(y_ref) + e) * dinv) + 2e-6 * np.abs(gated_ref) + 1e-7


def assert_gated(inp, y_ref, gated_gpu, z, w, eps, tol=TOL):
    """The gated output against the oracle's gated RMSNorm of the oracle's own
    y, within the scan bound propagated through the norm (``gated_bound``),
    and untouched on unowned token rows."""
    import oracle
    mask = covered_tokens(inp)
    want = oracle.gated_rmsnorm(y_ref[mask], z[mask], w, eps)
    got = gated_gpu[mask]
    assert np.isfinite(got).all()
    bound = gated_bound(inp, y_ref, z, w, eps, tol)[mask]
    err = np.abs(got - want)
    assert np.all(err <= bound), f"gated max err {err.max():.3e}, worst ratio {np.max(err / bound):.3f}"
    if (~mask).any():
        assert np.isnan(gated_gpu[~mask]).all()
