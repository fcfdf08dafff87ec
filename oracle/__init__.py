"""CPU oracle of the Mamba2 selective-state scan (test infrastructure).

Only the tests, the package smoke check and the bench's CPU-baseline leg use
this package.  Nothing in the product path imports it, and it imports nothing
from the product package.

Two independent forms are provided:

* ``scan``        -- the recurrence, run token by token in double precision by
                     the plain C code in ``ssm_oracle.c`` (threads over
                     independent (sequence, head) units only);
* ``matrix_form`` -- the same map written out as a sum over earlier tokens with
                     explicit decay factors (``matrix_form.py``, NumPy float64),
                     for tiny inputs.  It is used to pin the loop form;
* ``chunked_form`` -- the recurrence unrolled over chunks of tokens (the SSD
                     chunked matrix form with state passing between chunks,
                     ``chunked_form.py``, NumPy float64): the decomposition the
                     tensor-core kernels evaluate, checked against ``scan``;
* ``extensions``   -- the steps around the scan (dt discretisation, gated
                     RMSNorm, per-token state snapshots, causal conv1d + SiLU).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .chunked_form import chunked_form  # noqa: F401
from .extensions import conv1d_silu, discretize_dt, gated_rmsnorm, scan_with_snapshots  # noqa: F401
from .matrix_form import matrix_form  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libssm_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library and declare its entry point."""
    lib = ctypes.CDLL(path)
    f = lib.ssm_oracle_scan
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 13
                  + [ctypes.c_int, ctypes.c_long] + [ctypes.c_int] * 5)
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load_library(_LIB_PATH)
    return _lib


def _f64(a):
    a = a.detach().cpu().numpy() if hasattr(a, "detach") else np.asarray(a)
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    a = a.detach().cpu().numpy() if hasattr(a, "detach") else np.asarray(a)
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def scan(x, dt, A, B, C, D, state, seq_starts, seq_lens, resume, *,
         heads=None, n_threads=None, y_fill=np.nan, lib=None, dt_bias=None, dt_softplus=False):
    """Run the oracle.  Inputs may be torch tensors or arrays (any float type;
    they are widened to float64 exactly).  Shapes: x [T,H,P], dt [T,H], A [H],
    B/C [T,G,N], D [H], state [n,H,P,N] (read for resuming sequences only),
    seq_starts/seq_lens/resume [n].

    heads: optional iterable of head indices to compute (others stay NaN).
    lib: an already opened oracle library (default: the one built here).
    dt_bias [H], dt_softplus: discretise dt first (``extensions.discretize_dt``).
    Returns (y [T,H,P], state_out [n,H,P,N]) as float64 arrays.
    """
    if dt_bias is not None or dt_softplus:
        dt = discretize_dt(dt, dt_bias, dt_softplus)
    x, dt, A, B, C, D = map(_f64, (x, dt, A, B, C, D))
    state = _f64(state)
    seq_starts, seq_lens, resume = map(_i32, (seq_starts, seq_lens, resume))
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    n = seq_lens.shape[0]
    assert dt.shape == (T, H) and A.shape == (H,) and D.shape == (H,)
    assert B.shape == (T, G, N) and C.shape == (T, G, N)
    assert state.shape == (n, H, P, N)
    y = np.full((T, H, P), y_fill, dtype=np.float64)
    state_out = np.full((n, H, P, N), np.nan, dtype=np.float64)
    sel = None
    if heads is not None:
        sel = np.zeros(H, dtype=np.uint8)
        sel[np.asarray(list(heads), dtype=np.int64)] = 1
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    rc = (lib or _load()).ssm_oracle_scan(
        _ptr(state), _ptr(state_out), _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
        _ptr(C), _ptr(D), _ptr(y), _ptr(seq_starts), _ptr(seq_lens),
        _ptr(resume), _ptr(sel), int(n), int(T), int(H), int(P), int(N),
        int(G), int(n_threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return y, state_out


def scan_inputs(inp, **kw):
    """``scan`` on a ``ScanInputs`` bundle (from the workload generator)."""
    return scan(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.state,
                inp.seq_starts, inp.seq_lens, inp.resume, **kw)
