"""ctypes binding of libssmscan (argument marshalling only).

Every step of the scan runs in the CUDA kernels of ``libssmscan.so``; this
module checks tensor dtypes, devices and shapes, passes raw device pointers and
the current CUDA stream, and turns a nonzero status into an exception.  If the
library has not been built it raises: there is no other implementation.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libssmscan.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "ssmscan.h")

SSM_OK = 0
SSM_ERR_INVALID_ARG = -1
SSM_ERR_UNSUPPORTED = -2
SSM_ERR_CUDA = -3
SSM_ERR_TIMEOUT = -4

PATH_AUTO, PATH_DECODE, PATH_PREFILL, PATH_PREFILL_DIRECT = 0, 1, 2, 3
SEGMENT_STATE_AUTO, SEGMENT_STATE_FP32, SEGMENT_STATE_TENSOR = 0, 1, 2

_lib = None
_lock = threading.Lock()


class SsmScanError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Tuning(ctypes.Structure):
    """Launch-shape overrides (``ssm_scan_tuning``); zero fields mean automatic."""
    _fields_ = [("path", ctypes.c_int), ("lanes_per_row", ctypes.c_int),
                ("rows_per_thread", ctypes.c_int), ("rows_per_cta", ctypes.c_int),
                ("chunk_tokens", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("segment_tokens", ctypes.c_int), ("segment_state", ctypes.c_int)]


class Options(ctypes.Structure):
    """Optional steps around the scan (``ssm_scan_options``); zero fields mean off."""
    _fields_ = [("dt_bias", ctypes.c_void_p), ("dt_softplus", ctypes.c_int),
                ("state_snapshots", ctypes.c_void_p), ("gate_z", ctypes.c_void_p),
                ("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float),
                ("gated_y", ctypes.c_void_p), ("launch_events", ctypes.c_void_p),
                ("n_launch_events", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SCAN_ARGS = [_P] * 11 + [_I] * 6


def load():
    """Open libssmscan.so (built by ``state_space_model_ssm_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libssmscan is not built ({LIB_PATH} missing); run "
                    "`python -m state_space_model_ssm_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            lib.ssm_scan.restype = _I
            lib.ssm_scan.argtypes = _SCAN_ARGS + [_P]
            lib.ssm_scan_tuned.restype = _I
            lib.ssm_scan_tuned.argtypes = _SCAN_ARGS + [ctypes.POINTER(Tuning), _P]
            lib.ssm_scan_ws.restype = _I
            lib.ssm_scan_ws.argtypes = _SCAN_ARGS + [ctypes.POINTER(Tuning), _P, ctypes.c_size_t, _P]
            lib.ssm_scan_workspace_bytes.restype = ctypes.c_size_t
            lib.ssm_scan_workspace_bytes.argtypes = [_I] * 6 + [ctypes.POINTER(Tuning)]
            lib.ssm_scan_ex.restype = _I
            lib.ssm_scan_ex.argtypes = _SCAN_ARGS + [ctypes.POINTER(Tuning), ctypes.POINTER(Options), _P,
                                                     ctypes.c_size_t, _P]
            lib.ssm_scan_ex_workspace_bytes.restype = ctypes.c_size_t
            lib.ssm_scan_ex_workspace_bytes.argtypes = [_I] * 6 + [ctypes.POINTER(Tuning), ctypes.POINTER(Options)]
            lib.ssm_scan_ssd.restype = _I
            lib.ssm_scan_ssd.argtypes = _SCAN_ARGS + [_I, ctypes.POINTER(Options), _P, ctypes.c_size_t, _P]
            lib.ssm_scan_ssd_workspace_bytes.restype = ctypes.c_size_t
            lib.ssm_scan_ssd_workspace_bytes.argtypes = [_I] * 7
            lib.ssm_conv1d.restype = _I
            lib.ssm_conv1d.argtypes = [_P] * 8 + [_I] * 4 + [_P, _P]
            lib.ssm_status_string.restype = ctypes.c_char_p
            lib.ssm_status_string.argtypes = [_I]
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    try:
        return load().ssm_status_string(int(status)).decode()
    except Exception:  # library missing: still give a readable message
        return {0: "ok", -1: "invalid argument", -2: "unsupported geometry",
                -3: "CUDA error", -4: "device wait timed out"}.get(int(status), "unknown status")


def declared_functions(header: str = HEADER):
    """Names of the functions declared in the public C header."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(ssm_\w+)\s*\(", text, flags=re.M)))


def scan_raw(state, x, dt, A, B, C, D, y, seq_starts, seq_lens, resume,
             n_seqs, n_tokens, n_heads, head_dim, d_state, n_groups,
             stream=0, tuning: Tuning | None = None, workspace=None, workspace_bytes=0,
             options: Options | None = None) -> int:
    """Call the C ABI with integer pointers; returns the status code.
    With `options` the call goes through ssm_scan_ex, else with `workspace`
    (a device pointer) through ssm_scan_ws."""
    lib = load()
    args = [_P(int(p) if p else None) for p in
            (state, x, dt, A, B, C, D, y, seq_starts, seq_lens, resume)]
    args += [int(n_seqs), int(n_tokens), int(n_heads), int(head_dim), int(d_state), int(n_groups)]
    st = _P(int(stream) if stream else None)
    if options is not None:
        tp = ctypes.byref(tuning) if tuning is not None else None
        return lib.ssm_scan_ex(*args, tp, ctypes.byref(options), _P(int(workspace) if workspace else None),
                               ctypes.c_size_t(int(workspace_bytes)), st)
    if workspace is not None:
        tp = ctypes.byref(tuning) if tuning is not None else None
        return lib.ssm_scan_ws(*args, tp, _P(int(workspace) if workspace else None),
                               ctypes.c_size_t(int(workspace_bytes)), st)
    if tuning is None:
        return lib.ssm_scan(*args, st)
    return lib.ssm_scan_tuned(*args, ctypes.byref(tuning), st)


def workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, d_state, n_groups,
                    tuning: Tuning | None = None) -> int:
    """Bytes of workspace ssm_scan_ws uses for these sizes on the current device."""
    tp = ctypes.byref(tuning) if tuning is not None else None
    return int(load().ssm_scan_workspace_bytes(int(n_seqs), int(n_tokens), int(n_heads),
                                               int(head_dim), int(d_state), int(n_groups), tp))


def ssd_raw(state, x, dt, A, B, C, D, y, seq_starts, seq_lens, resume,
            n_seqs, n_tokens, n_heads, head_dim, d_state, n_groups, chunk,
            workspace, workspace_bytes, stream=0, options: Options | None = None) -> int:
    """ssm_scan_ssd with integer pointers; returns the status code."""
    args = [_P(int(p) if p else None) for p in
            (state, x, dt, A, B, C, D, y, seq_starts, seq_lens, resume)]
    args += [int(n_seqs), int(n_tokens), int(n_heads), int(head_dim), int(d_state), int(n_groups)]
    op = ctypes.byref(options) if options is not None else None
    return load().ssm_scan_ssd(*args, int(chunk), op, _P(int(workspace) if workspace else None),
                               ctypes.c_size_t(int(workspace_bytes)), _P(int(stream) if stream else None))


def ex_workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, d_state, n_groups,
                       tuning: Tuning | None = None, options: Options | None = None) -> int:
    """Bytes of workspace ssm_scan_ex uses (the discretised step of the dt options first)."""
    tp = ctypes.byref(tuning) if tuning is not None else None
    op = ctypes.byref(options) if options is not None else None
    return int(load().ssm_scan_ex_workspace_bytes(int(n_seqs), int(n_tokens), int(n_heads), int(head_dim),
                                                  int(d_state), int(n_groups), tp, op))


def make_options(dev, H, P, T, *, dt_bias=None, dt_softplus=False, snapshots=None, gate_z=None,
                 norm_weight=None, norm_eps=1e-6, gated_y=None, launch_events=None):
    """Options from tensors (checked for dtype, device and shape); None when all are off.

    launch_events: torch.cuda.Event objects (enable_timing=True), recorded by the
    call around its kernel launches in pairs (see ``ssm_scan_options``)."""
    f32 = torch.float32
    if (dt_bias is None and not dt_softplus and snapshots is None and gated_y is None
            and not launch_events):
        return None
    o = Options()
    if launch_events:
        handles = []
        for ev in launch_events:
            h = int(ev.cuda_event)
            if h == 0:                        # torch creates the CUDA event at its first record
                ev.record(torch.cuda.current_stream(dev))
                h = int(ev.cuda_event)
            handles.append(h)
        arr = (ctypes.c_void_p * len(handles))(*handles)
        o._events_keepalive = arr             # the array lives as long as the options
        o.launch_events = ctypes.cast(arr, ctypes.c_void_p)
        o.n_launch_events = len(handles)
    if dt_bias is not None:
        _check(dt_bias, "dt_bias", f32, dev, (H,))
        o.dt_bias = dt_bias.data_ptr()
    o.dt_softplus = 1 if dt_softplus else 0
    if snapshots is not None:
        _check(snapshots, "snapshots", f32, dev)
        if snapshots.shape[0] != T or snapshots.shape[1:3] != (H, P):
            raise ValueError("snapshots must be [n_tokens, n_heads, head_dim, d_state]")
        o.state_snapshots = snapshots.data_ptr()
    if gated_y is not None:
        for nm, t, shp in (("gated_y", gated_y, (T, H, P)), ("gate_z", gate_z, (T, H, P)),
                           ("norm_weight", norm_weight, (P,))):
            if t is None:
                raise ValueError(f"{nm} is required for the gated output")
            _check(t, nm, f32, dev, shp)
        o.gated_y, o.gate_z, o.norm_weight = gated_y.data_ptr(), gate_z.data_ptr(), norm_weight.data_ptr()
        o.norm_eps = float(norm_eps)
    return o


def ssd_workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, d_state, n_groups, chunk=0) -> int:
    """Bytes of workspace ssm_scan_ssd needs (0 for unsupported arguments)."""
    return int(load().ssm_scan_ssd_workspace_bytes(int(n_seqs), int(n_tokens), int(n_heads),
                                                   int(head_dim), int(d_state), int(n_groups),
                                                   int(chunk)))


def _check(t, name, dtype, device, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def ssm_scan(state_slots, x, dt, A, B, C, D, seq_starts, seq_lens, resume_flags,
             y=None, *, tuning: Tuning | None = None, stream=None, workspace=None,
             dt_bias=None, dt_softplus=False, snapshots=None, gate_z=None, norm_weight=None,
             norm_eps=1e-6, gated_y=None, launch_events=None):
    """Run the scan on the current CUDA stream (or ``stream``).

    state_slots [n,H,P,N] fp32 (updated in place), x [T,H,P], dt [T,H], A [H],
    B/C [T,G,N], D [H] fp32; seq_starts/seq_lens/resume_flags [n] int32; all on
    one CUDA device.  Returns y [T,H,P] (allocated if not given).
    workspace: optional uint8 CUDA tensor (see ``workspace_bytes``, or
    ``ex_workspace_bytes`` with options); lets long sequences run as parallel
    time segments.  With the dt options one is allocated when none of the
    needed size is given.
    dt_bias [H] / dt_softplus: discretise dt inside the scan; snapshots
    [T,H,P,N]: the state after every token; gated_y [T,H,P] with gate_z
    [T,H,P], norm_weight [P], norm_eps: the gated RMSNorm of y (see
    ``ssm_scan_options`` in the C header).  launch_events: torch.cuda.Event
    objects recorded in pairs around the call's kernel launches.
    """
    dev = state_slots.device
    if dev.type != "cuda":
        raise ValueError("the scan runs on CUDA tensors only")
    n, H, P, N = state_slots.shape
    T = x.shape[0]
    G = B.shape[1]
    f32, i32 = torch.float32, torch.int32
    _check(state_slots, "state_slots", f32, dev)
    _check(x, "x", f32, dev, (T, H, P))
    _check(dt, "dt", f32, dev, (T, H))
    _check(A, "A", f32, dev, (H,))
    _check(B, "B", f32, dev, (T, G, N))
    _check(C, "C", f32, dev, (T, G, N))
    _check(D, "D", f32, dev, (H,))
    for nm, t in (("seq_starts", seq_starts), ("seq_lens", seq_lens), ("resume_flags", resume_flags)):
        _check(t, nm, i32, dev, (n,))
    if y is None:
        y = torch.empty((T, H, P), dtype=f32, device=dev)
    _check(y, "y", f32, dev, (T, H, P))
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the scan's device")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    opts = make_options(dev, H, P, T, dt_bias=dt_bias, dt_softplus=dt_softplus, snapshots=snapshots,
                        gate_z=gate_z, norm_weight=norm_weight, norm_eps=norm_eps, gated_y=gated_y,
                        launch_events=launch_events)
    if opts is not None and (dt_bias is not None or dt_softplus):
        need = ex_workspace_bytes(n, T, H, P, N, G, tuning, opts)
        if ws_bytes < need:                   # the discretised step needs room in the workspace
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
            ws_ptr, ws_bytes = workspace.data_ptr(), need
    with torch.cuda.device(dev):
        rc = scan_raw(state_slots.data_ptr(), x.data_ptr(), dt.data_ptr(), A.data_ptr(),
                      B.data_ptr(), C.data_ptr(), D.data_ptr(), y.data_ptr(),
                      seq_starts.data_ptr(), seq_lens.data_ptr(), resume_flags.data_ptr(),
                      n, T, H, P, N, G, stream=handle, tuning=tuning,
                      workspace=ws_ptr, workspace_bytes=ws_bytes, options=opts)
    if rc != SSM_OK:
        raise SsmScanError(rc, "ssm_scan")
    return y


def ssm_scan_ssd(state_slots, x, dt, A, B, C, D, seq_starts, seq_lens, resume_flags,
                 y=None, *, chunk: int = 0, workspace=None, stream=None, dt_bias=None,
                 dt_softplus=False, gate_z=None, norm_weight=None, norm_eps=1e-6, gated_y=None,
                 launch_events=None):
    """The scan in chunked matrix form on the TF32 tensor cores (``ssm_scan_ssd``).

    Same tensors as ``ssm_scan``; y matches the exact scan to about
    5e-3 * (1 + |y|).  ``workspace`` is a contiguous CUDA tensor of at least
    ``ssd_workspace_bytes(...)`` bytes; if omitted one is allocated with torch
    for this call.
    """
    dev = state_slots.device
    if dev.type != "cuda":
        raise ValueError("the scan runs on CUDA tensors only")
    n, H, P, N = state_slots.shape
    T = x.shape[0]
    G = B.shape[1]
    f32, i32 = torch.float32, torch.int32
    _check(state_slots, "state_slots", f32, dev)
    _check(x, "x", f32, dev, (T, H, P))
    _check(dt, "dt", f32, dev, (T, H))
    _check(A, "A", f32, dev, (H,))
    _check(B, "B", f32, dev, (T, G, N))
    _check(C, "C", f32, dev, (T, G, N))
    _check(D, "D", f32, dev, (H,))
    for nm, t in (("seq_starts", seq_starts), ("seq_lens", seq_lens), ("resume_flags", resume_flags)):
        _check(t, nm, i32, dev, (n,))
    if y is None:
        y = torch.empty((T, H, P), dtype=f32, device=dev)
    _check(y, "y", f32, dev, (T, H, P))
    need = ssd_workspace_bytes(n, T, H, P, N, G, chunk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the scan's device")
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    opts = make_options(dev, H, P, T, dt_bias=dt_bias, dt_softplus=dt_softplus, gate_z=gate_z,
                        norm_weight=norm_weight, norm_eps=norm_eps, gated_y=gated_y,
                        launch_events=launch_events)
    with torch.cuda.device(dev):
        rc = ssd_raw(state_slots.data_ptr(), x.data_ptr(), dt.data_ptr(), A.data_ptr(),
                     B.data_ptr(), C.data_ptr(), D.data_ptr(), y.data_ptr(),
                     seq_starts.data_ptr(), seq_lens.data_ptr(), resume_flags.data_ptr(),
                     n, T, H, P, N, G, chunk, workspace.data_ptr(),
                     workspace.numel() * workspace.element_size(), stream=handle, options=opts)
    if rc != SSM_OK:
        raise SsmScanError(rc, "ssm_scan_ssd")
    return y


def conv1d_raw(x, weight, bias, conv_state, out, seq_starts, seq_lens, resume, n_seqs, n_tokens,
               channels, kernel_size, snapshots=None, stream=0) -> int:
    """ssm_conv1d with integer pointers; returns the status code."""
    ptrs = [_P(int(p) if p else None) for p in
            (x, weight, bias, conv_state, out, seq_starts, seq_lens, resume)]
    return load().ssm_conv1d(*ptrs, int(n_seqs), int(n_tokens), int(channels), int(kernel_size),
                             _P(int(snapshots) if snapshots else None), _P(int(stream) if stream else None))


def ssm_conv1d(x, weight, conv_state, seq_starts, seq_lens, resume_flags, out=None, *, bias=None,
               snapshots=None, stream=None):
    """Causal depthwise conv1d + SiLU with a rolling conv-state slot (``ssm_conv1d``).

    x [T, C], weight [C, K], conv_state [n, C, K-1] (updated in place), bias [C]
    or None, snapshots [T, C, K-1] or None; returns out [T, C]."""
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("the convolution runs on CUDA tensors only")
    T, C = x.shape
    K = weight.shape[1]
    n = seq_lens.shape[0]
    f32, i32 = torch.float32, torch.int32
    _check(x, "x", f32, dev)
    _check(weight, "weight", f32, dev, (C, K))
    _check(conv_state, "conv_state", f32, dev, (n, C, K - 1))
    if bias is not None:
        _check(bias, "bias", f32, dev, (C,))
    if snapshots is not None:
        _check(snapshots, "snapshots", f32, dev, (T, C, K - 1))
    for nm, t in (("seq_starts", seq_starts), ("seq_lens", seq_lens), ("resume_flags", resume_flags)):
        _check(t, nm, i32, dev, (n,))
    if out is None:
        out = torch.empty((T, C), dtype=f32, device=dev)
    _check(out, "out", f32, dev, (T, C))
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(dev):
        rc = conv1d_raw(x.data_ptr(), weight.data_ptr(), bias.data_ptr() if bias is not None else None,
                        conv_state.data_ptr(), out.data_ptr(), seq_starts.data_ptr(), seq_lens.data_ptr(),
                        resume_flags.data_ptr(), n, T, C, K,
                        snapshots.data_ptr() if snapshots is not None else None, stream=handle)
    if rc != SSM_OK:
        raise SsmScanError(rc, "ssm_conv1d")
    return out
