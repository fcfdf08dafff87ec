"""ssm_scan_static, the entry point for callers that cannot allocate device
memory (a runtime without a device allocator, a plugin whose host owns every
allocation, a path that must not enter cudaMalloc).  It runs the segmented
prefill with the library's own fixed device scratch instead of a caller
workspace, so it must give what ssm_scan_ws gives with a workspace the caller
allocated.  This file is collected last on purpose: if it fails, a run that
stops at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from state_space_model_ssm_gb300 import binding as bd
from state_space_model_ssm_gb300.workloads import workload
from tests.gpu_helpers import TOL

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 << 20     # SSM_SCAN_STATIC_SCRATCH_BYTES in include/ssmscan.h


@pytest.fixture(scope="module")
def lib():
    from state_space_model_ssm_gb300 import build
    build.build()
    lib = bd.load()
    f = lib.ssm_scan_static
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 11 + [ctypes.c_int] * 6 + [ctypes.c_void_p]
    return lib


def _ptrs(state, d, y):
    return [state.data_ptr(), d.x.data_ptr(), d.dt.data_ptr(), d.A.data_ptr(), d.B.data_ptr(),
            d.C.data_ptr(), d.D.data_ptr(), y.data_ptr(), d.seq_starts.data_ptr(),
            d.seq_lens.data_ptr(), d.resume.data_ptr()]


def _sizes(inp):
    g = inp.geom
    return [inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state, g.n_groups]


def _close(got, ref):
    got, ref = got.double().cpu().numpy(), ref.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert np.all(err <= TOL * (1.0 + np.abs(ref))), f"max err {err.max():.3e}"


@pytest.mark.parametrize("first,second,segmented", [("prefill_1x4096", 7, True), ("ragged_12", 8, True)])
def test_static_scratch_matches_caller_workspace(lib, first, second, segmented):
    """Two calls in a row (the second resumes every sequence from the first's
    slots): ssm_scan_static against ssm_scan_ws with a torch workspace.  The
    reference call segments both workloads; the static call runs the automatic
    plan on 1x4096 and, on ragged_12 (whose automatic plan needs more than the
    scratch), longer segments."""
    a = workload(first)
    b = workload(first, seed=second)
    b.resume.fill_(1)
    need = bd.workspace_bytes(*_sizes(a))
    if segmented:
        assert need > 0                         # the time-segmented path is the one exercised
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    da, db = a.to("cuda"), b.to("cuda")
    stream = torch.cuda.current_stream().cuda_stream

    state_ref = da.state.clone()
    state_new = da.state.clone()
    for d in (da, db):
        y_ref = torch.full_like(d.x, float("nan"))
        y_new = torch.full_like(d.x, float("nan"))
        bd.ssm_scan(state_ref, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens,
                    d.resume, y=y_ref, workspace=ws)
        rc = lib.ssm_scan_static(*_ptrs(state_new, d, y_new), *_sizes(a), stream)
        assert rc == bd.SSM_OK, bd.status_string(rc)
        torch.cuda.synchronize()
        _close(y_new, y_ref)
        _close(state_new, state_ref)


def _ragged_split_case():
    """A ragged batch (fresh and resuming, lengths 1 .. 1500) at 8 heads x 64 x
    128 state, 2 groups: small enough slots that the automatic time-segment
    plan fits the static scratch, so the static call runs that plan unchanged."""
    from state_space_model_ssm_gb300.workloads import Geometry, make_inputs
    return make_inputs(Geometry(8, 64, 128, 2), [1, 3, 40, 700, 1500, 9, 310], [0, 1, 0, 1, 1, 0, 1], seed=93)


def test_static_scratch_splits_ragged_sequences(lib):
    """The static call on a ragged batch whose automatic plan needs a workspace
    that fits the scratch: the long sequences are cut into time segments (the
    cross-segment combine runs), two calls in a row, the second resuming every
    sequence, against ssm_scan_ws with a caller workspace of that size."""
    a = _ragged_split_case()
    need = bd.workspace_bytes(*_sizes(a))
    assert 0 < need <= STATIC_SCRATCH_BYTES     # the automatic plan splits and is the one the static call runs
    b = _ragged_split_case()
    b.x.normal_(generator=torch.Generator().manual_seed(94))
    b.resume.fill_(1)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    da, db = a.to("cuda"), b.to("cuda")
    stream = torch.cuda.current_stream().cuda_stream
    state_ref, state_new = da.state.clone(), da.state.clone()
    for d in (da, db):
        y_ref = torch.full_like(d.x, float("nan"))
        y_new = torch.full_like(d.x, float("nan"))
        bd.ssm_scan(state_ref, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens,
                    d.resume, y=y_ref, workspace=ws)
        rc = lib.ssm_scan_static(*_ptrs(state_new, d, y_new), *_sizes(a), stream)
        assert rc == bd.SSM_OK, bd.status_string(rc)
        torch.cuda.synchronize()
        _close(y_new, y_ref)
        _close(state_new, state_ref)


def test_static_scratch_allocates_nothing(lib):
    """After one warm-up call per plan shape (which loads the kernels), further
    calls change neither the device's free memory nor torch's allocations."""
    from state_space_model_ssm_gb300.workloads import Geometry, make_inputs
    cases = [workload("prefill_1x4096"), workload("decode_16x1"), _ragged_split_case(),
             make_inputs(Geometry(24, 128, 1024, 24), [700, 1300], [0, 1], seed=91)]
    stream = torch.cuda.current_stream().cuda_stream
    devs = [(c, c.to("cuda")) for c in cases]
    outs = [(d.state.clone(), torch.empty_like(d.x)) for _, d in devs]

    def run_all():
        for (c, d), (state, y) in zip(devs, outs):
            rc = lib.ssm_scan_static(*_ptrs(state, d, y), *_sizes(c), stream)
            assert rc == bd.SSM_OK, bd.status_string(rc)
        torch.cuda.synchronize()

    run_all()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(3):
        run_all()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0


def test_static_scratch_without_segments(lib):
    """A decode batch needs no scratch; the entry point still runs it."""
    inp = workload("decode_16x1")
    d = inp.to("cuda")
    state_ref, state_new = d.state.clone(), d.state.clone()
    y_ref, y_new = torch.empty_like(d.x), torch.empty_like(d.x)
    bd.ssm_scan(state_ref, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume, y=y_ref)
    rc = lib.ssm_scan_static(*_ptrs(state_new, d, y_new), *_sizes(inp),
                             torch.cuda.current_stream().cuda_stream)
    assert rc == bd.SSM_OK
    torch.cuda.synchronize()
    _close(y_new, y_ref)
    _close(state_new, state_ref)


def test_static_scratch_fits_oversized_plans(lib):
    """A batch whose automatic plan needs more scratch than the static array
    (12 MiB state slots) runs with longer segments or none: same results as
    ssm_scan_ws with a caller workspace."""
    from state_space_model_ssm_gb300.workloads import Geometry, make_inputs
    inp = make_inputs(Geometry(24, 128, 1024, 24), [700, 1300], [0, 1], seed=91)
    g = inp.geom
    need = bd.workspace_bytes(*_sizes(inp))
    assert need > STATIC_SCRATCH_BYTES
    d = inp.to("cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    state_ref, state_new = d.state.clone(), d.state.clone()
    y_ref, y_new = torch.empty_like(d.x), torch.empty_like(d.x)
    bd.ssm_scan(state_ref, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume, y=y_ref,
                workspace=ws)
    rc = lib.ssm_scan_static(*_ptrs(state_new, d, y_new), *_sizes(inp), torch.cuda.current_stream().cuda_stream)
    assert rc == bd.SSM_OK, bd.status_string(rc)
    torch.cuda.synchronize()
    _close(y_new, y_ref)
    _close(state_new, state_ref)
