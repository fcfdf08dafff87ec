"""The bounded waits of the pipelined kernels give up cleanly (needs a GB300).

A child process runs with SSM_SCAN_TEST_FAIL_WAITS=1, so every pipeline wait of
the segments' tensor-core state pass and of the SSD kernels gives up at once,
and with SSM_SCAN_CHECK=1, so the library reads the status word back.  Both calls must report SSM_ERR_TIMEOUT (the kernels drain their copies
and products, free their tensor memory and return), and the same context must
then run a scan without such waits to oracle parity.  Nothing here stalls or
faults the GPU: the failure is a flag nothing sets."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import torch
    import oracle
    from state_space_model_ssm_gb300 import binding as bd
    from state_space_model_ssm_gb300.workloads import Geometry, make_inputs
    from tests.gpu_helpers import assert_parity

    bd.load()
    inp = make_inputs(Geometry(4, 32, 64, 2), [300, 40], [0, 1], seed=7)
    d = inp.to("cuda")
    g = inp.geom
    args = (d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume)

    t = bd.Tuning()
    t.path = bd.PATH_PREFILL
    t.segment_tokens = 64
    t.segment_state = bd.SEGMENT_STATE_TENSOR
    nbytes = bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state, g.n_groups, t)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for name, call in (
            ("segment state pass", lambda: bd.ssm_scan(d.state.clone(), *args, tuning=t, workspace=ws)),
            ("ssd output kernel", lambda: bd.ssm_scan_ssd(d.state.clone(), *args, chunk=128))):
        try:
            call()
        except bd.SsmScanError as e:
            assert e.status == bd.SSM_ERR_TIMEOUT, (name, e.status)
        else:
            raise SystemExit(name + ": no timeout reported")
    torch.cuda.synchronize()

    y_ref, s_ref = oracle.scan_inputs(inp)
    state = d.state.clone()
    y = bd.ssm_scan(state, *args)                  # no workspace: the prefill kernel alone, no pipeline waits
    torch.cuda.synchronize()
    assert_parity(inp, y.double().cpu().numpy(), state.double().cpu().numpy(), y_ref, s_ref)
    print("ok")
""")


CHILD_UNCHECKED = textwrap.dedent("""
    import torch
    from state_space_model_ssm_gb300 import binding as bd
    from state_space_model_ssm_gb300.workloads import Geometry, make_inputs
    from tests.gpu_helpers import covered_tokens

    bd.load()
    inp = make_inputs(Geometry(4, 32, 64, 2), [300, 40], [0, 1], seed=7)
    d = inp.to("cuda")
    g = inp.geom
    args = (d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume)
    owned = torch.from_numpy(covered_tokens(inp)).cuda()

    t = bd.Tuning()
    t.path = bd.PATH_PREFILL
    t.segment_tokens = 64
    t.segment_state = bd.SEGMENT_STATE_TENSOR
    nbytes = bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state, g.n_groups, t)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for name, run in (
            ("segment state pass", lambda s: bd.ssm_scan(s, *args, tuning=t, workspace=ws)),
            ("ssd chunk states", lambda s: bd.ssm_scan_ssd(s, *args, chunk=128))):
        state = d.state.clone()
        y = run(state)                             # no check: the call itself reports success
        torch.cuda.synchronize()
        assert torch.isnan(y[owned]).all(), name + ": y not marked NaN after a timeout"
        same = torch.equal(state.view(torch.int32), d.state.view(torch.int32))
        assert same, name + ": a slot changed after a timeout"
    print("ok")
""")


def test_timeout_without_check_marks_outputs():
    """Without SSM_SCAN_CHECK nothing reads the status word back, so a wait that
    gave up must show in the outputs: y NaN on every owned token, the slots
    bit-for-bit as they were before the call."""
    env = dict(os.environ, SSM_SCAN_TEST_FAIL_WAITS="1")
    env.pop("SSM_SCAN_CHECK", None)
    r = subprocess.run([sys.executable, "-c", CHILD_UNCHECKED], env=env, cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]


def test_bounded_waits_report_timeout_and_leave_the_context_usable():
    env = dict(os.environ, SSM_SCAN_CHECK="1", SSM_SCAN_TEST_FAIL_WAITS="1")
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
