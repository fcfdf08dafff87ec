"""Parity of the SSD chunked form on the TF32 tensor cores (ssm_scan_ssd) with
the CPU oracle (needs a GB300).

The oracle is the exact recurrence; the SSD form rounds the operands of its
contractions to TF32, so y (minus its exact D*x skip term) and the final state
are compared within 5e-3 * (1 + |ref|) elementwise."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_ssm_gb300 import binding as bd
from state_space_model_ssm_gb300.workloads import Geometry, make_inputs, workload
from tests.gpu_helpers import SSD_TOL, assert_parity, run_gpu_ssd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_model_ssm_gb300 import build
    build.build()
    bd.load()


@pytest.mark.parametrize("chunk", [64, 128])
@pytest.mark.parametrize("name", ["tiny", "ragged_12", "edge_p96_n100", "prefill_1x4096"])
def test_ssd_parity_workloads(name, chunk):
    inp = workload(name)
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu_ssd(inp, chunk=chunk)
    assert_parity(inp, y, s, y_ref, s_ref, tol=SSD_TOL)


def test_ssd_default_chunk_is_128():
    inp = workload("ragged_12")
    y0, s0 = run_gpu_ssd(inp, chunk=0)
    y1, s1 = run_gpu_ssd(inp, chunk=128)
    assert np.array_equal(y0, y1, equal_nan=True) and np.array_equal(s0, s1)


def test_ssd_long_4x16384_sampled_heads():
    """Full size (T = 65536, 512 chunks): three heads in three groups of every
    sequence are compared with the oracle element by element."""
    inp = workload("long_4x16384")
    heads = [0, 37, 63]
    y_ref, s_ref = oracle.scan_inputs(inp, heads=heads)
    y, s = run_gpu_ssd(inp, chunk=128)
    assert_parity(inp, y, s, y_ref, s_ref, heads=heads, tol=SSD_TOL)


@pytest.mark.parametrize("geom,chunk", [
    (Geometry(2, 16, 4, 1), 64),          # d_state padded from 4 to 8
    (Geometry(6, 32, 12, 3), 128),        # padded from 12 to 16, 3 groups
    (Geometry(3, 48, 36, 3), 64),         # head_dim 48: 6 column blocks
    (Geometry(4, 128, 128, 2), 128),      # the widest head_dim (mma.sync: tiles exceed one block)
    (Geometry(8, 96, 100, 2), 128),       # tcgen05 with d_state padded to 104
    (Geometry(4, 64, 256, 2), 64),        # the widest d_state that fits chunk 64
], ids=["n4", "n12_g3", "p48", "p128", "p96_n100", "n256"])
def test_ssd_odd_geometries(geom, chunk):
    inp = make_inputs(geom, [1, 70, 200, 129], [0, 1, 0, 1], seed=21)
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu_ssd(inp, chunk=chunk)
    assert_parity(inp, y, s, y_ref, s_ref, tol=SSD_TOL)


# head_dim 16 runs the output kernel on mma.sync; head_dim 32 and 64 at chunk
# 128 run it on tcgen05 (chunk 64 stays on mma.sync).
@pytest.mark.parametrize("geom", [Geometry(4, 16, 32, 2), Geometry(4, 32, 32, 2), Geometry(2, 64, 128, 1)],
                         ids=["p16", "p32", "p64"])
@pytest.mark.parametrize("dt_scale,a_value", [(1.0, -16.0), (60.0, -16.0), (1.0, 0.0), (0.5, 0.05)],
                         ids=["strong", "underflow", "no_decay", "growth"])
def test_ssd_extreme_decay(dt_scale, a_value, geom):
    """exp(a_t - a_s) only for s <= t: steep decay underflows to zero and never
    overflows; no decay and slow growth stay finite."""
    inp = make_inputs(geom, [150, 77, 256], [0, 1, 1], seed=31)
    inp.dt.mul_(dt_scale)
    inp.A.fill_(a_value)
    y_ref, s_ref = oracle.scan_inputs(inp)
    for chunk in (64, 128):
        y, s = run_gpu_ssd(inp, chunk=chunk)
        assert_parity(inp, y, s, y_ref, s_ref, tol=SSD_TOL)


@pytest.mark.parametrize("head_dim,chunk", [(16, 64), (32, 128)], ids=["mma_sync", "tcgen05"])
def test_ssd_zero_length_and_unowned_tokens(head_dim, chunk):
    """Zero-length sequences (fresh -> zero slot, resumed -> unchanged) and
    token rows owned by no sequence (never written)."""
    inp = make_inputs(Geometry(4, head_dim, 32, 2), [0, 0, 9, 4, 130], [0, 1, 0, 1, 1], seed=12,
                      starts=[0, 0, 3, 14, 20], n_tokens=160)
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu_ssd(inp, chunk=chunk)
    assert_parity(inp, y, s, y_ref, s_ref, tol=SSD_TOL)
    assert np.array_equal(s[0], np.zeros_like(s[0]))
    assert np.array_equal(s[1], inp.state[1].double().numpy())


@pytest.mark.parametrize("chunk", [64, 128])
def test_ssd_split_resume_equals_one_call(chunk):
    """A sequence run as two SSD calls (the second resuming from the slot the
    first left) matches one call and the oracle."""
    geom = Geometry(8, 32, 64, 2)
    inp = make_inputs(geom, [300], [1], seed=13)
    k = 123
    a = make_inputs(geom, [k], [1], seed=13)
    a.x, a.dt, a.B, a.C = inp.x[:k], inp.dt[:k], inp.B[:k], inp.C[:k]
    a.A, a.D, a.state = inp.A, inp.D, inp.state
    y1, s1 = run_gpu_ssd(a, chunk=chunk)
    b = make_inputs(geom, [300 - k], [1], seed=13)
    b.x, b.dt, b.B, b.C = inp.x[k:], inp.dt[k:], inp.B[k:], inp.C[k:]
    b.A, b.D = inp.A, inp.D
    b.state = torch.from_numpy(s1).float()
    y2, s2 = run_gpu_ssd(b, chunk=chunk)
    y_ref, s_ref = oracle.scan_inputs(inp)
    assert_parity(inp, np.concatenate([y1, y2]), s2, y_ref, s_ref, tol=SSD_TOL)


def test_ssd_runs_on_a_side_stream():
    inp = workload("ragged_12")
    y_ref, s_ref = oracle.scan_inputs(inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, st = run_gpu_ssd(inp, chunk=128, stream=s)
    assert_parity(inp, y, st, y_ref, s_ref, tol=SSD_TOL)


def _raw_call(inp, chunk, ws_bytes_override=None, geom_override=None):
    d = inp.to("cuda")
    g = geom_override or inp.geom
    need = bd.ssd_workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state,
                                  g.n_groups, chunk)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(d.x)
    nbytes = need if ws_bytes_override is None else ws_bytes_override
    return bd.ssd_raw(d.state.data_ptr(), d.x.data_ptr(), d.dt.data_ptr(), d.A.data_ptr(),
                      d.B.data_ptr(), d.C.data_ptr(), d.D.data_ptr(), y.data_ptr(),
                      d.seq_starts.data_ptr(), d.seq_lens.data_ptr(), d.resume.data_ptr(),
                      inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state, g.n_groups,
                      chunk, ws.data_ptr(), nbytes)


def test_ssd_rejections_before_launch():
    inp = workload("tiny")
    assert _raw_call(inp, 64, ws_bytes_override=1024) == bd.SSM_ERR_INVALID_ARG
    assert _raw_call(inp, 32) == bd.SSM_ERR_INVALID_ARG
    # d_state 1024 does not fit the shared-memory tiles of one block
    big = workload("edge_n1024")
    for chunk in (64, 128):
        assert _raw_call(big, chunk) == bd.SSM_ERR_UNSUPPORTED
    # d_state 256 fits chunk 64 only
    inp = make_inputs(Geometry(4, 64, 256, 2), [40], [0], seed=3)
    assert _raw_call(inp, 128) == bd.SSM_ERR_UNSUPPORTED
    assert _raw_call(inp, 64) == bd.SSM_OK
    torch.cuda.synchronize()


@pytest.mark.parametrize("geom,chunk", [(Geometry(4, 16, 32, 2), 64), (Geometry(4, 64, 128, 2), 128)],
                         ids=["mma_sync", "tcgen05"])
def test_ssd_fused_dt(geom, chunk):
    """dt + bias and softplus inside the kernels: against the oracle (a few
    steps above the softplus threshold), and against the same call on the
    step discretised on the host in fp32 (the same arithmetic, so far tighter
    than the TF32 bound)."""
    inp = make_inputs(geom, [1, 150, 300], [0, 1, 1], seed=44)
    g = torch.Generator().manual_seed(45)
    inp.dt = torch.randn(inp.dt.shape, generator=g) * 0.5 - 2.0
    inp.dt[::97] += 21.5                                                 # a few steps above 20
    bias = torch.rand(geom.n_heads, generator=g) - 0.5
    y_ref, s_ref = oracle.scan_inputs(inp, dt_bias=bias, dt_softplus=True)
    y, s = run_gpu_ssd(inp, chunk=chunk, dt_bias=bias, dt_softplus=True)
    assert_parity(inp, y, s, y_ref, s_ref, tol=SSD_TOL)
    host = make_inputs(geom, [1, 150, 300], [0, 1, 1], seed=44)
    v = inp.dt + bias[None, :]
    host.dt = torch.where(v > 20.0, v, torch.log1p(torch.exp(v)))      # fp32 on the host
    y_h, s_h = run_gpu_ssd(host, chunk=chunk)
    # A one-ulp difference of the step can flip TF32 roundings in the chunk-state
    # product, so the state agrees to about 1e-3, not to fp32 rounding; a fused
    # step that dropped the bias or the softplus would differ by percents.
    ok = ~np.isnan(y_h)
    assert np.allclose(y[ok], y_h[ok], rtol=1e-3, atol=1e-4)
    assert np.allclose(s, s_h, rtol=2e-3, atol=1e-4)


@pytest.mark.parametrize("geom,chunk", [(Geometry(4, 16, 32, 2), 64), (Geometry(4, 64, 128, 2), 128)],
                         ids=["mma_sync", "tcgen05"])
def test_ssd_gated_norm(geom, chunk):
    from tests.gpu_helpers import assert_gated, run_gpu_gated
    inp = make_inputs(geom, [3, 0, 200], [0, 1, 1], seed=48, starts=[0, 3, 5], n_tokens=210)
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s, gated, z, w = run_gpu_gated(inp, eps=1e-5, ssd_chunk=chunk)
    assert_parity(inp, y, s, y_ref, s_ref, tol=SSD_TOL)
    assert_gated(inp, y_ref, gated, z, w, 1e-5, tol=SSD_TOL)
