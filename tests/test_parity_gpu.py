"""Parity of the CUDA scan with the CPU oracle (needs a GB300).

Every case draws seeded inputs, runs libssmscan through the C ABI and the
oracle on the same inputs, and compares y (minus its exact D*x skip term) and
the final state elementwise within 1e-4 * (1 + |ref|)."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_ssm_gb300 import binding as bd
from state_space_model_ssm_gb300.workloads import Geometry, make_inputs, workload
from tests.gpu_helpers import SSD_TOL, assert_parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_model_ssm_gb300 import build
    build.build()
    bd.load()


def _tuning(path=0, lanes=0, rpt=0, rows=0, chunk=0, ctas=0, seg=0, seg_state=0):
    return bd.Tuning(path, lanes, rpt, rows, chunk, ctas, seg, seg_state)


PATHS = [("auto", None), ("decode", _tuning(path=bd.PATH_DECODE)),
         ("prefill", _tuning(path=bd.PATH_PREFILL)),
         ("prefill_direct", _tuning(path=bd.PATH_PREFILL_DIRECT))]


@pytest.mark.parametrize("name", ["tiny", "edge_p96_n100"])
@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
def test_parity_small_workloads(name, path):
    inp = workload(name)
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu(inp, tuning=path[1])
    assert_parity(inp, y, s, y_ref, s_ref)


def test_parity_skip_term_zero():
    """D = 0: y is the state readout alone."""
    inp = workload("tiny")
    inp.D.zero_()
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu(inp)
    assert_parity(inp, y, s, y_ref, s_ref)


def _decode_step_inputs(base, g):
    """Fresh x, dt, B, C for one decode step of `base` (A, D, lengths and slots
    kept), drawn with the workload's distributions."""
    import math
    from state_space_model_ssm_gb300.workloads import ScanInputs
    T, H, P = base.x.shape
    G, N = base.B.shape[1], base.B.shape[2]
    return ScanInputs(geom=base.geom, x=torch.randn(T, H, P, generator=g),
                      dt=torch.nn.functional.softplus(torch.randn(T, H, generator=g) * 0.5 - 2.0),
                      A=base.A, B=torch.randn(T, G, N, generator=g) / math.sqrt(N),
                      C=torch.randn(T, G, N, generator=g) / math.sqrt(N), D=base.D, state=base.state,
                      seq_starts=base.seq_starts, seq_lens=base.seq_lens, resume=base.resume)


def test_parity_decode_16x1_300_steps():
    """The decode configuration as it is measured: 300 chained steps on the same
    16 slots (Nemotron-H geometry), fresh x, dt, B and C every step.  The oracle
    carries its own float64 state through all 300 steps; y and the slots are
    compared after steps 1, 100 and 300, so any drift of the fp32 slots over
    the chain shows."""
    base = workload("decode_16x1")
    g = torch.Generator().manual_seed(300)
    state = base.to("cuda").state.clone()
    s_ref = base.state.double().numpy()
    for step in range(1, 301):
        inp = _decode_step_inputs(base, g)
        d = inp.to("cuda")
        y = bd.ssm_scan(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume)
        y_ref, s_ref = oracle.scan(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, s_ref, inp.seq_starts,
                                   inp.seq_lens, inp.resume)
        if step in (1, 100, 300):
            torch.cuda.synchronize()
            assert_parity(inp, y.double().cpu().numpy(), state.double().cpu().numpy(), y_ref, s_ref)


def test_parity_decode_16x1_multi_step():
    """Three consecutive decode steps on the same 16 slots (Nemotron-H geometry)."""
    inp = workload("decode_16x1")
    dev = inp.to("cuda")
    state = dev.state.clone()
    s_ref = inp.state.double().numpy()
    for step in range(3):
        step_inp = workload("decode_16x1", seed=100 + step)
        d = step_inp.to("cuda")
        y = bd.ssm_scan(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume)
        y_ref, s_ref = oracle.scan(step_inp.x, step_inp.dt, step_inp.A, step_inp.B, step_inp.C,
                                   step_inp.D, s_ref, step_inp.seq_starts, step_inp.seq_lens,
                                   step_inp.resume)
        torch.cuda.synchronize()
        assert_parity(step_inp, y.double().cpu().numpy(), state.double().cpu().numpy(), y_ref, s_ref)


def test_parity_prefill_1x4096():
    inp = workload("prefill_1x4096")
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu(inp)
    assert_parity(inp, y, s, y_ref, s_ref)


def test_parity_ragged_12():
    inp = workload("ragged_12")
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu(inp)
    assert_parity(inp, y, s, y_ref, s_ref)


def test_parity_edge_n1024():
    inp = workload("edge_n1024")
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu(inp)
    assert_parity(inp, y, s, y_ref, s_ref)


def test_parity_long_4x16384_sampled_heads():
    """Full size (T = 65536) without a workspace (one block walks each sequence):
    the oracle computes three heads (in three groups) of every sequence; those
    outputs are compared element by element."""
    inp = workload("long_4x16384")
    heads = [0, 37, 63]
    y_ref, s_ref = oracle.scan_inputs(inp, heads=heads)
    y, s = run_gpu(inp)
    assert_parity(inp, y, s, y_ref, s_ref, heads=heads)


def test_parity_long_4x16384_time_segments():
    """Full size (T = 65536) through the path callers with a workspace take:
    ssm_scan_ws with the workspace the library asks for (automatic time
    segments, tensor-core state pass, combine, full pass).  One head of each of
    the 8 groups is compared element by element with the oracle."""
    inp = workload("long_4x16384")
    g = inp.geom
    assert bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state, g.n_groups) > 0
    hpg = g.n_heads // g.n_groups
    heads = [grp * hpg + (grp % hpg) for grp in range(g.n_groups)]
    y_ref, s_ref = oracle.scan_inputs(inp, heads=heads)
    y, s = run_gpu(inp, workspace=True)
    assert_parity(inp, y, s, y_ref, s_ref, heads=heads)


# Launch shapes: every accepted (lanes, rows per thread, rows per block, chunk)
# must give the same result.
PREFILL_SHAPES = [
    (4, 1, 8, 32), (4, 1, 32, 32), (4, 1, 64, 7), (8, 1, 32, 16), (16, 1, 16, 5),
    (32, 1, 8, 1), (8, 2, 16, 32), (16, 4, 32, 32), (4, 2, 64, 32), (8, 2, 64, 13),
]


@pytest.mark.parametrize("lanes,rpt,rows,chunk", PREFILL_SHAPES)
def test_parity_prefill_direct_launch_shapes(lanes, rpt, rows, chunk):
    inp = workload("tiny")
    y_ref, s_ref = oracle.scan_inputs(inp)
    t = _tuning(path=bd.PATH_PREFILL_DIRECT, lanes=lanes, rpt=rpt, rows=rows, chunk=chunk)
    y, s = run_gpu(inp, tuning=t)
    assert_parity(inp, y, s, y_ref, s_ref)


SCALED_SHAPES = [(16, 4, 32, 32), (8, 2, 16, 32), (4, 4, 32, 7), (32, 8, 8, 1), (4, 1, 8, 32),
                 (4, 2, 16, 3), (16, 1, 8, 5), (8, 4, 32, 32), (4, 2, 64, 32), (16, 2, 16, 17),
                 (16, 4, 24, 16), (32, 8, 16, 9), (16, 8, 16, 16), (8, 8, 32, 16)]


@pytest.mark.parametrize("lanes,rpt,rows,chunk", SCALED_SHAPES)
def test_parity_prefill_launch_shapes(lanes, rpt, rows, chunk):
    inp = workload("tiny")
    y_ref, s_ref = oracle.scan_inputs(inp)
    t = _tuning(path=bd.PATH_PREFILL, lanes=lanes, rpt=rpt, rows=rows, chunk=chunk)
    y, s = run_gpu(inp, tuning=t)
    assert_parity(inp, y, s, y_ref, s_ref)


@pytest.mark.parametrize("dt_scale,a_value", [(1.0, -16.0), (8.0, -16.0), (60.0, -16.0),
                                              (1.0, 0.0), (0.5, 0.05)],
                         ids=["strong", "anchor_every_few", "underflow", "no_decay", "growth"])
@pytest.mark.parametrize("path", PATHS[2:], ids=[p[0] for p in PATHS[2:]])
def test_parity_extreme_decay(dt_scale, a_value, path):
    """Decay far outside the drawn range: re-anchoring of the rescaled state
    every few tokens, dA underflowing to zero, no decay at all, and growth."""
    inp = make_inputs(Geometry(4, 16, 32, 2), [150, 77], [0, 1], seed=31)
    inp.dt.mul_(dt_scale)
    inp.A.fill_(a_value)
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu(inp, tuning=path[1])
    assert_parity(inp, y, s, y_ref, s_ref)


DECODE_SHAPES = [(32, 1, 0), (32, 2, 0), (32, 4, 0), (32, 8, 0), (16, 2, 0), (16, 1, 0), (8, 1, 0), (32, 2, 1)]


@pytest.mark.parametrize("lanes,rpt,ctas", DECODE_SHAPES)
def test_parity_decode_launch_shapes(lanes, rpt, ctas):
    inp = make_inputs(Geometry(8, 24, 128, 2), [1, 3, 1, 0, 2], [1, 0, 1, 1, 0], seed=21)
    y_ref, s_ref = oracle.scan_inputs(inp)
    t = _tuning(path=bd.PATH_DECODE, lanes=lanes, rpt=rpt, ctas=ctas)
    y, s = run_gpu(inp, tuning=t)
    assert_parity(inp, y, s, y_ref, s_ref)


@pytest.mark.parametrize("geom", [Geometry(3, 5, 4, 1), Geometry(6, 7, 12, 3), Geometry(2, 33, 36, 2),
                                  Geometry(4, 10, 64, 4), Geometry(2, 8, 256, 1)],
                         ids=lambda g: f"H{g.n_heads}P{g.head_dim}N{g.d_state}G{g.n_groups}")
@pytest.mark.parametrize("path", PATHS[1:], ids=[p[0] for p in PATHS[1:]])
def test_parity_odd_geometries(geom, path):
    inp = make_inputs(geom, [19, 1, 0, 40], [0, 1, 1, 1], seed=8)
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu(inp, tuning=path[1])
    assert_parity(inp, y, s, y_ref, s_ref)


def test_zero_length_and_unowned_tokens():
    """Zero-length sequences (fresh -> zero slot, resumed -> unchanged) and
    token rows owned by no sequence (never written)."""
    inp = make_inputs(Geometry(4, 16, 32, 2), [0, 0, 9, 4], [0, 1, 0, 1], seed=12,
                      starts=[0, 0, 3, 14], n_tokens=20)
    y_ref, s_ref = oracle.scan_inputs(inp)
    for path in PATHS:
        y, s = run_gpu(inp, tuning=path[1])
        assert_parity(inp, y, s, y_ref, s_ref)
        assert np.array_equal(s[0], np.zeros_like(s[0]))
        assert np.array_equal(s[1], inp.state[1].double().numpy())


def test_split_resume_equals_one_call():
    """A sequence run as two calls (the second resuming) matches one call."""
    geom = Geometry(8, 32, 64, 2)
    inp = make_inputs(geom, [300], [1], seed=13)
    y_one, s_one = run_gpu(inp)
    k = 123
    a = make_inputs(geom, [k], [1], seed=13)
    a.x, a.dt, a.B, a.C = inp.x[:k], inp.dt[:k], inp.B[:k], inp.C[:k]
    a.A, a.D, a.state = inp.A, inp.D, inp.state
    y1, s1 = run_gpu(a)
    b = make_inputs(geom, [300 - k], [1], seed=13)
    b.x, b.dt, b.B, b.C = inp.x[k:], inp.dt[k:], inp.B[k:], inp.C[k:]
    b.A, b.D = inp.A, inp.D
    b.state = torch.from_numpy(s1).float()
    y2, s2 = run_gpu(b)
    y_ref, s_ref = oracle.scan_inputs(inp)
    assert_parity(inp, np.concatenate([y1, y2]), s2, y_ref, s_ref)
    assert_parity(inp, y_one, s_one, y_ref, s_ref)


def test_runs_on_a_side_stream():
    inp = workload("tiny")
    y_ref, s_ref = oracle.scan_inputs(inp)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        y, s = run_gpu(inp, stream=st)
    assert_parity(inp, y, s, y_ref, s_ref)


def test_bad_arguments_raise_before_launch():
    inp = workload("tiny").to("cuda")
    with pytest.raises(bd.SsmScanError) as e:
        bd.ssm_scan(inp.state, inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.seq_starts,
                    inp.seq_lens, inp.resume, tuning=_tuning(path=bd.PATH_PREFILL, lanes=4, rows=12))
    assert e.value.status == bd.SSM_ERR_INVALID_ARG
    with pytest.raises(TypeError):
        bd.ssm_scan(inp.state.double(), inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D,
                    inp.seq_starts, inp.seq_lens, inp.resume)


# Time segments (ssm_scan_ws): long sequences cut into segments that run in
# parallel, then combined.  Short segments make many segments per sequence.
# The segments' state pass runs on the tensor cores (automatic where d_state <=
# 128 and head_dim <= 256) or in the sequential kernel (SEGMENT_STATE_FP32).
SEGMENT_CASES = [("tiny", 16), ("tiny", 32), ("tiny", 48), ("edge_p96_n100", 64), ("edge_p96_n100", 112),
                 ("ragged_12", 256), ("edge_n1024", 512), ("prefill_1x4096", 0), ("ragged_12", 0)]
SEGMENT_STATE = [("auto", bd.SEGMENT_STATE_AUTO), ("fp32", bd.SEGMENT_STATE_FP32)]


@pytest.mark.parametrize("state_pass", SEGMENT_STATE, ids=[k for k, _ in SEGMENT_STATE])
@pytest.mark.parametrize("name,seg", SEGMENT_CASES, ids=[f"{n}-{s}" for n, s in SEGMENT_CASES])
def test_parity_time_segments(name, seg, state_pass):
    inp = workload(name)
    y_ref, s_ref = oracle.scan_inputs(inp)
    t = _tuning(path=bd.PATH_PREFILL, seg=seg, seg_state=state_pass[1])
    if seg > 0:
        g = inp.geom
        assert bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state,
                                  g.n_groups, t) > 0
    y, s = run_gpu(inp, tuning=t, workspace=True)
    assert_parity(inp, y, s, y_ref, s_ref)


@pytest.mark.parametrize("state_pass", SEGMENT_STATE, ids=[k for k, _ in SEGMENT_STATE])
@pytest.mark.parametrize("dt_scale,a_value", [(8.0, -16.0), (60.0, -16.0), (1.0, 0.0), (0.5, 0.05)],
                         ids=["anchor_every_few", "underflow", "no_decay", "growth"])
def test_parity_time_segments_extreme_decay(dt_scale, a_value, state_pass):
    inp = make_inputs(Geometry(4, 16, 32, 2), [150, 77, 0, 33], [0, 1, 1, 0], seed=32)
    inp.dt.mul_(dt_scale)
    inp.A.fill_(a_value)
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu(inp, tuning=_tuning(path=bd.PATH_PREFILL, seg=16, seg_state=state_pass[1]), workspace=True)
    assert_parity(inp, y, s, y_ref, s_ref)


# Head dims across the tensor-core state pass's register shapes (head_dim
# padded to 32, 64, ..., 256) and d_state below the 128 rows of its product.
TC_GEOMS = [(4, 32, 64, 2), (3, 64, 128, 1), (2, 160, 128, 1), (2, 256, 48, 2), (6, 224, 16, 3)]


@pytest.mark.parametrize("geom", TC_GEOMS, ids=[f"h{g[0]}_p{g[1]}_n{g[2]}" for g in TC_GEOMS])
def test_parity_tensor_state_pass_geometries(geom):
    inp = make_inputs(Geometry(*geom), [300, 97, 1, 160], [1, 0, 1, 1], seed=61)
    y_ref, s_ref = oracle.scan_inputs(inp)
    t = _tuning(path=bd.PATH_PREFILL, seg=48, seg_state=bd.SEGMENT_STATE_TENSOR)
    y, s = run_gpu(inp, tuning=t, workspace=True)
    assert_parity(inp, y, s, y_ref, s_ref)


def test_tensor_state_pass_refuses_large_d_state():
    """d_state 1024 is beyond the 128 rows of the product: an explicit request fails
    before any launch; the automatic choice takes the sequential kernel."""
    inp = workload("edge_n1024")
    t = _tuning(path=bd.PATH_PREFILL, seg=512, seg_state=bd.SEGMENT_STATE_TENSOR)
    with pytest.raises(bd.SsmScanError) as e:
        run_gpu(inp, tuning=t, workspace=True)
    assert e.value.status == bd.SSM_ERR_UNSUPPORTED


def test_time_segments_need_their_workspace():
    inp = workload("tiny").to("cuda")
    t = _tuning(path=bd.PATH_PREFILL, seg=16)
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(bd.SsmScanError) as e:
        bd.ssm_scan(inp.state, inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, inp.seq_starts,
                    inp.seq_lens, inp.resume, tuning=t, workspace=small)
    assert e.value.status == bd.SSM_ERR_INVALID_ARG


# ---- fused dt discretisation (dt + bias, softplus with the identity above 20) ----

def _raw_dt_case(geom, lens, resume, seed):
    inp = make_inputs(geom, lens, resume, seed=seed)
    g = torch.Generator().manual_seed(seed + 500)
    inp.dt = torch.randn(inp.dt.shape, generator=g) * 0.5 - 2.0          # pre-activation values
    inp.dt[::7] += 23.0                                                  # some rows above the threshold
    bias = torch.rand(geom.n_heads, generator=g) - 0.5
    return inp, bias


@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
@pytest.mark.parametrize("softplus", [True, False], ids=["softplus", "bias_only"])
def test_parity_fused_dt(path, softplus):
    inp, bias = _raw_dt_case(Geometry(4, 16, 32, 2), [1, 40, 77], [0, 1, 0], seed=41)
    if not softplus:                                                     # steps dt + bias stay small and positive
        inp.dt = inp.dt.abs() * 0.05
        bias = bias.abs() * 0.1
    y_ref, s_ref = oracle.scan_inputs(inp, dt_bias=bias, dt_softplus=softplus)
    if path[0] == "decode":
        dec = make_inputs(Geometry(4, 16, 32, 2), [1, 1, 1], [1, 0, 1], seed=42)
        dec.dt = inp.dt[:3].clone()
        y_ref, s_ref = oracle.scan_inputs(dec, dt_bias=bias, dt_softplus=softplus)
        inp = dec
    y, s = run_gpu(inp, tuning=path[1], dt_bias=bias, dt_softplus=softplus)
    assert_parity(inp, y, s, y_ref, s_ref)


def test_parity_fused_dt_time_segments():
    inp, bias = _raw_dt_case(Geometry(8, 64, 128, 2), [3000], [1], seed=43)
    y_ref, s_ref = oracle.scan_inputs(inp, dt_bias=bias, dt_softplus=True)
    y, s = run_gpu(inp, workspace=True, dt_bias=bias, dt_softplus=True)
    assert_parity(inp, y, s, y_ref, s_ref)


# ---- gated RMSNorm of y after the scan ----

@pytest.mark.parametrize("path", PATHS, ids=[p[0] for p in PATHS])
def test_parity_gated_norm(path):
    from tests.gpu_helpers import assert_gated, run_gpu_gated
    inp = make_inputs(Geometry(4, 16, 32, 2), [0, 9, 40], [0, 1, 1], seed=46,
                      starts=[0, 2, 11], n_tokens=60)
    if path[0] == "decode":
        inp = make_inputs(Geometry(4, 16, 32, 2), [1, 0, 1], [1, 0, 0], seed=46, starts=[0, 1, 2], n_tokens=4)
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s, gated, z, w = run_gpu_gated(inp, eps=1e-5, tuning=path[1])
    assert_parity(inp, y, s, y_ref, s_ref)
    assert_gated(inp, y_ref, gated, z, w, 1e-5)


def test_parity_gated_norm_odd_head_dim_and_segments():
    from tests.gpu_helpers import assert_gated, run_gpu_gated
    for geom, lens, ws in ((Geometry(3, 37, 12, 3), [5, 64], False),
                           (Geometry(8, 64, 128, 2), [2500], True)):
        inp = make_inputs(geom, lens, [1] * len(lens), seed=47)
        y_ref, s_ref = oracle.scan_inputs(inp)
        y, s, gated, z, w = run_gpu_gated(inp, eps=1e-6, workspace=ws, dt_softplus=False)
        assert_parity(inp, y, s, y_ref, s_ref)
        assert_gated(inp, y_ref, gated, z, w, 1e-6)


def test_parity_gated_norm_prefill_1x4096():
    """The gated output at the measured prefill workload through ssm_scan_ws
    (time segments): the full pass writes it itself (blocks of one head)."""
    from tests.gpu_helpers import assert_gated, run_gpu_gated
    inp = workload("prefill_1x4096")
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s, gated, z, w = run_gpu_gated(inp, eps=1e-5, workspace=True)
    assert_parity(inp, y, s, y_ref, s_ref)
    assert_gated(inp, y_ref, gated, z, w, 1e-5)


@pytest.mark.parametrize("chunk", [16, 32])
def test_parity_gated_norm_fused_two_consumer_warps(chunk):
    """The fused gated output with blocks of one 32-row head (two consumer
    warps, so a chunk's gating takes several rounds of eight-lane groups), with
    and without time segments."""
    from tests.gpu_helpers import assert_gated, run_gpu_gated
    inp = make_inputs(Geometry(4, 32, 128, 2), [300, 45, 0, 7], [1, 0, 1, 0], seed=58)
    y_ref, s_ref = oracle.scan_inputs(inp)
    for ws in (False, True):
        t = _tuning(path=bd.PATH_PREFILL, rows=32, chunk=chunk, seg=64 if ws else -1)
        y, s, gated, z, w = run_gpu_gated(inp, eps=1e-5, tuning=t, workspace=ws)
        assert_parity(inp, y, s, y_ref, s_ref)
        assert_gated(inp, y_ref, gated, z, w, 1e-5)


def test_parity_y_not_16_byte_aligned():
    """y only 4-byte aligned: the full pass's output tile falls back to scalar
    stores (same results)."""
    inp = make_inputs(Geometry(8, 64, 128, 2), [700, 3, 260], [1, 0, 1], seed=57)
    y_ref, s_ref = oracle.scan_inputs(inp)
    d = inp.to("cuda")
    buf = torch.full((d.x.numel() + 1,), float("nan"), device="cuda")
    y = buf[1:].view(d.x.shape)
    for ws in (False, True):
        state = d.state.clone()
        wsb = None
        if ws:
            g = inp.geom
            wsb = torch.empty(bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state,
                                                 g.n_groups), dtype=torch.uint8, device="cuda")
        bd.ssm_scan(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume, y=y, workspace=wsb)
        torch.cuda.synchronize()
        assert_parity(inp, y.double().cpu().numpy(), state.double().cpu().numpy(), y_ref, s_ref)


# ---- the self-staged full pass (four consumer warps stage their own chunks) ----

SELF_GEOMS = [Geometry(8, 64, 128, 2), Geometry(8, 64, 100, 2), Geometry(8, 64, 64, 2),
              Geometry(8, 32, 128, 2), Geometry(6, 48, 128, 3)]


@pytest.mark.parametrize("geom", SELF_GEOMS, ids=lambda g: f"h{g.n_heads}_p{g.head_dim}_n{g.d_state}_g{g.n_groups}")
def test_parity_self_staged_full_pass(geom):
    """Shapes whose full pass runs without a producer warp (8 lanes x 4 rows per
    lane, blocks of 64 rows, y through the two tiles): d_state 128 and 64 (every
    lane busy), 100 (lanes past d_state idle, the general staging walk), blocks
    holding two heads (head_dim 32) and heads that straddle blocks (head_dim
    48); a ragged, partly resuming batch with an empty sequence, through
    ssm_scan_ws (time segments) and with 64-row blocks and no segments."""
    inp = make_inputs(geom, [700, 3, 260, 1500, 0, 41], [1, 0, 1, 0, 1, 1], seed=71)
    y_ref, s_ref = oracle.scan_inputs(inp)
    y, s = run_gpu(inp, workspace=True)
    assert_parity(inp, y, s, y_ref, s_ref)
    y, s = run_gpu(inp, tuning=_tuning(path=bd.PATH_PREFILL, rows=64, seg=-1))
    assert_parity(inp, y, s, y_ref, s_ref)


@pytest.mark.parametrize("d_state", [128, 100, 64])
def test_parity_gated_self_staged(d_state):
    """The gated output of the self-staged full pass (blocks of one 64-row head:
    y and z through tiles, gated one chunk later by all four warps), with and
    without time segments, against the oracle's y."""
    from tests.gpu_helpers import assert_gated, run_gpu_gated
    inp = make_inputs(Geometry(8, 64, d_state, 2), [700, 3, 260, 1500, 0, 41], [1, 0, 1, 0, 1, 1], seed=72)
    y_ref, s_ref = oracle.scan_inputs(inp)
    for ws in (True, False):
        t = None if ws else _tuning(path=bd.PATH_PREFILL, rows=64, seg=-1)
        y, s, gated, z, w = run_gpu_gated(inp, eps=1e-5, tuning=t, workspace=ws)
        assert_parity(inp, y, s, y_ref, s_ref)
        assert_gated(inp, y_ref, gated, z, w, 1e-5)


# ---- per-token state snapshots (speculative verify) ----

@pytest.mark.parametrize("fused_dt", [False, True], ids=["plain", "fused_dt"])
def test_parity_state_snapshots(fused_dt):
    """Short multi-token sequences (fresh, resuming, empty, with gaps): every
    owned token row of the snapshots equals the oracle's state after that
    token; unowned rows stay untouched; y and the slots as in the scan."""
    from oracle import extensions as ext
    geom = Geometry(4, 64, 128, 2)
    inp = make_inputs(geom, [4, 1, 0, 6, 3], [1, 0, 1, 1, 0], seed=49,
                      starts=[0, 5, 6, 6, 13], n_tokens=17)
    kw = {}
    if fused_dt:
        g = torch.Generator().manual_seed(50)
        inp.dt = torch.randn(inp.dt.shape, generator=g) * 0.5 - 2.0
        kw = dict(dt_bias=torch.rand(geom.n_heads, generator=g) - 0.5, dt_softplus=True)
    y_ref, s_ref, snaps_ref = ext.scan_with_snapshots(oracle.scan, inp, n_threads=1, **kw)
    d = inp.to("cuda")
    state = d.state.clone()
    y = torch.full_like(d.x, float("nan"))
    snaps = torch.full((inp.n_tokens, geom.n_heads, geom.head_dim, geom.d_state), float("nan"), device="cuda")
    bd.ssm_scan(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume, y=y,
                snapshots=snaps, **{k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()})
    torch.cuda.synchronize()
    yg, sg, ng = y.double().cpu().numpy(), state.double().cpu().numpy(), snaps.double().cpu().numpy()
    assert_parity(inp, yg, sg, y_ref, s_ref)
    from tests.gpu_helpers import covered_tokens
    mask = covered_tokens(inp)
    err = np.abs(ng[mask] - snaps_ref[mask])
    assert np.all(err <= 1e-4 * (1.0 + np.abs(snaps_ref[mask]))), f"snapshot max err {err.max():.3e}"
    assert np.isnan(ng[~mask]).all()


def test_state_snapshots_refuse_prefill_paths():
    inp = make_inputs(Geometry(2, 16, 32, 1), [3], [0], seed=51)
    d = inp.to("cuda")
    snaps = torch.empty((3, 2, 16, 32), device="cuda")
    for path in (bd.PATH_PREFILL, bd.PATH_PREFILL_DIRECT):
        with pytest.raises(bd.SsmScanError) as e:
            bd.ssm_scan(d.state.clone(), d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume,
                        snapshots=snaps, tuning=_tuning(path=path))
        assert e.value.status == bd.SSM_ERR_UNSUPPORTED


def test_tensor_state_pass_needs_16_byte_aligned_x():
    """x only 4-byte aligned: the automatic choice takes the sequential state
    pass (same results); an explicit tensor-core request is refused."""
    inp = workload("tiny")
    y_ref, s_ref = oracle.scan_inputs(inp)
    d = inp.to("cuda")
    buf = torch.empty(d.x.numel() + 1, device="cuda")
    x = buf[1:].view(d.x.shape)
    x.copy_(d.x)
    g = inp.geom
    for mode in (bd.SEGMENT_STATE_AUTO, bd.SEGMENT_STATE_TENSOR):
        t = _tuning(path=bd.PATH_PREFILL, seg=16, seg_state=mode)
        nbytes = bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state, g.n_groups, t)
        ws = torch.empty(nbytes // 4, device="cuda")
        state = d.state.clone()
        call = lambda: bd.ssm_scan(state, x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume,
                                   tuning=t, workspace=ws)
        if mode == bd.SEGMENT_STATE_TENSOR:
            with pytest.raises(bd.SsmScanError) as e:
                call()
            assert e.value.status == bd.SSM_ERR_UNSUPPORTED
        else:
            y = call()
            torch.cuda.synchronize()
            assert_parity(inp, y.double().cpu().numpy(), state.double().cpu().numpy(), y_ref, s_ref)


def test_launch_events_bracket_each_kernel():
    """Timing events recorded around the segmented prefill's four launches (plan,
    state pass, combine, full pass) and the SSD call's four; results unchanged."""
    inp = workload("tiny")
    y_ref, s_ref = oracle.scan_inputs(inp)
    d = inp.to("cuda")
    g = inp.geom
    stream = torch.cuda.current_stream()

    def events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)
        return evs

    t = _tuning(path=bd.PATH_PREFILL, seg=16)
    nbytes = bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state, g.n_groups, t)
    ws = torch.empty(nbytes // 4, device="cuda")
    state = d.state.clone()
    evs = events(8)
    y = bd.ssm_scan(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume, tuning=t,
                    workspace=ws, launch_events=evs)
    torch.cuda.synchronize()
    assert_parity(inp, y.double().cpu().numpy(), state.double().cpu().numpy(), y_ref, s_ref)
    times = [evs[2 * k].elapsed_time(evs[2 * k + 1]) for k in range(4)]
    assert all(ms >= 0.0 for ms in times)
    # the pairs are in launch order: each launch starts after the previous one ended
    assert all(evs[2 * k + 1].elapsed_time(evs[2 * k + 2]) >= 0.0 for k in range(3))

    state = d.state.clone()
    evs = events(8)
    y = bd.ssm_scan_ssd(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume, chunk=64,
                        launch_events=evs)
    torch.cuda.synchronize()
    assert_parity(inp, y.double().cpu().numpy(), state.double().cpu().numpy(), y_ref, s_ref, tol=SSD_TOL)
    assert all(evs[2 * k].elapsed_time(evs[2 * k + 1]) >= 0.0 for k in range(4))
