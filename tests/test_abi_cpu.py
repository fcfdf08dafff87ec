"""The C ABI without a GPU: the library loads, exports every function the
public header declares, and rejects bad arguments on the host before any
launch (these calls never reach the device, so fake but aligned pointers are
safe: every case below fails a host check)."""
import ctypes

import pytest

from state_space_model_ssm_gb300 import binding as bd

GOOD = dict(n_seqs=2, n_tokens=8, n_heads=4, head_dim=16, d_state=32, n_groups=2)
PTR = 0x10000   # 16-byte aligned, never dereferenced (each call below fails a host check)


@pytest.fixture(scope="module")
def lib():
    from state_space_model_ssm_gb300 import build
    build.build()
    return bd.load()


def _call(lib, tuning=None, **over):
    ptrs = dict(state=PTR, x=PTR, dt=PTR, A=PTR, B=PTR, C=PTR, D=PTR, y=PTR,
                seq_starts=PTR, seq_lens=PTR, resume=PTR)
    sizes = dict(GOOD)
    for k, v in over.items():
        (ptrs if k in ptrs else sizes)[k] = v
    return bd.scan_raw(**ptrs, **sizes, tuning=tuning)


def test_header_declares_the_scan_entry_points():
    names = bd.declared_functions()
    assert {"ssm_scan", "ssm_scan_tuned", "ssm_scan_ws", "ssm_scan_workspace_bytes",
            "ssm_status_string"} <= set(names)


def test_workspace_bytes_is_zero_for_invalid_sizes(lib):
    assert bd.workspace_bytes(0, 8, 4, 16, 32, 2) == 0
    assert bd.workspace_bytes(2, 8, 4, 16, 30, 2) == 0
    assert bd.workspace_bytes(2, 8, 4, 16, 32, 3) == 0


def test_library_exports_every_declared_symbol(lib):
    for name in bd.declared_functions():
        assert hasattr(lib, name), f"libssmscan does not export {name}"


def test_status_strings(lib):
    for code, text in [(0, "ok"), (-1, "invalid argument"), (-2, "unsupported geometry"),
                       (-3, "CUDA error"), (-4, "device wait timed out"), (7, "unknown status")]:
        assert bd.status_string(code) == text


@pytest.mark.parametrize("over,expect", [
    (dict(n_seqs=-1), bd.SSM_ERR_INVALID_ARG),
    (dict(n_tokens=-3), bd.SSM_ERR_INVALID_ARG),
    (dict(n_heads=0), bd.SSM_ERR_INVALID_ARG),
    (dict(head_dim=0), bd.SSM_ERR_INVALID_ARG),
    (dict(n_groups=3), bd.SSM_ERR_INVALID_ARG),           # 4 heads % 3 groups
    (dict(d_state=30), bd.SSM_ERR_UNSUPPORTED),           # not a multiple of 4
    (dict(d_state=2048), bd.SSM_ERR_UNSUPPORTED),         # above the supported maximum
    (dict(state=0), bd.SSM_ERR_INVALID_ARG),
    (dict(x=0), bd.SSM_ERR_INVALID_ARG),
    (dict(y=0), bd.SSM_ERR_INVALID_ARG),
    (dict(seq_lens=0), bd.SSM_ERR_INVALID_ARG),
    (dict(resume=0), bd.SSM_ERR_INVALID_ARG),
    (dict(state=PTR + 4), bd.SSM_ERR_INVALID_ARG),        # state must be 16-byte aligned
    (dict(B=PTR + 8), bd.SSM_ERR_INVALID_ARG),
    (dict(C=PTR + 12), bd.SSM_ERR_INVALID_ARG),
    (dict(x=PTR + 2), bd.SSM_ERR_INVALID_ARG),            # 4-byte alignment for the rest
    (dict(seq_starts=PTR + 1), bd.SSM_ERR_INVALID_ARG),
])
def test_host_rejects_bad_arguments(lib, over, expect):
    assert _call(lib, **over) == expect


def test_empty_batch_is_a_noop(lib):
    # n_seqs == 0 returns before touching any pointer or the device
    assert _call(lib, n_seqs=0, state=0, x=0, y=0) == bd.SSM_OK


@pytest.mark.parametrize("field,value", [
    ("path", 4), ("path", -1), ("lanes_per_row", 3), ("lanes_per_row", 64),
    ("rows_per_thread", 3), ("chunk_tokens", 257), ("chunk_tokens", -1), ("ctas_per_sm", -2),
    ("segment_state", 3), ("segment_state", -1),
])
def test_host_rejects_bad_tuning(lib, field, value):
    t = bd.Tuning()
    setattr(t, field, value)
    # a misaligned-free, otherwise valid call: the tuning check alone must fail
    assert _call(lib, tuning=t) == bd.SSM_ERR_INVALID_ARG


def test_tuning_struct_layout_matches_header():
    import re
    text = open(bd.HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} ssm_scan_tuning;", text, re.S).group(1)
    fields = re.findall(r"int\s+(\w+);", body)
    assert fields == [f[0] for f in bd.Tuning._fields_]
    assert ctypes.sizeof(bd.Tuning) == 4 * len(fields)


def test_binding_refuses_cpu_tensors():
    import torch
    z = torch.zeros(1, 1, 1, 4)
    with pytest.raises(ValueError):
        bd.ssm_scan(z, z, z, z, z, z, z, z, z, z)


# ---- ssm_scan_ssd: host checks (never reach the device) ----
SSD_GOOD = dict(n_seqs=2, n_tokens=100, n_heads=4, head_dim=16, d_state=32, n_groups=2)


def _ssd_call(lib, chunk=64, ws=PTR, ws_bytes=None, **over):
    ptrs = dict(state=PTR, x=PTR, dt=PTR, A=PTR, B=PTR, C=PTR, D=PTR, y=PTR,
                seq_starts=PTR, seq_lens=PTR, resume=PTR)
    sizes = dict(SSD_GOOD)
    for k, v in over.items():
        (ptrs if k in ptrs else sizes)[k] = v
    if ws_bytes is None:
        ws_bytes = bd.ssd_workspace_bytes(**sizes, chunk=chunk)
    return bd.ssd_raw(**ptrs, **sizes, chunk=chunk, workspace=ws, workspace_bytes=ws_bytes)


def test_header_declares_the_ssd_entry_points():
    assert {"ssm_scan_ssd", "ssm_scan_ssd_workspace_bytes"} <= set(bd.declared_functions())


def test_ssd_workspace_bytes(lib):
    # units <= n_seqs + ceil(n_tokens / chunk); one fp32 state per unit and head
    for chunk, units in ((64, 2 + 2), (128, 2 + 1), (0, 2 + 1)):
        nbytes = bd.ssd_workspace_bytes(**SSD_GOOD, chunk=chunk)
        state_bytes = units * 4 * 16 * 32 * 4
        step_bytes = -(-100 * 4 * 4 // 256) * 256          # room for the discretised step
        assert state_bytes + step_bytes < nbytes <= state_bytes + step_bytes + 6 * 256 + units * (8 + 4 * 4) + 3 * 4
        assert nbytes % 256 == 0
    # 1 x 4096 tokens at 64 heads x 64 x 128: 33 units of 2 MiB
    big = bd.ssd_workspace_bytes(1, 4096, 64, 64, 128, 8, 128)
    assert 33 * (2 << 20) + 4096 * 64 * 4 < big < 33 * (2 << 20) + 4096 * 64 * 4 + 16384
    for bad in (dict(chunk=32), dict(chunk=-1), dict(head_dim=24), dict(head_dim=144),
                dict(d_state=30), dict(n_groups=3), dict(n_seqs=0)):
        args = dict(SSD_GOOD, chunk=64)
        args.update(bad)
        assert bd.ssd_workspace_bytes(**args) == 0, bad


@pytest.mark.parametrize("over,expect", [
    (dict(chunk=32), bd.SSM_ERR_INVALID_ARG),
    (dict(chunk=-1), bd.SSM_ERR_INVALID_ARG),
    (dict(head_dim=24), bd.SSM_ERR_UNSUPPORTED),         # not a multiple of 16
    (dict(head_dim=144), bd.SSM_ERR_UNSUPPORTED),        # above 128
    (dict(d_state=30), bd.SSM_ERR_UNSUPPORTED),
    (dict(n_groups=3), bd.SSM_ERR_INVALID_ARG),
    (dict(ws=0), bd.SSM_ERR_INVALID_ARG),                # no workspace
    (dict(ws=PTR + 16), bd.SSM_ERR_INVALID_ARG),         # workspace not 256-byte aligned
    (dict(ws_bytes=4096), bd.SSM_ERR_INVALID_ARG),       # workspace too small
    (dict(x=PTR + 4), bd.SSM_ERR_INVALID_ARG),           # x and y must be 16-byte aligned here
    (dict(y=PTR + 8), bd.SSM_ERR_INVALID_ARG),
    (dict(state=0), bd.SSM_ERR_INVALID_ARG),
    (dict(B=PTR + 4), bd.SSM_ERR_INVALID_ARG),
])
def test_ssd_host_rejects_bad_arguments(lib, over, expect):
    assert _ssd_call(lib, **over) == expect


def test_ssd_empty_batch_is_a_noop(lib):
    assert _ssd_call(lib, n_seqs=0, state=0, x=0, y=0, ws=0, ws_bytes=0) == bd.SSM_OK


# ---- ssm_scan_ex options: host checks ----

def _ex_call(lib, options):
    ptrs = dict(state=PTR, x=PTR, dt=PTR, A=PTR, B=PTR, C=PTR, D=PTR, y=PTR,
                seq_starts=PTR, seq_lens=PTR, resume=PTR)
    return bd.scan_raw(**ptrs, **GOOD, options=options)


def test_header_declares_the_options_entry_point_and_struct():
    import re
    assert "ssm_scan_ex" in bd.declared_functions()
    text = open(bd.HEADER).read()
    body = re.search(r"typedef struct \{([^{}]*?)\} ssm_scan_options;", text, re.S).group(1)
    fields = re.findall(r"\b(\w+);", body)
    assert fields == [f[0] for f in bd.Options._fields_]


@pytest.mark.parametrize("opts,expect", [
    (dict(dt_bias=PTR + 2), bd.SSM_ERR_INVALID_ARG),                   # 4-byte alignment
    (dict(state_snapshots=PTR + 8), bd.SSM_ERR_INVALID_ARG),           # 16-byte alignment
    (dict(gated_y=PTR), bd.SSM_ERR_INVALID_ARG),                       # no gate, no weight
    (dict(gated_y=PTR, gate_z=PTR, norm_weight=PTR, norm_eps=0.0), bd.SSM_ERR_INVALID_ARG),
    (dict(gated_y=PTR, gate_z=PTR + 4, norm_weight=PTR, norm_eps=1e-5), bd.SSM_ERR_INVALID_ARG),
    (dict(n_launch_events=-2), bd.SSM_ERR_INVALID_ARG),                # negative event count
    (dict(n_launch_events=2), bd.SSM_ERR_INVALID_ARG),                 # events without an array
])
def test_options_rejected_on_the_host(lib, opts, expect):
    o = bd.Options(**opts)
    assert _ex_call(lib, o) == expect


# ---- ssm_conv1d: host checks ----

@pytest.mark.parametrize("over,expect", [
    (dict(kernel_size=0), bd.SSM_ERR_INVALID_ARG),
    (dict(kernel_size=9), bd.SSM_ERR_INVALID_ARG),
    (dict(channels=0), bd.SSM_ERR_INVALID_ARG),
    (dict(n_tokens=-1), bd.SSM_ERR_INVALID_ARG),
    (dict(weight=0), bd.SSM_ERR_INVALID_ARG),
    (dict(conv_state=0), bd.SSM_ERR_INVALID_ARG),
    (dict(x=PTR + 2), bd.SSM_ERR_INVALID_ARG),
    (dict(bias=PTR + 1), bd.SSM_ERR_INVALID_ARG),
    (dict(n_tokens=1 << 20, channels=1 << 12), bd.SSM_ERR_UNSUPPORTED),
])
def test_conv1d_host_rejects(lib, over, expect):
    args = dict(x=PTR, weight=PTR, bias=None, conv_state=PTR, out=PTR, seq_starts=PTR, seq_lens=PTR,
                resume=PTR, n_seqs=2, n_tokens=8, channels=16, kernel_size=4, snapshots=None)
    args.update(over)
    assert bd.conv1d_raw(**args) == expect


def test_conv1d_empty_batch_is_a_noop(lib):
    assert bd.conv1d_raw(0, 0, 0, 0, 0, 0, 0, 0, 0, 8, 16, 4) == bd.SSM_OK


def test_ex_workspace_bytes_adds_the_discretised_step(lib):
    sizes = dict(GOOD)
    plain = bd.workspace_bytes(*sizes.values())
    assert bd.ex_workspace_bytes(*sizes.values()) == plain
    step = -(-GOOD["n_tokens"] * GOOD["n_heads"] * 4 // 256) * 256
    assert bd.ex_workspace_bytes(*sizes.values(), options=bd.Options(dt_softplus=1)) == step + plain
    assert bd.ex_workspace_bytes(*sizes.values(), options=bd.Options(dt_bias=PTR)) == step + plain
    assert bd.ex_workspace_bytes(*sizes.values(), options=bd.Options(dt_softplus=1, state_snapshots=PTR)) == step


def test_dt_options_need_a_workspace(lib):
    o = bd.Options(dt_softplus=1)
    assert _ex_call(lib, o) == bd.SSM_ERR_INVALID_ARG                     # none at all
    ptrs = dict(state=PTR, x=PTR, dt=PTR, A=PTR, B=PTR, C=PTR, D=PTR, y=PTR,
                seq_starts=PTR, seq_lens=PTR, resume=PTR)
    assert bd.scan_raw(**ptrs, **GOOD, options=o, workspace=PTR, workspace_bytes=64) == bd.SSM_ERR_INVALID_ARG
    assert bd.scan_raw(**ptrs, **GOOD, options=o, workspace=PTR + 16, workspace_bytes=1 << 20) == bd.SSM_ERR_INVALID_ARG
