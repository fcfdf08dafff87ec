"""Parity of the causal depthwise conv1d + SiLU (ssm_conv1d) with the oracle
(needs a GB300): outputs within fp32 rounding, and the conv-state slots and
snapshots (copies of inputs) exactly."""
import numpy as np
import pytest
import torch

from oracle import extensions as ext
from state_space_model_ssm_gb300 import binding as bd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from state_space_model_ssm_gb300 import build
    build.build()
    bd.load()


def _case(C, K, lens, resume, starts=None, n_tokens=None, seed=0):
    g = torch.Generator().manual_seed(seed)
    starts = starts if starts is not None else list(np.cumsum([0] + lens[:-1]))
    T = n_tokens if n_tokens is not None else int(sum(lens))
    x = torch.randn((T, C), generator=g)
    w = torch.randn((C, K), generator=g) * 0.5
    b = torch.randn((C,), generator=g) * 0.1
    st = torch.randn((len(lens), C, max(K - 1, 0)), generator=g)
    return x, w, b, st, starts, lens, resume


def _run(x, w, b, st, starts, lens, resume, use_bias, snaps):
    dev = "cuda"
    T, C = x.shape
    K = w.shape[1]
    i32 = torch.int32
    state = st.clone().to(dev)
    out = torch.full((T, C), float("nan"), device=dev)
    sn = torch.full((T, C, K - 1), float("nan"), device=dev) if snaps else None
    bd.ssm_conv1d(x.to(dev), w.to(dev), state, torch.tensor(starts, dtype=i32, device=dev),
                  torch.tensor(lens, dtype=i32, device=dev), torch.tensor(resume, dtype=i32, device=dev),
                  out=out, bias=b.to(dev) if use_bias else None, snapshots=sn)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), state.double().cpu().numpy(), (sn.double().cpu().numpy() if snaps else None)


@pytest.mark.parametrize("K", [1, 2, 4, 8])
@pytest.mark.parametrize("use_bias,snaps", [(True, True), (False, False)], ids=["bias_snaps", "plain"])
def test_conv1d_ragged(K, use_bias, snaps):
    """Ragged batch: an empty resuming sequence (slot kept), an empty fresh one
    (slot zeroed), sequences shorter than the k-1 history (slot shifted), and
    tokens no sequence owns."""
    x, w, b, st, starts, lens, resume = _case(37, K, [0, 1, 2, 9, 30, 0], [1, 0, 1, 1, 0, 0],
                                              starts=[0, 0, 3, 5, 15, 20], n_tokens=47, seed=K)
    out, state, sn = _run(x, w, b, st, starts, lens, resume, use_bias, snaps)
    o_ref, s_ref, sn_ref = ext.conv1d_silu(x, w, st, starts, lens, resume, bias=b if use_bias else None)
    own = ~np.isnan(o_ref[:, 0])
    assert np.all(np.abs(out[own] - o_ref[own]) <= 1e-5 * (1.0 + np.abs(o_ref[own])))
    assert np.isnan(out[~own]).all()                                   # tokens owned by no sequence
    assert np.array_equal(state, s_ref)
    if snaps:
        assert np.array_equal(sn[own], sn_ref[own])
        assert np.isnan(sn[~own]).all()


def test_conv1d_long_sequence_nemotron_width():
    """One sequence of 2048 tokens over 6144 channels (Nemotron-H's conv width:
    4096 of x plus 2 x 8 groups x 128 of B and C), resuming, k = 4."""
    x, w, b, st, starts, lens, resume = _case(6144, 4, [2048], [1], seed=11)
    out, state, _ = _run(x, w, b, st, starts, lens, resume, True, False)
    o_ref, s_ref, _ = ext.conv1d_silu(x, w, st, starts, lens, resume, bias=b)
    assert np.all(np.abs(out - o_ref) <= 1e-5 * (1.0 + np.abs(o_ref)))
    assert np.array_equal(state, s_ref)


def test_conv1d_split_resume_equals_one_call():
    x, w, b, st, starts, lens, resume = _case(64, 4, [50], [1], seed=12)
    out, s_full, _ = _run(x, w, b, st, starts, lens, resume, True, False)
    o1, s1, _ = _run(x[:17], w, b, st, [0], [17], [1], True, False)
    o2, s2, _ = _run(x[17:], w, b, torch.from_numpy(s1).float(), [0], [33], [1], True, False)
    assert np.array_equal(np.concatenate([o1, o2]), out)
    assert np.array_equal(s2, s_full)


@pytest.mark.parametrize("K", [2, 4, 7])
def test_conv1d_long_ragged_spans(K):
    """Sequences much longer than the average, so the blocks of one sequence
    walk several spans each, beside a short one; resuming and fresh."""
    x, w, b, st, starts, lens, resume = _case(264, K, [3000, 17, 1200], [1, 0, 1], seed=20 + K)
    out, state, _ = _run(x, w, b, st, starts, lens, resume, True, False)
    o_ref, s_ref, _ = ext.conv1d_silu(x, w, st, starts, lens, resume, bias=b)
    assert np.all(np.abs(out - o_ref) <= 1e-5 * (1.0 + np.abs(o_ref)))
    assert np.array_equal(state, s_ref)


def test_conv1d_no_tokens_rolls_the_slots():
    """A call with no tokens at all: fresh sequences' slots become zeros,
    resuming ones keep theirs."""
    x, w, b, st, starts, lens, resume = _case(40, 4, [0, 0, 0], [0, 1, 0], starts=[0, 0, 0], n_tokens=0, seed=5)
    out, state, _ = _run(x, w, b, st, starts, lens, resume, True, False)
    _, s_ref, _ = ext.conv1d_silu(x, w, st, starts, lens, resume, bias=b)
    assert np.array_equal(state, s_ref)
    assert np.all(state[0] == 0) and np.all(state[2] == 0)
    assert np.array_equal(state[1], st[1].double().numpy())
