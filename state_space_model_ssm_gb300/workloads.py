"""Seeded synthetic inputs for the Mamba2 selective-state scan.

This module draws inputs only; it holds none of the scan's arithmetic, so the
CUDA path and the CPU oracle can both be fed from it.

Shapes follow the packed ragged layout of the scan call:

    x      [T][H][P]        dt [T][H]        A [H]        D [H]
    B, C   [T][G][N]        state slots [n][H][P][N]
    seq_starts, seq_lens, resume_flags  [n] int32

Distributions (stated in the workload descriptions of the Nemotron-H scan
benchmarks; "N(mu, s)" is read as mean and standard deviation):

    x ~ N(0, 1);  B, C ~ N(0, 1/N);  dt = softplus(N(-2, 0.5));
    A = -exp(U(0, ln 16));  D ~ N(0, 1);  resumed slots ~ N(0, 0.1)

Fresh slots are filled with NaN: a fresh sequence must ignore its slot.
Draw order is fixed: x, dt, A, B, C, D, then the slots.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Geometry", "ScanInputs", "make_inputs", "WORKLOADS", "workload"]


@dataclass(frozen=True)
class Geometry:
    n_heads: int
    head_dim: int
    d_state: int
    n_groups: int


NEMOTRON_H = Geometry(n_heads=64, head_dim=64, d_state=128, n_groups=8)


@dataclass
class ScanInputs:
    geom: Geometry
    x: torch.Tensor
    dt: torch.Tensor
    A: torch.Tensor
    B: torch.Tensor
    C: torch.Tensor
    D: torch.Tensor
    state: torch.Tensor
    seq_starts: torch.Tensor
    seq_lens: torch.Tensor
    resume: torch.Tensor
    meta: dict = field(default_factory=dict)

    @property
    def n_tokens(self) -> int:
        return int(self.x.shape[0])

    @property
    def n_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    def tensors(self):
        return dict(x=self.x, dt=self.dt, A=self.A, B=self.B, C=self.C, D=self.D,
                    state=self.state, seq_starts=self.seq_starts,
                    seq_lens=self.seq_lens, resume=self.resume)

    def to(self, device) -> "ScanInputs":
        kw = {k: v.to(device) for k, v in self.tensors().items()}
        return ScanInputs(geom=self.geom, meta=dict(self.meta), **kw)


def make_inputs(geom: Geometry, lens, resume, seed: int, *,
                starts=None, n_tokens=None, a_zero=False, b_zero=False,
                fresh_fill=float("nan")) -> ScanInputs:
    """Draw one batch.

    lens    sequence lengths (tokens are packed back to back unless `starts`
            is given);
    resume  per-sequence flag, nonzero = continue from the slot;
    seed    torch CPU generator seed.
    """
    H, P, N, G = geom.n_heads, geom.head_dim, geom.d_state, geom.n_groups
    lens = [int(v) for v in lens]
    n = len(lens)
    resume = [int(bool(v)) for v in resume]
    assert len(resume) == n
    if starts is None:
        starts, acc = [], 0
        for L in lens:
            starts.append(acc)
            acc += L
        T = acc if n_tokens is None else int(n_tokens)
    else:
        starts = [int(v) for v in starts]
        T = int(n_tokens) if n_tokens is not None else max(
            [s + L for s, L in zip(starts, lens)] + [0])
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn(T, H, P, generator=g)
    dt = torch.nn.functional.softplus(torch.randn(T, H, generator=g) * 0.5 - 2.0)
    A = -torch.exp(torch.rand(H, generator=g) * math.log(16.0))
    B = torch.randn(T, G, N, generator=g) / math.sqrt(N)
    C = torch.randn(T, G, N, generator=g) / math.sqrt(N)
    D = torch.randn(H, generator=g)
    state = torch.randn(n, H, P, N, generator=g) * 0.1
    for i, r in enumerate(resume):
        if not r:
            state[i].fill_(fresh_fill)
    if a_zero:
        A.zero_()
    if b_zero:
        B.zero_()
    return ScanInputs(
        geom=geom, x=x, dt=dt, A=A, B=B, C=C, D=D, state=state,
        seq_starts=torch.tensor(starts, dtype=torch.int32),
        seq_lens=torch.tensor(lens, dtype=torch.int32),
        resume=torch.tensor(resume, dtype=torch.int32),
        meta=dict(seed=int(seed)))


def _alternate(n):
    # Even-indexed sequences start fresh, odd-indexed ones resume.
    return [i % 2 for i in range(n)]


# The workloads the scan is measured and checked on. Each entry gives the
# geometry, the per-sequence lengths and resume flags, and the seed.
WORKLOADS = {
    "tiny": dict(geom=Geometry(4, 16, 32, 2), lens=[37, 5], resume=[0, 1], seed=0,
                 what="2 sequences (fresh x37, resuming x5), 4 heads x 16 x d_state 32, 2 groups"),
    "decode_16x1": dict(geom=NEMOTRON_H, lens=[1] * 16, resume=[1] * 16, seed=1,
                        what="decode step, 16 resuming sequences x 1 token, 64 heads x 64 x 128 state, 8 groups"),
    "prefill_1x4096": dict(geom=NEMOTRON_H, lens=[4096], resume=[0], seed=2,
                           what="prefill, 1 fresh sequence x 4096 tokens, 64 heads x 64 x 128 state, 8 groups"),
    "ragged_12": dict(geom=NEMOTRON_H,
                      lens=[1, 1, 1, 1, 3, 25, 26, 150, 513, 1024, 2048, 4096],
                      resume=_alternate(12), seed=3,
                      what="ragged batch of 12 sequences (T=7889), alternately fresh and resuming"),
    "edge_p96_n100": dict(geom=Geometry(8, 96, 100, 2), lens=[777] * 4, resume=_alternate(4), seed=4,
                          what="8 heads x head_dim 96 x d_state 100, 2 groups, 4 x 777 tokens"),
    "edge_n1024": dict(geom=Geometry(16, 64, 1024, 4), lens=[2048] * 2, resume=_alternate(2), seed=4,
                       what="16 heads x 64 x d_state 1024, 4 groups, 2 x 2048 tokens"),
    "long_4x16384": dict(geom=NEMOTRON_H, lens=[16384] * 4, resume=_alternate(4), seed=4,
                         what="64 heads x 64 x 128 state, 8 groups, 4 sequences x 16384 tokens"),
}


def workload(name: str, **overrides) -> ScanInputs:
    w = dict(WORKLOADS[name])
    w.pop("what")
    w.update(overrides)
    inp = make_inputs(w.pop("geom"), w.pop("lens"), w.pop("resume"), w.pop("seed"), **w)
    inp.meta["workload"] = name
    return inp
