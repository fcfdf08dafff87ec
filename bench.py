#!/usr/bin/env python3
"""Benchmark of the Mamba2 selective-state scan on GB300 (libssmscan).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one scan call over the 1 x 4096-token prefill workload at
Nemotron-H geometry (64 heads x 64 x 128 state, 8 groups, fp32): state
load, chunk staging, discretisation, state update, y readout and state store,
all in the prefill kernel.  The same run also times the 16 x 1 decode step
(300 steps over rotating slot sets) and reports it under "decode", and the
chunked matrix form on the TF32 tensor cores (ssm_scan_ssd, chunk 128) on the
same prefill input under "ssd" (a lower-precision variant, not the headline).

Prints one JSON line (rank 0).  Under torchrun every rank scans its own
batch (weak scaling, no collective on the data path); the step time is the
maximum over ranks.  `--impl reference` times the CPU oracle instead, on the
host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from state_space_model_ssm_gb300.workloads import WORKLOADS, workload  # noqa: E402

METRIC = "scan tokens/s (1×4096 prefill), decode µs (16×1); % of HBM/FP32 roofline"
# gllm PR 90, "Results": 1 x 4096 prefill in 3.5 ms and 16 x 1 decode in 32 us on an
# RTX PRO 6000 (sm_120, 300 W cap); another machine's figures, quoted as context.
PAGE_PREFILL_MS = 3.5
PAGE_DECODE_US = 32.0
FP32_LANES_PER_SM = 128
TF32_PER_BF16 = 1.1 / 2.25    # nominal dense TF32 / BF16 tensor rate
L2_FLUSH_BYTES = 256 << 20
DECODE_STEPS = 300
DECODE_SLOT_SETS = 8          # 8 x 32 MiB of slots rotate, 2x the 129 MB L2
KERNEL_SOURCES = {
    "prefill_kernel": ["state_space_model_ssm_gb300/csrc/prefill_scaled.cu",
                       "state_space_model_ssm_gb300/csrc/segments.cu",
                       "state_space_model_ssm_gb300/csrc/scan_common.cuh"],
    "decode_kernel": ["state_space_model_ssm_gb300/csrc/decode.cu",
                      "state_space_model_ssm_gb300/csrc/scan_common.cuh"],
    "ssd_output_kernel": ["state_space_model_ssm_gb300/csrc/ssd_tc.cu",
                          "state_space_model_ssm_gb300/csrc/ssd_common.cuh",
                          "state_space_model_ssm_gb300/csrc/scan_common.cuh"],
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ssd", action="store_true")
    ap.add_argument("--no-next", action="store_true")
    ap.add_argument("--decode-launches", type=int, default=0,
                    help="run only this many 16x1 decode steps as plain launches (no graph) on the "
                         "rotating slot sets and exit: the command an ncu counter capture runs")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}, "fallback"


def source_hash(kernel: str) -> str:
    h = hashlib.sha1()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def ncu_traffic(kernel: str, workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since that capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = source_hash(kernel)
    for line in open(path):
        f = line.split()
        if len(f) >= 4 and f[0] == workload_name and f[1] == kernel:
            kv = dict(x.split("=", 1) for x in f[2:] if "=" in x)
            if kv.get("src") == want:
                return int(kv["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sms.append(float(f[0]))
                maxs.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sms:
            return None
        loaded = [s for s in sms if s > 0.5 * max(sms)] or sms
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(maxs),
                "reasons": sorted(reasons), "samples": len(sms)}


def event_pair():
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def launch_event_sets(n_sets, n_launches, stream):
    """n_sets lists of 2 * n_launches timing events for the library to record
    around a call's kernel launches (each recorded once here so that it exists)."""
    sets = []
    for _ in range(n_sets):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_launches)]
        for e in evs:
            e.record(stream)
        sets.append(evs)
    torch.cuda.synchronize()
    return sets


def launch_ms(sets):
    """Mean device ms of each launch over the recorded sets."""
    n = len(sets[0]) // 2
    return [sum(s[2 * k].elapsed_time(s[2 * k + 1]) for s in sets) / len(sets) for k in range(n)]


# ---------------------------------------------------------------- our arm

def prefill_workspace(inp, dev):
    """The workspace ssm_scan_ws asks for (time segments of the long sequence)."""
    from state_space_model_ssm_gb300 import binding as bd
    g = inp.geom
    nbytes = bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state, g.n_groups)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)


def prefill_launches_per_step(inp):
    """Kernels one prefill call launches: plan, state pass, combine and full pass
    with time segments, else the one prefill kernel."""
    from state_space_model_ssm_gb300 import binding as bd
    g = inp.geom
    segs = bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state, g.n_groups) > 0
    return 4 if segs else 1


def run_prefill(args, world, rank, dev):
    from state_space_model_ssm_gb300 import binding as bd

    inp = workload("prefill_1x4096", seed=WORKLOADS["prefill_1x4096"]["seed"] + 1000 * rank)
    d = inp.to(dev)
    state = d.state.clone()
    y = torch.empty_like(d.x)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ws = prefill_workspace(inp, dev)

    # the library records these around its launches (plan, state pass, combine, full pass)
    n_launch = prefill_launches_per_step(inp)
    kev = launch_event_sets(args.steps, n_launch, stream)

    def step(events=None):
        bd.ssm_scan(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume, y=y,
                    workspace=ws, launch_events=events)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    # The step as a caller runs it: no events between the library's launches
    # (recording them costs a few microseconds per launch boundary).
    evs = [event_pair() for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    for e0, e1 in evs:
        flush.zero_()                 # L2 flushed between timed steps
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    times_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    step_ms = sum(times_ms) / len(times_ms)
    # The same K steps again with the library recording events around each of
    # its launches: the per-kernel times of the rooflines.
    for ke in kev:
        flush.zero_()
        step(ke)
    torch.cuda.synchronize(dev)
    return inp, d, step_ms, times_ms, launch_ms(kev)


def run_prefill_fp32_state(args, dev, inp, d):
    """The same step with the segments' state pass in the sequential kernel
    (SEGMENT_STATE_FP32) instead of the tensor cores: mean ms per step."""
    from state_space_model_ssm_gb300 import binding as bd
    t = bd.Tuning()
    t.segment_state = bd.SEGMENT_STATE_FP32
    ws = prefill_workspace(inp, dev)
    state = d.state.clone()
    y = torch.empty_like(d.x)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    return _timed(lambda: bd.ssm_scan(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens,
                                      d.resume, y=y, workspace=ws, tuning=t),
                  max(5, args.steps // 2), flush)


def run_prefill_e2e(args, dev, inp):
    """Same metric through the public call with host buffers: every step copies
    the inputs from pinned host memory and reads y and the state back.

    Pipelined as a serving loop would run it: three streams (copies in, scan,
    copies out) and two device buffer sets, so the inputs of step i+1 and the
    results of step i-1 move while step i computes; every step's copies are
    inside the timed region.  (Splitting the copies in over two streams was
    slower: together with the copies out they already fill the host link.)
    Also returns the same steps run serially on one stream."""
    from state_space_model_ssm_gb300 import binding as bd

    host_in = {k: v.pin_memory() for k, v in inp.tensors().items()}
    sets = [({k: torch.empty_like(v, device=dev) for k, v in inp.tensors().items()},
             torch.empty(inp.x.shape, dtype=torch.float32, device=dev)) for _ in range(2)]
    y_host = torch.empty(inp.x.shape, dtype=torch.float32).pin_memory()
    s_host = torch.empty(inp.state.shape, dtype=torch.float32).pin_memory()
    in_keys = ["x", "dt", "A", "B", "C", "D", "seq_starts", "seq_lens", "resume"]
    if int(inp.resume.sum()) > 0:
        in_keys.append("state")
    h2d = sum(host_in[k].numel() * host_in[k].element_size() for k in in_keys)
    d2h = inp.x.numel() * 4 + inp.state.numel() * 4
    ws = prefill_workspace(inp, dev)
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
    for k in ev:                                   # every event exists before its first wait
        for e in ev[k]:
            e.record(torch.cuda.current_stream(dev))

    def scan(dbuf, y, stream):
        bd.ssm_scan(dbuf["state"], dbuf["x"], dbuf["dt"], dbuf["A"], dbuf["B"], dbuf["C"], dbuf["D"],
                    dbuf["seq_starts"], dbuf["seq_lens"], dbuf["resume"], y=y, workspace=ws, stream=stream)

    def step(i):
        b = i & 1
        dbuf, y = sets[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev["comp"][b])             # set b free: the scan of step i-2 is done
            for k in in_keys:
                dbuf[k].copy_(host_in[k], non_blocking=True)
            ev["in"][b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev["in"][b])
            s_comp.wait_event(ev["out"][b])            # y and the state of set b read back (step i-2)
            scan(dbuf, y, s_comp)
            ev["comp"][b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][b])
            y_host.copy_(y, non_blocking=True)
            s_host.copy_(dbuf["state"], non_blocking=True)
            ev["out"][b].record(s_out)

    def serial_step():
        dbuf, y = sets[0]
        cur = torch.cuda.current_stream(dev)
        for k in in_keys:
            dbuf[k].copy_(host_in[k], non_blocking=True)
        scan(dbuf, y, cur)
        y_host.copy_(y, non_blocking=True)
        s_host.copy_(dbuf["state"], non_blocking=True)

    n = max(3, min(args.steps, 20))
    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = event_pair()
    e0.record(s_in)
    for i in range(n):
        step(i)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / n

    for _ in range(3):
        serial_step()
    torch.cuda.synchronize(dev)
    f0, f1 = event_pair()
    f0.record()
    for _ in range(n):
        serial_step()
    f1.record()
    torch.cuda.synchronize(dev)
    return ms, h2d, d2h, f0.elapsed_time(f1) / n


def run_decode(dev, rank):
    """16 x 1 decode at Nemotron-H geometry, 300 steps captured in a CUDA graph
    (so host launch cost is not timed): cold = each step on the next of 8
    rotating 16-slot sets (256 MiB of slots, twice the L2); warm = every step on
    the same slots.  Per-step time = graph replay time / 300."""
    from state_space_model_ssm_gb300 import binding as bd

    base = workload("decode_16x1", seed=WORKLOADS["decode_16x1"]["seed"] + 1000 * rank)
    d = base.to(dev)
    sets = [d.state.clone() for _ in range(DECODE_SLOT_SETS)]
    y = torch.empty_like(d.x)
    stream = torch.cuda.current_stream(dev)

    def step(state):
        bd.ssm_scan(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume, y=y)

    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(10):
            step(sets[i % DECODE_SLOT_SETS])
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)

    def graph_us(rotate):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(DECODE_STEPS):
                step(sets[i % DECODE_SLOT_SETS] if rotate else sets[0])
        g.replay()
        torch.cuda.synchronize(dev)
        best = float("inf")
        for _ in range(5):
            e0, e1 = event_pair()
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            best = min(best, e0.elapsed_time(e1) * 1e3 / DECODE_STEPS)
        return best

    cold = graph_us(True)
    warm = graph_us(False)
    return dict(cold_us=cold, warm_graph_us=warm)


def decode_launches(n):
    """n decode steps (16 x 1, Nemotron-H geometry) as separate launches, each on
    the next of the rotating slot sets, then exit.  Under ncu with the L2 left
    alone between kernels, a launch's DRAM write counter shows the write-back
    of earlier launches' slots, which leave L2 as later launches stream through
    it, so the average over consecutive launches is the traffic per step."""
    from state_space_model_ssm_gb300 import binding as bd
    from state_space_model_ssm_gb300 import build as _build
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    base = workload("decode_16x1")
    d = base.to(dev)
    sets = [d.state.clone() for _ in range(DECODE_SLOT_SETS)]
    y = torch.empty_like(d.x)
    for i in range(n):
        bd.ssm_scan(sets[i % DECODE_SLOT_SETS], d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens,
                    d.resume, y=y)
    torch.cuda.synchronize(dev)
    print(json.dumps({"decode_launches": n, "slot_sets": DECODE_SLOT_SETS}))


def run_ssd(args, dev, inp, d, chunk=128):
    """ssm_scan_ssd (the chunked form on the TF32 tensor cores) on the same
    prefill input, timed like the prefill step (L2 flushed between steps)."""
    from state_space_model_ssm_gb300 import binding as bd
    g = inp.geom
    nbytes = bd.ssd_workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state,
                                    g.n_groups, chunk)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    state = d.state.clone()
    y = torch.empty_like(d.x)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    kev = launch_event_sets(args.steps, 4, stream)     # plan, chunk states, state pass, output

    def step(events=None):
        bd.ssm_scan_ssd(state, d.x, d.dt, d.A, d.B, d.C, d.D, d.seq_starts, d.seq_lens, d.resume,
                        y=y, chunk=chunk, workspace=ws, launch_events=events)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    evs = [event_pair() for _ in range(args.steps)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    times = [e0.elapsed_time(e1) for e0, e1 in evs]
    for ke in kev:                    # per-launch times from a second set of steps
        flush.zero_()
        step(ke)
    torch.cuda.synchronize(dev)
    return sum(times) / len(times), nbytes, launch_ms(kev)


def ssd_output_flops(inp, chunk):
    """Dense FLOPs of the output kernel alone: per chunk, G x 2 Q^2 N (C B^T)
    plus H x (2 Q^2 P (masked product with x) + 2 Q N P (C S_in^T))."""
    g = inp.geom
    H, P, N, G = g.n_heads, g.head_dim, g.d_state, g.n_groups
    chunks = sum((int(L) + chunk - 1) // chunk for L in inp.seq_lens.tolist())
    Q = chunk
    return chunks * (G * 2 * Q * Q * N + H * (2 * Q * Q * P + 2 * Q * N * P))


def ssd_algorithmic_flops(inp, chunk):
    """Dense FLOPs of the chunked form per call: per chunk, G groups x 2 Q^2 N
    (C B^T) plus H heads x (2 Q^2 P (masked product with x) + 2 Q N P (C S_in^T)
    + 2 Q N P (x^T B)), with Q = chunk (the causal half is not subtracted)."""
    g = inp.geom
    H, P, N, G = g.n_heads, g.head_dim, g.d_state, g.n_groups
    chunks = sum((int(L) + chunk - 1) // chunk for L in inp.seq_lens.tolist())
    Q = chunk
    return chunks * (G * 2 * Q * Q * N + H * (2 * Q * Q * P + 4 * Q * N * P))


def _timed(fn, steps, flush=None, warmup=3):
    """Mean ms of fn() over `steps` runs, CUDA events on the current stream,
    L2 flushed before each run when `flush` (a large tensor) is given."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        if flush is not None:
            flush.zero_()
        fn()
    torch.cuda.synchronize()
    evs = [event_pair() for _ in range(steps)]
    for e0, e1 in evs:
        if flush is not None:
            flush.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs) / steps


def run_next_rows(dev, inp, d, peaks, steps=10):
    """The steps around the scan, each timed on its own workload with its HBM
    roofline (bytes moved per call / time / measured copy bandwidth)."""
    from state_space_model_ssm_gb300 import binding as bd
    hbm = peaks["hbm_gbs"] * 1e9
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    g = torch.Generator().manual_seed(77)
    H, P, N = inp.geom.n_heads, inp.geom.head_dim, inp.geom.d_state
    T = inp.n_tokens
    ws = prefill_workspace(inp, dev)
    state = d.state.clone()
    y = torch.empty_like(d.x)
    out = {}

    def prefill(dt=None, **kw):
        dt = d.dt if dt is None else dt
        return lambda: bd.ssm_scan(state, d.x, dt, d.A, d.B, d.C, d.D, d.seq_starts,
                                   d.seq_lens, d.resume, y=y, workspace=ws, **kw)
    base = _timed(prefill(), steps, flush)

    # 1. fused dt: raw dt + bias with softplus inside the kernels
    raw = (torch.randn(d.dt.shape, generator=g) * 0.5 - 2.0).to(dev)
    bias = (torch.rand(H, generator=g) - 0.5).to(dev)
    fused = _timed(prefill(dt=raw, dt_bias=bias, dt_softplus=True), steps, flush)
    # the plain scan on the same steps, discretised beforehand (the rescaled
    # kernel's work depends on the steps through its re-anchoring)
    v = raw + bias[None, :]
    same = _timed(prefill(dt=torch.where(v > 20.0, v, torch.log1p(torch.exp(v)))), steps, flush)
    out["fused_dt"] = {"workload": "prefill_1x4096 with raw dt, dt_bias and softplus",
                       "ms": fused, "ms_plain": same, "overhead_pct": 100.0 * (fused - same) / same}

    # 2. gated RMSNorm of y: at this shape (blocks of one head) the full pass
    # applies it itself, so the step adds z read and the gated output written
    z = torch.randn((T, H, P), generator=g).to(dev)
    wn = (torch.rand(P, generator=g) + 0.5).to(dev)
    gated = torch.empty_like(d.x)
    with_norm = _timed(prefill(gate_z=z, norm_weight=wn, norm_eps=1e-5, gated_y=gated), steps, flush)
    nbytes = 2 * T * H * P * 4
    extra = max(with_norm - base, 1e-6)
    out["gated_norm"] = {"workload": "prefill_1x4096, RMSNorm(y) w silu(z) per (token, head) row",
                         "where": "fused into the full pass (consumer warps, from the y tile)",
                         "ms": with_norm, "ms_plain": base, "ms_added": extra,
                         "overhead_pct": 100.0 * extra / base, "bytes_added": nbytes,
                         "roofline": {"bound": "hbm", "achieved": nbytes / (extra * 1e-3) / 1e9,
                                      "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                      "frac": nbytes / (extra * 1e-3) / hbm,
                                      "basis": "bytes the gated output adds (z read, gated y written) "
                                               "over the step time it adds"}}

    # 3. state snapshots: a 16 x 4-token verify step at Nemotron-H geometry
    from state_space_model_ssm_gb300.workloads import Geometry, make_inputs
    vin = make_inputs(Geometry(64, 64, 128, 8), [4] * 16, [1] * 16, seed=78)
    vd = vin.to(dev)
    vstate = vd.state.clone()
    vy = torch.empty_like(vd.x)
    snaps = torch.empty((vin.n_tokens, 64, 64, 128), device=dev)
    verify = _timed(lambda: bd.ssm_scan(vstate, vd.x, vd.dt, vd.A, vd.B, vd.C, vd.D, vd.seq_starts,
                                        vd.seq_lens, vd.resume, y=vy, snapshots=snaps), steps, flush)
    slot = 64 * 64 * 128 * 4
    sbytes = 2 * 16 * slot + vin.n_tokens * slot
    out["state_snapshots"] = {"workload": "16 resuming sequences x 4 tokens, state after every token",
                              "ms": verify, "bytes": sbytes,
                              "roofline": {"bound": "hbm", "achieved": sbytes / (verify * 1e-3) / 1e9,
                                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                           "frac": sbytes / (verify * 1e-3) / hbm}}

    # 4. conv1d + SiLU: 1 x 4096 tokens over Nemotron-H's conv width 6144, k = 4
    Cc, K = 6144, 4
    xc = torch.randn((T, Cc), generator=g).to(dev)
    wc = (torch.randn((Cc, K), generator=g) * 0.5).to(dev)
    bc = (torch.randn((Cc,), generator=g) * 0.1).to(dev)
    cst = torch.randn((1, Cc, K - 1), generator=g).to(dev)
    oc = torch.empty_like(xc)
    one = torch.ones(1, dtype=torch.int32, device=dev)
    conv = _timed(lambda: bd.ssm_conv1d(xc, wc, cst, d.seq_starts, d.seq_lens, one, out=oc, bias=bc),
                  steps, flush)
    cbytes = 2 * T * Cc * 4 + Cc * (K + 1) * 4 + 2 * Cc * (K - 1) * 4
    out["conv1d"] = {"workload": "1 x 4096 tokens x 6144 channels, k = 4, resuming",
                     "ms": conv, "bytes": cbytes,
                     "roofline": {"bound": "hbm", "achieved": cbytes / (conv * 1e-3) / 1e9,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": cbytes / (conv * 1e-3) / hbm}}
    return out


def segment_units(inp):
    """(segments, segment length) of the library's automatic plan for a single
    sequence: its workspace holds one state per unit plus a few small tables."""
    from state_space_model_ssm_gb300 import binding as bd
    g = inp.geom
    slot = 4 * g.n_heads * g.head_dim * g.d_state
    ws = bd.workspace_bytes(inp.n_seqs, inp.n_tokens, g.n_heads, g.head_dim, g.d_state, g.n_groups)
    units = ws // slot - inp.n_seqs                # max_units = n_seqs + ceil(T / seg)
    T = int(inp.seq_lens.sum())
    seg = -(-T // units)
    seg = -(-seg // 16) * 16                       # a multiple of the prefill chunk
    return -(-T // seg), seg


def state_pass_report(inp, ms, peaks, peaks_src, fp32_step_ms, step_ms):
    """Roofline of the tensor-core state pass: every segment but the last, each
    L = sum_s w_s x_s B_s^T over its tokens (one multiply-add per token and state
    element), run as three TF32 products (hi*hi, hi*lo, lo*hi) with head_dim
    padded to a multiple of 32 and d_state to 128."""
    g = inp.geom
    H, P, N, G = g.n_heads, g.head_dim, g.d_state, g.n_groups
    units, seg = segment_units(inp)
    Ts = (units - 1) * seg
    alg_flops = 2 * Ts * H * P * N
    tc_flops = 3 * 2 * Ts * H * (-(-P // 32) * 32) * 128
    nbytes = 4 * (Ts * H * P + Ts * G * N + Ts * H + (units - 1) * H * P * N)
    tf32_peak = peaks["bf16_tflops"] * 1e12 * 1.1 / 2.25
    s = ms * 1e-3
    return {"what": "segment state pass on tcgen05 (3 split-TF32 products, fp32 accumulation)",
            "ms": ms, "tokens": Ts, "segments": units, "segment_tokens": seg,
            "roofline": {"bound": "hbm", "achieved": nbytes / s / 1e9, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": nbytes / s / 1e9 / peaks["hbm_gbs"], "peak_src": peaks_src,
                         "algorithmic": f"{nbytes} bytes per launch (x, B and dt of {Ts} tokens; the states out)",
                         "tensor_frac": tc_flops / s / tf32_peak,
                         "tensor_basis": f"{tc_flops} executed TF32 FLOPs vs measured bf16 burst x 1.1/2.25",
                         "algorithmic_tflops": alg_flops / s / 1e12},
            "step_ms_with_fp32_state_pass": fp32_step_ms,
            "step_speedup": fp32_step_ms / step_ms}


def prefill_algorithmic(inp):
    T = int(inp.seq_lens.sum())
    H, P, N, G = inp.geom.n_heads, inp.geom.head_dim, inp.geom.d_state, inp.geom.n_groups
    updates = T * H * P * N
    fp32_ops = 3 * updates                      # FMUL dt*x*B, FFMA decay, FFMA C-dot
    n = inp.n_seqs
    state_in = 4 * n * H * P * N * int(inp.resume.sum() > 0)
    bytes_ = 4 * (2 * T * H * P + 2 * T * G * N + T * H + 2 * H) + state_in + 4 * n * H * P * N
    return updates, fp32_ops, bytes_


def decode_algorithmic(inp):
    H, P, N, G = inp.geom.n_heads, inp.geom.head_dim, inp.geom.d_state, inp.geom.n_groups
    n = inp.n_seqs
    T = int(inp.seq_lens.sum())
    state_bytes = 2 * 4 * n * H * P * N
    other = 4 * (2 * T * H * P + 2 * T * G * N + T * H + 2 * H) + 3 * 4 * n
    return state_bytes, state_bytes + other


def cpu_baseline_prefill(inp, budget_s=20.0):
    """The oracle, as it stands, on the host cores: the full 1 x 4096 workload
    once with every core, then on one core for a head sample."""
    import oracle
    cores = os.cpu_count() or 1
    t = time.perf_counter()
    oracle.scan_inputs(inp, n_threads=cores)
    wall = time.perf_counter() - t
    T = int(inp.seq_lens.sum())
    heads = list(range(0, inp.geom.n_heads, 8))
    t = time.perf_counter()
    oracle.scan_inputs(inp, n_threads=1, heads=heads)
    wall1 = (time.perf_counter() - t) * inp.geom.n_heads / len(heads)
    return {"value": T / wall, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"full 1x{T} prefill workload, one run on {cores} threads (fp64 C oracle)",
            "single_core_value": T / wall1,
            "single_core_sample": f"{len(heads)} of {inp.geom.n_heads} heads on 1 thread, scaled"}


def ours(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    from state_space_model_ssm_gb300 import build as _build
    if rank == 0:
        _build.build()
    barrier(world)
    from state_space_model_ssm_gb300 import binding as bd
    bd.load()

    peaks, peaks_src = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    sampler = ClockSampler(local)
    sampler.start()
    inp, d, step_ms, times, kms = run_prefill(args, world, rank, dev)
    clocks = sampler.stop()
    step_ms_max = max_over_ranks(step_ms, world, dev)

    T = int(inp.seq_lens.sum())
    updates, fp32_ops, alg_bytes = prefill_algorithmic(inp)
    value = world * T / (step_ms_max * 1e-3)
    sm_max = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
    peak_ops = sms * FP32_LANES_PER_SM * sm_max * 1e6
    full_ms = kms[-1]                              # the full pass: the step's last launch
    achieved = fp32_ops / (full_ms * 1e-3)
    traffic = ncu_traffic("prefill_kernel", "prefill_1x4096")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": value / (world * 4096 / (PAGE_PREFILL_MS * 1e-3)),
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "prefill_1x4096", "what": WORKLOADS["prefill_1x4096"]["what"],
                   "n_seqs": 1, "tokens_per_rank": T, "geometry": "H=64 P=64 N=128 G=8",
                   "l2": "flushed between timed steps (256 MiB write)",
                   "path": "ssm_scan_ws: rescaled prefill kernel, time segments (workspace %.1f MiB)"
                           % (bd.workspace_bytes(1, T, 64, 64, 128, 8) / 2**20),
                   "parallelism": f"dp{world} (independent sequences per GPU)",
                   "vs_baseline_ref": "gllm PR 90: 3.5 ms on RTX PRO 6000 (context, another machine)"},
        "roofline": {"bound": "alu", "achieved": achieved / 1e12, "peak": peak_ops / 1e12,
                     "unit": "T fp32-ops/s", "frac": achieved / peak_ops,
                     "traffic": traffic,
                     "peak_basis": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x {sm_max:.0f} MHz (max clock)",
                     "algorithmic": f"{fp32_ops} FP32 ops per launch (3 per element-update)",
                     "hbm_frac": (alg_bytes / (full_ms * 1e-3)) / (peaks["hbm_gbs"] * 1e9),
                     "hbm_peak_src": peaks_src,
                     "timing": ("the full-pass kernel alone: CUDA events the library records around "
                                "its launch on the call's stream, mean over a second set of K steps "
                                "(the headline steps run without events between launches)"),
                     "kernel_ms": full_ms,
                     "step_frac": fp32_ops / (step_ms * 1e-3) / peak_ops},
        "gpu_launches": args.steps * prefill_launches_per_step(inp),
        "clocks": clocks,
        "step_ms_min": min(times),
        "step_ms_median": statistics.median(times),
    }
    if clocks and clocks.get("sm_mhz"):
        line["roofline"]["frac_at_sampled_clock"] = achieved / (sms * FP32_LANES_PER_SM * clocks["sm_mhz"] * 1e6)
    if len(kms) == 4:
        line["launches_ms"] = {"segment_plan": kms[0], "state_pass": kms[1], "combine": kms[2],
                               "full_pass": kms[3]}
        line["state_pass"] = state_pass_report(inp, kms[1], peaks, peaks_src,
                                               run_prefill_fp32_state(args, dev, inp, d), step_ms)

    if not args.no_e2e:
        e2e_ms, h2d, d2h, serial_ms = run_prefill_e2e(args, dev, inp)
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        line["e2e"] = {"value": world * T / (e2e_ms * 1e-3), "unit": "tokens/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e2e_ms,
                       "pipeline": ("copies in of step i+1 and out of step i-1 overlap the scan of step i "
                                    "(three streams, two device buffer sets); every copy in the timed region"),
                       "serial_ms_per_step": serial_ms,
                       "serial_value": world * T / (serial_ms * 1e-3)}
    if not args.no_decode:
        dec = run_decode(dev, rank)
        dinp = workload("decode_16x1")
        sbytes, dbytes = decode_algorithmic(dinp)
        cold_s = dec["cold_us"] * 1e-6
        line["decode"] = {
            "us_per_step": dec["cold_us"],
            "what": ("16 resuming sequences x 1 token; 300 steps replayed from a CUDA graph, "
                     "each on the next of 8 rotating slot sets (256 MiB, cold L2)"),
            "us_per_step_warm_graph": dec["warm_graph_us"],
            "roofline": {"bound": "hbm", "achieved": dbytes / cold_s / 1e9,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": dbytes / cold_s / 1e9 / peaks["hbm_gbs"],
                         "state_frac": sbytes / cold_s / 1e9 / peaks["hbm_gbs"],
                         "traffic": ncu_traffic("decode_kernel", "decode_16x1"),
                         "peak_src": peaks_src,
                         "timing": "graph replay / 300 (includes the gaps between kernels)",
                         "algorithmic": f"{dbytes} bytes per launch ({sbytes} of state)"},
            "vs_page": PAGE_DECODE_US / dec["cold_us"],
        }
    if not args.no_ssd:
        ssd_ms, ssd_ws, ssd_kms = run_ssd(args, dev, inp, d)
        flops = ssd_algorithmic_flops(inp, 128)
        out_flops = ssd_output_flops(inp, 128)
        tf32_peak = peaks["bf16_tflops"] * TF32_PER_BF16
        line["ssd"] = {
            "what": ("ssm_scan_ssd: chunked matrix form, chunk 128, TF32 operands (rounded to nearest), "
                     "fp32 accumulation and fp32 state pass; parity bound 5e-3 (1 + |ref|)"),
            "ms_per_step": ssd_ms,
            "value": T / (ssd_ms * 1e-3),
            "unit": "tokens/s",
            "dtype": "tf32",
            "workspace_mib": ssd_ws / 2**20,
            "launches_per_step": 4,
            "roofline": {"bound": "tensor", "achieved": flops / (ssd_ms * 1e-3) / 1e12,
                         "peak": tf32_peak, "unit": "TFLOP/s",
                         "frac": flops / (ssd_ms * 1e-3) / 1e12 / tf32_peak,
                         "peak_basis": "measured bf16 burst x 1.1/2.25 (nominal dense TF32/BF16)",
                         "algorithmic": f"{flops} dense FLOPs per call",
                         "hbm_frac": (alg_bytes / (ssd_ms * 1e-3)) / (peaks["hbm_gbs"] * 1e9),
                         "timing": "whole call (plan, chunk states, state pass, output)",
                         "traffic": ncu_traffic("ssd_output_kernel", "prefill_1x4096"),
                         "traffic_kernel": "the output kernel (tcgen05), DRAM bytes per launch"},
            "launches_ms": {"segment_plan": ssd_kms[0], "chunk_state": ssd_kms[1], "state_pass": ssd_kms[2],
                            "output": ssd_kms[3]},
            "output_kernel_roofline": {
                "bound": "tensor", "achieved": out_flops / (ssd_kms[3] * 1e-3) / 1e12, "peak": tf32_peak,
                "unit": "TFLOP/s", "frac": out_flops / (ssd_kms[3] * 1e-3) / 1e12 / tf32_peak,
                "algorithmic": f"{out_flops} dense FLOPs per launch",
                "timing": "CUDA events the library records around the output kernel's launch"},
        }
    if not args.no_next:
        line["next_rows"] = run_next_rows(dev, inp, d, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(inp)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------- reference arm

def reference(args):
    """The CPU oracle as it stands, on the host cores, on a bounded sample of
    the 1 x 4096 prefill workload: each step runs the oracle on a subset of
    heads sized so the whole run stays within about two minutes."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = workload("prefill_1x4096")
    H = inp.geom.n_heads
    cores = os.cpu_count() or 1
    t = time.perf_counter()
    oracle.scan_inputs(inp, n_threads=cores, heads=[0, 1, 2, 3])
    per_head = (time.perf_counter() - t) / 4
    total_steps = max(1, args.steps + args.warmup)
    heads_per_step = int(max(1, min(H, 120.0 / total_steps / max(per_head, 1e-6))))
    heads = list(range(heads_per_step))
    for _ in range(args.warmup):
        oracle.scan_inputs(inp, n_threads=cores, heads=heads)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan_inputs(inp, n_threads=cores, heads=heads)
    wall = (time.perf_counter() - t) / max(1, args.steps)
    T = int(inp.seq_lens.sum())
    value = T * (heads_per_step / H) / wall
    sample = (f"{heads_per_step} of {H} heads of the 1x{T} prefill per step "
              f"(tokens/s scaled by the head fraction), fp64 C oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wall * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill_1x4096", "what": WORKLOADS["prefill_1x4096"]["what"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference(args)
    elif args.decode_launches > 0:
        decode_launches(args.decode_launches)
    else:
        ours(args)


if __name__ == "__main__":
    main()
