"""The bench's multi-GPU host logic on CPU with two gloo ranks.

The scan shards by sequence with no data-path exchange: each rank scans its
own batch (its own seed) and only the step time is reduced (max over ranks).
Here two gloo ranks run that logic with the CPU oracle standing in for the
per-rank scan."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from state_space_model_ssm_gb300.workloads import WORKLOADS, workload
        w, r, lr = bench.dist_env()
        assert (w, r, lr) == (world, rank, rank)
        inp = workload("tiny", seed=WORKLOADS["tiny"]["seed"] + 1000 * r)
        y, s = oracle.scan_inputs(inp, n_threads=1)
        local_time = 1.0 + rank                       # a stand-in per-rank step time
        t_max = bench.max_over_ranks(local_time, w, torch.device("cpu"))
        bench.barrier(w)
        out[rank] = (t_max, float(inp.x.sum()), float(abs(y[:int(inp.seq_lens.sum())]).sum()))
    finally:
        dist.destroy_process_group()


def test_two_rank_weak_scaling_host_logic():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert set(out.keys()) == {0, 1}
    # both ranks see the slowest rank's time
    assert out[0][0] == out[1][0] == 2.0
    # each rank scanned a different batch (its own seed), no exchange of data
    assert out[0][1] != out[1][1]
    assert out[0][2] != out[1][2]
