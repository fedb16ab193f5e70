"""Host-side logic of the N-GPU benchmark, run as two gloo ranks on the CPU:
per-rank workloads differ only in their seed, the timing is the max over
ranks, and the reported rate counts every rank's tokens."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = bench.rank_workload(W.WORKLOADS[1], rank)
    lens = W.seq_lens(w)
    c, _ = W.sequence(w, 0, length=8)
    t_local = 10.0 + 5.0 * rank                       # ms: rank 1 is the slower one
    t_max = bench.max_over_ranks(t_local, world)
    rate = bench.job_throughput(w.B * w.s_q, world, t_max, steps=4)
    gathered = [None] * world
    dist.all_gather_object(gathered, (w.seed, w.B, w.H, lens.tolist(), c[0, :4].tolist()))
    if rank == 0:
        out.put((gathered, t_max, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_by_sequence_and_take_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered, t_max, rate = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (s0, B0, H0, l0, c0), (s1, B1, H1, l1, c1) = gathered
    assert (B0, H0) == (B1, H1)               # same shapes on every rank
    assert s0 != s1 and c0 != c1              # independent data per rank
    assert t_max == pytest.approx(15.0)       # slowest rank
    # 16 tokens per rank-step, 2 ranks, 4 steps in 15 ms
    assert rate == pytest.approx(16 * 2 * 4 / 0.015)
