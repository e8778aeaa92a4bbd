"""Multi-process host logic of the benchmark's data-parallel replicas (gloo, CPU).

Each rank processes its own batch (weak scaling, no data-path collective); the
only cross-rank steps are the barriers around the timed region and the max
over ranks of the elapsed time.  Run as two CPU processes with gloo.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from synth import Workload, make_inputs


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        wl = Workload("dp", T=4, K=16, H=16, seed=0)
        d = make_inputs(wl, seed=bench.rank_seed(wl.seed, rank))
        elapsed = 1.0 + rank  # rank 1 is the slow one
        bench.barrier()
        m = bench.max_over_ranks(elapsed)
        value = bench.whole_job_value(100.0, world, m)
        out[rank] = (m, value, int(d["x"].astype(np.int64).sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling_host_logic():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in (0, 1):
        m, value, _ = res[rank]
        assert m == 2.0                                  # the slowest rank's time
        assert value == pytest.approx(100.0 * world / 2.0)  # all ranks' units over it
    assert res[0][2] != res[1][2]                        # each replica draws its own batch


def test_single_process_helpers_without_a_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5
    bench.barrier()
    assert bench.whole_job_value(10.0, 1, 2.0) == 5.0
    assert bench.rank_seed(0, 0) != bench.rank_seed(0, 1)


def test_l2_flush_modes_on_cpu(monkeypatch):
    # the flush writes its own buffer; "clean" also reads a second buffer (into a scalar), "write" does not
    monkeypatch.setattr(bench, "FLUSH_BYTES", 1 << 16)
    f = bench.L2Flush("cpu", "clean")
    f.fill_(3.0)
    assert torch.all(f.buf == 3.0) and f.buf.numel() == (1 << 16) // 4
    assert float(f.sink) == float(f.src.numel())
    g = bench.L2Flush("cpu", "write")
    g.fill_(2.0)
    assert g.src is None and torch.all(g.buf == 2.0)
    assert set(bench.L2_FLUSH_NOTE) == {"clean", "write"}
