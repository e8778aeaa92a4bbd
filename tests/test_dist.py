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


def test_reference_arm_prints_the_gpu_arms_config():
    """Both arms describe the workload with the same dict, so a line-by-line comparison of their
    `config` matches (the plan the GPU arm tuned is reported beside it, not inside)."""
    import argparse
    from synth import workload
    args = argparse.Namespace(config="tiny", tokens=0, dtype="bf16", steps=1, warmup=3, ref_seconds=0.5,
                              l2_flush="clean")
    line = bench.run_reference(args)
    assert line["impl"] == "reference"
    assert line["config"] == bench.bench_config(workload("tiny"), "bf16", 1, "clean")
    assert "plan" not in line["config"]


def test_kernel_roofline_picks_the_slower_resource():
    from synth import workload
    peaks = {"bf16_tflops": 1000.0, "hbm_gbs": 5000.0}
    wl = workload("llama3_8b_oproj")
    # 4096^3 prefill: FLOPs dominate; achieved = FLOPs / time
    bound, ach, unit, frac = bench.kernel_roofline("gemm_fused", wl, 4096, 0.2, peaks)
    assert (bound, unit) == ("tensor", "TFLOP/s")
    assert ach == pytest.approx(2 * 4096 ** 3 / 0.2e-3 / 1e12)
    assert frac == pytest.approx(2 * 4096 ** 3 / 1e15 / 0.2e-3)
    # 8 tokens of a 70B o_proj: the weight bytes dominate
    wd = workload("llama70b_oproj_decode")
    bound, ach, unit, frac = bench.kernel_roofline("gemm_splitk", wd, 8, 0.03, peaks)
    nbytes = 2 * 8192 * 8192 + 2 * 8 * 8192
    assert (bound, unit) == ("hbm", "GB/s")
    assert ach == pytest.approx(nbytes / 0.03e-3 / 1e9)
    assert frac == pytest.approx(nbytes / 5e12 / 0.03e-3)
