"""The TPSP region's entry point on one GPU (one rank), through the C ABI.

With P = 1 the ReduceScatter and the AllGather are the identity, so the
region must give the undivided region: every element against the fp64
oracle, and bit for bit the PIPELINED path with the same tile width and
chunk (the same GEMM arithmetic per row, the same add + norm kernel).  The
multi-rank schedule itself is covered on CPU (tests/test_tp_region.py).
"""
import numpy as np
import pytest

import oracle
from synth import Workload, make_inputs

from .gpu_util import Run, dev_bf16, host_bits, plan
from .parity import compare

pytestmark = pytest.mark.gpu

fln = pytest.importorskip("decoder_layer_projection_gb300")

CASES = [
    (Workload("tp1_ragged", T=700, K=320, H=640, eps=1e-5, r_sigma=2.0, seed=61), 256),
    (Workload("tp1_small", T=130, K=200, H=264, eps=1e-6, seed=62), 0),
    (Workload("tp1_gemma", T=257, K=448, H=3584, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=63), 128),
    (Workload("tp1_one_token", T=1, K=64, H=2048, eps=1e-5, r_sigma=2.0, seed=64), 0),
    (Workload("tp1_four_slots", T=1000, K=128, H=512, eps=1e-5, r_sigma=2.0, seed=65), 100),
]


@pytest.fixture(scope="module")
def comm():
    fln.build()
    fln.load()
    c = fln.TpComm(1, 0)
    yield c
    c.close()


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_one_rank_region_matches_oracle_and_pipelined(comm, case):
    import torch
    wl, chunk = case
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    r = dev_bf16(d["r0"], extra_rows=2)
    out = dev_bf16(np.zeros((wl.T, wl.H), np.uint16), extra_rows=2, fill_bits=0x7FC2)
    fln.fused_proj_rs_add_rmsnorm_ag(run.x, run.W, r[:wl.T], run.gamma, wl.eps, wl.norm_kind, comm,
                                     microchunk_tokens=chunk, out=out[:wl.T])
    torch.cuda.synchronize()
    fln.fln_device_status()
    rb, ob = host_bits(r), host_bits(out)
    assert np.all(rb[wl.T:] == 0x7FC1) and np.all(ob[wl.T:] == 0x7FC2), "rows past T were written"
    rb, ob = rb[:wl.T], ob[:wl.T]
    r64, o64, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)
    compare(rb, r64, f"{wl.name} residual")
    compare(ob, o64, f"{wl.name} out")
    # the PIPELINED path with the same tile and chunk: the same numbers, bit for bit
    pr, po = run(plan(fln.PATH_PIPELINED, chunk=min(chunk or 1024, wl.T), tile_n=256))
    assert np.array_equal(rb, pr) and np.array_equal(ob, po)


def test_two_calls_in_a_row_and_argument_errors(comm):
    import torch
    wl, chunk = CASES[4]
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    r = dev_bf16(d["r0"])
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    fln.fused_proj_rs_add_rmsnorm_ag(run.x, run.W, r, run.gamma, wl.eps, wl.norm_kind, comm, chunk, out)
    first = host_bits(out)
    r.copy_(dev_bf16(d["r0"]))
    fln.fused_proj_rs_add_rmsnorm_ag(run.x, run.W, r, run.gamma, wl.eps, wl.norm_kind, comm, chunk, out)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out), first)
    rc = fln.fused_proj_rs_add_rmsnorm_ag_ptr(run.x.data_ptr(), run.W.data_ptr(), r.data_ptr(),
                                              run.gamma.data_ptr(), wl.eps, 0, wl.T, wl.K, wl.H, 0,
                                              out.data_ptr(), None, None)
    assert rc == fln.FLN_ERR_INVALID_ARG and "comm" in fln.fln_last_error()
    rc = fln.fused_proj_rs_add_rmsnorm_ag_ptr(run.x.data_ptr(), run.W.data_ptr(), r.data_ptr(),
                                              run.gamma.data_ptr(), wl.eps, 0, wl.T, wl.K, wl.H, 5000,
                                              out.data_ptr(), comm.handle, None)
    assert rc == fln.FLN_ERR_INVALID_ARG
    rc = fln.fused_proj_rs_add_rmsnorm_ag_ptr(run.x.data_ptr(), run.W.data_ptr(), r.data_ptr(),
                                              run.gamma.data_ptr(), wl.eps, 0, wl.T, wl.K, wl.H, 0,
                                              r.data_ptr(), comm.handle, None)
    assert rc == fln.FLN_ERR_INVALID_ARG and "overlap" in fln.fln_last_error()
    fln.fln_device_status()
