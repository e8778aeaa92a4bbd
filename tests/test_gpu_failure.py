"""Failure reporting on the GPU without a fault: a bounded wait that runs out.

The test switch makes one FUSED launch wait for a row-statistics value that no
CTA publishes; the wait gives up after about two seconds, the kernel unwinds
(copies in flight land, TMEM is freed) and the host reads
FLN_ERR_DEVICE_TIMEOUT.  The next call on the same context must be correct.
"""
import numpy as np
import pytest

import oracle
from synth import Workload, make_inputs

from .gpu_util import Run, plan
from .parity import compare

pytestmark = pytest.mark.gpu

fln = pytest.importorskip("decoder_layer_projection_gb300")


@pytest.mark.parametrize("epi_warps", [4, 8])
def test_bounded_wait_timeout_is_reported_and_the_context_survives(epi_warps):
    fln.build()
    fln.load()
    wl = Workload("stall", T=300, K=256, H=512, eps=1e-5, r_sigma=2.0, seed=31)
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    fln.fln_device_status()  # nothing pending
    fln.fln_debug_stall_next_call(True)
    with pytest.raises(fln.FlnError) as e:
        run(plan(fln.PATH_FUSED, chunk=4096, tile_n=256, epi_warps=epi_warps))
    assert e.value.status == fln.FLN_ERR_DEVICE_TIMEOUT
    assert "bounded wait" in str(e.value)
    # the error word was read and cleared; the context still computes correctly
    fln.fln_device_status()
    rb, ob = run(plan(fln.PATH_FUSED, chunk=4096, tile_n=256, epi_warps=epi_warps))
    r, o, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)
    compare(rb, r, "after timeout: residual")
    compare(ob, o, "after timeout: out")


def test_split_k_tail_wait_timeout_is_reported_and_counters_recover():
    """The UNFUSED path's split-K tail waits for every 128-row block of W to be reduced; with the
    test switch it waits for one block more than there are.  The wait gives up, the status is
    reported, and the next calls (eager, then again) are correct: the tail's counters start over."""
    fln.build()
    fln.load()
    wl = Workload("stall_tail", T=16, K=4096, H=1024, eps=1e-5, r_sigma=2.0, seed=32)
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    unfused = plan(fln.PATH_FUSED, threshold=257)
    fln.fln_set_splitk_tail_tokens(256)
    try:
        fln.fln_device_status()
        fln.fln_debug_stall_next_call(True)
        with pytest.raises(fln.FlnError) as e:
            run(unfused)
        assert e.value.status == fln.FLN_ERR_DEVICE_TIMEOUT
        fln.fln_device_status()
        r, o, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)
        for i in range(2):
            rb, ob = run(unfused)
            compare(rb, r, f"after tail timeout, call {i}: residual")
            compare(ob, o, f"after tail timeout, call {i}: out")
    finally:
        fln.fln_set_splitk_tail_tokens(0)
