"""The entry point that never allocates device memory.

Some callers cannot let a library call cudaMalloc: a serving runtime that has
reserved all device memory for its own pool (an allocation outside the pool can
fail or break its accounting), or a latency-critical loop where an allocation
would synchronise the device.  fused_proj_add_rmsnorm_noalloc keeps its
scratch (the cross-tile row statistics) in a static device array instead of
the growable workspace.  Its results are checked against the ordinary entry
point (within the parity tolerance: the two run different kernels) and against
the fp64 oracle, on two calls in a row.  This file runs last so that a failure
here cannot hide the other tests' results; it passes alone in a fresh process
too.
"""
import numpy as np
import pytest

import oracle
from synth import Workload, bf16_bits_to_f32, make_inputs

from .gpu_util import Run, dev_bf16, host_bits, plan
from .parity import ATOL, MEAN_TOL, bf16_ulp, compare

pytestmark = pytest.mark.gpu

fln = pytest.importorskip("decoder_layer_projection_gb300")

TIMEOUT_ROWSTAT = 0x8  # device error bit: cross-CTA row statistics never arrived


def _close(a_bits, b_bits, name):
    a = bf16_bits_to_f32(a_bits).astype(np.float64)
    b = bf16_bits_to_f32(b_bits).astype(np.float64)
    d = np.abs(a - b)
    assert np.all(np.isfinite(a)), name
    assert np.all(d <= np.maximum(ATOL, bf16_ulp(b))), (name, float(d.max()))
    assert d.mean() <= MEAN_TOL, (name, float(d.mean()))


def _noalloc(run, d, wl, err=None):
    """One call on fresh residual / output buffers with guard rows; returns (residual bits, out bits)."""
    import torch
    r = dev_bf16(d["r0"], extra_rows=2)
    out = dev_bf16(np.zeros((wl.T, wl.H), np.uint16), extra_rows=2, fill_bits=0x7FC2)
    fln.fused_proj_add_rmsnorm_noalloc(run.x, run.W, r[:wl.T], run.gamma, wl.eps, wl.norm_kind,
                                       out=out[:wl.T], device_error=err)
    torch.cuda.synchronize()
    rb, ob = host_bits(r), host_bits(out)
    assert np.all(rb[wl.T:] == 0x7FC1) and np.all(ob[wl.T:] == 0x7FC2), "guard rows were written"
    return rb[:wl.T], ob[:wl.T]


@pytest.mark.parametrize("wl", [
    Workload("noalloc", T=600, K=512, H=1024, eps=1e-5, r_sigma=2.0, seed=21),
    Workload("noalloc_gemma", T=130, K=264, H=3584, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=22),
    # more than one 4096-token chunk: the second launch starts at row 4096 and reuses the scratch
    Workload("noalloc_two_chunks", T=4100, K=192, H=520, eps=1e-5, r_sigma=2.0, seed=23),
], ids=lambda w: w.name)
def test_noalloc_matches_existing_entry_point_on_two_calls(wl):
    import torch
    fln.build()
    fln.load()
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    # the existing entry point, FUSED path with the same tile width and chunking
    ref_r, ref_o = run(plan(fln.PATH_FUSED, chunk=4096, tile_n=256))
    r64, o64, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        rb, ob = _noalloc(run, d, wl, err)
        assert int(err.item()) == 0
        _close(rb, ref_r, f"residual vs fused_proj_add_rmsnorm, call {call}")
        _close(ob, ref_o, f"out vs fused_proj_add_rmsnorm, call {call}")
        compare(rb, r64, f"{wl.name} residual vs oracle, call {call}")
        compare(ob, o64, f"{wl.name} out vs oracle, call {call}")


def test_noalloc_reports_a_bounded_wait_that_ran_out():
    """The test switch makes one launch wait for row statistics nobody publishes: after about two
    seconds the kernel gives up, ORs its bit into the caller's word (or, without one, into the
    static scratch's word that fln_device_status reads), and the next call is correct."""
    import torch
    fln.build()
    fln.load()
    wl = Workload("noalloc_stall", T=300, K=256, H=512, eps=1e-5, r_sigma=2.0, seed=24)
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    r64, o64, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)
    fln.fln_device_status()  # nothing pending before the test
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fln.fln_debug_stall_next_call(True)
    _noalloc(run, d, wl, err)
    assert int(err.item()) & TIMEOUT_ROWSTAT
    fln.fln_device_status()  # the caller's word took the bits: the library's words are clear
    # no caller word: the bits land in the static scratch and fln_device_status reports them
    fln.fln_debug_stall_next_call(True)
    _noalloc(run, d, wl, None)
    with pytest.raises(fln.FlnError) as e:
        fln.fln_device_status()
    assert e.value.status == fln.FLN_ERR_DEVICE_TIMEOUT
    fln.fln_device_status()  # read and cleared
    rb, ob = _noalloc(run, d, wl, None)
    fln.fln_device_status()
    compare(rb, r64, "residual after a timed-out call")
    compare(ob, o64, "out after a timed-out call")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fln.build()
    fln.load()
    # 32 row blocks x 65 N-tiles = 2080 tiles > 2048: refused before any launch
    rc = fln.fused_proj_add_rmsnorm_noalloc_ptr(None, None, None, None, 1e-5, 0, 4096, 64, 16392, None, None, None)
    assert rc == fln.FLN_ERR_UNSUPPORTED
    assert "static scratch" in fln.fln_last_error()
