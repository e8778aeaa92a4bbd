"""The entry point that never allocates device memory, checked against the
ordinary entry point.

Some callers cannot let a library call cudaMalloc: a serving runtime that has
reserved all device memory for its own pool, or a latency-critical loop where
an allocation would synchronise the device.  fused_proj_add_rmsnorm_noalloc
keeps its scratch (the cross-tile row statistics) in a static device array
instead of the growable workspace.  This file runs last so that a failure here
cannot hide the other tests' results; it passes alone in a fresh process too.
"""
import numpy as np
import pytest

from synth import Workload, bf16_bits_to_f32, make_inputs

from .gpu_util import Run, dev_bf16, host_bits, plan
from .parity import ATOL, MEAN_TOL, bf16_ulp

pytestmark = pytest.mark.gpu

fln = pytest.importorskip("decoder_layer_projection_gb300")


def _close(a_bits, b_bits, name):
    a = bf16_bits_to_f32(a_bits).astype(np.float64)
    b = bf16_bits_to_f32(b_bits).astype(np.float64)
    d = np.abs(a - b)
    assert np.all(np.isfinite(a)), name
    assert np.all(d <= np.maximum(ATOL, bf16_ulp(b))), (name, float(d.max()))
    assert d.mean() <= MEAN_TOL, (name, float(d.mean()))


@pytest.mark.parametrize("wl", [
    Workload("noalloc", T=600, K=512, H=1024, eps=1e-5, r_sigma=2.0, seed=21),
    Workload("noalloc_gemma", T=130, K=264, H=3584, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=22),
], ids=lambda w: w.name)
def test_noalloc_matches_existing_entry_point_on_two_calls(wl):
    import torch
    fln.build()
    fln.load()
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    # the existing entry point, FUSED path with the same tile width and chunking
    ref_r, ref_o = run(plan(fln.PATH_FUSED, chunk=4096, tile_n=256))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        r = dev_bf16(d["r0"], extra_rows=2)
        out = dev_bf16(np.zeros((wl.T, wl.H), np.uint16), extra_rows=2, fill_bits=0x7FC2)
        fln.fused_proj_add_rmsnorm_noalloc(run.x, run.W, r[:wl.T], run.gamma, wl.eps, wl.norm_kind,
                                           out=out[:wl.T], device_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        rb, ob = host_bits(r), host_bits(out)
        assert np.all(rb[wl.T:] == 0x7FC1) and np.all(ob[wl.T:] == 0x7FC2)
        _close(rb[:wl.T], ref_r, f"residual, call {call}")
        _close(ob[:wl.T], ref_o, f"out, call {call}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fln.build()
    fln.load()
    # 32 row blocks x 65 N-tiles = 2080 tiles > 2048: refused before any launch
    rc = fln.fused_proj_add_rmsnorm_noalloc_ptr(None, None, None, None, 1e-5, 0, 4096, 64, 16392, None, None, None)
    assert rc == fln.FLN_ERR_UNSUPPORTED
    assert "static scratch" in fln.fln_last_error()
