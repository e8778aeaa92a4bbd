"""GPU parity of fused_proj_add_rmsnorm_host: x, residual and out in host
memory, streamed through the GPU in transfer chunks whose copies overlap the
compute of the chunk before, through the C ABI.

Results are held to the oracle's bar on every row; with the FUSED plan on a
K below the split threshold the per-row arithmetic is the device entry
point's, so the two agree bit for bit.  Covers page-locked and pageable host
memory, ragged chunks (T not a multiple of the chunk, T below one chunk, one
token), every path, two chained calls on one host residual buffer, argument
errors, and the Llama-3-8B o_proj prefill at full size on sampled rows.
"""
import numpy as np
import pytest

import oracle
from synth import Workload, make_inputs, workload

from .gpu_util import dev_bf16, host_bits, plan
from .parity import compare

pytestmark = pytest.mark.gpu

fln = pytest.importorskip("decoder_layer_projection_gb300")
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fln.build()
    fln.load()
    yield


def _host(a, pinned):
    t = torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pinned else t.clone()


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _run_host(d, wl, tt, pinned, W=None, gamma=None, r_host=None):
    W = dev_bf16(d["W"]) if W is None else W
    gamma = torch.from_numpy(np.ascontiguousarray(d["gamma"], np.float32)).cuda() if gamma is None else gamma
    x_h = _host(d["x"], pinned)
    r_h = _host(d["r0"], pinned) if r_host is None else r_host
    o_h = torch.full(r_h.shape, float("nan"), dtype=torch.bfloat16)
    if pinned:
        o_h = o_h.pin_memory()
    fln.fused_proj_add_rmsnorm_host(x_h, W, r_h, gamma, wl.eps, wl.norm_kind, tt, o_h)
    torch.cuda.synchronize()
    fln.fln_device_status()
    return r_h, o_h


WL = Workload("host", T=300, K=320, H=640, eps=1e-5, r_sigma=2.0, seed=41)
FUSED = plan(fln.PATH_FUSED, chunk=4096, tile_n=256)
PIPE = plan(fln.PATH_PIPELINED, chunk=64, tile_n=128)


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("tt,p", [(128, None), (128, FUSED), (0, FUSED), (100, PIPE), (7, None), (1000, FUSED)],
                         ids=["128-default", "128-fused", "auto-fused", "100-pipelined", "7-unfused", "1000-fused"])
def test_host_entry_matches_the_oracle(pinned, tt, p):
    d = make_inputs(WL)
    if p is not None:
        fln.fln_set_plan(WL.K, WL.H, WL.norm_kind, p)
    try:
        r_h, o_h = _run_host(d, WL, tt, pinned)
    finally:
        if p is not None:
            fln.fln_set_plan(WL.K, WL.H, WL.norm_kind, None)
    r, o, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], WL.eps, WL.norm_kind)
    compare(_bits(r_h), r, f"host tt={tt} residual")
    compare(_bits(o_h), o, f"host tt={tt} out")


def _device_call(d, wl, W, gamma, r_dev):
    x = dev_bf16(d["x"])
    out = torch.empty_like(r_dev)
    fln.fused_proj_add_rmsnorm(x, W, r_dev, gamma, wl.eps, wl.norm_kind, 0, out)
    torch.cuda.synchronize()
    fln.fln_device_status()
    return out


def test_host_entry_equals_the_device_entry_and_chains():
    """FUSED plan, K = 320 (no split): per-row arithmetic is the same, so every chunking gives the device
    entry point's bits.  A second call (another layer's x and W) on the same host residual buffer picks up
    the first call's residual, as the device entry point does with its device residual."""
    wl2 = Workload("host2", T=300, K=320, H=640, eps=1e-5, r_sigma=2.0, seed=42)
    d1, d2 = make_inputs(WL), make_inputs(wl2)
    W1, W2 = dev_bf16(d1["W"]), dev_bf16(d2["W"])
    g1 = torch.from_numpy(np.ascontiguousarray(d1["gamma"], np.float32)).cuda()
    g2 = torch.from_numpy(np.ascontiguousarray(d2["gamma"], np.float32)).cuda()
    fln.fln_set_plan(WL.K, WL.H, WL.norm_kind, FUSED)
    try:
        r_dev = dev_bf16(d1["r0"])
        o1 = host_bits(_device_call(d1, WL, W1, g1, r_dev))
        r1 = host_bits(r_dev)
        o2 = host_bits(_device_call(d2, wl2, W2, g2, r_dev))
        r2 = host_bits(r_dev)
        for tt in (64, 128, 300):
            r_h = _host(d1["r0"], True)
            _, o_h1 = _run_host(d1, WL, tt, True, W1, g1, r_h)
            assert np.array_equal(_bits(r_h), r1) and np.array_equal(_bits(o_h1), o1), tt
            _, o_h2 = _run_host(d2, wl2, tt, True, W2, g2, r_h)
            assert np.array_equal(_bits(r_h), r2) and np.array_equal(_bits(o_h2), o2), tt
    finally:
        fln.fln_set_plan(WL.K, WL.H, WL.norm_kind, None)


@pytest.mark.parametrize("T", [1, 5, 129])
def test_host_entry_short_calls(T):
    wl = Workload("host_short", T=T, K=256, H=512, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=43 + T)
    d = make_inputs(wl)
    r_h, o_h = _run_host(d, wl, 64, True)
    r, o, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)
    compare(_bits(r_h), r, f"host T={T} residual")
    compare(_bits(o_h), o, f"host T={T} out")


def test_host_entry_argument_errors():
    d = make_inputs(WL)
    W = dev_bf16(d["W"])
    gamma = torch.from_numpy(np.ascontiguousarray(d["gamma"], np.float32)).cuda()
    x_h, r_h = _host(d["x"], True), _host(d["r0"], True)
    o_h = torch.empty_like(r_h).pin_memory()
    T, K, H = WL.T, WL.K, WL.H
    s = torch.cuda.current_stream().cuda_stream
    call = fln.fused_proj_add_rmsnorm_host_ptr
    # activations on the device where host memory is expected
    x_d = dev_bf16(d["x"])
    assert call(x_d.data_ptr(), W.data_ptr(), r_h.data_ptr(), gamma.data_ptr(), WL.eps, 0, T, K, H, 0,
                o_h.data_ptr(), s) == fln.FLN_ERR_INVALID_ARG
    # weights in host memory where device memory is expected
    W_h = _host(d["W"], True)
    assert call(x_h.data_ptr(), W_h.data_ptr(), r_h.data_ptr(), gamma.data_ptr(), WL.eps, 0, T, K, H, 0,
                o_h.data_ptr(), s) == fln.FLN_ERR_INVALID_ARG
    # out overlapping the residual
    assert call(x_h.data_ptr(), W.data_ptr(), r_h.data_ptr(), gamma.data_ptr(), WL.eps, 0, T, K, H, 0,
                r_h.data_ptr(), s) == fln.FLN_ERR_INVALID_ARG
    assert fln.fln_last_error()
    # nothing was written: the residual still holds r0
    torch.cuda.synchronize()
    assert np.array_equal(_bits(r_h), np.ascontiguousarray(d["r0"], np.uint16))


def test_host_entry_full_size_oproj_sampled_rows():
    wl = workload("llama3_8b_oproj")
    d = make_inputs(wl)
    r_h, o_h = _run_host(d, wl, 0, True)
    rows = np.array(sorted(set([0, 1, 1023, 1024, 2047, 2048, 3071, 3072, 4094, 4095]
                               + list(np.random.default_rng(5).integers(0, wl.T, 22)))))
    r, o, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind, rows=rows)
    compare(_bits(r_h)[rows], r, "host o_proj residual")
    compare(_bits(o_h)[rows], o, "host o_proj out")
