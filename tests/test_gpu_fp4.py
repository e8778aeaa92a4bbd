"""GPU parity of the NVFP4-weight region against the fp64 oracle, through the C ABI.

Same bar as the bf16 paths (tests/parity.py): the split-K path that reads W
packed and dequantises it on the SM (1 to 256 tokens, several tile
widths of the token side), the FUSED and PIPELINED paths after the whole
weight is converted to bf16, ragged T and H, chunk invariance bit for bit,
the tuner, full-size workloads on sampled rows, guard rows after T untouched.
"""
import numpy as np
import pytest

import oracle
from synth import Workload, make_inputs_nvfp4, workload

from .gpu_util import dev_bf16, host_bits, plan
from .parity import compare

pytestmark = pytest.mark.gpu

fln = pytest.importorskip("decoder_layer_projection_gb300")
torch = pytest.importorskip("torch")

NV = fln.DTYPE_NVFP4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fln.build()
    fln.load()
    yield
    fln.fln_set_overrides(0, 0)


def unfused():
    return plan(fln.PATH_FUSED, threshold=257)


class Run4:
    """One call of fused_proj_add_rmsnorm_nvfp4 on uploaded inputs with guard rows."""

    GUARD = 3

    def __init__(self, d, eps, kind):
        self.T, self.K = d["x"].shape
        self.H = d["Wq"].shape[0]
        self.eps, self.kind = eps, kind
        self.x = dev_bf16(d["x"])
        self.W = torch.from_numpy(np.ascontiguousarray(d["Wq"])).cuda()
        self.S = torch.from_numpy(np.ascontiguousarray(d["S"])).cuda()
        self.gs = d["gs"]
        self.r0 = d["r0"]
        self.gamma = torch.from_numpy(np.ascontiguousarray(d["gamma"], np.float32)).cuda()

    def __call__(self, plan_dict=None, chunk=0, T=None):
        T = self.T if T is None else T
        if plan_dict is not None:
            fln.fln_set_plan(self.K, self.H, self.kind, plan_dict, dtype=NV)
        try:
            r = dev_bf16(self.r0[:T], extra_rows=self.GUARD)
            out = dev_bf16(np.zeros((T, self.H), np.uint16), extra_rows=self.GUARD, fill_bits=0x7FC2)
            fln.fused_proj_add_rmsnorm_nvfp4(self.x[:T], self.W, self.S, self.gs, r[:T], self.gamma, self.eps,
                                             self.kind, chunk, out[:T])
            fln.fln_device_status()
        finally:
            if plan_dict is not None:
                fln.fln_set_plan(self.K, self.H, self.kind, None, dtype=NV)
        rb, ob = host_bits(r), host_bits(out)
        assert np.all(rb[T:] == 0x7FC1), "residual guard rows were written"
        assert np.all(ob[T:] == 0x7FC2), "output guard rows were written"
        return rb[:T], ob[:T]


def check(rb, ob, d, wl, rows=None, name="", T=None):
    T = d["x"].shape[0] if T is None else T
    r, o, _ = oracle.proj_add_rmsnorm_nvfp4(d["x"][:T], d["Wq"], d["S"], d["gs"], d["r0"][:T], d["gamma"], wl.eps,
                                            wl.norm_kind, rows=rows)
    if rows is not None:
        rb, ob = rb[rows], ob[rows]
    compare(rb, r, name + " residual")
    compare(ob, o, name + " out")


SMALL = [
    Workload("ragged", T=300, K=320, H=640, eps=1e-5, r_sigma=2.0, seed=1),
    Workload("ragged_h", T=130, K=192, H=264, eps=1e-6, r_sigma=1.0, seed=2),
    Workload("gemma_small", T=257, K=448, H=3584, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=3),
    Workload("wide_k", T=129, K=2048, H=512, eps=1e-5, r_sigma=2.0, seed=4),
]


def test_tiny_all_paths():
    wl = workload("tiny")
    d = make_inputs_nvfp4(wl)
    run = Run4(d, wl.eps, wl.norm_kind)
    for p in (unfused(), plan(fln.PATH_FUSED, chunk=16), plan(fln.PATH_FUSED, chunk=16, tile_n=224),
              plan(fln.PATH_FUSED, chunk=16, tile_n=128), plan(fln.PATH_PIPELINED, chunk=16)):
        rb, ob = run(p)
        check(rb, ob, d, wl, name=f"tiny nvfp4 {p}")


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("T", [1, 7, 16, 33, 128, 256])
def test_split_k_dequant_full_parity(wl, T):
    d = make_inputs_nvfp4(wl, T=T)
    run = Run4(d, wl.eps, wl.norm_kind)
    rb, ob = run(unfused())
    check(rb, ob, d, wl, name=f"{wl.name} nvfp4 unfused T={T}")
    rb2, ob2 = run(unfused())
    assert np.array_equal(rb, rb2) and np.array_equal(ob, ob2)


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("path,tile", [(1, 256), (1, 224), (2, 256), (2, 128)])
def test_converted_weight_paths_full_parity(wl, path, tile):
    d = make_inputs_nvfp4(wl)
    run = Run4(d, wl.eps, wl.norm_kind)
    rb, ob = run(plan(path, chunk=128, tile_n=tile))
    check(rb, ob, d, wl, name=f"{wl.name} nvfp4 path={path} tile={tile}")


def test_chunk_invariance_is_bitwise():
    wl = Workload("chunks", T=700, K=256, H=512, eps=1e-5, r_sigma=2.0, seed=9)
    d = make_inputs_nvfp4(wl)
    run = Run4(d, wl.eps, wl.norm_kind)
    for path in (fln.PATH_FUSED, fln.PATH_PIPELINED):
        res = [run(plan(path, chunk=c)) for c in (128, 256, 384, 700)]
        for rb, ob in res[1:]:
            assert np.array_equal(rb, res[0][0]) and np.array_equal(ob, res[0][1])
        check(res[0][0], res[0][1], d, wl, name=f"nvfp4 chunks path={path}")


def test_autotune_then_auto_calls():
    wl = Workload("tune4", T=1024, K=512, H=1024, eps=1e-5, r_sigma=2.0, seed=7)
    fln.fln_autotune(wl.K, wl.H, wl.norm_kind, wl.T, dtype=NV)
    try:
        assert fln.fln_get_plan(wl.K, wl.H, wl.norm_kind, wl.T, dtype=NV)["tuned_max_tokens"] == wl.T
        d = make_inputs_nvfp4(wl)
        run = Run4(d, wl.eps, wl.norm_kind)
        for T in (1, 64, 300, 1024):
            rb, ob = run(None, chunk=0, T=T)
            check(rb, ob, d, wl, name=f"nvfp4 tuned T={T}", T=T)
    finally:
        fln.fln_set_plan(wl.K, wl.H, wl.norm_kind, None, dtype=NV)


def test_rejects_bad_arguments():
    wl = workload("tiny")
    d = make_inputs_nvfp4(wl)
    run = Run4(d, wl.eps, wl.norm_kind)
    r = dev_bf16(d["r0"])
    out = torch.empty_like(r)
    lib = fln.load()
    rc = lib.fused_proj_add_rmsnorm_nvfp4(run.x.data_ptr(), run.W.data_ptr(), run.S.data_ptr(), 0.5, r.data_ptr(),
                                          run.gamma.data_ptr(), 1e-6, 0, 16, 224, 256, 0, out.data_ptr(), None)
    assert rc == fln.FLN_ERR_INVALID_ARG and "64" in fln.fln_last_error()
    rc = lib.fused_proj_add_rmsnorm_nvfp4(run.x.data_ptr(), run.W.data_ptr(), run.S.data_ptr(), float("inf"),
                                          r.data_ptr(), run.gamma.data_ptr(), 1e-6, 0, 16, 256, 256, 0,
                                          out.data_ptr(), None)
    assert rc == fln.FLN_ERR_INVALID_ARG
    fln.fln_device_status()


# every row of the full-size workloads is compared with the oracle


@pytest.mark.parametrize("name", ["llama70b_oproj_decode", "llama70b_down_decode"])
@pytest.mark.parametrize("T", [1, 8, 256])
def test_full_size_decode_every_row(name, T):
    wl = workload(name)
    d = make_inputs_nvfp4(wl, T=T)
    run = Run4(d, wl.eps, wl.norm_kind)
    rb, ob = run(unfused())
    check(rb, ob, d, wl, name=f"{name} nvfp4 T={T} unfused")


def test_full_size_prefill_every_row():
    wl = workload("llama3_8b_oproj")
    d = make_inputs_nvfp4(wl)
    run = Run4(d, wl.eps, wl.norm_kind)
    rb, ob = run(plan(fln.PATH_FUSED, chunk=4096))
    check(rb, ob, d, wl, name="oproj nvfp4 fused")
