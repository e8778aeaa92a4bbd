"""GPU parity of the FP8 (E4M3) region against the fp64 oracle, through the C ABI.

Same bar as the bf16 paths (tests/parity.py): every path (FUSED tiles 128 /
192 / 224 / 256, PIPELINED 128 / 256, UNFUSED with static and dynamic split-K),
per-tensor and per-token / per-channel scales, ragged T, K (multiple of 16,
not of the 128-element K-block) and H, chunk invariance bit for bit, full-size
workloads on sampled rows, guard rows after T untouched.
"""
import numpy as np
import pytest

import oracle
from synth import Workload, make_inputs_fp8, workload

from .gpu_util import dev_bf16, host_bits, plan
from .parity import compare

pytestmark = pytest.mark.gpu

fln = pytest.importorskip("decoder_layer_projection_gb300")
torch = pytest.importorskip("torch")

E4M3 = fln.DTYPE_E4M3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fln.build()
    fln.load()
    yield
    fln.fln_set_overrides(0, 0)


def unfused():
    return plan(fln.PATH_FUSED, threshold=257)


class Run8:
    """One call of fused_proj_add_rmsnorm_fp8 on uploaded inputs with guard rows."""

    GUARD = 3

    def __init__(self, d, eps, kind):
        self.T, self.K = d["x8"].shape
        self.H = d["W8"].shape[0]
        self.eps, self.kind = eps, kind
        self.x = torch.from_numpy(np.ascontiguousarray(d["x8"])).cuda()
        self.W = torch.from_numpy(np.ascontiguousarray(d["W8"])).cuda()
        self.sx = torch.from_numpy(np.ascontiguousarray(d["x_scale"])).cuda()
        self.sw = torch.from_numpy(np.ascontiguousarray(d["w_scale"])).cuda()
        self.r0 = d["r0"]
        self.gamma = torch.from_numpy(np.ascontiguousarray(d["gamma"], np.float32)).cuda()

    def __call__(self, plan_dict=None, chunk=0, T=None, sx=None):
        T = self.T if T is None else T
        sx = self.sx if sx is None else sx
        if sx.numel() == self.T and T < self.T:
            sx = sx[:T]
        if plan_dict is not None:
            fln.fln_set_plan(self.K, self.H, self.kind, plan_dict, dtype=E4M3)
        try:
            r = dev_bf16(self.r0[:T], extra_rows=self.GUARD)
            out = dev_bf16(np.zeros((T, self.H), np.uint16), extra_rows=self.GUARD, fill_bits=0x7FC2)
            fln.fused_proj_add_rmsnorm_fp8(self.x[:T], sx, self.W, self.sw, r[:T], self.gamma, self.eps, self.kind,
                                           chunk, out[:T])
            fln.fln_device_status()
        finally:
            if plan_dict is not None:
                fln.fln_set_plan(self.K, self.H, self.kind, None, dtype=E4M3)
        rb, ob = host_bits(r), host_bits(out)
        assert np.all(rb[T:] == 0x7FC1), "residual guard rows were written"
        assert np.all(ob[T:] == 0x7FC2), "output guard rows were written"
        return rb[:T], ob[:T]


def check(rb, ob, d, wl, rows=None, name="", T=None):
    T = d["x8"].shape[0] if T is None else T
    sx = d["x_scale"] if d["x_scale"].size == 1 else d["x_scale"][:T]
    r, o, _ = oracle.proj_add_rmsnorm_fp8(d["x8"][:T], sx, d["W8"], d["w_scale"], d["r0"][:T], d["gamma"], wl.eps,
                                          wl.norm_kind, rows=rows)
    if rows is not None:
        rb, ob = rb[rows], ob[rows]
    compare(rb, r, name + " residual")
    compare(ob, o, name + " out")


SMALL = [
    Workload("ragged", T=300, K=320, H=640, eps=1e-5, r_sigma=2.0, seed=1),
    Workload("ragged_k_h", T=130, K=208, H=264, eps=1e-6, r_sigma=1.0, seed=2),
    Workload("gemma_small", T=257, K=448, H=3584, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=3),
    Workload("wide_k", T=129, K=2048, H=512, eps=1e-5, r_sigma=2.0, seed=4),
]


def test_tiny_all_paths():
    wl = workload("tiny")
    d = make_inputs_fp8(wl)
    run = Run8(d, wl.eps, wl.norm_kind)
    for p in (plan(fln.PATH_FUSED, chunk=16), plan(fln.PATH_FUSED, chunk=16, tile_n=128),
              plan(fln.PATH_FUSED, chunk=16, tile_n=192), plan(fln.PATH_FUSED, chunk=16, tile_n=224),
              plan(fln.PATH_PIPELINED, chunk=16), plan(fln.PATH_PIPELINED, chunk=16, tile_n=128), unfused()):
        rb, ob = run(p)
        check(rb, ob, d, wl, name=f"tiny fp8 {p}")


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("path,tile", [(1, 256), (1, 224), (1, 192), (1, 128), (2, 256), (2, 128), (2, 64)])
def test_small_paths_full_parity(wl, path, tile):
    d = make_inputs_fp8(wl)
    run = Run8(d, wl.eps, wl.norm_kind)
    rb, ob = run(plan(path, chunk=128, tile_n=tile))
    check(rb, ob, d, wl, name=f"{wl.name} fp8 path={path} tile={tile}")


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("tile,ew", [(256, 8), (224, 8), (256, 4)])
def test_epilogue_warps_full_parity(wl, tile, ew):
    d = make_inputs_fp8(wl)
    run = Run8(d, wl.eps, wl.norm_kind)
    rb, ob = run(plan(fln.PATH_FUSED, chunk=128, tile_n=tile, epi_warps=ew))
    check(rb, ob, d, wl, name=f"{wl.name} fp8 tile={tile} epi_warps={ew}")


@pytest.mark.parametrize("wl", SMALL[:3], ids=lambda w: w.name)
@pytest.mark.parametrize("per_token,per_channel", [(False, False), (True, False), (False, True)])
def test_scale_granularities(wl, per_token, per_channel):
    d = make_inputs_fp8(wl, x_scale_per_token=per_token, w_scale_per_channel=per_channel)
    run = Run8(d, wl.eps, wl.norm_kind)
    for p in (plan(fln.PATH_FUSED, chunk=128), plan(fln.PATH_PIPELINED, chunk=128)):
        rb, ob = run(p)
        check(rb, ob, d, wl, name=f"{wl.name} fp8 scales {per_token}/{per_channel} path={p['path']}")
    rb, ob = run(unfused(), T=33)
    check(rb, ob, d, wl, name=f"{wl.name} fp8 unfused scales {per_token}/{per_channel}", T=33)


def test_tensor_scale_equals_repeated_token_scale_bitwise():
    wl = SMALL[0]
    d = make_inputs_fp8(wl, x_scale_per_token=False)
    run = Run8(d, wl.eps, wl.norm_kind)
    rep = torch.full((wl.T,), float(d["x_scale"][0]), dtype=torch.float32, device="cuda")
    for p in (plan(fln.PATH_FUSED, chunk=128), plan(fln.PATH_PIPELINED, chunk=128)):
        a = run(p)
        b = run(p, sx=rep)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("wl", SMALL[:3], ids=lambda w: w.name)
@pytest.mark.parametrize("T", [1, 7, 16, 33, 128, 256])
@pytest.mark.parametrize("tail", [256, 0], ids=["tail", "reducer"])
def test_small_unfused_full_parity(wl, T, tail):
    d = make_inputs_fp8(wl, T=T)
    run = Run8(d, wl.eps, wl.norm_kind)
    fln.fln_set_splitk_tail_tokens(tail)
    try:
        rb, ob = run(unfused())
    finally:
        fln.fln_set_splitk_tail_tokens(0)
    check(rb, ob, d, wl, name=f"{wl.name} fp8 unfused T={T} tail={tail}")


@pytest.mark.parametrize("T", [1, 9, 32, 64])
@pytest.mark.parametrize("tail", [256, 0], ids=["tail", "reducer"])
def test_unfused_dynamic_chunks(T, tail):
    # K >= 16384: at <= 32 tokens the last fifth of each m-tile's K-blocks is drawn at run time
    wl = Workload("deep_k_fp8", T=64, K=16400, H=392, eps=1e-5, r_sigma=2.0, seed=13)
    d = make_inputs_fp8(wl, T=T)
    run = Run8(d, wl.eps, wl.norm_kind)
    fln.fln_set_splitk_tail_tokens(tail)
    try:
        rb, ob = run(unfused())
        check(rb, ob, d, wl, name=f"deep_k fp8 unfused T={T} tail={tail}")
        rb2, ob2 = run(unfused())
        assert np.array_equal(rb, rb2) and np.array_equal(ob, ob2)
    finally:
        fln.fln_set_splitk_tail_tokens(0)


def test_chunk_invariance_is_bitwise():
    wl = Workload("chunks", T=700, K=256, H=512, eps=1e-5, r_sigma=2.0, seed=9)
    d = make_inputs_fp8(wl)
    run = Run8(d, wl.eps, wl.norm_kind)
    for path in (fln.PATH_FUSED, fln.PATH_PIPELINED):
        res = [run(plan(path, chunk=c)) for c in (128, 256, 384, 700)]
        for rb, ob in res[1:]:
            assert np.array_equal(rb, res[0][0]) and np.array_equal(ob, res[0][1])
        check(res[0][0], res[0][1], d, wl, name=f"fp8 chunks path={path}")


def test_dtype_plans_are_separate():
    K, H = 1024, 768
    fln.fln_set_plan(K, H, 0, plan(fln.PATH_PIPELINED, chunk=512, tile_n=128), dtype=E4M3)
    try:
        assert fln.fln_get_plan(K, H, 0, 4096, dtype=E4M3)["path"] == fln.PATH_PIPELINED
        assert fln.fln_get_plan(K, H, 0, 4096)["path"] == fln.PATH_FUSED
    finally:
        fln.fln_set_plan(K, H, 0, None, dtype=E4M3)


def test_autotune_fp8_then_auto_calls():
    wl = Workload("tune8", T=1024, K=512, H=1024, eps=1e-5, r_sigma=2.0, seed=7)
    fln.fln_autotune(wl.K, wl.H, wl.norm_kind, wl.T, dtype=E4M3)
    try:
        p = fln.fln_get_plan(wl.K, wl.H, wl.norm_kind, wl.T, dtype=E4M3)
        assert p["tuned_max_tokens"] == wl.T
        d = make_inputs_fp8(wl)
        run = Run8(d, wl.eps, wl.norm_kind)
        for T in (1, 64, 300, 1024):
            rb, ob = run(None, chunk=0, T=T)
            check(rb, ob, d, wl, name=f"fp8 tuned T={T}", T=T)
    finally:
        fln.fln_set_plan(wl.K, wl.H, wl.norm_kind, None, dtype=E4M3)


def test_rejects_bad_fp8_arguments():
    wl = workload("tiny")
    d = make_inputs_fp8(wl)
    run = Run8(d, wl.eps, wl.norm_kind)
    r = dev_bf16(d["r0"])
    out = torch.empty_like(r)
    lib = fln.load()
    # K not a multiple of 16
    rc = lib.fused_proj_add_rmsnorm_fp8(run.x.data_ptr(), run.sx.data_ptr(), 1, run.W.data_ptr(), run.sw.data_ptr(),
                                        1, r.data_ptr(), run.gamma.data_ptr(), 1e-6, 0, 16, 248, 256, 0,
                                        out.data_ptr(), None)
    assert rc == fln.FLN_ERR_INVALID_ARG and "16" in fln.fln_last_error()
    # scale on the host
    host = torch.ones(16, dtype=torch.float32)
    rc = lib.fused_proj_add_rmsnorm_fp8(run.x.data_ptr(), host.data_ptr(), 1, run.W.data_ptr(), run.sw.data_ptr(),
                                        1, r.data_ptr(), run.gamma.data_ptr(), 1e-6, 0, 16, 256, 256, 0,
                                        out.data_ptr(), None)
    assert rc == fln.FLN_ERR_INVALID_ARG and "x_scale" in fln.fln_last_error()
    # out aliasing a scale
    rc = lib.fused_proj_add_rmsnorm_fp8(run.x.data_ptr(), run.sx.data_ptr(), 1, run.W.data_ptr(), run.sw.data_ptr(),
                                        1, r.data_ptr(), run.gamma.data_ptr(), 1e-6, 0, 16, 256, 256, 0,
                                        run.sw.data_ptr(), None)
    assert rc == fln.FLN_ERR_INVALID_ARG
    fln.fln_device_status()


# --------------------------------------------------------------- full sizes
# every row of the full-size workloads is compared with the oracle


@pytest.mark.parametrize("name", ["llama3_8b_oproj", "gemma2_9b_down"])
def test_full_size_prefill_every_row(name):
    wl = workload(name)
    d = make_inputs_fp8(wl)
    run = Run8(d, wl.eps, wl.norm_kind)
    # the oracle once, shared by both paths
    r, o, _ = oracle.proj_add_rmsnorm_fp8(d["x8"], d["x_scale"], d["W8"], d["w_scale"], d["r0"], d["gamma"], wl.eps,
                                          wl.norm_kind)
    for p in (plan(fln.PATH_FUSED, chunk=min(wl.T, 4096)), plan(fln.PATH_PIPELINED, chunk=1024)):
        rb, ob = run(p)
        compare(rb, r, f"{name} fp8 path={p['path']} residual")
        compare(ob, o, f"{name} fp8 path={p['path']} out")


@pytest.mark.parametrize("name", ["llama70b_oproj_decode", "llama70b_down_decode"])
@pytest.mark.parametrize("T", [1, 8, 256])
def test_full_size_decode_every_row(name, T):
    wl = workload(name)
    d = make_inputs_fp8(wl, T=T)
    run = Run8(d, wl.eps, wl.norm_kind)
    rb, ob = run(unfused())
    check(rb, ob, d, wl, name=f"{name} fp8 T={T} unfused")
