"""GPU parity: every path of libfusedln against the fp64 oracle, through the C ABI.

Every element is compared with the oracle: small cases (several tiles,
ragged tails in T, K and H) and the five full-size workloads alike, on the
FUSED and UNFUSED paths (and PIPELINED for the prefill shapes).  Chunk
invariance is bitwise (K below the 128 K-blocks from which a last round of
tiles is split).  Guard rows after T must stay untouched on every call.
"""
import numpy as np
import pytest

import oracle
from synth import Workload, make_inputs, workload

from .gpu_util import UNFUSED, Run, plan
from .parity import compare

pytestmark = pytest.mark.gpu

fln = pytest.importorskip("decoder_layer_projection_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fln.build()
    fln.load()
    yield
    fln.fln_set_overrides(0, 0)


def check_rows(rb, ob, d, wl, rows=None, tight=True, name=""):
    r, o, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind, rows=rows)
    if rows is not None:
        rb, ob = rb[rows], ob[rows]
    sr = compare(rb, r, name + " residual", tight=tight)
    so = compare(ob, o, name + " out", tight=tight)
    return sr, so


SMALL = [
    Workload("ragged", T=300, K=320, H=640, eps=1e-5, r_sigma=2.0, seed=1),
    Workload("ragged_k_h", T=130, K=200, H=264, eps=1e-6, r_sigma=1.0, seed=2),
    Workload("gemma_small", T=257, K=448, H=3584, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=3),
    Workload("wide_k", T=129, K=2048, H=512, eps=1e-5, x_mode="silu_gu", r_sigma=2.0, seed=4),
]


def test_tiny_config_all_paths():
    wl = workload("tiny")
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    for p in (plan(fln.PATH_FUSED, chunk=16), plan(fln.PATH_PIPELINED, chunk=16),
              plan(fln.PATH_FUSED, chunk=16, tile_n=128), plan(fln.PATH_FUSED, chunk=16, tile_n=192),
              plan(fln.PATH_FUSED, chunk=16, tile_n=224), UNFUSED):
        rb, ob = run(p)
        check_rows(rb, ob, d, wl, name=f"tiny {p}")


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("path,tile", [(1, 256), (1, 224), (1, 192), (1, 128), (2, 256), (2, 128), (2, 64)])
def test_small_prefill_paths_full_parity(wl, path, tile):
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    rb, ob = run(plan(path, chunk=128, tile_n=tile))
    check_rows(rb, ob, d, wl, name=f"{wl.name} path={path} tile={tile}")


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("tile", [256, 224])
def test_eight_epilogue_warps_full_parity(wl, tile):
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    rb, ob = run(plan(1, chunk=128, tile_n=tile, epi_warps=8))
    check_rows(rb, ob, d, wl, name=f"{wl.name} fused tile={tile} epi_warps=8")


def test_epilogue_width_does_not_change_the_layout_of_work():
    # four or eight epilogue warps: same tiles, same rows, results within the gate
    wl = Workload("ew", T=700, K=320, H=1024, eps=1e-5, r_sigma=2.0, seed=21)
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    for c in (128, 700):
        a = run(plan(1, chunk=c, tile_n=256, epi_warps=4))
        b = run(plan(1, chunk=c, tile_n=256, epi_warps=8))
        check_rows(a[0], a[1], d, wl, name=f"ew4 chunk={c}")
        check_rows(b[0], b[1], d, wl, name=f"ew8 chunk={c}")
        # the same arithmetic per row, only the warps differ: bit-identical
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


class tail_tokens:
    """Within the block, UNFUSED calls of at most n tokens reduce in the split-K GEMM's tail (0: the
    separate reducer kernel for every call)."""

    def __init__(self, n):
        self.n = n

    def __enter__(self):
        fln.fln_set_splitk_tail_tokens(self.n)

    def __exit__(self, *exc):
        fln.fln_set_splitk_tail_tokens(0)
        return False


@pytest.mark.parametrize("wl", SMALL[:3], ids=lambda w: w.name)
@pytest.mark.parametrize("T", [1, 7, 16, 33, 128, 256])
@pytest.mark.parametrize("tail", [256, 0], ids=["tail", "reducer"])
def test_small_unfused_full_parity(wl, T, tail):
    d = make_inputs(wl, T=T)
    run = Run(d, wl.eps, wl.norm_kind)
    with tail_tokens(tail):
        rb, ob = run(UNFUSED)
    check_rows(rb, ob, d, wl, name=f"{wl.name} unfused T={T} tail={tail}")


# K long enough (>= 256 K-blocks) that for <= 32 tokens the split-K GEMM hands
# the last fifth of every m-tile's K-blocks out at run time
DEEP = [
    Workload("deep_k_ragged", T=64, K=16392, H=392, eps=1e-5, r_sigma=2.0, seed=11),
    Workload("deep_k_gemma", T=64, K=28672, H=1024, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=12),
]


@pytest.mark.parametrize("wl", DEEP, ids=lambda w: w.name)
@pytest.mark.parametrize("T", [1, 9, 32, 64])
@pytest.mark.parametrize("tail", [256, 0], ids=["tail", "reducer"])
def test_unfused_dynamic_chunks_full_parity(wl, T, tail):
    d = make_inputs(wl, T=T)
    run = Run(d, wl.eps, wl.norm_kind)
    with tail_tokens(tail):
        rb, ob = run(UNFUSED)
        check_rows(rb, ob, d, wl, name=f"{wl.name} unfused T={T} tail={tail}")
        # the chunk counter (and the tail's counters) return to zero after every launch: repeats are
        # bitwise equal
        for _ in range(3):
            rb2, ob2 = run(UNFUSED)
            assert np.array_equal(rb, rb2) and np.array_equal(ob, ob2)


@pytest.mark.parametrize("tail", [0, 256], ids=["reducer", "tail"])
def test_unfused_graph_replay_is_bitwise(tail):
    """The split-K path captured in a CUDA graph and replayed gives the eager
    result on every replay (nothing of one launch is baked into the next: the
    dynamic-chunk counter and the tail's counters return to zero)."""
    import torch
    from .gpu_util import dev_bf16, host_bits
    wl = DEEP[0]
    T = 16
    d = make_inputs(wl, T=T)
    x, W = dev_bf16(d["x"]), dev_bf16(d["W"])
    gamma = torch.from_numpy(np.ascontiguousarray(d["gamma"], np.float32)).cuda()
    r0 = dev_bf16(d["r0"])
    fln.fln_set_plan(wl.K, wl.H, wl.norm_kind, UNFUSED)
    fln.fln_set_splitk_tail_tokens(tail)
    try:
        r = r0.clone()
        out = torch.empty_like(r)
        fln.fused_proj_add_rmsnorm(x, W, r, gamma, wl.eps, wl.norm_kind, 0, out)  # eager; sizes the workspace
        fln.fln_device_status()
        r_eager, o_eager = host_bits(r), host_bits(out)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        r.copy_(r0)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            fln.fused_proj_add_rmsnorm(x, W, r, gamma, wl.eps, wl.norm_kind, 0, out)
        for _ in range(3):
            r.copy_(r0)
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            fln.fln_device_status()
            assert np.array_equal(host_bits(r), r_eager) and np.array_equal(host_bits(out), o_eager)
    finally:
        fln.fln_set_plan(wl.K, wl.H, wl.norm_kind, None)
        fln.fln_set_splitk_tail_tokens(0)
    check_rows(r_eager, o_eager, d, wl, name=f"graph replay tail={tail}")


def test_chunk_invariance_is_bitwise():
    wl = Workload("chunks", T=700, K=256, H=512, eps=1e-5, r_sigma=2.0, seed=9)
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    for path in (fln.PATH_FUSED, fln.PATH_PIPELINED):
        res = [run(plan(path, chunk=c)) for c in (128, 256, 384, 700)]
        for rb, ob in res[1:]:
            assert np.array_equal(rb, res[0][0]) and np.array_equal(ob, res[0][1])
        check_rows(res[0][0], res[0][1], d, wl, name=f"chunks path={path}")


def test_call_microchunk_argument_and_overrides():
    wl = Workload("args", T=520, K=128, H=256, eps=1e-5, seed=5)
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    rb0, ob0 = run(plan(fln.PATH_FUSED, chunk=4096), chunk=0)
    rb1, ob1 = run(plan(fln.PATH_FUSED, chunk=4096), chunk=200)   # the call's chunk wins
    assert np.array_equal(rb0, rb1) and np.array_equal(ob0, ob1)
    fln.fln_set_overrides(100, 0)
    try:
        rb2, ob2 = run(None, chunk=0)
    finally:
        fln.fln_set_overrides(0, 0)
    assert np.array_equal(rb0, rb2) and np.array_equal(ob0, ob2)
    check_rows(rb0, ob0, d, wl, name="args")


def test_add_rmsnorm_matches_oracle():
    import torch
    from .gpu_util import dev_bf16, host_bits
    for T, H, kind, eps in [(1, 256, 0, 1e-6), (37, 4096, 0, 1e-5), (300, 3584, 1, 1e-6), (5, 8192, 0, 1e-5),
                            (3, 8, 1, 0.0), (2, 32768, 0, 1e-5)]:
        wl = Workload("n", T=T, K=8, H=H, norm_kind=kind, eps=eps, r_sigma=2.0, seed=T,
                      gamma_mode="plain" if kind else "one_plus")
        d = make_inputs(wl)
        y = make_inputs(wl, seed=100 + T)["r0"]
        r_dev = dev_bf16(d["r0"], extra_rows=2)
        out = dev_bf16(np.zeros_like(d["r0"]), extra_rows=2, fill_bits=0x7FC2)
        fln.add_rmsnorm(dev_bf16(y), r_dev[:T], torch.from_numpy(d["gamma"]).cuda(), eps, kind, out=out[:T])
        fln.fln_device_status()
        rb, ob = host_bits(r_dev), host_bits(out)
        assert np.all(rb[T:] == 0x7FC1) and np.all(ob[T:] == 0x7FC2)
        r, o, _ = oracle.add_rmsnorm(y, d["r0"], d["gamma"], eps, kind)
        compare(rb[:T], r, f"add_rmsnorm T={T} H={H} residual")
        compare(ob[:T], o, f"add_rmsnorm T={T} H={H} out")


def test_minimal_shapes():
    for T, K, H in [(1, 8, 8), (2, 64, 16), (129, 8, 24)]:
        wl = Workload("min", T=T, K=K, H=H, eps=1e-5, seed=T + K)
        d = make_inputs(wl)
        run = Run(d, wl.eps, wl.norm_kind)
        for p in (plan(fln.PATH_FUSED), plan(fln.PATH_PIPELINED, tile_n=128), UNFUSED):
            if p is UNFUSED and T > 256:
                continue
            rb, ob = run(p)
            check_rows(rb, ob, d, wl, name=f"min {T}x{K}x{H} {p['path']}")


def test_errors_reported_on_device():
    import torch
    wl = workload("tiny")
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    out = torch.empty((16, 256), dtype=torch.bfloat16, device="cuda")
    host_x = torch.zeros((16, 256), dtype=torch.bfloat16)
    r = run.x.clone()
    rc = fln.fused_proj_add_rmsnorm_ptr(host_x.data_ptr(), run.W.data_ptr(), r.data_ptr(), run.gamma.data_ptr(),
                                        1e-6, 0, 16, 256, 256, 0, out.data_ptr(), 0)
    assert rc == fln.FLN_ERR_INVALID_ARG and "device pointer" in fln.fln_last_error()
    rc = fln.fused_proj_add_rmsnorm_ptr(run.x.data_ptr() + 2, run.W.data_ptr(), r.data_ptr(), run.gamma.data_ptr(),
                                        1e-6, 0, 16, 256, 256, 0, out.data_ptr(), 0)
    assert rc == fln.FLN_ERR_INVALID_ARG and "aligned" in fln.fln_last_error()
    rc = fln.fused_proj_add_rmsnorm_ptr(run.x.data_ptr(), run.W.data_ptr(), r.data_ptr(), run.gamma.data_ptr(),
                                        1e-6, 0, 16, 256, 256, 0, r.data_ptr(), 0)
    assert rc == fln.FLN_ERR_INVALID_ARG and "overlap" in fln.fln_last_error()
    fln.fln_set_plan(256, 256, 0, plan(fln.PATH_FUSED, tuned_max=8))
    try:
        rc = fln.fused_proj_add_rmsnorm_ptr(run.x.data_ptr(), run.W.data_ptr(), r.data_ptr(), run.gamma.data_ptr(),
                                            1e-6, 0, 16, 256, 256, 0, out.data_ptr(), 0)
        assert rc == fln.FLN_ERR_NOT_TUNED
    finally:
        fln.fln_set_plan(256, 256, 0, None)
    fln.fln_device_status()


def test_autotune_then_auto_calls():
    wl = Workload("tune", T=1024, K=512, H=1024, eps=1e-5, r_sigma=2.0, seed=7)
    fln.fln_autotune(wl.K, wl.H, wl.norm_kind, wl.T)
    try:
        p = fln.fln_get_plan(wl.K, wl.H, wl.norm_kind, wl.T)
        assert p["tuned_max_tokens"] == wl.T
        assert p["path"] in (fln.PATH_FUSED, fln.PATH_PIPELINED)
        d = make_inputs(wl)
        run = Run(d, wl.eps, wl.norm_kind)
        for T in (1, 64, 300, 1024):
            rb, ob = run(None, chunk=0, T=T)
            dd = {k: (v[:T] if k in ("x", "r0") else v) for k, v in d.items()}
            check_rows(rb, ob, dd, wl, name=f"tuned T={T}")
        with pytest.raises(fln.FlnError) as e:
            fln.fln_get_plan(wl.K, wl.H, wl.norm_kind, 1025)
        assert e.value.status == fln.FLN_ERR_NOT_TUNED
    finally:
        fln.fln_set_plan(wl.K, wl.H, wl.norm_kind, None)


# --------------------------------------------------------------- full sizes
# Every element of every full-size workload is compared with the oracle (the
# OpenMP oracle does the largest, 8192 x 14336 x 4096, in about half a minute
# on 16 host cores).  One oracle result is kept at a time and shared by the
# paths that are checked against it.
_full_cache = {}


def _full(name, T=None):
    key = (name, T)
    if key not in _full_cache:
        _full_cache.clear()
        wl = workload(name)
        d = make_inputs(wl, T=T) if T else make_inputs(wl)
        r, o, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)
        _full_cache[key] = (wl, d, r, o)
    return _full_cache[key]


def _check_full(rb, ob, ref_r, ref_o, name):
    sr = compare(rb, ref_r, name + " residual")
    so = compare(ob, ref_o, name + " out")
    return sr, so


FULL = ["llama3_8b_oproj", "llama3_8b_down", "gemma2_9b_down"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_prefill_every_row(name):
    wl, d, ref_r, ref_o = _full(name)
    run = Run(d, wl.eps, wl.norm_kind)
    for p in (plan(fln.PATH_FUSED, chunk=min(wl.T, 4096)), plan(fln.PATH_PIPELINED, chunk=1024)):
        rb, ob = run(p)
        _check_full(rb, ob, ref_r, ref_o, f"{name} path={p['path']}")


def test_full_size_chunk_sweep_bitwise():
    """K = 4096 is below the K-blocks from which the fused kernel splits a last round, so every chunk size
    runs the same arithmetic per tile: bit for bit the same results."""
    wl, d, ref_r, ref_o = _full("llama3_8b_oproj")
    run = Run(d, wl.eps, wl.norm_kind)
    base = run(plan(fln.PATH_FUSED, chunk=4096))
    for c in (256, 512, 1024):
        rb, ob = run(plan(fln.PATH_FUSED, chunk=c))
        assert np.array_equal(rb, base[0]) and np.array_equal(ob, base[1]), c
    _check_full(base[0], base[1], ref_r, ref_o, "oproj chunk sweep")


@pytest.mark.parametrize("name", ["llama70b_oproj_decode", "llama70b_down_decode"])
@pytest.mark.parametrize("T", [1, 8, 32, 128, 256])
def test_full_size_decode_every_row(name, T):
    wl, d, ref_r, ref_o = _full(name, T)
    run = Run(d, wl.eps, wl.norm_kind)
    for tail in (256, 0):
        with tail_tokens(tail):
            rb, ob = run(UNFUSED)
        _check_full(rb, ob, ref_r, ref_o, f"{name} T={T} unfused tail={tail}")
    rb, ob = run(plan(fln.PATH_FUSED, chunk=T))
    _check_full(rb, ob, ref_r, ref_o, f"{name} T={T} fused")


# --------------------------------------------------------------- SM split of the PIPELINED path
@pytest.mark.parametrize("wl", [
    Workload("split_ragged", T=700, K=320, H=640, eps=1e-5, r_sigma=2.0, seed=41),
    Workload("split_gemma", T=333, K=448, H=3584, norm_kind=1, eps=1e-6, gamma_mode="plain", seed=42),
], ids=lambda w: w.name)
@pytest.mark.parametrize("gemm_ctas", [0, 8, 64])
def test_pipelined_sm_split_full_parity(wl, gemm_ctas):
    """The PIPELINED path with the GEMM grid held to a CTA target and the second-stream add + norm
    capped at 1, 8 or a quarter of the SMs (the SM-count split the tuner sweeps), on ragged shapes with
    more chunks than slots: every element against the oracle, and bitwise equal to the uncapped run
    (the cap changes which CTA handles a row, not the row's arithmetic)."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    d = make_inputs(wl)
    run = Run(d, wl.eps, wl.norm_kind)
    r, o, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind)
    base = None
    for norm_ctas in (0, 1, 8, sms // 4):
        for tile in (256, 128):
            rb, ob = run(plan(fln.PATH_PIPELINED, chunk=128, tile_n=tile, gemm_ctas=gemm_ctas, norm_ctas=norm_ctas))
            _check_full(rb, ob, r, o, f"{wl.name} pipelined tile={tile} gemm_ctas={gemm_ctas} norm_ctas={norm_ctas}")
            if tile == 256:
                if base is None:
                    base = (rb, ob)
                assert np.array_equal(rb, base[0]) and np.array_equal(ob, base[1]), norm_ctas
