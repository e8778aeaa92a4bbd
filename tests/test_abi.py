"""Host-side checks of the C ABI (no GPU needed).

The library builds for sm_103a, loads, exports every entry point the public
header declares, and its host logic (argument validation, overrides, plans,
token threshold, the profiled-maximum rule) answers without launching
anything.
"""
import os
import re
import subprocess

import pytest

import decoder_layer_projection_gb300 as fln

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "libfusedln.h")


@pytest.fixture(scope="module")
def lib():
    fln.build()
    return fln.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set()
    for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", src, flags=re.M):
        line = src[m.start():src.index("\n", m.start())]
        if line.lstrip().startswith(("typedef", "#", "return")):
            continue
        names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fused_proj_add_rmsnorm", "add_rmsnorm", "fln_autotune", "fln_set_overrides",
              "fln_last_error", "fln_release_workspace"):
        assert n in names
    assert set(names) == set(fln.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fln.lib_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)


def test_version_and_counters(lib):
    assert fln.fln_version() == 100
    assert fln.fln_launch_count() == 0


def test_overrides_validation(lib):
    assert lib.fln_set_overrides(-1, 0) == fln.FLN_ERR_INVALID_ARG
    assert lib.fln_set_overrides(5000, 0) == fln.FLN_ERR_INVALID_ARG
    assert "microchunk" in fln.fln_last_error()
    assert lib.fln_set_overrides(0, 300) == fln.FLN_ERR_INVALID_ARG
    fln.fln_set_overrides(256, 64)
    try:
        p = fln.fln_get_plan(512, 512, 0, 1000)
        assert p["microchunk_tokens"] == 256 and p["threshold_tokens"] == 64
        assert p["path"] == fln.PATH_FUSED
        assert fln.fln_get_plan(512, 512, 0, 63)["path"] == fln.PATH_UNFUSED
        # both overrides: autotune skips its scan and check, touching no device
        fln.fln_autotune(512, 512, 0, 1024, stream=0)
    finally:
        fln.fln_set_overrides(0, 0)


def test_plans_thresholds_and_profiled_maximum(lib):
    K, H = 1024, 768
    assert fln.fln_get_plan(K, H, 0, 4096)["path"] == fln.PATH_FUSED       # default plan
    assert fln.fln_get_plan(K, H, 0, 256)["path"] == fln.PATH_UNFUSED      # below default threshold
    bad = dict(path=fln.PATH_FUSED, microchunk_tokens=512, tile_n=96, gemm_ctas=0, norm_ctas=0,
               threshold_tokens=1, tuned_max_tokens=0)
    with pytest.raises(fln.FlnError) as e:
        fln.fln_set_plan(K, H, 0, bad)
    assert e.value.status == fln.FLN_ERR_INVALID_ARG
    with pytest.raises(fln.FlnError):
        fln.fln_set_plan(K, H, 0, dict(bad, tile_n=192, path=fln.PATH_PIPELINED))  # 192: FUSED only
    with pytest.raises(fln.FlnError):
        fln.fln_set_plan(K, H, 0, dict(bad, tile_n=64))  # 64: PIPELINED only
    good = dict(bad, tile_n=128, path=fln.PATH_PIPELINED, threshold_tokens=33, tuned_max_tokens=2048)
    fln.fln_set_plan(K, H, 0, good)
    try:
        assert fln.fln_get_plan(K, H, 0, 40)["path"] == fln.PATH_PIPELINED
        assert fln.fln_get_plan(K, H, 0, 32)["path"] == fln.PATH_UNFUSED
        assert fln.fln_get_plan(K, H, 1, 40)["path"] == fln.PATH_UNFUSED  # other group: default plan
        with pytest.raises(fln.FlnError) as e:
            fln.fln_get_plan(K, H, 0, 4096)  # automatic choice above the profiled maximum
        assert e.value.status == fln.FLN_ERR_NOT_TUNED
        assert fln.fln_get_plan(K, H, 0, 4096, microchunk_tokens=1024)["microchunk_tokens"] == 1024
    finally:
        fln.fln_set_plan(K, H, 0, None)
    assert fln.fln_get_plan(K, H, 0, 4096)["tuned_max_tokens"] == 0


@pytest.mark.parametrize("kw,status", [
    (dict(norm_kind=2), fln.FLN_ERR_INVALID_ARG),
    (dict(eps=-1.0), fln.FLN_ERR_INVALID_ARG),
    (dict(eps=float("nan")), fln.FLN_ERR_INVALID_ARG),
    (dict(eps=float("inf")), fln.FLN_ERR_INVALID_ARG),
    (dict(K=12), fln.FLN_ERR_INVALID_ARG),
    (dict(H=4), fln.FLN_ERR_INVALID_ARG),
    (dict(T=-1), fln.FLN_ERR_INVALID_ARG),
    (dict(microchunk_tokens=4097), fln.FLN_ERR_INVALID_ARG),
    (dict(H=32776), fln.FLN_ERR_UNSUPPORTED),
])
def test_fused_rejects_bad_arguments_before_any_launch(lib, kw, status):
    a = dict(eps=1e-5, norm_kind=0, T=16, K=256, H=256, microchunk_tokens=0)
    a.update(kw)
    rc = fln.fused_proj_add_rmsnorm_ptr(None, None, None, None, a["eps"], a["norm_kind"], a["T"], a["K"], a["H"],
                                        a["microchunk_tokens"], None, None)
    assert rc == status, fln.fln_last_error()
    assert fln.fln_last_error()
    assert fln.fln_launch_count() == 0


@pytest.mark.parametrize("kw,status", [
    (dict(norm_kind=2), fln.FLN_ERR_INVALID_ARG),
    (dict(eps=-1.0), fln.FLN_ERR_INVALID_ARG),
    (dict(K=12), fln.FLN_ERR_INVALID_ARG),
    (dict(H=4), fln.FLN_ERR_INVALID_ARG),
    (dict(T=-1), fln.FLN_ERR_INVALID_ARG),
    (dict(transfer_tokens=4097), fln.FLN_ERR_INVALID_ARG),
    (dict(transfer_tokens=-1), fln.FLN_ERR_INVALID_ARG),
    (dict(T=0), fln.FLN_OK),                      # empty call: nothing to copy or launch
])
def test_host_entry_rejects_bad_arguments_before_any_copy(lib, kw, status):
    a = dict(eps=1e-5, norm_kind=0, T=16, K=256, H=256, transfer_tokens=0)
    a.update(kw)
    rc = fln.fused_proj_add_rmsnorm_host_ptr(None, None, None, None, a["eps"], a["norm_kind"], a["T"], a["K"],
                                             a["H"], a["transfer_tokens"], None, None)
    assert rc == status, fln.fln_last_error()
    assert fln.fln_launch_count() == 0


def test_host_entry_refuses_untuned_chunks_before_any_copy(lib):
    # a group profiled up to 256 tokens: automatic chunks of 1024 exceed it, chunks of 256 do not
    K, H = 512, 256
    fln.fln_set_plan(K, H, 0, dict(path=fln.PATH_FUSED, microchunk_tokens=4096, tile_n=256, gemm_ctas=0,
                                   norm_ctas=0, threshold_tokens=1, tuned_max_tokens=256))
    try:
        rc = fln.fused_proj_add_rmsnorm_host_ptr(None, None, None, None, 1e-5, 0, 2048, K, H, 0, None, None)
        assert rc == fln.FLN_ERR_NOT_TUNED, fln.fln_last_error()
        rc = fln.fused_proj_add_rmsnorm_host_ptr(None, None, None, None, 1e-5, 0, 2048, K, H, 256, None, None)
        assert rc == fln.FLN_ERR_INVALID_ARG   # past the plan check, stopped at the NULL pointers
    finally:
        fln.fln_set_plan(K, H, 0, None)
    assert fln.fln_launch_count() == 0


@pytest.mark.parametrize("kw,status", [
    (dict(K=24), fln.FLN_ERR_INVALID_ARG),        # FP8 rows must be 16 bytes: K multiple of 16
    (dict(K=8), fln.FLN_ERR_INVALID_ARG),
    (dict(norm_kind=5), fln.FLN_ERR_INVALID_ARG),
    (dict(T=-3), fln.FLN_ERR_INVALID_ARG),
    (dict(H=12), fln.FLN_ERR_INVALID_ARG),
    (dict(microchunk_tokens=-1), fln.FLN_ERR_INVALID_ARG),
])
def test_fp8_rejects_bad_arguments_before_any_launch(lib, kw, status):
    a = dict(eps=1e-5, norm_kind=0, T=16, K=256, H=256, microchunk_tokens=0)
    a.update(kw)
    rc = lib.fused_proj_add_rmsnorm_fp8(None, None, 1, None, None, 1, None, None, a["eps"], a["norm_kind"], a["T"],
                                        a["K"], a["H"], a["microchunk_tokens"], None, None)
    assert rc == status, fln.fln_last_error()
    assert fln.fln_launch_count() == 0


def test_dtype_plans_validation(lib):
    p = fln.Plan(path=fln.PATH_FUSED, microchunk_tokens=512, tile_n=256, gemm_ctas=0, norm_ctas=0,
                 threshold_tokens=1, tuned_max_tokens=0)
    import ctypes
    assert lib.fln_set_plan_dtype(1024, 768, 0, 7, ctypes.byref(p)) == fln.FLN_ERR_INVALID_ARG
    fln.fln_set_plan(1024, 768, 0, p, dtype=fln.DTYPE_E4M3)
    try:
        assert fln.fln_get_plan(1024, 768, 0, 4096, dtype=fln.DTYPE_E4M3)["microchunk_tokens"] == 512
        assert fln.fln_get_plan(1024, 768, 0, 4096)["microchunk_tokens"] == 4096   # bf16 group untouched
    finally:
        fln.fln_set_plan(1024, 768, 0, None, dtype=fln.DTYPE_E4M3)
    assert fln.fln_get_plan(1024, 768, 0, 4096, dtype=fln.DTYPE_E4M3)["microchunk_tokens"] == 4096


def test_empty_call_is_a_no_op(lib):
    assert fln.fused_proj_add_rmsnorm_ptr(None, None, None, None, 1e-5, 0, 0, 256, 256, 0, None, None) == 0
    assert fln.add_rmsnorm_ptr(None, None, None, 1e-5, 0, 0, 256, None, None) == 0


def test_add_rmsnorm_rejects_bad_arguments(lib):
    assert fln.add_rmsnorm_ptr(None, None, None, 1e-5, 3, 4, 256, None, None) == fln.FLN_ERR_INVALID_ARG
    assert fln.add_rmsnorm_ptr(None, None, None, 1e-5, 0, 4, 100, None, None) == fln.FLN_ERR_INVALID_ARG


def test_product_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "decoder_layer_projection_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "liboracle" not in text and "oracle.c" not in text, f


def test_epilogue_warps_plan_validation(lib):
    base = dict(path=fln.PATH_FUSED, microchunk_tokens=512, tile_n=256, gemm_ctas=0, norm_ctas=0,
                threshold_tokens=1, tuned_max_tokens=0)
    for bad in (dict(epi_warps=5), dict(epi_warps=8, tile_n=128), dict(epi_warps=8, path=fln.PATH_PIPELINED)):
        with pytest.raises(fln.FlnError) as e:
            fln.fln_set_plan(1024, 768, 0, {**base, **bad})
        assert e.value.status == fln.FLN_ERR_INVALID_ARG and "epi_warps" in e.value.message
    fln.fln_set_plan(1024, 768, 0, {**base, "epi_warps": 8})
    try:
        assert fln.fln_get_plan(1024, 768, 0, 4096)["epi_warps"] == 8
    finally:
        fln.fln_set_plan(1024, 768, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(K=96), fln.FLN_ERR_INVALID_ARG),        # NVFP4 K-blocks: K multiple of 64
    (dict(K=32), fln.FLN_ERR_INVALID_ARG),
    (dict(norm_kind=4), fln.FLN_ERR_INVALID_ARG),
    (dict(T=-1), fln.FLN_ERR_INVALID_ARG),
    (dict(gs=float("nan")), fln.FLN_ERR_INVALID_ARG),
    (dict(gs=2.0 ** 101), fln.FLN_ERR_INVALID_ARG),  # the reducer scales the split-K sum by gs * 2^8
])
def test_nvfp4_rejects_bad_arguments_before_any_launch(lib, kw, status):
    a = dict(eps=1e-5, norm_kind=0, T=16, K=256, H=256, microchunk_tokens=0, gs=0.5)
    a.update(kw)
    rc = lib.fused_proj_add_rmsnorm_nvfp4(None, None, None, a["gs"], None, None, a["eps"], a["norm_kind"], a["T"],
                                          a["K"], a["H"], a["microchunk_tokens"], None, None)
    assert rc == status, fln.fln_last_error()
    assert fln.fln_launch_count() == 0


@pytest.mark.parametrize("kw,status", [
    (dict(K=192), fln.FLN_ERR_INVALID_ARG),       # MXFP4: K multiple of 128 (whole 4-byte words of scales)
    (dict(K=64), fln.FLN_ERR_INVALID_ARG),
    (dict(norm_kind=2), fln.FLN_ERR_INVALID_ARG),
    (dict(H=0), fln.FLN_ERR_INVALID_ARG),
    (dict(microchunk_tokens=5000), fln.FLN_ERR_INVALID_ARG),
])
def test_mxfp4_rejects_bad_arguments_before_any_launch(lib, kw, status):
    a = dict(eps=1e-5, norm_kind=0, T=16, K=256, H=256, microchunk_tokens=0)
    a.update(kw)
    rc = lib.fused_proj_add_rmsnorm_mxfp4(None, None, None, None, None, a["eps"], a["norm_kind"], a["T"], a["K"],
                                          a["H"], a["microchunk_tokens"], None, None)
    assert rc == status, fln.fln_last_error()
    assert fln.fln_launch_count() == 0


def test_mxfp4_plan_group_is_its_own(lib):
    import ctypes
    p = fln.Plan()
    assert lib.fln_get_plan_dtype(1024, 768, 0, fln.DTYPE_MXFP4, 64, 0, ctypes.byref(p)) == fln.FLN_OK
    assert lib.fln_get_plan_dtype(1024, 768, 0, 4, 64, 0, ctypes.byref(p)) == fln.FLN_ERR_INVALID_ARG
