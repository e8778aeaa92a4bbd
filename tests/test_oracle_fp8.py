"""Pins for the oracle's FP8 (E4M3) region, independent of the oracle's own code.

* the value of every one of the 256 codes against PyTorch's float8_e4m3fn
  conversion (a library routine), plus hand-checked codes of the format;
* a hand-worked 2x2 case with per-token and per-channel scales;
* at unit scales the FP8 region equals the bf16 region (pinned separately in
  test_oracle.py) on the same values, bit for bit: every E4M3 value is a bf16
  value;
* exact scale laws: power-of-two scales multiply y exactly; a per-token
  (per-channel) scale acts on its row (column) alone; one scale per tensor
  equals the same value repeated per row.
Runs on the CPU only.
"""
import math

import numpy as np
import pytest

import oracle
from synth import Workload, f32_to_bf16_bits, make_inputs_fp8

torch = pytest.importorskip("torch")


def _lib_decode(codes):
    t = torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_every_code_matches_library_decode():
    codes = np.arange(256, dtype=np.uint8)
    ours = np.array([oracle.e4m3_to_double(c) for c in codes])
    ref = _lib_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert sorted(np.nonzero(nan)[0].tolist()) == [0x7F, 0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, oracle.e4m3_to_double(0x80)) == -1.0


@pytest.mark.parametrize("code,value", [
    (0x38, 1.0), (0x40, 2.0), (0x44, 3.0), (0x48, 4.0), (0x3C, 1.5), (0xB8, -1.0),
    (0x7E, 448.0),                 # largest finite: 1.75 * 2^8
    (0x08, 2.0 ** -6),             # smallest normal
    (0x01, 2.0 ** -9),             # smallest subnormal: 1/8 * 2^-6
    (0x07, 7 * 2.0 ** -9),         # largest subnormal
    (0x00, 0.0),
])
def test_format_facts(code, value):
    assert oracle.e4m3_to_double(code) == value


def test_hand_worked_scaled_case():
    # x = [[1,2],[3,4]], W = [[1,0],[1,1]], r0 = [[1,-1],[0,2]]; x.W^T = [[1,3],[3,7]]
    x8 = np.array([[0x38, 0x40], [0x44, 0x48]], np.uint8)
    W8 = np.array([[0x38, 0x00], [0x38, 0x38]], np.uint8)
    r0 = f32_to_bf16_bits(np.array([[1, -1], [0, 2]], np.float32))
    sx = np.array([0.5, 2.0], np.float32)     # per token
    sw = np.array([1.0, 0.25], np.float32)    # per output row of W
    gamma = np.array([1.0, 1.0], np.float32)
    r, o, ms = oracle.proj_add_rmsnorm_fp8(x8, sx, W8, sw, r0, gamma, 0.0, 0)
    # y = [[0.5*1*1, 0.5*0.25*3], [2*1*3, 2*0.25*7]] = [[0.5, 0.375], [6, 3.5]]
    np.testing.assert_array_equal(r, [[1.5, -0.625], [6.0, 5.5]])
    ms_ref = [(1.5 ** 2 + 0.625 ** 2) / 2, (36 + 30.25) / 2]
    np.testing.assert_allclose(ms, ms_ref, rtol=1e-15)
    o_ref = np.array([[1.5, -0.625], [6.0, 5.5]]) / np.sqrt(np.array(ms_ref))[:, None]
    np.testing.assert_allclose(o, o_ref, rtol=2e-15, atol=0)


def _small(T=5, K=48, H=24, seed=3, per_token=True, per_channel=True, kind=0):
    wl = Workload("fp8pin", T=T, K=K, H=H, norm_kind=kind, eps=1e-5, r_sigma=2.0, seed=seed,
                  gamma_mode="plain" if kind else "one_plus")
    return wl, make_inputs_fp8(wl, x_scale_per_token=per_token, w_scale_per_channel=per_channel)


@pytest.mark.parametrize("kind", [0, 1])
def test_unit_scales_equal_bf16_region(kind):
    wl, d = _small(kind=kind)
    # the E4M3 values as bf16 bit patterns (exact: 3 fraction bits, exponents 2^-9..2^8)
    xv = _lib_decode(d["x8"]).astype(np.float32)
    wv = _lib_decode(d["W8"]).astype(np.float32)
    xb, wb = f32_to_bf16_bits(xv), f32_to_bf16_bits(wv)
    back = (xb.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, xv)
    one = np.ones(1, np.float32)
    r8, o8, ms8 = oracle.proj_add_rmsnorm_fp8(d["x8"], one, d["W8"], one, d["r0"], d["gamma"], wl.eps, kind)
    rb, ob, msb = oracle.proj_add_rmsnorm(xb, wb, d["r0"], d["gamma"], wl.eps, kind)
    assert np.array_equal(r8, rb) and np.array_equal(o8, ob) and np.array_equal(ms8, msb)


def test_power_of_two_scales_are_exact():
    wl, d = _small()
    one = np.ones(1, np.float32)
    r1, _, _ = oracle.proj_add_rmsnorm_fp8(d["x8"], one, d["W8"], one, d["r0"], d["gamma"], wl.eps, 0)
    y1 = r1 - _r0(d)
    r2, _, _ = oracle.proj_add_rmsnorm_fp8(d["x8"], np.float32([0.25]), d["W8"], np.float32([8.0]), d["r0"],
                                           d["gamma"], wl.eps, 0)
    np.testing.assert_array_equal(r2 - _r0(d), 2.0 * y1)


def _r0(d):
    return (d["r0"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_per_token_and_per_channel_scales_act_on_their_row_and_column():
    wl, d = _small()
    T, H = d["r0"].shape
    one = np.ones(1, np.float32)
    r1, _, _ = oracle.proj_add_rmsnorm_fp8(d["x8"], one, d["W8"], one, d["r0"], d["gamma"], wl.eps, 0)
    y1 = r1 - _r0(d)
    sx = np.exp2(np.arange(T) % 3 - 1).astype(np.float32)    # 1/2, 1, 2, ...
    sw = np.exp2(-(np.arange(H) % 4)).astype(np.float32)     # 1, 1/2, 1/4, 1/8, ...
    r, _, _ = oracle.proj_add_rmsnorm_fp8(d["x8"], sx, d["W8"], sw, d["r0"], d["gamma"], wl.eps, 0)
    np.testing.assert_array_equal(r - _r0(d), y1 * sx[:, None].astype(np.float64) * sw[None, :].astype(np.float64))


def test_tensor_scale_equals_repeated_row_scale():
    wl, d = _small(per_token=False, per_channel=False)
    T, H = d["r0"].shape
    a = oracle.proj_add_rmsnorm_fp8(d["x8"], d["x_scale"], d["W8"], d["w_scale"], d["r0"], d["gamma"], wl.eps, 0)
    b = oracle.proj_add_rmsnorm_fp8(d["x8"], np.repeat(d["x_scale"], T), d["W8"], np.repeat(d["w_scale"], H),
                                    d["r0"], d["gamma"], wl.eps, 0)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_selected_rows_match_full_run():
    wl, d = _small(T=9)
    full = oracle.proj_add_rmsnorm_fp8(d["x8"], d["x_scale"], d["W8"], d["w_scale"], d["r0"], d["gamma"], wl.eps, 0)
    rows = [7, 0, 4]
    part = oracle.proj_add_rmsnorm_fp8(d["x8"], d["x_scale"], d["W8"], d["w_scale"], d["r0"], d["gamma"], wl.eps, 0,
                                       rows=rows)
    for u, v in zip(full, part):
        assert np.array_equal(u[rows], v)


def test_projection_against_float64_matmul():
    wl, d = _small(T=6, K=80, H=40)
    xv = _lib_decode(d["x8"])
    wv = _lib_decode(d["W8"])
    y = (xv @ wv.T) * d["x_scale"].astype(np.float64)[:, None] * d["w_scale"].astype(np.float64)[None, :]
    r, _, _ = oracle.proj_add_rmsnorm_fp8(d["x8"], d["x_scale"], d["W8"], d["w_scale"], d["r0"], d["gamma"], wl.eps, 0)
    np.testing.assert_allclose(r - _r0(d), y, rtol=1e-12, atol=1e-12)
