"""Pins for the oracle's NVFP4-weight region, independent of the oracle's own code.

* the sixteen E2M1 codes against the OCP element table, written out here;
* a hand-worked 2x2 case (nibble order, block scale, tensor scale);
* with unit scales the region equals the bf16 region (pinned in
  test_oracle.py) on the same weight values, bit for bit: every E2M1 value
  times an E4M3 scale is a bf16 value;
* exact scale laws: a power-of-two tensor scale multiplies y exactly; scaling
  every block scale of one weight row by two doubles that column of y;
* a float64 matmul on weights dequantised here from the table and PyTorch's
  float8_e4m3fn decoding of the scales.
Runs on the CPU only.
"""
import numpy as np
import pytest

import oracle
from synth import Workload, f32_to_bf16_bits, make_inputs_nvfp4

torch = pytest.importorskip("torch")

# OCP FP4 E2M1: sign | 2 exponent bits (bias 1) | 1 fraction bit
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_table():
    for code in range(16):
        v = oracle.e2m1_to_double(code)
        mag = E2M1[code & 7]
        assert abs(v) == mag
        assert (np.signbit(v) if v == 0 else v < 0) == bool(code & 8)


def _e4m3(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _dequant(d):
    Wq, S, gs = d["Wq"], d["S"], d["gs"]
    H, half = Wq.shape
    K = 2 * half
    codes = np.empty((H, K), np.int64)
    codes[:, 0::2] = Wq & 0xF
    codes[:, 1::2] = Wq >> 4
    vals = np.array(E2M1)[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    scale = _e4m3(S)[:, np.arange(K) // 16]
    return np.float64(np.float32(gs)) * scale * vals


def test_hand_worked_case():
    # x = [[1,2],[3,4]]; W row 0 = [1, 1.5] (codes 2, 3 -> byte 0x32), row 1 = [-2, 6] (codes 0xC, 7 -> 0x7C);
    # block scales 1.0 (0x38) and 0.5 (0x30); tensor scale 2 -> w = [[2, 3], [-2, 6]]
    x = f32_to_bf16_bits(np.array([[1, 2], [3, 4]], np.float32))
    Wq = np.array([[0x32], [0x7C]], np.uint8)
    S = np.array([[0x38], [0x30]], np.uint8)
    r0 = f32_to_bf16_bits(np.zeros((2, 2), np.float32))
    g = np.ones(2, np.float32)
    r, o, ms = oracle.proj_add_rmsnorm_nvfp4(x, Wq, S, 2.0, r0, g, 0.0, 0)
    np.testing.assert_array_equal(r, [[8.0, 10.0], [18.0, 18.0]])
    np.testing.assert_allclose(ms, [82.0, 324.0], rtol=1e-15)
    np.testing.assert_allclose(o, np.array([[8, 10], [18, 18]]) / np.sqrt([[82.0], [324.0]]), rtol=2e-15)


def _small(T=5, K=96, H=24, seed=5, kind=0):
    wl = Workload("fp4pin", T=T, K=K, H=H, norm_kind=kind, eps=1e-5, r_sigma=2.0, seed=seed,
                  gamma_mode="plain" if kind else "one_plus")
    return wl, make_inputs_nvfp4(wl)


def _r0(d):
    return (d["r0"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("kind", [0, 1])
def test_unit_scales_equal_bf16_region(kind):
    wl, d = _small(kind=kind)
    d = dict(d)
    d["S"] = np.full_like(d["S"], 0x38)   # every block scale 1.0
    w = _dequant({**d, "gs": 1.0})
    wb = f32_to_bf16_bits(w.astype(np.float32))
    assert np.array_equal((wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), w)
    a = oracle.proj_add_rmsnorm_nvfp4(d["x"], d["Wq"], d["S"], 1.0, d["r0"], d["gamma"], wl.eps, kind)
    b = oracle.proj_add_rmsnorm(d["x"], wb, d["r0"], d["gamma"], wl.eps, kind)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_tensor_scale_power_of_two_is_exact():
    wl, d = _small()
    r1, _, _ = oracle.proj_add_rmsnorm_nvfp4(d["x"], d["Wq"], d["S"], d["gs"], d["r0"], d["gamma"], wl.eps, 0)
    r2, _, _ = oracle.proj_add_rmsnorm_nvfp4(d["x"], d["Wq"], d["S"], 4.0 * d["gs"], d["r0"], d["gamma"], wl.eps, 0)
    np.testing.assert_array_equal(r2 - _r0(d), 4.0 * (r1 - _r0(d)))


def test_row_block_scales_act_on_their_column():
    wl, d = _small()
    r1, _, _ = oracle.proj_add_rmsnorm_nvfp4(d["x"], d["Wq"], d["S"], d["gs"], d["r0"], d["gamma"], wl.eps, 0)
    S2 = d["S"].copy()
    S2[3] = S2[3] + 8          # E4M3 exponent field + 1: every scale of row 3 doubled
    r2, _, _ = oracle.proj_add_rmsnorm_nvfp4(d["x"], d["Wq"], S2, d["gs"], d["r0"], d["gamma"], wl.eps, 0)
    y1, y2 = r1 - _r0(d), r2 - _r0(d)
    np.testing.assert_array_equal(y2[:, 3], 2.0 * y1[:, 3])
    cols = [h for h in range(y1.shape[1]) if h != 3]
    np.testing.assert_array_equal(y2[:, cols], y1[:, cols])


def test_projection_against_float64_matmul():
    wl, d = _small(T=6, K=160, H=40)
    xv = (d["x"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y = xv @ _dequant(d).T
    r, _, _ = oracle.proj_add_rmsnorm_nvfp4(d["x"], d["Wq"], d["S"], d["gs"], d["r0"], d["gamma"], wl.eps, 0)
    np.testing.assert_allclose(r - _r0(d), y, rtol=1e-12, atol=1e-12)


def test_selected_rows_match_full_run():
    wl, d = _small(T=9)
    full = oracle.proj_add_rmsnorm_nvfp4(d["x"], d["Wq"], d["S"], d["gs"], d["r0"], d["gamma"], wl.eps, 0)
    rows = [8, 0, 5]
    part = oracle.proj_add_rmsnorm_nvfp4(d["x"], d["Wq"], d["S"], d["gs"], d["r0"], d["gamma"], wl.eps, 0,
                                         rows=rows)
    for u, v in zip(full, part):
        assert np.array_equal(u[rows], v)
