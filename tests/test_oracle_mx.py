"""Pins for the oracle's MXFP4-weight region, independent of the oracle's own code.

* every E8M0 code against the closed form 2^(E-127), and 255 as NaN;
* a hand-worked 2x2 case (nibble order, two scales, no tensor scale);
* with every scale 1 (E = 127) the region equals the bf16 region (pinned in
  test_oracle.py) on the same weight values, bit for bit;
* exact scale laws: E + 1 on every block of one weight row doubles that
  column of y; a change of the scale of elements 32..63 of a row changes y by
  x[:, 32:64] times the weight change there, so blocks are 32 wide;
* a NaN scale turns exactly its row's column of y into NaN;
* a float64 matmul on weights decoded here from the E2M1 table and the
  closed form of the scales.
Runs on the CPU only.
"""
import math

import numpy as np
import pytest

import oracle
from synth import Workload, f32_to_bf16_bits, make_inputs_mxfp4

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e8m0_closed_form():
    for E in range(255):
        assert oracle.e8m0_to_double(E) == math.ldexp(1.0, E - 127)
    assert math.isnan(oracle.e8m0_to_double(255))


def _dequant(Wq, S):
    H, half = Wq.shape
    K = 2 * half
    codes = np.empty((H, K), np.int64)
    codes[:, 0::2] = Wq & 0xF
    codes[:, 1::2] = Wq >> 4
    vals = np.array(E2M1)[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    scale = np.ldexp(1.0, S.astype(np.int64) - 127)[:, np.arange(K) // 32]
    return scale * vals


def test_hand_worked_case():
    # x = [[1,2],[3,4]]; W row 0 = [1, 1.5] (codes 2, 3 -> byte 0x32) with scale 2 (E = 128) -> [2, 3];
    # row 1 = [-2, 6] (codes 0xC, 7 -> byte 0x7C) with scale 0.5 (E = 126) -> [-1, 3]
    x = f32_to_bf16_bits(np.array([[1, 2], [3, 4]], np.float32))
    Wq = np.array([[0x32], [0x7C]], np.uint8)
    S = np.array([[128], [126]], np.uint8)
    r0 = f32_to_bf16_bits(np.zeros((2, 2), np.float32))
    g = np.ones(2, np.float32)
    r, o, ms = oracle.proj_add_rmsnorm_mxfp4(x, Wq, S, r0, g, 0.0, 0)
    np.testing.assert_array_equal(r, [[8.0, 5.0], [18.0, 9.0]])
    np.testing.assert_allclose(ms, [44.5, 202.5], rtol=1e-15)
    np.testing.assert_allclose(o, np.array([[8, 5], [18, 9]]) / np.sqrt([[44.5], [202.5]]), rtol=2e-15)


def _small(T=5, K=96, H=24, seed=5, kind=0):
    wl = Workload("mxpin", T=T, K=K, H=H, norm_kind=kind, eps=1e-5, r_sigma=2.0, seed=seed,
                  gamma_mode="plain" if kind else "one_plus")
    return wl, make_inputs_mxfp4(wl)


def _r0(d):
    return (d["r0"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _run(d, wl, S=None, kind=0):
    return oracle.proj_add_rmsnorm_mxfp4(d["x"], d["Wq"], d["S"] if S is None else S, d["r0"], d["gamma"], wl.eps,
                                         kind)


@pytest.mark.parametrize("kind", [0, 1])
def test_unit_scales_equal_bf16_region(kind):
    wl, d = _small(kind=kind)
    S = np.full_like(d["S"], 127)
    w = _dequant(d["Wq"], S)
    wb = f32_to_bf16_bits(w.astype(np.float32))
    assert np.array_equal((wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), w)
    a = oracle.proj_add_rmsnorm_mxfp4(d["x"], d["Wq"], S, d["r0"], d["gamma"], wl.eps, kind)
    b = oracle.proj_add_rmsnorm(d["x"], wb, d["r0"], d["gamma"], wl.eps, kind)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_row_scales_double_their_column():
    wl, d = _small()
    r1, _, _ = _run(d, wl)
    S2 = d["S"].copy()
    S2[3] += 1
    r2, _, _ = _run(d, wl, S2)
    y1, y2 = r1 - _r0(d), r2 - _r0(d)
    np.testing.assert_array_equal(y2[:, 3], 2.0 * y1[:, 3])
    cols = [h for h in range(y1.shape[1]) if h != 3]
    np.testing.assert_array_equal(y2[:, cols], y1[:, cols])


def test_blocks_are_32_wide():
    wl, d = _small(K=128)
    r1, _, _ = _run(d, wl)
    S2 = d["S"].copy()
    S2[0, 1] += 2  # elements 32..63 of row 0 times 4
    r2, _, _ = _run(d, wl, S2)
    xv = (d["x"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    dw = _dequant(d["Wq"], S2)[0] - _dequant(d["Wq"], d["S"])[0]
    assert np.all(dw[:32] == 0) and np.all(dw[64:] == 0) and np.any(dw[32:64] != 0)
    np.testing.assert_allclose((r2 - r1)[:, 0], xv @ dw, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal((r2 - r1)[:, 1:], 0.0)


def test_nan_scale_poisons_its_column():
    wl, d = _small()
    S2 = d["S"].copy()
    S2[5, 0] = 255
    r, _, _ = _run(d, wl, S2)
    assert np.all(np.isnan(r[:, 5]))
    assert not np.any(np.isnan(np.delete(r, 5, axis=1)))


def test_projection_against_float64_matmul():
    wl, d = _small(T=6, K=160, H=40)
    xv = (d["x"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y = xv @ _dequant(d["Wq"], d["S"]).T
    r, _, _ = _run(d, wl)
    np.testing.assert_allclose(r - _r0(d), y, rtol=1e-12, atol=1e-12)


def test_selected_rows_match_full_run():
    wl, d = _small(T=9)
    full = _run(d, wl)
    rows = [8, 0, 5]
    part = oracle.proj_add_rmsnorm_mxfp4(d["x"], d["Wq"], d["S"], d["r0"], d["gamma"], wl.eps, 0, rows=rows)
    for u, v in zip(full, part):
        assert np.array_equal(u[rows], v)
