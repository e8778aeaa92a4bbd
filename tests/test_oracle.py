"""Pins for the fp64 oracle, independent of the oracle's own code.

Each check is a hand-worked value, a closed form, an invariant of the
definition, or a library routine (numpy float64 matmul) on a special case.
Runs on the CPU only.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from synth import Workload, bf16_bits_to_f32, f32_to_bf16_bits, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _bf16(a):
    return f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def _ev(expr):
    return float(eval(expr, {"__builtins__": {}}, {"sqrt": math.sqrt}))


def _evm(m):
    return np.array([[_ev(e) for e in row] for row in m], dtype=np.float64)


def _load_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _load_cases(), ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    x = _bf16(case["x"])
    W = _bf16(case["W"])
    r0 = _bf16(case["r0"])
    gamma = np.array(case["gamma"], np.float32)
    # the fixtures are exactly representable in bf16
    assert np.array_equal(bf16_bits_to_f32(x), np.array(case["x"], np.float32))
    r, o, ms = oracle.proj_add_rmsnorm(x, W, r0, gamma, _ev(case["eps"]), case["norm_kind"])
    np.testing.assert_allclose(r, _evm(case["r"]), rtol=0, atol=0)
    np.testing.assert_allclose(ms, [_ev(e) for e in case["ms"]], rtol=1e-15, atol=0)
    np.testing.assert_allclose(o, _evm(case["o"]), rtol=2e-15, atol=1e-15)


def test_bf16_rounding_fixed_points():
    cases = [
        (1.0, 0x3F80),
        (-2.5, 0xC020),
        (1.0 + 2.0 ** -8, 0x3F80),                 # tie -> even (down)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),             # tie -> even (up)
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),    # above the tie -> up
        (2.0 ** -133, 0x0001),                     # smallest subnormal
        (2.0 ** -134, 0x0000),                     # half of it, tie -> even zero
        (3.4e38, 0x7F80),                          # beyond the last tie -> inf
        (3.3895313892515355e38, 0x7F7F),           # largest finite bf16
        (0.0, 0x0000),
        (-0.0, 0x8000),
    ]
    for v, bits in cases:
        assert oracle.round_to_bf16(np.array([v]))[0] == bits, (v, hex(bits))


def test_bf16_rounding_is_nearest_by_brute_force():
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        rng.standard_normal(2000) * 1e-39])
    b = oracle.round_to_bf16(v).astype(np.int64)
    dec = lambda bits: bf16_bits_to_f32(np.asarray(bits, np.int64).astype(np.uint16)).astype(np.float64)
    here = np.abs(v - dec(b))
    # neighbours one code up / down in magnitude (sign kept)
    mag = b & 0x7FFF
    sign = b & 0x8000
    up = dec(sign | np.minimum(mag + 1, 0x7F7F))
    dn = dec(sign | np.maximum(mag - 1, 0))
    assert np.all(here <= np.abs(v - up))
    assert np.all(here <= np.abs(v - dn))
    ties = (here == np.abs(v - up)) | (here == np.abs(v - dn))
    assert np.all((b[ties] & 1) == 0)


def _small(T=8, K=96, H=80, kind=0, eps=1e-5, seed=3, gamma_mode="one_plus"):
    wl = Workload("t", T=T, K=K, H=H, norm_kind=kind, eps=eps, r_sigma=2.0, seed=seed,
                  gamma_mode=gamma_mode)
    return wl, make_inputs(wl)


def test_projection_matches_numpy_matmul():
    wl, d = _small(T=12, K=200, H=72)
    zero = np.zeros_like(d["r0"])
    r, _, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], zero, d["gamma"], wl.eps, 0)
    x = bf16_bits_to_f32(d["x"]).astype(np.float64)
    W = bf16_bits_to_f32(d["W"]).astype(np.float64)
    ref = x @ W.T
    np.testing.assert_allclose(r, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_unit_rms_invariant_standard_and_gemma():
    for kind, gval in ((0, 1.0), (1, 0.0)):
        wl, d = _small(kind=kind, eps=1e-6)
        g = np.full(wl.H, gval, np.float32)
        _, o, ms = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], g, wl.eps, kind)
        rms = np.sqrt(np.mean(o * o, axis=1))
        np.testing.assert_allclose(rms, np.sqrt(ms / (ms + wl.eps)), rtol=1e-12)
        assert np.all(np.abs(rms - 1.0) <= wl.eps / (2 * ms) + 1e-12)


def test_gemma_zero_equals_standard_one_bitwise():
    wl, d = _small()
    _, o_std, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], np.ones(wl.H, np.float32), wl.eps, 0)
    _, o_gem, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], np.zeros(wl.H, np.float32), wl.eps, 1)
    assert np.array_equal(o_std, o_gem)


def test_gemma_shifts_weight_by_one():
    wl, d = _small()
    gam = (np.round(d["gamma"].astype(np.float64) * 64) / 64 - 1).astype(np.float32)  # 1+gam exact
    _, o_gem, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], gam, wl.eps, 1)
    _, o_std, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], (gam + 1).astype(np.float32), wl.eps, 0)
    assert np.array_equal(o_std, o_gem)


def test_residual_add_is_linear():
    wl, d = _small(T=6, K=64, H=48)
    _, d2 = _small(T=6, K=64, H=48, seed=11)
    r1, _, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, 0)
    r2, _, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d2["r0"], d["gamma"], wl.eps, 0)
    dr = bf16_bits_to_f32(d["r0"]).astype(np.float64) - bf16_bits_to_f32(d2["r0"]).astype(np.float64)
    np.testing.assert_allclose(r1 - r2, dr, rtol=0, atol=1e-12)
    # doubling x (exact in bf16) doubles y = r - r0
    x2 = _bf16(bf16_bits_to_f32(d["x"]) * 2)
    r3, _, _ = oracle.proj_add_rmsnorm(x2, d["W"], d["r0"], d["gamma"], wl.eps, 0)
    r0 = bf16_bits_to_f32(d["r0"]).astype(np.float64)
    np.testing.assert_allclose(r3 - r0, 2 * (r1 - r0), rtol=1e-13, atol=1e-13)


def test_scale_invariance_without_eps():
    wl, d = _small()
    _, o1, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], 0.0, 0)
    x4 = _bf16(bf16_bits_to_f32(d["x"]) * 4)
    r4 = _bf16(bf16_bits_to_f32(d["r0"]) * 4)
    _, o4, _ = oracle.proj_add_rmsnorm(x4, d["W"], r4, d["gamma"], 0.0, 0)
    np.testing.assert_allclose(o1, o4, rtol=1e-14, atol=1e-14)


def test_rows_are_independent_and_selectable():
    wl, d = _small(T=10)
    r, o, ms = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, 0)
    rows = [7, 0, 3, 3]
    rs, os_, mss = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, 0, rows=rows)
    assert np.array_equal(rs, r[rows]) and np.array_equal(os_, o[rows]) and np.array_equal(mss, ms[rows])
    # permuting token rows permutes the outputs
    p = np.random.default_rng(0).permutation(wl.T)
    rp, op, _ = oracle.proj_add_rmsnorm(d["x"][p], d["W"], d["r0"][p], d["gamma"], wl.eps, 0)
    assert np.array_equal(rp, r[p]) and np.array_equal(op, o[p])


def test_joint_k_permutation_leaves_projection_unchanged():
    wl, d = _small(T=5, K=128, H=40)
    r, _, _ = oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, 0)
    p = np.random.default_rng(1).permutation(wl.K)
    rp, _, _ = oracle.proj_add_rmsnorm(d["x"][:, p], d["W"][:, p], d["r0"], d["gamma"], wl.eps, 0)
    np.testing.assert_allclose(rp, r, rtol=1e-13, atol=1e-13)


def test_zero_input_and_identity_weight_are_exact():
    wl, d = _small(T=4, K=64, H=64)
    r, _, _ = oracle.proj_add_rmsnorm(np.zeros_like(d["x"]), d["W"], d["r0"], d["gamma"], wl.eps, 0)
    assert np.array_equal(r, bf16_bits_to_f32(d["r0"]).astype(np.float64))
    eye = _bf16(np.eye(64))
    r, o, _ = oracle.proj_add_rmsnorm(d["x"], eye, d["r0"], d["gamma"], wl.eps, 0)
    exp = bf16_bits_to_f32(d["r0"]).astype(np.float64) + bf16_bits_to_f32(d["x"]).astype(np.float64)
    assert np.array_equal(r, exp)
    # the add+norm oracle on y = x agrees bit for bit with the projection through W = I
    r2, o2, _ = oracle.add_rmsnorm(d["x"], d["r0"], d["gamma"], wl.eps, 0)
    assert np.array_equal(r2, r) and np.array_equal(o2, o)


def test_constant_row_closed_form():
    H = 64
    for a in (0.5, 3.0, -7.0):
        r0 = _bf16(np.full((1, H), a))
        y = np.zeros((1, H), np.uint16)
        g = np.linspace(-2, 2, H).astype(np.float32)
        _, o, ms = oracle.add_rmsnorm(y, r0, g, a * a, 0)      # eps = a^2
        assert ms[0] == a * a
        np.testing.assert_allclose(o[0], np.sign(a) * g.astype(np.float64) / math.sqrt(2), rtol=1e-15, atol=1e-15)


def test_bad_arguments_are_rejected():
    wl, d = _small(T=2, K=16, H=16)
    with pytest.raises(ValueError):
        oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], -1.0, 0)
    with pytest.raises(ValueError):
        oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], 1e-5, 2)
    with pytest.raises(ValueError):
        oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], 1e-5, 0, rows=[5])
