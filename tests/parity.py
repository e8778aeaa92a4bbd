"""Parity gate between a bf16 GPU result and the fp64 oracle.

Tolerance (spec: max-abs <= 2e-2 and mean-abs <= 2e-3 on the normed
output and the residual), read for bf16 outputs:
  * each GPU value is compared with the oracle value rounded to bf16;
  * per element |gpu - oracle_bf16| <= max(2e-2, one bf16 ulp of oracle_bf16):
    two correct fp32 evaluations that land on opposite sides of a rounding
    midpoint differ by one ulp, and for |value| >= 4 that ulp (>= 2^-5)
    exceeds 2e-2 by itself;
  * mean |gpu - oracle_bf16| <= 2e-3.
  * "tight" (paths that keep y and r in fp32 until the final rounding):
    |gpu - oracle_fp64| <= half a bf16 ulp + 2^-12 * max(|oracle|, 1), i.e.
    the GPU value is the correctly rounded exact result up to fp32-level
    error; a path that rounded r to bf16 before normalising fails it.
Raw errors against the unrounded fp64 values are returned too.
"""
from __future__ import annotations

import numpy as np

import oracle
from synth import bf16_bits_to_f32

ATOL = 2e-2
MEAN_TOL = 2e-3
TIGHT_REL = 2.0 ** -12


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    out = np.zeros_like(a)
    nz = a > 0
    e = np.floor(np.log2(a[nz]))
    e = np.maximum(e, -126.0)
    out[nz] = 2.0 ** (e - 7)
    return out


def compare(gpu_bits: np.ndarray, ref64: np.ndarray, name: str = "", tight: bool = True) -> dict:
    g = bf16_bits_to_f32(gpu_bits).astype(np.float64)
    ref64 = np.asarray(ref64, np.float64)
    assert g.shape == ref64.shape, (g.shape, ref64.shape)
    rb = bf16_bits_to_f32(oracle.round_to_bf16(ref64)).astype(np.float64)
    d = np.abs(g - rb)
    allowed = np.maximum(ATOL, bf16_ulp(rb))
    raw = np.abs(g - ref64)
    stats = {
        "name": name,
        "n": int(g.size),
        "max_abs_vs_rounded": float(d.max()) if d.size else 0.0,
        "mean_abs_vs_rounded": float(d.mean()) if d.size else 0.0,
        "max_abs_vs_fp64": float(raw.max()) if raw.size else 0.0,
        "mean_abs_vs_fp64": float(raw.mean()) if raw.size else 0.0,
        "ulp_flips": int(np.count_nonzero(d > 0)),
    }
    if not np.all(np.isfinite(g)):
        raise AssertionError(f"{name}: non-finite GPU values")
    bad = d > allowed
    if bad.any():
        i = np.flatnonzero(bad.reshape(-1))[0]
        idx = np.unravel_index(i, g.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} elements beyond tolerance; first at {idx}: "
                             f"gpu={g[idx]!r} oracle={ref64[idx]!r} stats={stats}")
    if d.size and d.mean() > MEAN_TOL:
        raise AssertionError(f"{name}: mean abs error {d.mean()} > {MEAN_TOL}; stats={stats}")
    if tight:
        lim = 0.5 * bf16_ulp(ref64) + TIGHT_REL * np.maximum(np.abs(ref64), 1.0)
        badt = raw > lim
        if badt.any():
            i = np.flatnonzero(badt.reshape(-1))[0]
            idx = np.unravel_index(i, g.shape)
            raise AssertionError(f"{name}: {int(badt.sum())} elements are not the fp32-accurate rounding; first at "
                                 f"{idx}: gpu={g[idx]!r} oracle={ref64[idx]!r} stats={stats}")
    return stats
