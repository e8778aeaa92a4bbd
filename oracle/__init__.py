"""fp64 CPU oracle for y = x.W^T, r = r0 + y, out = RMSNorm(r), with bf16
operands, FP8 (E4M3) operands and their dequantisation scales, or FP4
weights (E2M1 codes with E4M3 block scales and an fp32 tensor scale, or
E8M0 block scales); and for the MoE region: top-k routing, grouping of the
(token, slot) pairs by expert, the gather into grouped order, the grouped
down projection, the gated unpermute, add and norm.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg may import this package; the library under
``decoder_layer_projection_gb300`` never does.  The arithmetic lives in
``oracle.c`` (plain C, fp64); this module compiles it with gcc and marshals
numpy arrays through ctypes.  It shares no code with the CUDA path.

The definitions it follows are cited in ``oracle.c``'s header (vLLM "TPSP
Design", sections 1, 3 and 4; torch-spyre "Plugin Architecture", the
GemmaRMSNorm / RowParallelLinear rows and "Transformers backend").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

NORM_STANDARD = 0
NORM_GEMMA = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    L = ctypes.c_long
    lib.oracle_proj_add_rmsnorm.argtypes = [
        p, p, p, p, ctypes.c_double, ctypes.c_int, L, L, L, p, L, p, p, p, ctypes.c_int]
    lib.oracle_proj_add_rmsnorm.restype = ctypes.c_int
    lib.oracle_add_rmsnorm.argtypes = [
        p, p, p, ctypes.c_double, ctypes.c_int, L, L, p, p, p, ctypes.c_int]
    lib.oracle_add_rmsnorm.restype = ctypes.c_int
    lib.oracle_round_to_bf16.argtypes = [p, L, p]
    lib.oracle_round_to_bf16.restype = None
    lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_double_to_bf16.restype = ctypes.c_uint16
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_proj_add_rmsnorm_fp8.argtypes = [
        p, p, ctypes.c_int, p, p, ctypes.c_int, p, p, ctypes.c_double, ctypes.c_int, L, L, L, p, L, p, p, p,
        ctypes.c_int]
    lib.oracle_proj_add_rmsnorm_fp8.restype = ctypes.c_int
    lib.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1_to_double.restype = ctypes.c_double
    lib.oracle_proj_add_rmsnorm_nvfp4.argtypes = [
        p, p, p, ctypes.c_float, p, p, ctypes.c_double, ctypes.c_int, L, L, L, p, L, p, p, p, ctypes.c_int]
    lib.oracle_proj_add_rmsnorm_nvfp4.restype = ctypes.c_int
    lib.oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e8m0_to_double.restype = ctypes.c_double
    lib.oracle_proj_add_rmsnorm_mxfp4.argtypes = [
        p, p, p, p, p, ctypes.c_double, ctypes.c_int, L, L, L, p, L, p, p, p, ctypes.c_int]
    lib.oracle_proj_add_rmsnorm_mxfp4.restype = ctypes.c_int
    lib.oracle_moe_route.argtypes = [p, L, L, L, p, p]
    lib.oracle_moe_route.restype = ctypes.c_int
    lib.oracle_moe_permute.argtypes = [p, L, L, L, p, p, p, p]
    lib.oracle_moe_permute.restype = ctypes.c_int
    lib.oracle_moe_down_region.argtypes = [
        p, p, p, p, p, p, p, ctypes.c_double, ctypes.c_int, L, L, L, L, L, p, p, p, ctypes.c_int]
    lib.oracle_moe_down_region.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


class using_library:
    """Temporarily route this module's functions to another build of oracle.c
    (the tests use it to check that the pins catch planted mistakes)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _u16(a, shape):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands are passed as their uint16 bit patterns")
    if a.shape != shape:
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


def proj_add_rmsnorm(x, W, r0, gamma, eps, norm_kind, rows=None, nthreads=0):
    """Return (r, o, ms) in float64 for the selected token rows (all if None).

    x [T,K], W [H,K], r0 [T,H] are bf16 bit patterns (uint16); gamma [H] is
    float32.  r = r0 + x.W^T, o = RMSNorm(r), ms = mean_h r^2.
    """
    lib = _load()
    T, K = np.shape(x)
    H = np.shape(W)[0]
    x = _u16(x, (T, K))
    W = _u16(W, (H, K))
    r0 = _u16(r0, (T, H))
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    if gamma.shape != (H,):
        raise ValueError("gamma must be [H]")
    rows_arr = None
    n = T
    if rows is not None:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.shape[0]
    r = np.empty((n, H), np.float64)
    o = np.empty((n, H), np.float64)
    ms = np.empty((n,), np.float64)
    rc = lib.oracle_proj_add_rmsnorm(_ptr(x), _ptr(W), _ptr(r0), _ptr(gamma), float(eps),
                                     int(norm_kind), T, K, H, _ptr(rows_arr), n,
                                     _ptr(r), _ptr(o), _ptr(ms), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return r, o, ms


def _u8(a, shape):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError("FP8 operands are passed as their uint8 E4M3 codes")
    if a.shape != shape:
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


def _scales(s, n, what):
    s = np.ascontiguousarray(np.atleast_1d(s), dtype=np.float32)
    if s.ndim != 1 or s.shape[0] not in (1, n):
        raise ValueError(f"{what} must hold 1 or {n} values")
    return s, int(s.shape[0] == n and n > 1)


def e4m3_to_double(code: int) -> float:
    """Value of one FP8 E4M3 code."""
    return float(_load().oracle_e4m3_to_double(int(code) & 0xFF))


def proj_add_rmsnorm_fp8(x, x_scale, W, w_scale, r0, gamma, eps, norm_kind, rows=None, nthreads=0):
    """Return (r, o, ms) in float64 for FP8 operands.

    x [T,K] and W [H,K] are E4M3 codes (uint8); x_scale holds 1 value (tensor)
    or T (per token), w_scale 1 (tensor) or H (per output row of W), fp32;
    r0 [T,H] bf16 bits; gamma [H] fp32.  y = sx * sw * sum_k x.W.
    """
    lib = _load()
    T, K = np.shape(x)
    H = np.shape(W)[0]
    x = _u8(x, (T, K))
    W = _u8(W, (H, K))
    r0 = _u16(r0, (T, H))
    sx, sx_row = _scales(x_scale, T, "x_scale")
    sw, sw_row = _scales(w_scale, H, "w_scale")
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    if gamma.shape != (H,):
        raise ValueError("gamma must be [H]")
    rows_arr = None
    n = T
    if rows is not None:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.shape[0]
    r = np.empty((n, H), np.float64)
    o = np.empty((n, H), np.float64)
    ms = np.empty((n,), np.float64)
    rc = lib.oracle_proj_add_rmsnorm_fp8(_ptr(x), _ptr(sx), sx_row, _ptr(W), _ptr(sw), sw_row, _ptr(r0),
                                         _ptr(gamma), float(eps), int(norm_kind), T, K, H, _ptr(rows_arr), n,
                                         _ptr(r), _ptr(o), _ptr(ms), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return r, o, ms


def e2m1_to_double(code: int) -> float:
    """Value of one FP4 E2M1 code (low four bits)."""
    return float(_load().oracle_e2m1_to_double(int(code) & 0xF))


def proj_add_rmsnorm_nvfp4(x, Wq, S, gs, r0, gamma, eps, norm_kind, rows=None, nthreads=0):
    """Return (r, o, ms) in float64 for NVFP4 weights and bf16 activations.

    x [T,K] bf16 bits; Wq [H,K/2] uint8 (E2M1 codes, element 2j in the low
    nibble of byte j); S [H,ceil(K/16)] uint8 E4M3 block scales; gs the fp32
    tensor scale; w = gs * S * e2m1(W).
    """
    lib = _load()
    T, K = np.shape(x)
    H = np.shape(Wq)[0]
    x = _u16(x, (T, K))
    Wq = _u8(Wq, (H, K // 2))
    S = _u8(S, (H, (K + 15) // 16))
    r0 = _u16(r0, (T, H))
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    if gamma.shape != (H,):
        raise ValueError("gamma must be [H]")
    rows_arr = None
    n = T
    if rows is not None:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.shape[0]
    r = np.empty((n, H), np.float64)
    o = np.empty((n, H), np.float64)
    ms = np.empty((n,), np.float64)
    rc = lib.oracle_proj_add_rmsnorm_nvfp4(_ptr(x), _ptr(Wq), _ptr(S), float(gs), _ptr(r0), _ptr(gamma), float(eps),
                                           int(norm_kind), T, K, H, _ptr(rows_arr), n, _ptr(r), _ptr(o), _ptr(ms),
                                           int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return r, o, ms


def e8m0_to_double(E):
    """Value of an OCP E8M0 scale code (2^(E-127); NaN for 255)."""
    return _load().oracle_e8m0_to_double(int(E) & 0xFF)


def proj_add_rmsnorm_mxfp4(x, Wq, S, r0, gamma, eps, norm_kind, rows=None, nthreads=0):
    """Return (r, o, ms) in float64 for MXFP4 weights and bf16 activations.

    x [T,K] bf16 bits; Wq [H,K/2] uint8 (E2M1 codes, element 2j in the low
    nibble of byte j); S [H,ceil(K/32)] uint8 E8M0 block scales; w = S * e2m1(W).
    """
    lib = _load()
    T, K = np.shape(x)
    H = np.shape(Wq)[0]
    x = _u16(x, (T, K))
    Wq = _u8(Wq, (H, K // 2))
    S = _u8(S, (H, (K + 31) // 32))
    r0 = _u16(r0, (T, H))
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    if gamma.shape != (H,):
        raise ValueError("gamma must be [H]")
    rows_arr = None
    n = T
    if rows is not None:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.shape[0]
    r = np.empty((n, H), np.float64)
    o = np.empty((n, H), np.float64)
    ms = np.empty((n,), np.float64)
    rc = lib.oracle_proj_add_rmsnorm_mxfp4(_ptr(x), _ptr(Wq), _ptr(S), _ptr(r0), _ptr(gamma), float(eps),
                                           int(norm_kind), T, K, H, _ptr(rows_arr), n, _ptr(r), _ptr(o), _ptr(ms),
                                           int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return r, o, ms


def moe_route(logits, k):
    """Top-k experts per token (larger logit first, equal logits: smaller index first) and
    their softmax weights over the chosen logits.  logits [T,E] float32 -> (ids [T,k] int32,
    w [T,k] float64)."""
    lib = _load()
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    if lib.oracle_moe_route(_ptr(logits), T, E, int(k), _ptr(ids), _ptr(w)) != 0:
        raise ValueError("oracle rejected its arguments")
    return ids, w


def moe_permute(ids, E):
    """Rows grouped by expert (tokens ascending within an expert).  ids [T,k] int32 ->
    (offsets [E+1], row_token [T*k], row_slot [T*k], row_of [T,k]) int32."""
    lib = _load()
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, np.int32)
    row_token = np.empty(T * k, np.int32)
    row_slot = np.empty(T * k, np.int32)
    row_of = np.empty((T, k), np.int32)
    if lib.oracle_moe_permute(_ptr(ids), T, int(E), k, _ptr(offsets), _ptr(row_token), _ptr(row_slot),
                              _ptr(row_of)) != 0:
        raise ValueError("oracle rejected its arguments")
    return offsets, row_token, row_slot, row_of


def moe_gather(x, row_token):
    """The permute step of the MoE region's input side: grouped row r is token row_token[r] of x
    ([T,H] bf16 bits) -> [T*k,H] bf16 bits."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    row_token = np.ascontiguousarray(row_token, dtype=np.int64)
    if row_token.size and (row_token.min() < 0 or row_token.max() >= x.shape[0]):
        raise ValueError("row_token out of range")
    out = np.empty((row_token.size, x.shape[1]), np.uint16)
    for r in range(row_token.size):
        out[r] = x[row_token[r]]
    return out


def moe_down_region(hg, offsets, row_of, wt, We, r0, gamma, eps, norm_kind, nthreads=0):
    """Return (r, o, ms) in float64: grouped down projection of hg [T*k,K] (bf16 bits, grouped by
    expert per offsets) by We [E,H,K] (bf16 bits), unpermuted through row_of [T,k] with gate
    weights wt [T,k] (float32), added to r0 [T,H] and normalised."""
    lib = _load()
    row_of = np.ascontiguousarray(row_of, dtype=np.int32)
    T, k = row_of.shape
    E, H, K = np.shape(We)
    hg = _u16(hg, (T * k, K))
    We = _u16(We, (E, H, K))
    offsets = np.ascontiguousarray(offsets, dtype=np.int32)
    wt = np.ascontiguousarray(wt, dtype=np.float32)
    r0 = _u16(r0, (T, H))
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    if offsets.shape != (E + 1,) or wt.shape != (T, k) or gamma.shape != (H,):
        raise ValueError("shape mismatch")
    r = np.empty((T, H), np.float64)
    o = np.empty((T, H), np.float64)
    ms = np.empty((T,), np.float64)
    rc = lib.oracle_moe_down_region(_ptr(hg), _ptr(offsets), _ptr(row_of), _ptr(wt), _ptr(We), _ptr(r0),
                                    _ptr(gamma), float(eps), int(norm_kind), T, K, H, E, k, _ptr(r), _ptr(o),
                                    _ptr(ms), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return r, o, ms


def add_rmsnorm(y, r0, gamma, eps, norm_kind, nthreads=0):
    """Return (r, o, ms) in float64: r = r0 + y (both bf16), o = RMSNorm(r)."""
    lib = _load()
    T, H = np.shape(y)
    y = _u16(y, (T, H))
    r0 = _u16(r0, (T, H))
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    if gamma.shape != (H,):
        raise ValueError("gamma must be [H]")
    r = np.empty((T, H), np.float64)
    o = np.empty((T, H), np.float64)
    ms = np.empty((T,), np.float64)
    rc = lib.oracle_add_rmsnorm(_ptr(y), _ptr(r0), _ptr(gamma), float(eps), int(norm_kind),
                                T, H, _ptr(r), _ptr(o), _ptr(ms), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return r, o, ms


def round_to_bf16(v):
    """Round float64 values to bf16 bit patterns (nearest, ties to even)."""
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    lib.oracle_round_to_bf16(_ptr(v), v.size, _ptr(out))
    return out


def max_threads() -> int:
    return int(_load().oracle_max_threads())
