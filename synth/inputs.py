"""Workload table and seeded input generator.

Every value is drawn in float64 from numpy's PCG64, scaled to the stated
spread, and rounded to its storage type: bf16 tensors go float64 -> float32
(numpy cast, nearest-even) -> bf16 (nearest-even on the bit pattern); the fp32
norm weight goes float64 -> float32.  That two-step cast is part of this
generator's definition only: both the oracle and the GPU path receive the same
bytes, so nothing downstream depends on it.

Each tensor has its own stream, SeedSequence([seed, stream_id]) spawned into
fixed 1 Mi-element blocks, so the draws are reproducible independently of the
thread count used to make them.

Spreads follow the workloads of the vLLM "TPSP Design" page's two fusion
regions (o_proj and down_proj shapes of Llama-3-8B, Gemma-2-9B and a
70B-class model); ``N(0, s)`` in the workload list is read with ``s`` the
variance, so W ~ N(0, 1/K) has standard deviation 1/sqrt(K) and
gamma = 1 + N(0, 0.1) has perturbation standard deviation sqrt(0.1).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

BLOCK = 1 << 20

STREAM_X, STREAM_U, STREAM_W, STREAM_R, STREAM_GAMMA = 0, 1, 2, 3, 4
STREAM_X8, STREAM_W8, STREAM_SX, STREAM_SW = 5, 6, 7, 8
STREAM_W4, STREAM_S4 = 9, 10
STREAM_S5 = 11
STREAM_LOGITS, STREAM_IDS, STREAM_GATE, STREAM_HG, STREAM_WE = 12, 13, 14, 15, 16

# FP8 operands are drawn as values of spread FP8_SPREAD and stored as E4M3
# codes (see _fill_e4m3); the dequantisation scales bring them back to the
# bf16 workloads' spreads.
FP8_SPREAD = 16.0

NORM_STANDARD = 0
NORM_GEMMA = 1

DECODE_TOKENS = (1, 8, 32, 128, 256)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    K: int
    H: int
    norm_kind: int = NORM_STANDARD
    eps: float = 1e-5
    x_mode: str = "normal"          # "normal" or "silu_gu" (x = silu(g) * u)
    x_sigma: float = 1.0
    r_sigma: float = 1.0
    gamma_mode: str = "one_plus"    # "one_plus": 1 + N(0, v); "plain": N(0, v)
    gamma_var: float = 0.1
    microchunks: tuple = field(default_factory=tuple)
    seed: int = 0

    @property
    def w_sigma(self) -> float:
        return 1.0 / math.sqrt(self.K)

    def with_tokens(self, T: int) -> "Workload":
        return replace(self, T=int(T))

    def flops(self) -> float:
        return 2.0 * self.T * self.K * self.H

    def algorithmic_bytes(self, operand_bytes: int = 2) -> float:
        """x read + W read once + residual read and written + out written + gamma
        (operand_bytes = 1 for FP8 x and W, whose scales add 4T + 4H at most;
        operand_bytes = 0 for NVFP4 weights: bf16 x, W at half a byte per
        weight plus one scale byte per 16; operand_bytes = -1 for MXFP4
        weights: one scale byte per 32)."""
        T, K, H = self.T, self.K, self.H
        rest = 4.0 * T * H + 2.0 * T * H + 4.0 * H
        if operand_bytes == 0:
            return 2.0 * T * K + 0.5 * H * K + H * K / 16.0 + rest
        if operand_bytes == -1:
            return 2.0 * T * K + 0.5 * H * K + H * K / 32.0 + rest
        b = float(operand_bytes)
        extra = 4.0 * T + 4.0 * H if operand_bytes == 1 else 0.0
        return b * T * K + b * H * K + rest + extra


CONFIGS = {
    "tiny": Workload("tiny", T=16, K=256, H=256, eps=1e-6, r_sigma=1.0,
                     microchunks=(16,)),
    "llama3_8b_oproj": Workload("llama3_8b_oproj", T=4096, K=4096, H=4096, eps=1e-5,
                                r_sigma=2.0, microchunks=(256, 512, 1024, 4096)),
    "llama3_8b_down": Workload("llama3_8b_down", T=8192, K=14336, H=4096, eps=1e-5,
                               x_mode="silu_gu", r_sigma=2.0,
                               microchunks=(256, 512, 1024, 4096)),
    "gemma2_9b_down": Workload("gemma2_9b_down", T=2048, K=14336, H=3584,
                               norm_kind=NORM_GEMMA, eps=1e-6, r_sigma=1.0,
                               gamma_mode="plain", microchunks=(256, 512, 1024, 2048)),
    "llama70b_oproj_decode": Workload("llama70b_oproj_decode", T=256, K=8192, H=8192,
                                      eps=1e-5, r_sigma=2.0),
    "llama70b_down_decode": Workload("llama70b_down_decode", T=256, K=28672, H=8192,
                                     eps=1e-5, r_sigma=2.0),
}


# MoE down-projection regions: (workload with K = expert width, H = hidden; experts E; top-k)
MOE_CONFIGS = {
    "moe_tiny": (Workload("moe_tiny", T=24, K=256, H=256, eps=1e-6, r_sigma=1.0), 4, 2),
    "mixtral_8x7b_down": (Workload("mixtral_8x7b_down", T=4096, K=14336, H=4096, eps=1e-5, r_sigma=2.0), 8, 2),
    "mixtral_8x7b_down_decode": (Workload("mixtral_8x7b_down_decode", T=8, K=14336, H=4096, eps=1e-5,
                                          r_sigma=2.0), 8, 2),
}


def workload(name: str, **overrides) -> Workload:
    wl = CONFIGS[name]
    return replace(wl, **overrides) if overrides else wl


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, nearest-even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _block_gens(seed: int, stream: int, nblocks: int):
    ss = np.random.SeedSequence([int(seed), int(stream)])
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(nblocks)]


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _fill_bf16(out: np.ndarray, seed: int, stream: int, sigma: float, mean: float = 0.0):
    flat = out.reshape(-1)
    n = flat.size
    nb = (n + BLOCK - 1) // BLOCK
    gens = _block_gens(seed, stream, nb)

    def work(i):
        s, e = i * BLOCK, min(n, (i + 1) * BLOCK)
        v = gens[i].standard_normal(e - s) * sigma + mean
        flat[s:e] = f32_to_bf16_bits(v.astype(np.float32))

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(nb)))


def _fill_silu_gu(out: np.ndarray, seed: int):
    """x = silu(g) * u with g, u ~ N(0,1) rounded to bf16 first; product in float64."""
    flat = out.reshape(-1)
    n = flat.size
    nb = (n + BLOCK - 1) // BLOCK
    gg = _block_gens(seed, STREAM_X, nb)
    gu = _block_gens(seed, STREAM_U, nb)

    def work(i):
        s, e = i * BLOCK, min(n, (i + 1) * BLOCK)
        g = bf16_bits_to_f32(f32_to_bf16_bits(gg[i].standard_normal(e - s).astype(np.float32)))
        u = bf16_bits_to_f32(f32_to_bf16_bits(gu[i].standard_normal(e - s).astype(np.float32)))
        g = g.astype(np.float64)
        v = g / (1.0 + np.exp(-g)) * u.astype(np.float64)
        flat[s:e] = f32_to_bf16_bits(v.astype(np.float32))

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(nb)))


def make_inputs(wl: Workload, seed: int | None = None, T: int | None = None):
    """Return dict(x=[T,K] u16, W=[H,K] u16, r0=[T,H] u16, gamma=[H] f32) for a workload.

    ``T`` overrides the token count (the decode sweep and the parity sizes).
    The draws for a tensor depend only on (seed, tensor, element index), so a
    smaller T gives a prefix of the larger-T tensors' rows.
    """
    seed = wl.seed if seed is None else int(seed)
    T = wl.T if T is None else int(T)
    K, H = wl.K, wl.H
    x = np.empty((T, K), np.uint16)
    if wl.x_mode == "normal":
        _fill_bf16(x, seed, STREAM_X, wl.x_sigma)
    elif wl.x_mode == "silu_gu":
        _fill_silu_gu(x, seed)
    else:
        raise ValueError(wl.x_mode)
    W = np.empty((H, K), np.uint16)
    _fill_bf16(W, seed, STREAM_W, wl.w_sigma)
    r0 = np.empty((T, H), np.uint16)
    _fill_bf16(r0, seed, STREAM_R, wl.r_sigma)
    g = _block_gens(seed, STREAM_GAMMA, 1)[0].standard_normal(H) * math.sqrt(wl.gamma_var)
    if wl.gamma_mode == "one_plus":
        g = 1.0 + g
    elif wl.gamma_mode != "plain":
        raise ValueError(wl.gamma_mode)
    gamma = g.astype(np.float32)
    return {"x": x, "W": W, "r0": r0, "gamma": gamma}


def _fill_e4m3(out: np.ndarray, seed: int, stream: int, spread: float):
    """Codes of FP8 E4M3 values drawn as N(0, spread^2).

    A drawn value v is stored by truncation toward zero to an E4M3 code: the
    sign bit, the exponent field floor(log2|v|) + 7 (0 below 2^-6, where the
    3-bit fraction counts units of 2^-9), and the top three fraction bits,
    clamped below the largest finite code 0x7E; the NaN codes 0x7F/0xFF never
    occur.
    """
    flat = out.reshape(-1)
    n = flat.size
    nb = (n + BLOCK - 1) // BLOCK
    gens = _block_gens(seed, stream, nb)

    def work(i):
        s, e = i * BLOCK, min(n, (i + 1) * BLOCK)
        v = gens[i].standard_normal(e - s) * spread
        a = np.abs(v)
        with np.errstate(divide="ignore"):
            ex = np.floor(np.log2(np.where(a > 0, a, 1.0)))
        normal = (a >= 2.0 ** -6)
        ef = np.clip(ex + 7, 1, 15)
        frac_n = np.floor((a / np.exp2(ef - 7) - 1.0) * 8.0)
        frac_s = np.floor(a / 2.0 ** -9)
        frac = np.clip(np.where(normal, frac_n, frac_s), 0, 7)
        efield = np.where(normal, ef, 0)
        code = (efield.astype(np.int64) << 3) | frac.astype(np.int64)
        code = np.minimum(code, 0x7E)
        code |= (v < 0).astype(np.int64) << 7
        flat[s:e] = code.astype(np.uint8)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(nb)))


def make_inputs_fp8(wl: Workload, seed: int | None = None, T: int | None = None,
                    x_scale_per_token: bool = True, w_scale_per_channel: bool = True):
    """FP8 operands for a workload: dict(x8=[T,K] u8, x_scale=[T] or [1] f32,
    W8=[H,K] u8, w_scale=[H] or [1] f32, r0=[T,H] u16, gamma=[H] f32).

    x8 and W8 are E4M3 codes of N(0, FP8_SPREAD^2) draws; the scales are
    1/FP8_SPREAD (x) and 1/(FP8_SPREAD sqrt(K)) (W) times 2^u, u ~ U(-1/2, 1/2)
    per token / per output row (per-tensor: u = 0), so the dequantised
    operands have the bf16 workload's spreads.  r0 and gamma are the bf16
    workload's tensors (same streams).
    """
    seed = wl.seed if seed is None else int(seed)
    T = wl.T if T is None else int(T)
    K, H = wl.K, wl.H
    base = make_inputs(wl, seed=seed, T=T)
    x8 = np.empty((T, K), np.uint8)
    _fill_e4m3(x8, seed, STREAM_X8, FP8_SPREAD)
    W8 = np.empty((H, K), np.uint8)
    _fill_e4m3(W8, seed, STREAM_W8, FP8_SPREAD)
    sx0 = 1.0 / FP8_SPREAD
    sw0 = 1.0 / (FP8_SPREAD * math.sqrt(K))
    if x_scale_per_token:
        u = _block_gens(seed, STREAM_SX, 1)[0].uniform(-0.5, 0.5, T)
        x_scale = (sx0 * np.exp2(u)).astype(np.float32)
    else:
        x_scale = np.array([sx0], np.float32)
    if w_scale_per_channel:
        u = _block_gens(seed, STREAM_SW, 1)[0].uniform(-0.5, 0.5, H)
        w_scale = (sw0 * np.exp2(u)).astype(np.float32)
    else:
        w_scale = np.array([sw0], np.float32)
    return {"x8": x8, "x_scale": x_scale, "W8": W8, "w_scale": w_scale, "r0": base["r0"], "gamma": base["gamma"]}


def _fill_e2m1_packed(out: np.ndarray, seed: int, stream: int, spread: float):
    """E2M1 codes of N(0, spread^2) draws, two per byte along a row (element
    2j in the low nibble of byte j).  A draw is stored by truncation toward
    zero onto the E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (the code is the
    index of the largest magnitude not above |v|), with its sign bit."""
    flat = out.reshape(-1)
    n = flat.size
    nb = (n + BLOCK - 1) // BLOCK
    gens = _block_gens(seed, stream, nb)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])

    def work(i):
        s0, e = i * BLOCK, min(n, (i + 1) * BLOCK)
        v = gens[i].standard_normal(2 * (e - s0)) * spread
        idx = np.searchsorted(grid, np.abs(v), side="right") - 1
        code = idx.astype(np.int64) | ((v < 0).astype(np.int64) << 3)
        flat[s0:e] = (code[0::2] | (code[1::2] << 4)).astype(np.uint8)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(nb)))


def make_inputs_nvfp4(wl: Workload, seed: int | None = None, T: int | None = None):
    """NVFP4 weights for a workload: dict(x=[T,K] u16 bf16, Wq=[H,K/2] u8,
    S=[H,ceil(K/16)] u8 E4M3 block scales, gs=float, r0, gamma).

    W codes are E2M1 codes of N(0, 2^2) draws; each block scale is an E4M3
    code 2^e * (1 + m/8) with e uniform in {-1, 0, 1} and m uniform in 0..7;
    gs = 1 / (2 sqrt(K)), so the dequantised weights have about the bf16
    workload's spread.  x, r0 and gamma are the bf16 workload's tensors.
    """
    seed = wl.seed if seed is None else int(seed)
    T = wl.T if T is None else int(T)
    K, H = wl.K, wl.H
    if K % 2:
        raise ValueError("NVFP4 rows pack two elements per byte: K must be even")
    base = make_inputs(wl, seed=seed, T=T)
    Wq = np.empty((H, K // 2), np.uint8)
    _fill_e2m1_packed(Wq, seed, STREAM_W4, 2.0)
    nblk = (K + 15) // 16
    g = _block_gens(seed, STREAM_S4, 1)[0]
    e = g.integers(-1, 2, size=(H, nblk))
    m = g.integers(0, 8, size=(H, nblk))
    S = (((e + 7) << 3) | m).astype(np.uint8)
    gs = float(np.float32(1.0 / (2.0 * math.sqrt(K))))
    return {"x": base["x"], "Wq": Wq, "S": S, "gs": gs, "r0": base["r0"], "gamma": base["gamma"]}


def make_inputs_mxfp4(wl: Workload, seed: int | None = None, T: int | None = None):
    """MXFP4 weights for a workload: dict(x=[T,K] u16 bf16, Wq=[H,K/2] u8,
    S=[H,ceil(K/32)] u8 E8M0 block scales, r0, gamma).

    W codes are those of make_inputs_nvfp4 (E2M1 codes of N(0, 2^2) draws);
    each block scale is the E8M0 code of 2^(e0 + u), u uniform in {-1, 0, 1},
    e0 = round(log2(1 / (2 sqrt(K)))), so the dequantised weights have about
    the bf16 workload's spread.  x, r0 and gamma are the bf16 workload's tensors.
    """
    seed = wl.seed if seed is None else int(seed)
    T = wl.T if T is None else int(T)
    K, H = wl.K, wl.H
    if K % 2:
        raise ValueError("MXFP4 rows pack two elements per byte: K must be even")
    base = make_inputs(wl, seed=seed, T=T)
    Wq = np.empty((H, K // 2), np.uint8)
    _fill_e2m1_packed(Wq, seed, STREAM_W4, 2.0)
    nblk = (K + 31) // 32
    e0 = int(round(math.log2(1.0 / (2.0 * math.sqrt(K)))))
    u = _block_gens(seed, STREAM_S5, 1)[0].integers(-1, 2, size=(H, nblk))
    S = (127 + e0 + u).astype(np.uint8)
    return {"x": base["x"], "Wq": Wq, "S": S, "r0": base["r0"], "gamma": base["gamma"]}


def make_inputs_moe(wl: Workload, E: int, k: int, seed: int | None = None, T: int | None = None):
    """MoE down-projection region inputs for a workload (K = expert width, H = hidden):
    dict(logits=[T,E] f32, ids=[T,k] i32, wt=[T,k] f32, hg=[T*k,K] u16 bf16, We=[E,H,K] u16 bf16,
    r0, gamma).

    logits are N(0, 1) draws (router output); ids are k distinct experts per token drawn
    uniformly (an assignment given to the down region directly, not a routing of the logits);
    wt are U(0.05, 1) gate weights; hg holds the expert activations, one N(0, x_sigma^2) row
    per (token, slot) pair in the grouped order; We[e] is an [H, K] bf16 weight with the
    workload's W spread.  r0 and gamma are the bf16 workload's tensors.
    """
    seed = wl.seed if seed is None else int(seed)
    T = wl.T if T is None else int(T)
    K, H = wl.K, wl.H
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    base = make_inputs(wl, seed=seed, T=T)
    logits = _block_gens(seed, STREAM_LOGITS, 1)[0].standard_normal((T, E)).astype(np.float32)
    g = _block_gens(seed, STREAM_IDS, 1)[0]
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else np.zeros((0, k), np.int32)
    wt = _block_gens(seed, STREAM_GATE, 1)[0].uniform(0.05, 1.0, (T, k)).astype(np.float32)
    hg = np.empty((T * k, K), np.uint16)
    _fill_bf16(hg, seed, STREAM_HG, wl.x_sigma)
    We = np.empty((E, H, K), np.uint16)
    _fill_bf16(We.reshape(E * H, K), seed, STREAM_WE, wl.w_sigma)
    return {"logits": logits, "ids": ids, "wt": wt, "hg": hg, "We": We, "r0": base["r0"], "gamma": base["gamma"]}

