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

    def algorithmic_bytes(self) -> float:
        """x read + W read once + residual read and written + out written + gamma."""
        T, K, H = self.T, self.K, self.H
        return 2.0 * T * K + 2.0 * H * K + 4.0 * T * H + 2.0 * T * H + 4.0 * H


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
