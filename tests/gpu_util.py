"""Device helpers for the GPU tests: upload seeded inputs, run a path through
the C ABI, bring results back as bf16 bit patterns."""
from __future__ import annotations

import numpy as np
import torch

import decoder_layer_projection_gb300 as fln


def dev_bf16(a: np.ndarray, extra_rows: int = 0, fill_bits: int = 0x7FC1) -> torch.Tensor:
    """Upload uint16 bf16 bits; optional guard rows filled with a NaN pattern."""
    a = np.ascontiguousarray(a, np.uint16)
    if extra_rows:
        g = np.full((extra_rows,) + a.shape[1:], fill_bits, np.uint16)
        a = np.concatenate([a, g], axis=0)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def plan(path, chunk=4096, tile_n=256, gemm_ctas=0, norm_ctas=0, threshold=1, tuned_max=0, epi_warps=0):
    return dict(path=path, microchunk_tokens=chunk, tile_n=tile_n, gemm_ctas=gemm_ctas, norm_ctas=norm_ctas,
                threshold_tokens=threshold, tuned_max_tokens=tuned_max, epi_warps=epi_warps)


UNFUSED = plan(fln.PATH_FUSED, threshold=257)  # every T <= 256 takes the UNFUSED path


class Run:
    """One call of fused_proj_add_rmsnorm on uploaded inputs with guard rows."""

    GUARD = 3

    def __init__(self, d: dict, eps: float, norm_kind: int):
        self.T, self.K = d["x"].shape
        self.H = d["W"].shape[0]
        self.eps, self.kind = eps, norm_kind
        self.x = dev_bf16(d["x"])
        self.W = dev_bf16(d["W"])
        self.r0 = d["r0"]
        self.gamma = torch.from_numpy(np.ascontiguousarray(d["gamma"], np.float32)).cuda()

    def __call__(self, plan_dict=None, chunk=0, T=None):
        T = self.T if T is None else T
        if plan_dict is not None:
            fln.fln_set_plan(self.K, self.H, self.kind, plan_dict)
        try:
            r = dev_bf16(self.r0[:T], extra_rows=self.GUARD)
            out = dev_bf16(np.zeros((T, self.H), np.uint16), extra_rows=self.GUARD, fill_bits=0x7FC2)
            fln.fused_proj_add_rmsnorm(self.x[:T], self.W, r[:T], self.gamma, self.eps, self.kind, chunk, out[:T])
            fln.fln_device_status()
        finally:
            if plan_dict is not None:
                fln.fln_set_plan(self.K, self.H, self.kind, None)
        rb, ob = host_bits(r), host_bits(out)
        # rows at or beyond T must be untouched
        assert np.all(rb[T:] == 0x7FC1), "residual guard rows were written"
        assert np.all(ob[T:] == 0x7FC2), "output guard rows were written"
        return rb[:T], ob[:T]
