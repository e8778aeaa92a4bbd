"""GB300-native fused projection + residual add + RMSNorm (libfusedln).

A thin ctypes binding over the C ABI declared in ``include/libfusedln.h``.
The functions here carry the same names as the C entry points and only
marshal arguments: tensor shapes and device pointers in, status codes out.
Every step of the computation runs in the library's CUDA kernels; if the
shared library is missing, the first call raises -- there is no CPU path.

PyTorch provides the device memory and the streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfusedln.so")

FLN_OK = 0
FLN_ERR_INVALID_ARG = -1
FLN_ERR_UNSUPPORTED = -2
FLN_ERR_CUDA = -3
FLN_ERR_DEVICE_TIMEOUT = -4
FLN_ERR_NOT_TUNED = -5
FLN_ERR_COMM = -6

NORM_STANDARD = 0
NORM_GEMMA = 1

PATH_FUSED = 1
PATH_PIPELINED = 2
PATH_UNFUSED = 3

DTYPE_BF16 = 0
DTYPE_E4M3 = 1
DTYPE_NVFP4 = 2
DTYPE_MXFP4 = 3

KERNEL_NAMES = ("gemm_fused", "gemm_slot", "gemm_splitk", "norm_bf16", "norm_slot", "norm_splitk", "w4_dequant",
                "moe_route", "moe_gemm", "moe_norm", "moe_gather")

EXPORTED_SYMBOLS = (
    "fused_proj_add_rmsnorm", "add_rmsnorm", "fln_autotune", "fln_set_overrides", "fln_set_plan",
    "fln_get_plan", "fln_device_status", "fln_last_error", "fln_release_workspace", "fln_launch_count",
    "fln_profile_enable", "fln_profile_read", "fln_version", "fused_proj_add_rmsnorm_noalloc",
    "fln_debug_stall_next_call", "fused_proj_add_rmsnorm_fp8", "fln_autotune_dtype", "fln_set_plan_dtype",
    "fln_get_plan_dtype", "fused_proj_add_rmsnorm_nvfp4", "fused_proj_add_rmsnorm_mxfp4", "fln_moe_route",
    "fused_moe_down_add_rmsnorm", "fln_moe_gather", "fused_proj_add_rmsnorm_host",
    "fln_tp_unique_id", "fln_tp_comm_init", "fln_tp_comm_destroy", "fln_tp_layout", "fln_tp_chunk_rows",
    "fused_proj_rs_add_rmsnorm_ag", "fln_set_splitk_tail_tokens",
)


class FlnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libfusedln status {status}: {message}")
        self.status = status
        self.message = message


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("microchunk_tokens", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("gemm_ctas", ctypes.c_int), ("norm_ctas", ctypes.c_int), ("threshold_tokens", ctypes.c_int),
                ("tuned_max_tokens", ctypes.c_int), ("epi_warps", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class ProfileStats(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_uint64 * len(KERNEL_NAMES)), ("total_ms", ctypes.c_double * len(KERNEL_NAMES))]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return LIB_PATH


def load(path: str | None = None):
    """Load libfusedln.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it first (python -m decoder_layer_projection_gb300._build)")
        lib = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.fused_proj_add_rmsnorm.argtypes = [vp, vp, vp, vp, f, i, i, i, i, i, vp, vp]
        lib.fused_proj_add_rmsnorm.restype = i
        lib.add_rmsnorm.argtypes = [vp, vp, vp, f, i, i, i, vp, vp]
        lib.add_rmsnorm.restype = i
        lib.fln_autotune.argtypes = [i, i, i, i, vp]
        lib.fln_autotune.restype = i
        lib.fln_set_overrides.argtypes = [i, i]
        lib.fln_set_overrides.restype = i
        lib.fln_set_plan.argtypes = [i, i, i, ctypes.POINTER(Plan)]
        lib.fln_set_plan.restype = i
        lib.fln_get_plan.argtypes = [i, i, i, i, i, ctypes.POINTER(Plan)]
        lib.fln_get_plan.restype = i
        lib.fln_device_status.argtypes = [vp]
        lib.fln_device_status.restype = i
        lib.fln_last_error.argtypes = []
        lib.fln_last_error.restype = ctypes.c_char_p
        lib.fln_release_workspace.argtypes = []
        lib.fln_release_workspace.restype = None
        lib.fln_launch_count.argtypes = []
        lib.fln_launch_count.restype = ctypes.c_uint64
        lib.fln_profile_enable.argtypes = [i]
        lib.fln_profile_enable.restype = i
        lib.fln_profile_read.argtypes = [ctypes.POINTER(ProfileStats)]
        lib.fln_profile_read.restype = i
        lib.fln_version.argtypes = []
        lib.fln_version.restype = i
        lib.fln_debug_stall_next_call.argtypes = [i]
        lib.fln_debug_stall_next_call.restype = i
        lib.fused_proj_add_rmsnorm_host.argtypes = [vp, vp, vp, vp, f, i, i, i, i, i, vp, vp]
        lib.fused_proj_add_rmsnorm_host.restype = i
        lib.fused_proj_add_rmsnorm_noalloc.argtypes = [vp, vp, vp, vp, f, i, i, i, i, vp, vp, vp]
        lib.fused_proj_add_rmsnorm_noalloc.restype = i
        lib.fused_proj_add_rmsnorm_fp8.argtypes = [vp, vp, i, vp, vp, i, vp, vp, f, i, i, i, i, i, vp, vp]
        lib.fused_proj_add_rmsnorm_fp8.restype = i
        lib.fused_proj_add_rmsnorm_nvfp4.argtypes = [vp, vp, vp, f, vp, vp, f, i, i, i, i, i, vp, vp]
        lib.fused_proj_add_rmsnorm_nvfp4.restype = i
        lib.fused_proj_add_rmsnorm_mxfp4.argtypes = [vp, vp, vp, vp, vp, f, i, i, i, i, i, vp, vp]
        lib.fused_proj_add_rmsnorm_mxfp4.restype = i
        lib.fln_moe_route.argtypes = [vp, i, i, i, vp, vp, vp, vp, vp, vp, vp]
        lib.fln_moe_route.restype = i
        lib.fused_moe_down_add_rmsnorm.argtypes = [vp, vp, vp, vp, vp, vp, vp, f, i, i, i, i, i, i, vp, vp]
        lib.fused_moe_down_add_rmsnorm.restype = i
        lib.fln_moe_gather.argtypes = [vp, vp, i, i, i, vp, vp]
        lib.fln_moe_gather.restype = i
        lib.fln_autotune_dtype.argtypes = [i, i, i, i, i, vp]
        lib.fln_autotune_dtype.restype = i
        lib.fln_set_plan_dtype.argtypes = [i, i, i, i, ctypes.POINTER(Plan)]
        lib.fln_set_plan_dtype.restype = i
        lib.fln_get_plan_dtype.argtypes = [i, i, i, i, i, i, ctypes.POINTER(Plan)]
        lib.fln_get_plan_dtype.restype = i
        lib.fln_set_splitk_tail_tokens.argtypes = [i]
        lib.fln_set_splitk_tail_tokens.restype = i
        ip = ctypes.POINTER(ctypes.c_int)
        lib.fln_tp_unique_id.argtypes = [vp]
        lib.fln_tp_unique_id.restype = i
        lib.fln_tp_comm_init.argtypes = [i, i, vp, ctypes.POINTER(vp)]
        lib.fln_tp_comm_init.restype = i
        lib.fln_tp_comm_destroy.argtypes = [vp]
        lib.fln_tp_comm_destroy.restype = i
        lib.fln_tp_layout.argtypes = [i, i, i, ip, ip, ip]
        lib.fln_tp_layout.restype = i
        lib.fln_tp_chunk_rows.argtypes = [i, i, i, i, i, ip, ip, ip]
        lib.fln_tp_chunk_rows.restype = i
        lib.fused_proj_rs_add_rmsnorm_ag.argtypes = [vp, vp, vp, vp, f, i, i, i, i, i, vp, vp, vp]
        lib.fused_proj_rs_add_rmsnorm_ag.restype = i
        _lib = lib
        return lib


def _check(status: int):
    if status != FLN_OK:
        raise FlnError(status, load().fln_last_error().decode(errors="replace"))


def _stream_ptr(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def fused_proj_add_rmsnorm(x, W, residual, gamma, eps: float, norm_kind: int = NORM_STANDARD,
                           microchunk_tokens: int = 0, out=None, stream=None):
    """residual += x @ W^T; out = RMSNorm(residual).  Tensors: x [T,K] bf16,
    W [H,K] bf16, residual [T,H] bf16 (in place), gamma [H] fp32, out [T,H] bf16.
    Returns out."""
    T, K = x.shape
    H = W.shape[0]
    if out is None:
        import torch
        out = torch.empty((T, H), dtype=residual.dtype, device=residual.device)
    _check(load().fused_proj_add_rmsnorm(_ptr(x), _ptr(W), _ptr(residual), _ptr(gamma), float(eps),
                                         int(norm_kind), int(T), int(K), int(H), int(microchunk_tokens),
                                         _ptr(out), _stream_ptr(stream)))
    return out


def fused_proj_add_rmsnorm_ptr(x_ptr, W_ptr, residual_ptr, gamma_ptr, eps, norm_kind, T, K, H,
                               microchunk_tokens, out_ptr, stream_ptr) -> int:
    """Raw-pointer form: returns the status code without raising."""
    return load().fused_proj_add_rmsnorm(x_ptr, W_ptr, residual_ptr, gamma_ptr, float(eps), int(norm_kind),
                                         int(T), int(K), int(H), int(microchunk_tokens), out_ptr, stream_ptr)


def fused_proj_add_rmsnorm_host(x_host, W, residual_host, gamma, eps: float, norm_kind: int = NORM_STANDARD,
                                transfer_tokens: int = 0, out_host=None, stream=None):
    """The same region with x, residual (in place) and out in HOST memory (CPU
    tensors; pinned ones let the copies overlap) and W, gamma on the device.
    Asynchronous on `stream`: synchronize it before reading residual_host or
    out_host.  Returns out_host."""
    T, K = x_host.shape
    H = W.shape[0]
    if out_host is None:
        import torch
        out_host = torch.empty((T, H), dtype=residual_host.dtype, pin_memory=residual_host.is_pinned())
    _check(load().fused_proj_add_rmsnorm_host(_ptr(x_host), _ptr(W), _ptr(residual_host), _ptr(gamma), float(eps),
                                              int(norm_kind), int(T), int(K), int(H), int(transfer_tokens),
                                              _ptr(out_host), _stream_ptr(stream)))
    return out_host


def fused_proj_add_rmsnorm_host_ptr(x_ptr, W_ptr, residual_ptr, gamma_ptr, eps, norm_kind, T, K, H,
                                    transfer_tokens, out_ptr, stream_ptr) -> int:
    """Raw-pointer form: returns the status code without raising."""
    return load().fused_proj_add_rmsnorm_host(x_ptr, W_ptr, residual_ptr, gamma_ptr, float(eps), int(norm_kind),
                                              int(T), int(K), int(H), int(transfer_tokens), out_ptr, stream_ptr)


def fused_proj_add_rmsnorm_noalloc(x, W, residual, gamma, eps: float, norm_kind: int = NORM_STANDARD, out=None,
                                   device_error=None, stream=None):
    """Same result as fused_proj_add_rmsnorm, through the entry point that never
    allocates device memory (static scratch; FUSED path).  `out` must be given by
    callers that cannot allocate; `device_error` is an optional int32/uint32
    device tensor of one element that receives device error bits.  Returns out."""
    T, K = x.shape
    H = W.shape[0]
    if out is None:
        import torch
        out = torch.empty((T, H), dtype=residual.dtype, device=residual.device)
    _check(load().fused_proj_add_rmsnorm_noalloc(_ptr(x), _ptr(W), _ptr(residual), _ptr(gamma), float(eps),
                                                 int(norm_kind), int(T), int(K), int(H), _ptr(out),
                                                 _ptr(device_error), _stream_ptr(stream)))
    return out


def fused_proj_add_rmsnorm_noalloc_ptr(x_ptr, W_ptr, residual_ptr, gamma_ptr, eps, norm_kind, T, K, H, out_ptr,
                                       device_error_ptr, stream_ptr) -> int:
    """Raw-pointer form: returns the status code without raising."""
    return load().fused_proj_add_rmsnorm_noalloc(x_ptr, W_ptr, residual_ptr, gamma_ptr, float(eps),
                                                 int(norm_kind), int(T), int(K), int(H), out_ptr,
                                                 device_error_ptr, stream_ptr)


def fused_proj_add_rmsnorm_fp8(x, x_scale, W, w_scale, residual, gamma, eps: float,
                               norm_kind: int = NORM_STANDARD, microchunk_tokens: int = 0, out=None, stream=None):
    """FP8 operands: residual += (x . W^T) * x_scale * w_scale; out = RMSNorm(residual).
    x [T,K] and W [H,K] hold E4M3 codes (torch.uint8 or torch.float8_e4m3fn);
    x_scale fp32 with T values (per token) or 1 (tensor); w_scale fp32 with H
    values (per output row of W) or 1.  Returns out."""
    T, K = x.shape
    H = W.shape[0]
    if out is None:
        import torch
        out = torch.empty((T, H), dtype=residual.dtype, device=residual.device)
    x_per_token = 1 if (x_scale.numel() == T and T > 1) else 0
    w_per_channel = 1 if (w_scale.numel() == H and H > 1) else 0
    if x_scale.numel() not in (1, T) or w_scale.numel() not in (1, H):
        raise ValueError("x_scale must hold 1 or T values and w_scale 1 or H values")
    _check(load().fused_proj_add_rmsnorm_fp8(_ptr(x), _ptr(x_scale), x_per_token, _ptr(W), _ptr(w_scale),
                                             w_per_channel, _ptr(residual), _ptr(gamma), float(eps),
                                             int(norm_kind), int(T), int(K), int(H), int(microchunk_tokens),
                                             _ptr(out), _stream_ptr(stream)))
    return out


def fused_proj_add_rmsnorm_nvfp4(x, W, W_scale, w_global_scale: float, residual, gamma, eps: float,
                                 norm_kind: int = NORM_STANDARD, microchunk_tokens: int = 0, out=None, stream=None):
    """NVFP4 weights, bf16 activations: w = w_global_scale * e4m3(W_scale[h, k/16]) * e2m1(W[h, k]);
    residual += x . w^T; out = RMSNorm(residual).  x [T,K] bf16; W [H,K/2] uint8 (element 2j in
    the low nibble of byte j); W_scale [H,K/16] uint8 E4M3 codes.  Returns out."""
    T, K = x.shape
    H = W.shape[0]
    if out is None:
        import torch
        out = torch.empty((T, H), dtype=residual.dtype, device=residual.device)
    _check(load().fused_proj_add_rmsnorm_nvfp4(_ptr(x), _ptr(W), _ptr(W_scale), float(w_global_scale),
                                               _ptr(residual), _ptr(gamma), float(eps), int(norm_kind), int(T),
                                               int(K), int(H), int(microchunk_tokens), _ptr(out),
                                               _stream_ptr(stream)))
    return out



def fused_proj_add_rmsnorm_mxfp4(x, W, W_scale, residual, gamma, eps: float, norm_kind: int = NORM_STANDARD,
                                 microchunk_tokens: int = 0, out=None, stream=None):
    """MXFP4 weights, bf16 activations: w = 2^(W_scale[h, k/32] - 127) * e2m1(W[h, k]);
    residual += x . w^T; out = RMSNorm(residual).  x [T,K] bf16; W [H,K/2] uint8 (element 2j in
    the low nibble of byte j); W_scale [H,K/32] uint8 E8M0 codes.  Returns out."""
    T, K = x.shape
    H = W.shape[0]
    if out is None:
        import torch
        out = torch.empty((T, H), dtype=residual.dtype, device=residual.device)
    _check(load().fused_proj_add_rmsnorm_mxfp4(_ptr(x), _ptr(W), _ptr(W_scale), _ptr(residual), _ptr(gamma),
                                               float(eps), int(norm_kind), int(T), int(K), int(H),
                                               int(microchunk_tokens), _ptr(out), _stream_ptr(stream)))
    return out

def add_rmsnorm(y, residual, gamma, eps: float, norm_kind: int = NORM_STANDARD, out=None, stream=None):
    """residual += y; out = RMSNorm(residual).  y, residual, out [T,H] bf16; gamma [H] fp32."""
    T, H = y.shape
    if out is None:
        import torch
        out = torch.empty((T, H), dtype=residual.dtype, device=residual.device)
    _check(load().add_rmsnorm(_ptr(y), _ptr(residual), _ptr(gamma), float(eps), int(norm_kind), int(T), int(H),
                              _ptr(out), _stream_ptr(stream)))
    return out


def add_rmsnorm_ptr(y_ptr, residual_ptr, gamma_ptr, eps, norm_kind, T, H, out_ptr, stream_ptr) -> int:
    return load().add_rmsnorm(y_ptr, residual_ptr, gamma_ptr, float(eps), int(norm_kind), int(T), int(H),
                              out_ptr, stream_ptr)


def fln_autotune(K: int, H: int, norm_kind: int, max_tokens: int, stream=None, dtype: int = DTYPE_BF16):
    _check(load().fln_autotune_dtype(int(K), int(H), int(norm_kind), int(dtype), int(max_tokens),
                                     _stream_ptr(stream)))


def fln_set_overrides(microchunk_tokens: int = 0, threshold_tokens: int = 0):
    _check(load().fln_set_overrides(int(microchunk_tokens), int(threshold_tokens)))


def fln_set_plan(K: int, H: int, norm_kind: int, plan: Plan | dict | None, dtype: int = DTYPE_BF16):
    if isinstance(plan, dict):
        plan = Plan(**plan)
    _check(load().fln_set_plan_dtype(int(K), int(H), int(norm_kind), int(dtype),
                                     ctypes.byref(plan) if plan is not None else None))


def fln_get_plan(K: int, H: int, norm_kind: int, T: int, microchunk_tokens: int = 0,
                 dtype: int = DTYPE_BF16) -> dict:
    p = Plan()
    _check(load().fln_get_plan_dtype(int(K), int(H), int(norm_kind), int(dtype), int(T), int(microchunk_tokens),
                                     ctypes.byref(p)))
    return p.as_dict()


def fln_device_status(stream=None):
    _check(load().fln_device_status(_stream_ptr(stream)))


def fln_last_error() -> str:
    return load().fln_last_error().decode(errors="replace")


def fln_release_workspace():
    load().fln_release_workspace()


def fln_launch_count() -> int:
    return int(load().fln_launch_count())


def fln_profile_enable(enable: bool = True):
    _check(load().fln_profile_enable(1 if enable else 0))


def fln_profile_read() -> dict:
    s = ProfileStats()
    _check(load().fln_profile_read(ctypes.byref(s)))
    return {name: {"launches": int(s.launches[i]), "total_ms": float(s.total_ms[i])}
            for i, name in enumerate(KERNEL_NAMES)}


def fln_debug_stall_next_call(enable: bool = True):
    """Test switch: the next FUSED launch's bounded row-statistics wait runs out."""
    _check(load().fln_debug_stall_next_call(1 if enable else 0))


def fln_set_splitk_tail_tokens(max_tokens: int):
    """UNFUSED calls with at most max_tokens tokens reduce, add and normalise in the split-K GEMM's tail."""
    _check(load().fln_set_splitk_tail_tokens(int(max_tokens)))


def fln_version() -> int:
    return int(load().fln_version())


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def fln_moe_route(logits, k: int, stream=None):
    """MoE routing and grouping on the device: logits [T,E] float32 CUDA tensor -> dict of int32 /
    float32 CUDA tensors ids [T,k], gates [T,k], offsets [E+1], row_token [T*k], row_slot [T*k],
    row_of [T,k] (expert e owns grouped rows offsets[e]..offsets[e+1]-1, tokens ascending)."""
    import torch
    T, E = logits.shape
    dev = logits.device
    res = {"ids": torch.empty((T, k), dtype=torch.int32, device=dev),
           "gates": torch.empty((T, k), dtype=torch.float32, device=dev),
           "offsets": torch.empty((E + 1,), dtype=torch.int32, device=dev),
           "row_token": torch.empty((T * k,), dtype=torch.int32, device=dev),
           "row_slot": torch.empty((T * k,), dtype=torch.int32, device=dev),
           "row_of": torch.empty((T, k), dtype=torch.int32, device=dev)}
    _check(load().fln_moe_route(_ptr(logits), int(T), int(E), int(k), _ptr(res["ids"]), _ptr(res["gates"]),
                                _ptr(res["offsets"]), _ptr(res["row_token"]), _ptr(res["row_slot"]),
                                _ptr(res["row_of"]), _stream_ptr(stream)))
    return res


def fused_moe_down_add_rmsnorm(hg, offsets, row_of, gates, We, residual, gamma, eps: float,
                               norm_kind: int = NORM_STANDARD, out=None, stream=None):
    """MoE region after the experts: y = hg . We[e(row)]^T per grouped row; residual += sum_j gates[t,j] *
    y[row_of[t,j]]; out = RMSNorm(residual).  hg [T*k,K] bf16; offsets [E+1], row_of [T,k] int32;
    gates [T,k] float32; We [E,H,K] bf16.  Returns out."""
    T, k = row_of.shape
    E, H, K = We.shape
    if out is None:
        import torch
        out = torch.empty((T, H), dtype=residual.dtype, device=residual.device)
    _check(load().fused_moe_down_add_rmsnorm(_ptr(hg), _ptr(offsets), _ptr(row_of), _ptr(gates), _ptr(We),
                                             _ptr(residual), _ptr(gamma), float(eps), int(norm_kind), int(T), int(K),
                                             int(H), int(E), int(k), _ptr(out), _stream_ptr(stream)))
    return out


def fln_moe_gather(x, row_token, k: int, out=None, stream=None):
    """Grouped copy of the hidden states: out[r] = x[row_token[r]] (x [T,H] bf16, row_token [T*k] int32)."""
    T, H = x.shape
    if out is None:
        import torch
        out = torch.empty((T * k, H), dtype=x.dtype, device=x.device)
    _check(load().fln_moe_gather(_ptr(x), _ptr(row_token), int(T), int(k), int(H), _ptr(out), _stream_ptr(stream)))
    return out



# ------------------------------------------------------------------ TPSP region across ranks
def _nccl_in_process():
    """The TP calls use the NCCL that PyTorch loads into the process."""
    import torch  # noqa: F401  (loads libnccl with the CUDA libraries)


def fln_tp_unique_id() -> bytes:
    """128-byte NCCL unique id for fln_tp_comm_init (made on one rank, sent to the others)."""
    _nccl_in_process()
    buf = ctypes.create_string_buffer(128)
    _check(load().fln_tp_unique_id(buf))
    return buf.raw


class TpComm:
    """One rank's TP communicator handle (current CUDA device); close() frees it."""

    def __init__(self, nranks: int, rank: int, unique_id: bytes | None = None):
        _nccl_in_process()
        h = ctypes.c_void_p()
        idbuf = None if unique_id is None else ctypes.create_string_buffer(bytes(unique_id), 128)
        _check(load().fln_tp_comm_init(int(nranks), int(rank), idbuf, ctypes.byref(h)))
        self.handle = h
        self.nranks, self.rank = int(nranks), int(rank)

    def close(self):
        if self.handle:
            _check(load().fln_tp_comm_destroy(self.handle))
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False


def fln_tp_layout(T: int, nranks: int, microchunk_tokens: int = 0) -> tuple:
    """(shard rows S, chunk tokens per rank, number of chunks); host only."""
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(load().fln_tp_layout(int(T), int(nranks), int(microchunk_tokens), ctypes.byref(a), ctypes.byref(b),
                                ctypes.byref(c)))
    return a.value, b.value, c.value


def fln_tp_chunk_rows(T: int, nranks: int, microchunk_tokens: int, chunk: int, rank: int) -> tuple:
    """(first token, block rows, valid rows) of chunk `chunk` of rank `rank`; host only."""
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(load().fln_tp_chunk_rows(int(T), int(nranks), int(microchunk_tokens), int(chunk), int(rank),
                                    ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def fused_proj_rs_add_rmsnorm_ag(x, W, residual_shard, gamma, eps: float, norm_kind: int, comm: TpComm,
                                 microchunk_tokens: int = 0, out=None, stream=None):
    """One rank's TPSP region: x [T,K] and W [H,K] are this rank's K-shards (bf16), residual_shard
    [ceil(T/P), H] its token shard (bf16, in place); returns out [T,H] bf16, the gathered normalised
    tensor."""
    T, K = x.shape
    H = W.shape[0]
    if out is None:
        import torch
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(load().fused_proj_rs_add_rmsnorm_ag(_ptr(x), _ptr(W), _ptr(residual_shard), _ptr(gamma), float(eps),
                                               int(norm_kind), int(T), int(K), int(H), int(microchunk_tokens),
                                               _ptr(out), comm.handle, _stream_ptr(stream)))
    return out


def fused_proj_rs_add_rmsnorm_ag_ptr(x_ptr, W_ptr, residual_ptr, gamma_ptr, eps, norm_kind, T, K, H,
                                     microchunk_tokens, out_ptr, comm_handle, stream_ptr) -> int:
    """Raw-pointer form: returns the status code without raising."""
    return load().fused_proj_rs_add_rmsnorm_ag(x_ptr, W_ptr, residual_ptr, gamma_ptr, float(eps), int(norm_kind),
                                               int(T), int(K), int(H), int(microchunk_tokens), out_ptr,
                                               comm_handle, stream_ptr)
