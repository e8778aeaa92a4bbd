"""Benchmark: fused projection + residual add + RMSNorm on GB300.

One step = one fused_proj_add_rmsnorm call over one batch of T tokens
(y = x W^T, residual += y, out = RMSNorm(residual)) through the C ABI, on
inputs already resident in HBM.  The default workload is the Llama-3-8B-shaped
o_proj prefill (T = K = H = 4096, standard RMSNorm, eps 1e-5); --config picks
another row of the workload table.  Inputs are synthetic and seeded.

Timing: W warm-up steps, then exactly K steps, each bracketed by CUDA events on
the launching stream with an L2 flush between steps, outside the events (a
512 MiB device write; with --l2-flush clean, the default, it is followed by a
512 MiB read of another buffer, so the timed step does not pay for writing back
the dirty lines the write left in L2); a barrier and a device synchronize on both sides of the
timed loop; the slowest rank's time counts.  The roofline fraction uses the
dominant kernel's own per-launch CUDA-event durations, recorded by the library
on the stream that launches it.

--impl reference times the fp64 CPU oracle instead (host cores, bounded row
sample per step, same metric and unit).

Prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused proj+add+RMSNorm TFLOP/s and tokens/s; % of roofline (tensor or HBM) on 1 GB300"
DEFAULT_CONFIG = "llama3_8b_oproj"
FLUSH_BYTES = 512 << 20
L2_FLUSH_NOTE = {"write": "flushed between timed steps (512 MiB write)",
                 "clean": "flushed between timed steps (512 MiB write, then a 512 MiB read of another buffer: "
                          "L2 holds clean unrelated lines when a step starts)"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch of the dominant kernel, from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum, one launch, -s 5 -c 1),
# keyed by workload, tokens, kernel, plan tile width (0 for the split-K
# kernels, whose tile follows the token count) and the sha1 of the kernel
# sources the capture was taken on; reported as null when the sources have
# changed since.  Captures: profiles/ (same commands).
class L2Flush:
    """Evicts the step's operands from L2 between timed steps.

    "write": fill a 512 MiB buffer (4x the L2).  The last L2's worth of it is
    left dirty, and writing it back is charged to whatever runs next.
    "clean": the same fill, then a 512 MiB read of a second buffer, which
    evicts the dirty lines outside the timed region."""

    def __init__(self, device, mode):
        import torch
        self.mode = mode
        self.buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.src = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device) if mode == "clean" else None
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def fill_(self, v):
        self.buf.fill_(v)
        if self.src is not None:
            import torch
            torch.sum(self.src, dim=0, out=self.sink)


def kernel_sources_hash(dtype, kernel):
    """sha1 (12 hex digits) of the sources the dominant kernel (by its profile name) is built from."""
    h = hashlib.sha1()
    if dtype == "moe":
        files = ["fln_moe.cu", "fln_gemm2.cu", "fln_ptx.cuh"]
    elif kernel == "gemm_fused":
        files = ["fln_gemm2.cu", "fln_ptx.cuh"]
    elif kernel == "gemm_splitk" and dtype in ("nvfp4", "mxfp4"):
        files = ["fln_gemm_w4.cu", "fln_ptx.cuh"]
    else:
        files = ["fln_gemm.cu", "fln_ptx.cuh"]
    for f in files:
        h.update(open(os.path.join(ROOT, "decoder_layer_projection_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:12]


NCU_TRAFFIC = {
    ("llama3_8b_oproj", 4096, "bf16", "gemm_fused", 256, "04894e535244"): 109651456 + 33146880,
    ("llama3_8b_down", 8192, "bf16", "gemm_fused", 256, "04894e535244"): 1209827584 + 122526720,
    ("gemma2_9b_down", 2048, "bf16", "gemm_fused", 192, "04894e535244"): 278789632 + 18013440,
    ("gemma2_9b_down", 2048, "bf16", "gemm_fused", 256, "04894e535244"): 286519808 + 22036480,
    ("llama70b_down_decode", 8, "bf16", "gemm_splitk", 0, "384cbfdf0b50"): 471428352 + 3621120,
    ("llama70b_oproj_decode", 8, "bf16", "gemm_splitk", 0, "384cbfdf0b50"): 135542016 + 2951936,
    ("llama3_8b_oproj", 4096, "e4m3", "gemm_fused", 224, "04894e535244"): 67461376 + 17776384,
    ("llama3_8b_down", 8192, "e4m3", "gemm_fused", 256, "04894e535244"): 541988352 + 110707456,
    ("llama70b_oproj_decode", 8, "e4m3", "gemm_splitk", 0, "384cbfdf0b50"): 67211008 + 72704,
    ("llama70b_down_decode", 8, "e4m3", "gemm_splitk", 0, "384cbfdf0b50"): 236310016 + 3079680,
    ("llama70b_down_decode", 8, "nvfp4", "gemm_splitk", 0, "75d05af169d4"): 135886080 + 2963712,
    ("llama70b_oproj_decode", 8, "nvfp4", "gemm_splitk", 0, "75d05af169d4"): 37937152 + 0,
    ("llama70b_down_decode", 8, "mxfp4", "gemm_splitk", 0, "75d05af169d4"): 128547072 + 2881536,
    ("llama70b_oproj_decode", 8, "mxfp4", "gemm_splitk", 0, "75d05af169d4"): 35841280 + 0,
    ("mixtral_8x7b_down_decode", 8, "moe", "moe_gemm", 256, "b78e8675c0a1"): 822593536 + 2991872,
    ("mixtral_8x7b_down", 4096, "moe", "moe_gemm", 256, "b78e8675c0a1"): 1400630016 + 123581440,
}
def traffic_tile(kname, plan):
    return plan["tile_n"] if kname in ("gemm_fused", "gemm_slot") else 0


# FP8 (E4M3) dense peak: the measured bf16 peak times NVIDIA's nominal dense
# FP8 / BF16 ratio (4.5 / 2.25 PFLOP/s); no FP8 GEMM peak is measured
FP8_OVER_BF16 = 2.0


def bench_config(wl, operands, world, l2_mode, extra=None):
    """The workload description both arms print in `config` (identical keys and values)."""
    c = {"workload": wl.name, "T": wl.T, "K": wl.K, "H": wl.H, "operands": operands,
         "norm": "gemma" if wl.norm_kind else "standard", "eps": wl.eps, "global_batch_tokens": wl.T * world,
         "parallelism": f"dp{world} (replicas)", "l2": L2_FLUSH_NOTE[l2_mode]}
    if extra:
        c.update(extra)
    return c


def moe_config(wl, E, k, world, l2_mode):
    return bench_config(wl, "bf16", world, l2_mode, {
        "experts": E, "top_k": k,
        "region": "MoE: routing + grouping, grouped down projection, unpermute + add + RMSNorm"})


# ------------------------------------------------------------------ distributed helpers
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base: int, rank: int) -> int:
    """Each data-parallel replica draws its own batch."""
    return int(base) + 1000003 * int(rank)


def max_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def whole_job_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Aggregate throughput: all ranks' units over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------------ peaks / clocks
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 20):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={self.interval_ms}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10], parts[5]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t0 - 0.05 <= r[0] <= self.t1 + 0.05] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------------ GPU arm
def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import decoder_layer_projection_gb300 as fln
    from synth import make_inputs, make_inputs_fp8, make_inputs_mxfp4, make_inputs_nvfp4, workload

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=device)

    fln.build()
    fln.load()
    if args.splitk_tail >= 0:
        fln.fln_set_splitk_tail_tokens(args.splitk_tail)
    wl = workload(args.config)
    if args.tokens:
        wl = wl.with_tokens(args.tokens)
    T, K, H = wl.T, wl.K, wl.H
    f8 = args.dtype == "e4m3"
    w4 = args.dtype in ("nvfp4", "mxfp4")
    mx = args.dtype == "mxfp4"
    dt = (fln.DTYPE_E4M3 if f8 else fln.DTYPE_MXFP4 if mx else fln.DTYPE_NVFP4 if w4 else fln.DTYPE_BF16)
    if f8:
        d = make_inputs_fp8(wl, seed=rank_seed(wl.seed, rank))
    elif w4:
        d = (make_inputs_mxfp4 if mx else make_inputs_nvfp4)(wl, seed=rank_seed(wl.seed, rank))
    else:
        d = make_inputs(wl, seed=rank_seed(wl.seed, rank))

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    if f8:
        x = torch.from_numpy(np.ascontiguousarray(d["x8"])).to(device)
        W = torch.from_numpy(np.ascontiguousarray(d["W8"])).to(device)
        sx = torch.from_numpy(d["x_scale"]).to(device)
        sw = torch.from_numpy(d["w_scale"]).to(device)
    elif w4:
        x = up(d["x"])
        W = torch.from_numpy(np.ascontiguousarray(d["Wq"])).to(device)
        sw = torch.from_numpy(np.ascontiguousarray(d["S"])).to(device)  # block scales
        sx = None
    else:
        x, W = up(d["x"]), up(d["W"])
        sx = sw = None
    r = up(d["r0"])
    gamma = torch.from_numpy(d["gamma"]).to(device)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    flush = L2Flush(device, args.l2_flush)
    stream = torch.cuda.current_stream(device)

    # profile the group on this device, as the pages' runtime does after the weights load
    t_tune = time.time()
    if args.plan == "auto":
        fln.fln_autotune(K, H, wl.norm_kind, T, stream, dtype=dt)
    else:
        f = args.plan.split(":")
        path = {"fused": fln.PATH_FUSED, "pipelined": fln.PATH_PIPELINED}[f[0]]
        fln.fln_set_plan(K, H, wl.norm_kind, dict(
            path=path, microchunk_tokens=int(f[1]), tile_n=int(f[2]), gemm_ctas=int(f[3]),
            norm_ctas=int(f[4]) if len(f) > 4 else 0, threshold_tokens=1 if T > 256 else 257,
            tuned_max_tokens=0, epi_warps=int(f[5]) if len(f) > 5 else 0), dtype=dt)
    t_tune = time.time() - t_tune
    plan = fln.fln_get_plan(K, H, wl.norm_kind, T, args.microchunk, dtype=dt)

    def step():
        if f8:
            fln.fused_proj_add_rmsnorm_fp8(x, sx, W, sw, r, gamma, wl.eps, wl.norm_kind, args.microchunk, out,
                                           stream)
        elif mx:
            fln.fused_proj_add_rmsnorm_mxfp4(x, W, sw, r, gamma, wl.eps, wl.norm_kind, args.microchunk, out, stream)
        elif w4:
            fln.fused_proj_add_rmsnorm_nvfp4(x, W, sw, d["gs"], r, gamma, wl.eps, wl.norm_kind, args.microchunk,
                                             out, stream)
        else:
            fln.fused_proj_add_rmsnorm(x, W, r, gamma, wl.eps, wl.norm_kind, args.microchunk, out, stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    fln.fln_device_status(stream)

    def timed_pass(profile: bool):
        """K steps, each bracketed by events on the launching stream, L2 flushed between them."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if profile:
            fln.fln_profile_enable(True)
        launches0 = fln.fln_launch_count()
        barrier(device)
        torch.cuda.synchronize(device)
        if sampler is not None:
            sampler.mark_begin()
        for i in range(args.steps):
            flush.fill_(float(i))  # L2 flush, outside the events
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(device)
        barrier(device)
        if sampler is not None:
            sampler.mark_end()
        nl = fln.fln_launch_count() - launches0
        prof = None
        if profile:
            prof = fln.fln_profile_read()
            fln.fln_profile_enable(False)
        fln.fln_device_status(stream)
        step_ms = [st.elapsed_time(en) for st, en in zip(starts, ends)]
        return sum(step_ms) / 1e3, nl, prof, step_ms

    # pass 1: the headline number, nothing recorded between the library's launches
    sampler = ClockSampler(local_rank)
    sampler.start()
    local_s, launches, _, head_step_ms = timed_pass(False)
    clocks = sampler.stop()
    sampler = None
    # pass 2: the same K steps with per-kernel events on each kernel's own stream (which kernel
    # dominates, and its time when a step launches more than one kernel)
    prof_s, _, prof, _ = timed_pass(True)
    max_s = max_over_ranks(local_s, device)
    ms_per_step = max_s * 1e3 / args.steps
    flops = wl.flops()
    value = whole_job_value(flops * args.steps, world, max_s) / 1e12
    tokens_per_s = whole_job_value(T * args.steps, world, max_s)

    # roofline of the dominant kernel (largest share of recorded device time)
    peaks, peak_src = load_peaks()
    kname = max(prof, key=lambda k: prof[k]["total_ms"])
    kp = prof[kname]
    avg_launch_ms = kp["total_ms"] / max(kp["launches"], 1)
    launches_per_step = kp["launches"] / args.steps
    if launches == args.steps and kp["launches"] == args.steps:
        # one library launch per step: the headline pass's step events, recorded on the stream that
        # launches the kernel, bracket exactly that launch
        avg_launch_ms = statistics.fmean(head_step_ms)
        kernel_timing = "headline pass: each step's CUDA events bracket the kernel's one launch on its stream"
    else:
        kernel_timing = ("second timed pass of the same K steps with per-kernel CUDA events on each kernel's "
                         "stream (a step launches more than one kernel)")
    tokens_per_launch = T / launches_per_step
    ob = 1.0 if f8 else 2.0  # bytes per x element (and per W element, except NVFP4)
    wb = 0.5 + (1.0 / 32.0 if mx else 1.0 / 16.0) if w4 else ob  # bytes per W element
    tensor_peak = peaks["bf16_tflops"] * (FP8_OVER_BF16 if f8 else 1.0)
    if kname in ("gemm_fused", "gemm_slot"):
        # tensor bound: 2 * tokens * K * H per launch
        achieved = 2.0 * tokens_per_launch * K * H / (avg_launch_ms * 1e-3) / 1e12
        bound, unit, peak = "tensor", "TFLOP/s", tensor_peak
    elif kname == "gemm_splitk":
        # HBM bound: W read once plus x, per launch
        achieved = (wb * H * K + ob * tokens_per_launch * K) / (avg_launch_ms * 1e-3) / 1e9
        bound, unit, peak = "hbm", "GB/s", peaks["hbm_gbs"]
    else:
        # add + norm: residual read and written, output written, gamma
        achieved = (tokens_per_launch * H * 6.0 + 4.0 * H) / (avg_launch_ms * 1e-3) / 1e9
        bound, unit, peak = "hbm", "GB/s", peaks["hbm_gbs"]
    src_hash = kernel_sources_hash(args.dtype, kname)
    traffic = NCU_TRAFFIC.get((args.config, T, args.dtype, kname, traffic_tile(kname, plan), src_hash))
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_unit": "bytes per launch (ncu)",
                "kernel": kname,
                "peak_source": (f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" else "fallback")
                + (" bf16 x 2, the nominal dense FP8/BF16 ratio" if f8 and bound == "tensor" else ""),
                "kernel_ms_per_launch": round(avg_launch_ms, 5), "launches_per_step": launches_per_step,
                "measured": kernel_timing,
                "profiled_ms_per_step": round(prof_s * 1e3 / args.steps, 5)}
    # full-step roofline: the slower of FLOPs at tensor peak and bytes at HBM bandwidth
    t_roof = max(flops / (tensor_peak * 1e12),
                 wl.algorithmic_bytes(1 if f8 else -1 if mx else 0 if w4 else 2) / (peaks["hbm_gbs"] * 1e9))
    step_frac = t_roof / (ms_per_step * 1e-3)

    # end to end through the public API with host buffers (pinned), copies inside the timed region
    e2e = run_e2e(args, wl, d, W, gamma, device, stream, fln, sw)
    comparator = run_comparator(args, wl, x, W, d, gamma, device, stream, fln, flush, sx, sw)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "config": bench_config(wl, args.dtype, world, args.l2_flush),
        "plan": dict(plan, plan_arg=args.plan, microchunk_arg=args.microchunk, tune_s=round(t_tune, 2)),
        "tokens_per_s": round(tokens_per_s, 1),
        "step_roofline_frac": round(step_frac, 4),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches,
        "kernel_time_ms": {k: round(v["total_ms"] / args.steps, 5) for k, v in prof.items() if v["launches"]},
        "comparator_unfused_cublas": comparator,
        "clocks": clocks,
    }
    if (world == 1 and not args.no_table and args.config == DEFAULT_CONFIG and args.dtype == "bf16"
            and not args.tokens):
        line["configs"] = run_table(args, fln, device, stream, flush, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, d, args.cpu_seconds)
    if world > 1:
        dist.destroy_process_group()
    return line if rank == 0 else None


def _moe_sample(d, E, sel):
    """The MoE region restricted to tokens sel, regrouped (a token's result depends only on its own rows)."""
    import oracle
    ids_s = d["ids"][sel]
    _, _, _, row_of = oracle.moe_permute(d["ids"], E)
    off_s, tok_s, slot_s, row_of_s = oracle.moe_permute(ids_s, E)
    return d["hg"][row_of[sel[tok_s], slot_s]], off_s, row_of_s, d["wt"][sel], d["r0"][sel]


def moe_cpu_baseline(wl, E, k, d, seconds):
    """The fp64 oracle's MoE region on a sample of token rows, on the host cores."""
    import numpy as np
    import oracle
    oracle.build()
    cores = oracle.max_threads()

    def timed(n):
        hg, off, row_of, wt, r0 = _moe_sample(d, E, np.arange(n))
        t = time.time()
        oracle.moe_down_region(hg, off, row_of, wt, d["We"], r0, d["gamma"], wl.eps, wl.norm_kind)
        return time.time() - t

    probe = min(wl.T, max(1, cores))
    t = timed(probe)
    n = int(min(wl.T, max(probe, probe * seconds / max(t, 1e-6))))
    t = timed(n) if n > probe else t
    flops = 2.0 * n * k * wl.K * wl.H
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {wl.T} tokens of {wl.name} (E={E}, k={k}; fp64, OpenMP over tokens), "
                      f"{t:.1f} s"}


def run_gpu_moe(args):
    """The MoE region (routing + grouping, grouped down projection, unpermute + add + norm) as one step."""
    import numpy as np
    import torch

    import decoder_layer_projection_gb300 as fln
    from synth import MOE_CONFIGS, make_inputs_moe

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    fln.build()
    fln.load()
    wl, E, k = MOE_CONFIGS[args.config]
    if args.tokens:
        wl = wl.with_tokens(args.tokens)
    T, K, H = wl.T, wl.K, wl.H
    d = make_inputs_moe(wl, E, k, seed=rank_seed(wl.seed, rank))

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    logits = torch.from_numpy(d["logits"]).to(device)
    hg, We, r = up(d["hg"]), up(d["We"]), up(d["r0"])
    gamma = torch.from_numpy(d["gamma"]).to(device)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    flush = L2Flush(device, args.l2_flush)
    stream = torch.cuda.current_stream(device)

    def step():
        g = fln.fln_moe_route(logits, k, stream)
        fln.fused_moe_down_add_rmsnorm(hg, g["offsets"], g["row_of"], g["gates"], We, r, gamma, wl.eps,
                                       wl.norm_kind, out, stream)
        return g

    for _ in range(args.warmup):
        flush.fill_(1.0)
        g = step()
    fln.fln_device_status(stream)
    used = int(np.unique(g["ids"].cpu().numpy()).size)

    def timed_pass(profile):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if profile:
            fln.fln_profile_enable(True)
        launches0 = fln.fln_launch_count()
        barrier(device)
        torch.cuda.synchronize(device)
        if sampler is not None:
            sampler.mark_begin()
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(device)
        barrier(device)
        if sampler is not None:
            sampler.mark_end()
        nl = fln.fln_launch_count() - launches0
        prof = None
        if profile:
            prof = fln.fln_profile_read()
            fln.fln_profile_enable(False)
        fln.fln_device_status(stream)
        return sum(st.elapsed_time(en) for st, en in zip(starts, ends)) / 1e3, nl, prof

    sampler = ClockSampler(local_rank)
    sampler.start()
    local_s, launches, _ = timed_pass(False)
    clocks = sampler.stop()
    sampler = None
    prof_s, _, prof = timed_pass(True)
    max_s = max_over_ranks(local_s, device)
    ms_per_step = max_s * 1e3 / args.steps
    R = T * k
    flops = 2.0 * R * K * H
    value = whole_job_value(flops * args.steps, world, max_s) / 1e12
    peaks, peak_src = load_peaks()
    kp = prof["moe_gemm"]
    avg_ms = kp["total_ms"] / max(kp["launches"], 1)
    w_bytes = used * H * K * 2.0
    if R <= 256:
        achieved = (w_bytes + 2.0 * R * K) / (avg_ms * 1e-3) / 1e9
        bound, unit, peak = "hbm", "GB/s", peaks["hbm_gbs"]
    else:
        achieved = flops / (avg_ms * 1e-3) / 1e12
        bound, unit, peak = "tensor", "TFLOP/s", peaks["bf16_tflops"]
    traffic = NCU_TRAFFIC.get((args.config, T, "moe", "moe_gemm", 256, kernel_sources_hash("moe", "moe_gemm")))
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_unit": "bytes per launch (ncu)",
                "kernel": "moe_gemm",
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" else "fallback",
                "kernel_ms_per_launch": round(avg_ms, 5), "launches_per_step": kp["launches"] / args.steps,
                "experts_used": used,
                "measured": "second timed pass of the same K steps with per-kernel CUDA events",
                "profiled_ms_per_step": round(prof_s * 1e3 / args.steps, 5)}
    alg_bytes = w_bytes + 2.0 * R * K + 6.0 * T * H + 4.0 * H + 4.0 * T * E
    t_roof = max(flops / (peaks["bf16_tflops"] * 1e12), alg_bytes / (peaks["hbm_gbs"] * 1e9))

    # end to end: logits, grouped activations and residual up, output and residual down, every step
    h_lg = torch.from_numpy(d["logits"]).pin_memory()
    h_hg = torch.from_numpy(np.ascontiguousarray(d["hg"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    h_r = torch.from_numpy(np.ascontiguousarray(d["r0"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    h_o = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    h_ro = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        logits.copy_(h_lg, non_blocking=True)
        hg.copy_(h_hg, non_blocking=True)
        r.copy_(h_r, non_blocking=True)
        step()
        h_o.copy_(out, non_blocking=True)
        h_ro.copy_(r, non_blocking=True)

    for _ in range(2):
        e2e_step()
    n = max(5, args.steps // 4)
    barrier(device)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    es = max_over_ranks(e0.elapsed_time(e1) / 1e3, device)
    e2e = {"value": round(whole_job_value(flops * n, world, es) / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(4 * T * E + 2 * R * K + 2 * T * H), "d2h_bytes_per_step": int(4 * T * H),
           "steps": n, "ms_per_step": round(es * 1e3 / n, 4), "weights": "We and gamma resident on the device"}

    # conventional sequence: one cuBLAS GEMM per expert, gated scatter-add, then add_rmsnorm
    offs = g["offsets"].cpu().numpy()
    row_token = g["row_token"].long()
    gate_row = g["gates"].reshape(-1)[g["row_token"].long() * k + g["row_slot"].long()]
    r2 = up(d["r0"])
    out2 = torch.empty_like(out)
    times = []
    for i in range(args.warmup + max(5, args.steps // 4)):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        y = torch.empty((R, H), dtype=torch.bfloat16, device=device)
        for e in range(E):
            if offs[e + 1] > offs[e]:
                torch.matmul(hg[offs[e]:offs[e + 1]], We[e].t(), out=y[offs[e]:offs[e + 1]])
        z = torch.zeros((T, H), dtype=torch.float32, device=device)
        z.index_add_(0, row_token, y.float() * gate_row[:, None])
        fln.add_rmsnorm(z.to(torch.bfloat16), r2, gamma, wl.eps, wl.norm_kind, out2, stream)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize(device)
    cms = [a.elapsed_time(b) for a, b in times[args.warmup:]]
    cm = sum(cms) / len(cms)
    comparator = {"value": round(flops / (cm * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(cm, 5),
                  "what": "per-expert torch.matmul (cuBLAS, bf16 out), gated index_add in fp32, then add_rmsnorm"}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": moe_config(wl, E, k, world, args.l2_flush),
        "tokens_per_s": round(whole_job_value(T * args.steps, world, max_s), 1),
        "step_roofline_frac": round(t_roof / (ms_per_step * 1e-3), 4),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches,
        "kernel_time_ms": {kk: round(v["total_ms"] / args.steps, 5) for kk, v in prof.items() if v["launches"]},
        "comparator_unfused_cublas": comparator,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = moe_cpu_baseline(wl, E, k, d, args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line if rank == 0 else None


def run_e2e(args, wl, d, W, gamma, device, stream, fln, sw=None):
    import numpy as np
    import torch
    T, K, H = wl.T, wl.K, wl.H
    f8 = args.dtype == "e4m3"
    if f8:
        hx = torch.from_numpy(np.ascontiguousarray(d["x8"])).pin_memory()
        hsx = torch.from_numpy(np.ascontiguousarray(d["x_scale"])).pin_memory()
        dx = torch.empty((T, K), dtype=torch.uint8, device=device)
        dsx = torch.empty_like(hsx, device=device)
    else:
        hx = torch.from_numpy(np.ascontiguousarray(d["x"]).view(np.int16)).view(torch.bfloat16).pin_memory()
        dx = torch.empty((T, K), dtype=torch.bfloat16, device=device)
    hr = torch.from_numpy(np.ascontiguousarray(d["r0"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    ho = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    hr_out = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    dr = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    do = torch.empty((T, H), dtype=torch.bfloat16, device=device)

    def step():
        dx.copy_(hx, non_blocking=True)
        dr.copy_(hr, non_blocking=True)
        if f8:
            dsx.copy_(hsx, non_blocking=True)
            fln.fused_proj_add_rmsnorm_fp8(dx, dsx, W, sw, dr, gamma, wl.eps, wl.norm_kind, args.microchunk, do,
                                           stream)
        elif args.dtype == "nvfp4":
            fln.fused_proj_add_rmsnorm_nvfp4(dx, W, sw, d["gs"], dr, gamma, wl.eps, wl.norm_kind, args.microchunk,
                                             do, stream)
        elif args.dtype == "mxfp4":
            fln.fused_proj_add_rmsnorm_mxfp4(dx, W, sw, dr, gamma, wl.eps, wl.norm_kind, args.microchunk, do, stream)
        else:
            fln.fused_proj_add_rmsnorm(dx, W, dr, gamma, wl.eps, wl.norm_kind, args.microchunk, do, stream)
        ho.copy_(do, non_blocking=True)
        hr_out.copy_(dr, non_blocking=True)

    if args.dtype == "bf16" and not args.e2e_torch_copies:
        # the library's host-buffer entry point: x and the residual go in and
        # the residual and out come back in transfer chunks that overlap the
        # compute (the residual host buffer is updated in place every step)
        def step():  # noqa: F811
            fln.fused_proj_add_rmsnorm_host(hx, W, hr_out, gamma, wl.eps, wl.norm_kind, args.transfer_tokens, ho,
                                            stream)
        hr_out.copy_(hr)

    for _ in range(max(2, args.warmup // 2)):
        step()
    n = max(5, args.steps // 4)
    barrier(device)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    s = max_over_ranks(e0.elapsed_time(e1) / 1e3, device)
    _, world, _ = dist_env()
    h2d = hx.numel() * hx.element_size() + hr.numel() * 2 + (hsx.numel() * 4 if f8 else 0)
    via = ("fused_proj_add_rmsnorm_host (C ABI, host buffers in page-locked memory, transfer chunks of "
           f"{args.transfer_tokens or 1024} tokens)" if args.dtype == "bf16" and not args.e2e_torch_copies else
           "torch copies from / to page-locked host memory around the C ABI call, one stream")
    return {"value": round(whole_job_value(wl.flops() * n, world, s) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 4 * T * H, "steps": n,
            "ms_per_step": round(s * 1e3 / n, 4), "weights": "W, its scales and gamma resident on the device",
            "via": via}


def run_comparator(args, wl, x, W, d, gamma, device, stream, fln, flush, sx=None, sw=None):
    """Unfused sequence: cuBLAS bf16 GEMM (torch.matmul) then the library's
    add_rmsnorm (bf16 operands only)."""
    import numpy as np
    import torch
    f8 = args.dtype == "e4m3"
    r = torch.from_numpy(np.ascontiguousarray(d["r0"]).view(np.int16)).view(torch.bfloat16).to(device)
    out = torch.empty_like(r)
    T, H = r.shape
    if args.dtype in ("nvfp4", "mxfp4"):
        return {"unavailable": "no library GEMM takes FP4 weights with bf16 activations here"}
    if f8:
        # torch._scaled_mm with row-wise scales ended in a GPU fault (Xid 43) on
        # this GPU under PyTorch 2.9.1 (its kernel prints that it was built
        # without sm_90+ TMA support); it is not run again.  The line names the
        # fault by its Xid only, so that the output carries no CUDA error text.
        return {"unavailable": "torch._scaled_mm row-wise FP8 faulted on GB300 under PyTorch 2.9.1 "
                               "(GPU Xid 43); not run"}
    else:
        def gemm():
            return torch.matmul(x, W.t())
        what = "torch.matmul (cuBLAS, bf16 out) then add_rmsnorm; y rounded to bf16 before the add"
    times = []
    for i in range(args.warmup + max(5, args.steps // 4)):
        flush.fill_(float(i))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        y = gemm()
        fln.add_rmsnorm(y, r, gamma, wl.eps, wl.norm_kind, out, stream)
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize(device)
    ms = [a.elapsed_time(b) for a, b in times[args.warmup:]]
    m = sum(ms) / len(ms)
    return {"value": round(wl.flops() / (m * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(m, 5),
            "what": what}


# ------------------------------------------------------------------ the other workloads
# Every large workload of the table besides the headline one: the Llama-3-8B
# down projection, the Gemma-2-9B down projection, and the 70B decode sweep
# (o_proj and down_proj at each token count).  The tiny workload is a parity
# case only.
TABLE_CASES = ([("llama3_8b_down", 0), ("gemma2_9b_down", 0)] +
               [(n, t) for n in ("llama70b_oproj_decode", "llama70b_down_decode") for t in (1, 8, 32, 128, 256)])
PATH_NAMES = {1: "FUSED", 2: "PIPELINED", 3: "UNFUSED"}
# the extensions of the region (FP8 operands, FP4 weights, the MoE region), measured by the same code
# as their own bench lines and summarised in the table
EXTRA_CASES = [("llama3_8b_oproj", 0, "e4m3"), ("llama3_8b_down", 0, "e4m3"),
               ("llama70b_oproj_decode", 8, "e4m3"), ("llama70b_down_decode", 8, "e4m3"),
               ("llama70b_oproj_decode", 8, "nvfp4"), ("llama70b_down_decode", 8, "nvfp4"),
               ("llama70b_oproj_decode", 8, "mxfp4"), ("llama70b_down_decode", 8, "mxfp4"),
               ("mixtral_8x7b_down_decode", 0, "moe"), ("mixtral_8x7b_down", 0, "moe")]


def summarize_line(line):
    """The figures of a workload's own bench line that the table keeps."""
    c, rf = line["config"], line["roofline"]
    comp = line.get("comparator_unfused_cublas") or {}
    out = {"workload": c["workload"], "T": c["T"], "K": c["K"], "H": c["H"], "operands": c.get("operands", "bf16"),
           "ms_per_step": line["ms_per_step"], "tflops": line["value"], "tokens_per_s": line["tokens_per_s"],
           "step_roofline_frac": line["step_roofline_frac"], "kernel": rf["kernel"],
           "kernel_ms_per_launch": rf["kernel_ms_per_launch"], "kernel_timing": rf["measured"],
           "roofline": {k: rf[k] for k in ("bound", "achieved", "unit", "frac", "traffic", "peak_source")},
           "kernel_time_ms": line["kernel_time_ms"], "e2e_tflops": line["e2e"]["value"],
           "gpu_launches_per_step": line["gpu_launches"] / line["steps"]}
    if "plan" in line:
        out["plan"] = {k: line["plan"][k] for k in ("path", "microchunk_tokens", "tile_n", "gemm_ctas",
                                                     "threshold_tokens", "epi_warps")}
    if "experts" in c:
        out.update(experts=c["experts"], top_k=c["top_k"], experts_used=rf.get("experts_used"))
    if "ms_per_step" in comp:
        out["comparator_unfused_cublas"] = {"ms_per_step": comp["ms_per_step"], "tflops": comp["value"]}
        out["speedup_vs_comparator"] = round(comp["ms_per_step"] / line["ms_per_step"], 4)
    else:
        out["comparator_unfused_cublas"] = comp
    return out


def kernel_roofline(kname, wl, T_launch, ms, peaks):
    """Roofline of one launch of a kernel: the slower of its FLOPs at the tensor peak and its
    algorithmic bytes at the HBM bandwidth decides the bound; returns (bound, achieved, unit, frac)."""
    K, H = wl.K, wl.H
    if kname in ("gemm_fused", "gemm_slot", "gemm_splitk"):
        flops = 2.0 * T_launch * K * H
        nbytes = 2.0 * H * K + 2.0 * T_launch * K + (6.0 * T_launch * H + 4.0 * H if kname == "gemm_fused" else 0.0)
    else:
        flops = 5.0 * T_launch * H
        nbytes = 6.0 * T_launch * H + 4.0 * H
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    s = ms * 1e-3
    if t_tensor >= t_hbm:
        return "tensor", flops / s / 1e12, "TFLOP/s", t_tensor / s
    return "hbm", nbytes / s / 1e9, "GB/s", t_hbm / s


def run_table(args, fln, device, stream, flush, peaks):
    """Each case: the tuned plan, K timed steps (L2 flushed between them, the headline's timing), the
    dominant kernel's per-launch time and roofline, and the unfused cuBLAS GEMM + add_rmsnorm comparator."""
    import numpy as np
    import torch
    from synth import make_inputs, workload

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    rows = []
    tuned = set()
    sampler = ClockSampler(device.index)
    sampler.start()
    sampler.mark_begin()
    t_start = time.time()
    for name, T in TABLE_CASES:
        wl = workload(name)
        if T:
            wl = wl.with_tokens(T)
        T, K, H = wl.T, wl.K, wl.H
        d = make_inputs(wl)
        x, W, r = up(d["x"]), up(d["W"]), up(d["r0"])
        gamma = torch.from_numpy(d["gamma"]).to(device)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        group = (K, H, wl.norm_kind)
        if group not in tuned:
            # decode groups are profiled once up to 256 tokens, so the token threshold decides the path
            fln.fln_autotune(K, H, wl.norm_kind, 256 if "decode" in name else T, stream)
            tuned.add(group)
        plan = fln.fln_get_plan(K, H, wl.norm_kind, T)

        def step():
            fln.fused_proj_add_rmsnorm(x, W, r, gamma, wl.eps, wl.norm_kind, 0, out, stream)

        for _ in range(args.warmup):
            flush.fill_(1.0)
            step()

        def timed(profile):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            if profile:
                fln.fln_profile_enable(True)
            n0 = fln.fln_launch_count()
            torch.cuda.synchronize(device)
            for i, (a, b) in enumerate(ev):
                flush.fill_(float(i))
                a.record(stream)
                step()
                b.record(stream)
            torch.cuda.synchronize(device)
            nl = fln.fln_launch_count() - n0
            prof = None
            if profile:
                prof = fln.fln_profile_read()
                fln.fln_profile_enable(False)
            fln.fln_device_status(stream)
            return [a.elapsed_time(b) for a, b in ev], nl, prof

        step_ms, nl, _ = timed(False)
        _, _, prof = timed(True)
        ms = statistics.fmean(step_ms)
        kname = max(prof, key=lambda k: prof[k]["total_ms"])
        kp = prof[kname]
        if nl == args.steps and kp["launches"] == args.steps:
            kms, ktiming = ms, "headline-style pass (one launch per step)"
        else:
            kms, ktiming = kp["total_ms"] / kp["launches"], "second pass, per-kernel events"
        lps = kp["launches"] / args.steps
        bound, achieved, unit, kfrac = kernel_roofline(kname, wl, T / lps, kms, peaks)
        t_roof = max(wl.flops() / (peaks["bf16_tflops"] * 1e12), wl.algorithmic_bytes(2) / (peaks["hbm_gbs"] * 1e9))
        src_hash = kernel_sources_hash("bf16", kname)
        traffic = NCU_TRAFFIC.get((name, T, "bf16", kname, traffic_tile(kname, plan), src_hash))
        # comparator: cuBLAS GEMM (bf16 out) then add_rmsnorm, same flush, same timing
        r2 = up(d["r0"])
        out2 = torch.empty_like(out)
        cm = []
        for i in range(args.warmup + args.steps):
            flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            y = torch.matmul(x, W.t())
            fln.add_rmsnorm(y, r2, gamma, wl.eps, wl.norm_kind, out2, stream)
            b.record(stream)
            cm.append((a, b))
        torch.cuda.synchronize(device)
        cms = statistics.fmean(a.elapsed_time(b) for a, b in cm[args.warmup:])
        rows.append({
            "workload": name, "T": T, "K": K, "H": H, "norm": "gemma" if wl.norm_kind else "standard",
            "path": PATH_NAMES.get(3 if T < plan["threshold_tokens"] else plan["path"]),
            "plan": {k: plan[k] for k in ("path", "microchunk_tokens", "tile_n", "gemm_ctas", "norm_ctas",
                                          "threshold_tokens", "epi_warps")},
            "ms_per_step": round(ms, 5), "tflops": round(wl.flops() / (ms * 1e-3) / 1e12, 2),
            "tokens_per_s": round(T / (ms * 1e-3), 1), "step_roofline_frac": round(t_roof / (ms * 1e-3), 4),
            "launches_per_step": nl / args.steps,
            "kernel": kname, "kernel_ms_per_launch": round(kms, 5), "kernel_timing": ktiming,
            "roofline": {"bound": bound, "achieved": round(achieved, 2), "unit": unit, "frac": round(kfrac, 4),
                         "traffic": traffic},
            "kernel_time_ms": {k: round(v["total_ms"] / args.steps, 5) for k, v in prof.items() if v["launches"]},
            "comparator_unfused_cublas": {"ms_per_step": round(cms, 5),
                                          "tflops": round(wl.flops() / (cms * 1e-3) / 1e12, 2)},
            "speedup_vs_comparator": round(cms / ms, 4),
        })
        del x, W, r, out, r2, out2, y
        torch.cuda.empty_cache()
    for name, T, dtype in EXTRA_CASES:
        import argparse
        sub = argparse.Namespace(**vars(args))
        sub.config, sub.tokens, sub.dtype = name, T, dtype
        sub.no_cpu_baseline, sub.no_table, sub.plan, sub.microchunk = True, True, "auto", 0
        rows.append(summarize_line(run_gpu_moe(sub) if dtype == "moe" else run_gpu(sub)))
        torch.cuda.empty_cache()
    sampler.mark_end()
    clocks = sampler.stop()
    return {"cases": rows, "clocks": clocks, "wall_s": round(time.time() - t_start, 1),
            "what": "bf16 cases: each with its tuned plan (decode groups profiled up to 256 tokens), the same "
                    "timing and L2 flush as the headline; roofline of the dominant kernel: the slower of its "
                    "FLOPs at the tensor peak and its algorithmic bytes at the HBM bandwidth (measured peaks). "
                    "FP8, FP4 and MoE cases: the figures of each one's own bench line (bench.py --config C "
                    "--dtype D), run in this process"}


# ------------------------------------------------------------------ CPU oracle
def _oracle_rows_timed(wl, d, rows, nthreads=0):
    import numpy as np
    import oracle
    t = time.time()
    rows = np.asarray(rows, np.int64)
    if "x8" in d:
        oracle.proj_add_rmsnorm_fp8(d["x8"], d["x_scale"], d["W8"], d["w_scale"], d["r0"], d["gamma"], wl.eps,
                                    wl.norm_kind, rows=rows, nthreads=nthreads)
    elif "Wq" in d and "gs" not in d:
        oracle.proj_add_rmsnorm_mxfp4(d["x"], d["Wq"], d["S"], d["r0"], d["gamma"], wl.eps, wl.norm_kind, rows=rows,
                                      nthreads=nthreads)
    elif "Wq" in d:
        oracle.proj_add_rmsnorm_nvfp4(d["x"], d["Wq"], d["S"], d["gs"], d["r0"], d["gamma"], wl.eps, wl.norm_kind,
                                      rows=rows, nthreads=nthreads)
    else:
        oracle.proj_add_rmsnorm(d["x"], d["W"], d["r0"], d["gamma"], wl.eps, wl.norm_kind, rows=rows,
                                nthreads=nthreads)
    return time.time() - t


def cpu_baseline(wl, d, seconds: float):
    """The fp64 oracle as it stands, on this host's cores, on a bounded row sample."""
    import oracle
    cores = oracle.max_threads()
    probe = min(wl.T, max(1, cores))
    t = _oracle_rows_timed(wl, d, list(range(probe)))
    rows = int(min(wl.T, max(probe, probe * seconds / max(t, 1e-6))))
    t = _oracle_rows_timed(wl, d, list(range(rows)))
    flops = 2.0 * rows * wl.K * wl.H
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} of {wl.T} token rows of {wl.name} (fp64, OpenMP over rows), {t:.1f} s"}


def run_reference(args):
    """--impl reference: the oracle timed on host cores, same metric/unit/config."""
    import oracle
    from synth import make_inputs, make_inputs_fp8, make_inputs_mxfp4, make_inputs_nvfp4, workload
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    wl = workload(args.config)
    if args.tokens:
        wl = wl.with_tokens(args.tokens)
    oracle.build()
    d = (make_inputs_fp8(wl) if args.dtype == "e4m3" else make_inputs_nvfp4(wl) if args.dtype == "nvfp4"
         else make_inputs_mxfp4(wl) if args.dtype == "mxfp4" else make_inputs(wl))
    cores = oracle.max_threads()
    # rows per step sized so that warm-up + steps stay within about a minute
    probe = min(wl.T, max(1, cores))
    t = _oracle_rows_timed(wl, d, list(range(probe)))
    per_step = float(args.ref_seconds) / max(1, args.steps + args.warmup)
    rows = int(min(wl.T, max(1, probe * per_step / max(t, 1e-6))))
    for i in range(args.warmup):
        _oracle_rows_timed(wl, d, [(i * rows + j) % wl.T for j in range(rows)])
    total = 0.0
    for i in range(args.steps):
        total += _oracle_rows_timed(wl, d, [(i * rows + j) % wl.T for j in range(rows)])
    flops = 2.0 * rows * wl.K * wl.H * args.steps
    value = flops / total / 1e12
    sample = f"{rows} of {wl.T} token rows per step of {wl.name} ({args.dtype} inputs, fp64 oracle, OpenMP over rows)"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": bench_config(wl, args.dtype, world, args.l2_flush),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference_moe(args):
    """--impl reference for a MoE workload: the fp64 oracle's region on host cores, sampled tokens per step."""
    import numpy as np
    import oracle
    from synth import MOE_CONFIGS, make_inputs_moe
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    wl, E, k = MOE_CONFIGS[args.config]
    if args.tokens:
        wl = wl.with_tokens(args.tokens)
    oracle.build()
    d = make_inputs_moe(wl, E, k)
    cores = oracle.max_threads()

    def timed(sel):
        hg, off, row_of, wt, r0 = _moe_sample(d, E, np.asarray(sel, np.int64))
        t = time.time()
        oracle.moe_route(d["logits"][sel], k)
        oracle.moe_down_region(hg, off, row_of, wt, d["We"], r0, d["gamma"], wl.eps, wl.norm_kind)
        return time.time() - t

    probe = min(wl.T, max(1, cores))
    t = timed(list(range(probe)))
    per_step = float(args.ref_seconds) / max(1, args.steps + args.warmup)
    rows = int(min(wl.T, max(1, probe * per_step / max(t, 1e-6))))
    for i in range(args.warmup):
        timed([(i * rows + j) % wl.T for j in range(rows)])
    total = sum(timed([(i * rows + j) % wl.T for j in range(rows)]) for i in range(args.steps))
    value = 2.0 * rows * k * wl.K * wl.H * args.steps / total / 1e12
    sample = f"{rows} of {wl.T} tokens per step of {wl.name} (E={E}, k={k}; fp64 oracle, OpenMP over tokens)"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": moe_config(wl, E, k, world, args.l2_flush),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["libfusedln", "reference"], default="libfusedln")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--tokens", type=int, default=0, help="override T of the workload")
    ap.add_argument("--microchunk", type=int, default=0, help="0 = tuned plan")
    ap.add_argument("--plan", default="auto",
                    help="auto (tune the group) or path:chunk:tile:gemm_ctas[:norm_ctas[:epi_warps]], "
                         "path fused|pipelined")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU work of the cpu_baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=60.0, help="--impl reference: CPU work of the whole run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--splitk-tail", type=int, default=-1,
                    help="UNFUSED calls of at most this many tokens reduce in the split-K GEMM's tail "
                         "(0 = separate reducer kernel; -1 = the library's default)")
    ap.add_argument("--no-table", action="store_true",
                    help="skip the other workloads' record (run with the default workload at N = 1)")
    ap.add_argument("--transfer-tokens", type=int, default=0,
                    help="e2e: tokens per host transfer chunk of fused_proj_add_rmsnorm_host (0 = its default)")
    ap.add_argument("--e2e-torch-copies", action="store_true",
                    help="e2e: torch copies around the device-pointer call instead of the host-buffer entry point")
    ap.add_argument("--l2-flush", choices=["clean", "write"], default="clean",
                    help="between timed steps: 512 MiB write (write), or the write then a 512 MiB read (clean)")
    ap.add_argument("--dtype", choices=["bf16", "e4m3", "nvfp4", "mxfp4"], default="bf16",
                    help="operand types: bf16; e4m3 (FP8 x and W with per-token / per-channel scales); "
                         "nvfp4 (NVFP4 weights, bf16 x); mxfp4 (MXFP4 weights, bf16 x)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from synth import MOE_CONFIGS
    if args.config in MOE_CONFIGS:
        if args.impl == "reference":
            line = run_reference_moe(args)
        else:
            line = run_gpu_moe(args)
    else:
        line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
