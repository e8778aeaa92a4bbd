/*
 * libfusedln.h -- C ABI of the GB300 (sm_103a) library for the dense
 * decoder-layer region
 *
 *     y   = x . W^T                    row-parallel projection (o_proj / down_proj)
 *     r   = r + y                      residual add, in place
 *     out = RMSNorm(r)                 standard:  r / sqrt(mean_h r^2 + eps) * gamma
 *                                      Gemma:     r / sqrt(mean_h r^2 + eps) * (1 + gamma)
 *
 * Sources (web pages; cited by title and section):
 *   - vLLM "TPSP Design", section 1 "Motivation": the projection is followed by a
 *     residual add and a norm that keeps the complete hidden dimension of every
 *     token; section 3 "Fusion regions": o_proj -> add + post-attention norm and
 *     down_proj -> add + next input norm; section 3 "Microchunk pipeline": per
 *     chunk GEMM then add/norm on a second stream through three reusable slots,
 *     only valid rows written; section 3 "Profiling and fallback": tuning of the
 *     microchunk size and SM-count targets, candidate numerical checks, a
 *     token-threshold search, overrides, errors that propagate; section 4
 *     "Constraints": BF16, standard RMSNorm without bias, microchunks capped at
 *     4096 tokens, calls must fit the profiled token maximum, a shared
 *     workspace that assumes sequential calls.
 *   - torch-spyre "Plugin Architecture": F.linear semantics, W stored [out, in]
 *     ("Transposed linear weights"); GemmaRMSNorm's trailing fp32 weight
 *     multiply and the fp32 upcast of RMSNorm ("Custom Op Replacement" table,
 *     "Transformers backend").
 *   On one GPU the pages' ReduceScatter / AllGather between the GEMM and the
 *   add/norm are absent; everything else keeps its meaning.
 *
 * Conventions for every call
 *   - Tensors are row-major with the last dimension contiguous.  bf16 tensors
 *     are passed as pointers to their 16-bit storage (fln_bf16).  gamma is fp32.
 *   - Pointers are CUDA device pointers on the current device, 16-byte
 *     aligned (fused_proj_add_rmsnorm_host takes its activations in host
 *     memory).  The caller owns every tensor; the library never frees them.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Work the library puts on its internal second stream is joined back into
 *     `stream` before the call returns; nothing is synchronised on the host.
 *   - Return value: FLN_OK, or a negative fln_status.  On an error nothing has
 *     been launched, except FLN_ERR_CUDA from a failed launch in the middle of
 *     a call.  fln_last_error() gives a message for the calling thread.
 *     Errors are reported, never retried or routed around.
 *   - The library owns a per-device workspace (row statistics, pipeline slots,
 *     split-K partials, a device error word).  It is grown on demand with
 *     cudaMalloc the first time a shape needs more (so make the first call for
 *     a shape outside CUDA-graph capture), it is shared by all calls on a
 *     device, and calls must therefore be issued sequentially: two host
 *     threads calling concurrently on one device is unsupported.
 */
#ifndef LIBFUSEDLN_H
#define LIBFUSEDLN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t fln_bf16;               /* storage of one bfloat16 value */
typedef struct CUstream_st* fln_stream_t; /* identical to cudaStream_t */

typedef enum {
  FLN_OK = 0,
  FLN_ERR_INVALID_ARG = -1,    /* null/misaligned/host pointer, bad size, bad kind, bad eps, aliasing */
  FLN_ERR_UNSUPPORTED = -2,    /* valid but outside what the kernels support (e.g. H > 32768) */
  FLN_ERR_CUDA = -3,           /* a CUDA runtime call or launch failed */
  FLN_ERR_DEVICE_TIMEOUT = -4, /* a kernel's bounded wait expired (reported by fln_device_status) */
  FLN_ERR_NOT_TUNED = -5,      /* automatic choice requested for T above the tuned token maximum */
  FLN_ERR_COMM = -6            /* the collective library (NCCL) is missing or a collective failed */
} fln_status;

typedef enum { FLN_NORM_STANDARD = 0, FLN_NORM_GEMMA = 1 } fln_norm_kind;

/* Execution paths (vLLM "TPSP Design", section 3 "Microchunk pipeline" and
 * "Profiling and fallback").
 *   FUSED      one persistent tcgen05 GEMM whose epilogue does the residual
 *              add, the full-row sum of squares (combined across the row's
 *              N-tiles through global partial sums) and the norm.  Microchunks
 *              run back to back inside one launch of up to 16384 tokens (as
 *              many whole chunks as fit; tiles in row-block order, so one
 *              chunk's add + norm overlaps the next chunk's GEMM on other
 *              CTA pairs).  From 128 K-blocks (K >= 8192 bf16, 16384 E4M3;
 *              32 K-blocks with eight epilogue warps) a last round of tiles
 *              that would leave half of the CTA pairs idle is split into
 *              K-halves on two pairs (fp32 halves added in a fixed order).  A row wider than the grid has CTA pairs (N-tiles >
 *              pairs) runs the PIPELINED path instead.
 *   PIPELINED  per microchunk, the GEMM writes y (fp32) into one of three
 *              reusable slots on the caller's stream; the add + norm of that
 *              chunk runs on a second stream, overlapping the next GEMM.
 *   UNFUSED    the conventional sequence for small token counts: a split-K
 *              GEMM (H on the MMA's M side) then a separate add + norm pass. */
typedef enum { FLN_PATH_FUSED = 1, FLN_PATH_PIPELINED = 2, FLN_PATH_UNFUSED = 3 } fln_path;

/* How calls for one projection group (K, H, norm kind) execute. */
typedef struct {
  int path;              /* fln_path used when T >= threshold_tokens (FUSED or PIPELINED) */
  int microchunk_tokens; /* 1..4096, the chunk of tokens per pipeline step */
  int tile_n;            /* GEMM tile width on H: 64 (PIPELINED only), 128, 192 or 224 (FUSED only), 256 */
  int gemm_ctas;         /* SM-count target of the persistent GEMM grid; 0 = all SMs */
  int norm_ctas;         /* CTA cap of the second-stream add + norm (PIPELINED); 0 = no cap */
  int threshold_tokens;  /* T < threshold -> UNFUSED; 1..257 (UNFUSED handles T <= 256) */
  int tuned_max_tokens;  /* largest T the plan was profiled for; 0 = not profiled */
  int epi_warps;         /* FUSED: epilogue warps per CTA, 4, or 8 = two groups of four taking
                            alternate tiles (tile 224 or 256 only); 0 = automatic (8 for FP8
                            operands with K <= 6144 on tiles 224 / 256, else 4) */
} fln_plan;

/*
 * fused_proj_add_rmsnorm -- y = x . W^T; residual += y; out = RMSNorm(residual)
 *
 *   x          [T, K] bf16 activations (input of o_proj / down_proj)
 *   W          [H, K] bf16 weight, F.linear layout [out, in]
 *   residual   [T, H] bf16, read and overwritten with r0 + y (rounded to bf16)
 *   gamma      [H] fp32 norm weight
 *   eps        finite, >= 0, added to the mean square inside the square root
 *   norm_kind  FLN_NORM_STANDARD (x gamma) or FLN_NORM_GEMMA (x (1 + gamma))
 *   T          tokens, 0 <= T <= 2^24 (T = 0 is an empty call)
 *   K, H       multiples of 8 (16-byte rows); 8 <= K <= 2^20, 8 <= H <= 32768
 *   microchunk_tokens  0 = automatic (the group's plan); else 1..4096
 *   out        [T, H] bf16 normalised output; must not overlap x, W, residual
 *
 * The norm statistics and the normalised output are computed from the fp32
 * sum r0 + y, before the residual is rounded to bf16.  Rows at or beyond T
 * are never written.  With microchunk_tokens = 0 and a profiled plan whose
 * tuned_max_tokens < T the call returns FLN_ERR_NOT_TUNED.
 */
int fused_proj_add_rmsnorm(const fln_bf16* x, const fln_bf16* W, fln_bf16* residual, const float* gamma,
                           float eps, int norm_kind, int T, int K, int H, int microchunk_tokens, fln_bf16* out,
                           fln_stream_t stream);

/*
 * fused_proj_add_rmsnorm_host -- the same region for activations held in host
 * memory.  The microchunk pipeline of vLLM "TPSP Design" (section 3: per chunk,
 * compute on one stream while the chunk before is exchanged on another) with
 * the host link in place of the collectives.
 *
 *   x_host         [T, K] bf16 in HOST memory (page-locked memory lets the
 *                  copies overlap; pageable memory works, without overlap)
 *   W, gamma       DEVICE pointers as in fused_proj_add_rmsnorm (weights stay
 *                  resident)
 *   residual_host  [T, H] bf16 in HOST memory, read and overwritten with r0 + y
 *   out_host       [T, H] bf16 in HOST memory, must not overlap x_host or
 *                  residual_host
 *   transfer_tokens  tokens per transfer chunk: 0 = 1024, else 1..4096
 *   eps, norm_kind, T, K, H as in fused_proj_add_rmsnorm
 *
 * The tokens stream through the GPU in chunks of transfer_tokens: the copy of
 * chunk i + 1 to the device, the projection + add + norm of chunk i (on
 * `stream`, with the group's plan for that chunk's token count) and the copy
 * of chunk i - 1 back to the host run at the same time on three streams,
 * through three device staging slots the library owns (allocated on first
 * use and grown as needed; fln_release_workspace frees them).  Asynchronous
 * on `stream` like the other calls: the copies start after the work queued
 * on `stream` before the call, the host buffers must stay valid and unchanged
 * until `stream` completes, and only then do residual_host and out_host hold
 * the results.  Calls are sequential-use like the workspace (one host thread
 * at a time).  Errors: FLN_ERR_INVALID_ARG for NULL or device host-side
 * pointers, host or misaligned device-side pointers, bad sizes;
 * FLN_ERR_NOT_TUNED, before any copy, when a transfer chunk exceeds the
 * group's profiled token maximum; FLN_ERR_CUDA for a failing copy or launch.
 */
int fused_proj_add_rmsnorm_host(const fln_bf16* x_host, const fln_bf16* W, fln_bf16* residual_host,
                                const float* gamma, float eps, int norm_kind, int T, int K, int H,
                                int transfer_tokens, fln_bf16* out_host, fln_stream_t stream);

/* Operand element types of a projection group. */
typedef enum { FLN_DTYPE_BF16 = 0, FLN_DTYPE_E4M3 = 1, FLN_DTYPE_NVFP4 = 2, FLN_DTYPE_MXFP4 = 3 } fln_dtype;

/*
 * fused_proj_add_rmsnorm_fp8 -- the same region with FP8 operands ("TPSP
 * Design", section 5 "To-do": FP8 dense, quantized projections and scale
 * handling across microchunks):
 *
 *     y[t,h] = sx[t] * sw[h] * sum_k x[t,k] * W[h,k];  residual += y;  out = RMSNorm(residual)
 *
 *   x          [T, K] FP8 E4M3 codes (OCP "FN" form: bias 7, max 448, no
 *              infinities), one byte per element, produced by the caller
 *   x_scale    fp32 dequantisation scale(s) of x: [T] (x_scale_per_token != 0)
 *              or [1] (one scale for the tensor)
 *   W          [H, K] E4M3 codes, F.linear layout [out, in]
 *   w_scale    fp32 scale(s) of W: [H] (w_scale_per_channel != 0, one per
 *              output row) or [1]
 *   K          multiple of 16 (16-byte rows), 16 <= K <= 2^20; H multiple of 8
 *   the rest   as in fused_proj_add_rmsnorm (bf16 residual and out, fp32 gamma)
 *
 * The products are accumulated in fp32 by the tensor cores (tcgen05
 * kind::f8f6f4) and scaled in fp32 before the residual add.  A microchunk
 * uses its own tokens' scales, so the chunking changes no result bit.  Every
 * path exists for FP8 (FUSED, PIPELINED, UNFUSED); plans, tuning and the
 * threshold are kept per (K, H, norm_kind, FLN_DTYPE_E4M3) group.  The scale
 * pointers must be device pointers, 16-byte aligned; the library does not
 * quantise x (the producing operation supplies E4M3 codes and their scales).
 */
int fused_proj_add_rmsnorm_fp8(const uint8_t* x, const float* x_scale, int x_scale_per_token, const uint8_t* W,
                               const float* w_scale, int w_scale_per_channel, fln_bf16* residual,
                               const float* gamma, float eps, int norm_kind, int T, int K, int H,
                               int microchunk_tokens, fln_bf16* out, fln_stream_t stream);

/*
 * fused_proj_add_rmsnorm_nvfp4 -- the region with NVFP4 weights and bf16
 * activations ("TPSP Design", section 5 "To-do": MXFP4 / NVFP4 dense, low-bit
 * weight layouts and their scaling):
 *
 *     w[h,k] = w_global_scale * e4m3(W_scale[h, k/16]) * e2m1(W[h,k])
 *     residual += x . w^T;  out = RMSNorm(residual)
 *
 *   x           [T, K] bf16
 *   W           [H, K/2] bytes: E2M1 codes, element 2j of a row in the low
 *               nibble of byte j, element 2j + 1 in the high nibble
 *   W_scale     [H, K/16] E4M3 codes, one per 16 consecutive elements of a
 *               row (finite)
 *   w_global_scale  the fp32 tensor scale
 *   K           multiple of 64; the rest as in fused_proj_add_rmsnorm
 *
 * e2m1 * e4m3 is exact in bf16, so the tensor cores multiply bf16 x by exact
 * bf16 weights with fp32 accumulation, and the tensor scale multiplies the
 * fp32 result.  Below the threshold (few tokens) the split-K GEMM reads W
 * packed (0.5625 bytes per weight) and dequantises it on the SM; at and
 * above it the call first converts the whole weight to bf16 in the
 * workspace (H * K * 2 bytes) and runs the bf16 FUSED or PIPELINED path.
 * Plans, tuning and the threshold are kept per (K, H, norm_kind,
 * FLN_DTYPE_NVFP4) group.  |w_global_scale| must not exceed 2^100
 * (FLN_ERR_INVALID_ARG otherwise).
 */
int fused_proj_add_rmsnorm_nvfp4(const fln_bf16* x, const uint8_t* W, const uint8_t* W_scale,
                                 float w_global_scale, fln_bf16* residual, const float* gamma, float eps,
                                 int norm_kind, int T, int K, int H, int microchunk_tokens, fln_bf16* out,
                                 fln_stream_t stream);

/*
 * fused_proj_add_rmsnorm_mxfp4 -- the region with MXFP4 weights (the OCP
 * microscaling FP4 layout) and bf16 activations (the same "MXFP4 / NVFP4
 * dense" to-do item):
 *
 *     w[h,k] = e8m0(W_scale[h, k/32]) * e2m1(W[h,k]),  e8m0(E) = 2^(E - 127)
 *     residual += x . w^T;  out = RMSNorm(residual)
 *
 *   x           [T, K] bf16
 *   W           [H, K/2] bytes, packed as for fused_proj_add_rmsnorm_nvfp4
 *   W_scale     [H, K/32] E8M0 codes, one per 32 consecutive elements of a
 *               row; the code 255 (NaN) makes its row's outputs NaN
 *   K           multiple of 128; the rest as in fused_proj_add_rmsnorm
 *
 * Every w is a bf16 value as long as |w| stays below the bf16 maximum
 * (E <= 252 always does): the tensor cores multiply bf16 x by exact bf16
 * weights with fp32 accumulation.  Paths, workspace and plans as for NVFP4,
 * per (K, H, norm_kind, FLN_DTYPE_MXFP4) group.
 */
int fused_proj_add_rmsnorm_mxfp4(const fln_bf16* x, const uint8_t* W, const uint8_t* W_scale, fln_bf16* residual,
                                 const float* gamma, float eps, int norm_kind, int T, int K, int H,
                                 int microchunk_tokens, fln_bf16* out, fln_stream_t stream);

/*
 * fln_moe_route -- routing and expert grouping of the MoE region ("TPSP
 * Design", section 3 "Fusion regions": routing and permute before the
 * grouped GEMM; section 5 "To-do": MoE).
 *
 *   logits     [T, E] fp32 router outputs (finite), device
 *   ids        [T, k] int32 out: the k experts of largest logit per token,
 *              largest first, equal logits: smaller expert index first
 *   gates      [T, k] fp32 out: softmax over the token's k chosen logits
 *   offsets    [E + 1] int32 out: expert e owns grouped rows
 *              [offsets[e], offsets[e + 1]); offsets[E] = T * k
 *   row_token  [T * k] int32 out: the token of each grouped row
 *   row_slot   [T * k] int32 out: its slot j (ids[token, j] is the row's expert)
 *   row_of     [T, k] int32 out: the grouped row of pair (t, j)
 *   1 <= E <= 256, 1 <= k <= min(8, E), T * k < 2^31.
 *
 * Rows of an expert are ordered by token.  All arrays are caller-owned device
 * memory, 16-byte aligned; nothing is allocated.  The up-projection of the
 * MoE layer (gather by row_token, expert MLP) is the caller's; its grouped
 * output feeds fused_moe_down_add_rmsnorm.
 */
int fln_moe_route(const float* logits, int T, int E, int k, int* ids, float* gates, int* offsets, int* row_token,
                  int* row_slot, int* row_of, fln_stream_t stream);

/*
 * fln_moe_gather -- the permute step of the MoE region's input side: gathers
 * the (normalised) hidden states into the grouped order fln_moe_route wrote,
 *
 *   xg[r, :] = x[row_token[r], :]      r < T * k
 *
 *   x          [T, H] bf16; row_token [T * k] int32 (fln_moe_route's, every
 *              entry in [0, T)); xg [T * k, H] bf16 out, must not overlap x
 *   H % 8 == 0; 1 <= k <= 8.  Bit-exact copy; device memory, 16-byte aligned.
 *   A row_token entry outside [0, T) leaves its row of xg unwritten and makes
 *   fln_device_status return FLN_ERR_INVALID_ARG.
 * The expert MLP (the caller's) turns xg into the grouped activations hg of
 * fused_moe_down_add_rmsnorm.
 */
int fln_moe_gather(const fln_bf16* x, const int* row_token, int T, int k, int H, fln_bf16* xg, fln_stream_t stream);

/*
 * fused_moe_down_add_rmsnorm -- the MoE region after the experts: grouped
 * down projection, unpermute, residual add and RMSNorm ("TPSP Design",
 * section 3: grouped GEMM -> unpermute -> add / next norm):
 *
 *   y[r, :]  = hg[r, :] . We[e(r)]^T          (e(r): the expert owning row r)
 *   residual[t, :] += sum_j gates[t, j] * y[row_of[t, j], :]   (slot order, fp32)
 *   out[t, :] = RMSNorm(residual[t, :])
 *
 *   hg         [T * k, K] bf16 grouped expert activations (rows as offsets)
 *   offsets    [E + 1], row_of [T, k], gates [T, k]: as fln_moe_route writes
 *   We         [E, H, K] bf16 down-projection weights (F.linear layout)
 *   residual, gamma, eps, norm_kind, out: as in fused_proj_add_rmsnorm
 *   K % 8 == 0; H % 8 == 0, H <= 16384; E, k as in fln_moe_route.
 *
 * y is kept in fp32 in the library workspace ([T * k, H]); the grouped GEMM
 * is a persistent tcgen05 kernel over (expert, 128-row tile, 256-column tile)
 * items read from the device offsets (with T * k >= 256 E: over (expert,
 * 256-row block, 256-column tile) tiles on CTA pairs), so no host
 * synchronisation is needed.
 * Offsets that are not a grouping of the T * k rows (0 first, T * k last,
 * non-decreasing) make the call write nothing, a row_of entry outside
 * [0, T * k) leaves that token's residual and out rows untouched; either
 * makes fln_device_status return FLN_ERR_INVALID_ARG.
 */
int fused_moe_down_add_rmsnorm(const fln_bf16* hg, const int* offsets, const int* row_of, const float* gates,
                               const fln_bf16* We, fln_bf16* residual, const float* gamma, float eps, int norm_kind,
                               int T, int K, int H, int E, int k, fln_bf16* out, fln_stream_t stream);

/*
 * add_rmsnorm -- residual += y; out = RMSNorm(residual)   (the add/norm step alone)
 *
 *   y [T, H] bf16 addend; residual [T, H] bf16 in/out; gamma [H] fp32;
 *   out [T, H] bf16, must not overlap y or residual.  Other arguments as above.
 */
int add_rmsnorm(const fln_bf16* y, fln_bf16* residual, const float* gamma, float eps, int norm_kind, int T,
                int H, fln_bf16* out, fln_stream_t stream);

/*
 * fln_autotune -- profile a projection group on the current device ("TPSP
 * Design", section 3 "Profiling and fallback").  Sweeps path x microchunk x
 * tile width x SM-count target on synthetic data of shape [max_tokens, K],
 * [H, K]; checks every timed candidate numerically against the UNFUSED path;
 * then searches the token threshold below which UNFUSED is faster.  Stores the
 * winning plan for (K, H, norm_kind) with tuned_max_tokens = max_tokens.
 * Synchronises `stream`.  Skipped (returns FLN_OK, plan untouched) when both
 * overrides are set (fln_set_overrides).  1 <= max_tokens <= 65536.
 */
int fln_autotune(int K, int H, int norm_kind, int max_tokens, fln_stream_t stream);

/*
 * fln_set_overrides -- global overrides of the automatic choices ("TPSP
 * Design", section 3: --tpsp-microchunk-tokens / --tpsp-threshold-tokens).
 * 0 clears an override.  microchunk_tokens in 0..4096; threshold_tokens in
 * 0..257.  An override is not evidence of benefit; when both are set,
 * fln_autotune skips its scan and numerical check.
 */
int fln_set_overrides(int microchunk_tokens, int threshold_tokens);

/* Install (or, with plan = NULL, remove) the plan of a group explicitly. */
int fln_set_plan(int K, int H, int norm_kind, const fln_plan* plan);

/* The plan a call with these arguments would use after overrides (path is
 * FLN_PATH_UNFUSED when T is below the threshold).  Writes *plan. */
int fln_get_plan(int K, int H, int norm_kind, int T, int microchunk_tokens, fln_plan* plan);

/* The three calls above for groups of a given operand type (fln_dtype); the
 * calls without a dtype act on FLN_DTYPE_BF16 groups.  FP8 groups are tuned on
 * synthetic E4M3 data with per-tensor scales. */
int fln_autotune_dtype(int K, int H, int norm_kind, int dtype, int max_tokens, fln_stream_t stream);
int fln_set_plan_dtype(int K, int H, int norm_kind, int dtype, const fln_plan* plan);
int fln_get_plan_dtype(int K, int H, int norm_kind, int dtype, int T, int microchunk_tokens, fln_plan* plan);

/* Synchronise `stream` and the internal stream, read and clear the device
 * error words of the current device: the workspace's (if the device has a
 * workspace; this call never creates one) and the one in the static scratch
 * of fused_proj_add_rmsnorm_noalloc (if that entry point has run on the
 * device).  FLN_ERR_DEVICE_TIMEOUT if a kernel gave up a bounded wait;
 * FLN_ERR_INVALID_ARG if an MoE kernel met a device-resident index out of
 * range (offsets that are not a grouping of the T * k rows, a row_of entry
 * outside [0, T * k), a row_token entry outside [0, T)): the kernel then
 * wrote none of the rows that index touches. */
int fln_device_status(fln_stream_t stream);

/* Message for the last error on the calling thread ("" if none). */
const char* fln_last_error(void);

/* Free the workspace, streams and events of every device (synchronises the
 * devices first).  The next call allocates again. */
void fln_release_workspace(void);

/* Number of kernels this library has launched since load (all devices). */
uint64_t fln_launch_count(void);

/* Per-kernel timing with CUDA events recorded on each kernel's own stream. */
enum {
  FLN_KERNEL_GEMM_FUSED = 0,   /* GEMM with the fused add + norm epilogue */
  FLN_KERNEL_GEMM_SLOT = 1,    /* GEMM writing a pipeline slot */
  FLN_KERNEL_GEMM_SPLITK = 2,  /* split-K GEMM of the UNFUSED path */
  FLN_KERNEL_NORM_BF16 = 3,    /* add_rmsnorm */
  FLN_KERNEL_NORM_SLOT = 4,    /* pipeline second stage */
  FLN_KERNEL_NORM_SPLITK = 5,  /* split-K reduce + add + norm */
  FLN_KERNEL_W4_DEQUANT = 6,   /* FP4 weights to bf16 (paths with many tokens) */
  FLN_KERNEL_MOE_ROUTE = 7,    /* MoE routing + grouping */
  FLN_KERNEL_MOE_GEMM = 8,     /* MoE grouped down projection */
  FLN_KERNEL_MOE_NORM = 9,     /* MoE unpermute + add + norm */
  FLN_KERNEL_MOE_GATHER = 10,  /* MoE gather of hidden states into grouped order */
  FLN_KERNEL_KINDS = 11
};
typedef struct {
  uint64_t launches[FLN_KERNEL_KINDS];
  double total_ms[FLN_KERNEL_KINDS];
} fln_profile_stats;

/* enable != 0 starts recording (and clears earlier records); 0 stops. */
int fln_profile_enable(int enable);
/* Synchronise the recorded events and return their per-kind sums; clears them. */
int fln_profile_read(fln_profile_stats* stats);

/*
 * fused_proj_add_rmsnorm_noalloc -- the same projection + residual add + norm
 * as fused_proj_add_rmsnorm, for callers that must not allocate device memory.
 * (The pages have no counterpart; it exists for integration.)
 *
 * Who needs it: runtimes that own every byte of device memory through their
 * own pool or budget (an inference server that reserved the GPU up front, where
 * a cudaMalloc outside the pool can fail or break its accounting), and
 * latency-critical loops where cudaMalloc / cudaFree would synchronise the
 * device.  fused_proj_add_rmsnorm grows a library workspace with cudaMalloc the
 * first time a shape needs more; this entry point never does, and never
 * creates a stream or an event.
 *
 *   x, W, residual, gamma, eps, norm_kind, T, K, H, out, stream: as in
 *   fused_proj_add_rmsnorm.  It always runs one kernel: the single-CTA
 *   tcgen05 GEMM with the fused add + norm epilogue (tile 128 x 256, chunks
 *   of 4096 tokens, one CTA per SM, row statistics exchanged through the
 *   static scratch).  That is not the CTA-pair kernel of the FUSED path, so
 *   its results agree with fused_proj_add_rmsnorm within the parity
 *   tolerance (max-abs 2e-2 or one bf16 ulp, mean-abs 2e-3, both against the
 *   fp64 reference), not bit for bit.  Plans, tuning, the token threshold and
 *   the overrides do not apply.
 *   device_error: NULL, or a device pointer to one 4-byte word owned by the
 *   caller; a kernel that gives up a bounded wait ORs its error bits into it
 *   (the caller clears it and reads it after synchronising).  With NULL the
 *   bits go to a word in the static scratch instead, which fln_device_status
 *   reads and clears (that call allocates nothing either).  A bounded wait
 *   gives up only if the kernel's CTAs cannot all be resident at once (for
 *   example while other streams hold SMs); the rows it did not finish are
 *   left unwritten.
 *
 * Scratch: a static device array of 1 057 024 bytes, held by every GPU that
 * loads the library until the process exits.  It holds the row statistics of
 * at most 2048 tiles: ceil(min(T, 4096) / 128) * ceil(H / 256) <= 2048, i.e.
 * H <= 16384 once T >= 3969.  Larger problems return FLN_ERR_UNSUPPORTED with a
 * message before anything is launched, as do rows with more 256-wide N-tiles
 * than the GPU has SMs (the N-tiles of a row block must run on distinct,
 * co-resident CTAs).
 * The first call on a device looks up where the array lives on that device
 * (cudaGetSymbolAddress) and sets the kernel's shared-memory limit; make that
 * first call before any stream capture.
 * Every call on a device shares the one array and it keeps the last call's
 * contents: the publication flags start at zero when the library loads and
 * each call writes a new per-device value into them, so stale flags are never
 * taken for this call's; the partial sums are written before they are read.
 * Calls whose GPU work overlaps (for example, issued on two streams without
 * ordering) race on the array and give undefined results: order them.
 */
int fused_proj_add_rmsnorm_noalloc(const fln_bf16* x, const fln_bf16* W, fln_bf16* residual, const float* gamma,
                                   float eps, int norm_kind, int T, int K, int H, fln_bf16* out,
                                   unsigned int* device_error, fln_stream_t stream);

/*
 * The TPSP region across P tensor-parallel ranks (vLLM "TPSP Design": section
 * 1 "Motivation", section 3 "Microchunk pipeline", section 4 "Constraints").
 * Each rank holds a K-shard of the projection's input and weight; the
 * AllReduce after the row-parallel projection becomes a ReduceScatter over
 * tokens, the residual add and norm run on the rank's token shard only, and an
 * AllGather hands every rank the full normalised [T, H] tensor:
 *
 *   y_p   = x_p . W_p^T                      (this rank's partial projection, all T tokens)
 *   y     = sum_p y_p                        (ReduceScatter: rank p receives its token shard)
 *   r_p  += y[shard p];  o_p = RMSNorm(r_p)  (local, rank p's tokens only)
 *   out   = AllGather(o_p)                   ([T, H] on every rank)
 *
 * Token partition: S = ceil(T / P) rows per rank, rank p owning tokens
 * [p S, min((p + 1) S, T)) (the last shards are padded: their rows past T are
 * never read or written).  A microchunk of c tokens per rank (c <= 4096) is
 * chunk i of every shard at once: rank p's shard rows [i c, i c + n_i),
 * n_i = min(c, S - i c).  Per chunk: the GEMM writes the partial y of every
 * rank's rows into a rank-major fp32 slot [P, n_i, H] on the caller's stream;
 * on the communicator's second stream the ReduceScatter (fp32 sum), the add +
 * norm of this rank's valid rows and the AllGather (bf16) follow, and the
 * gathered rows are written to `out` in token order; three slots guarded by
 * events let the next chunks' GEMMs overlap.  The collectives are NCCL's,
 * found at run time in the process (PyTorch loads it) or at the path in the
 * environment variable FLN_NCCL_LIBRARY; without it these calls return
 * FLN_ERR_COMM.  bf16 operands only.
 */
typedef struct fln_tp_comm fln_tp_comm;  /* one rank's communicator, stream, slots and events */

/* Writes a 128-byte unique id (on one rank; the caller hands it to the others). */
int fln_tp_unique_id(void* id);

/* Collective over the nranks ranks (each calls it with the same id and its own
 * rank, with its device current).  nranks = 1 may pass id = NULL (no
 * rendezvous).  The handle belongs to the current device; free it with
 * fln_tp_comm_destroy. */
int fln_tp_comm_init(int nranks, int rank, const void* id, fln_tp_comm** comm);
int fln_tp_comm_destroy(fln_tp_comm* comm);

/* Host-only partition of T tokens over nranks ranks in microchunks of
 * microchunk_tokens per rank (0 = 1024, the default; at most 4096): shard rows
 * S, the chunk size used and the number of chunks; and, for chunk `chunk` of
 * rank `rank`, its first token, its block rows n_i (the same on every rank)
 * and how many of those rows are valid tokens (< T).  Needs no GPU. */
int fln_tp_layout(int T, int nranks, int microchunk_tokens, int* shard_rows, int* chunk_tokens, int* num_chunks);
int fln_tp_chunk_rows(int T, int nranks, int microchunk_tokens, int chunk, int rank, int* token0, int* rows,
                      int* valid);

/*
 * fused_proj_rs_add_rmsnorm_ag -- one rank's part of the TPSP region.
 *
 *   x               [T, K] bf16, this rank's K-shard of the projection input (all T tokens)
 *   W               [H, K] bf16, this rank's K-shard of the weight (F.linear layout)
 *   residual_shard  [S, H] bf16, this rank's token shard of the residual (S = ceil(T / P));
 *                   its valid rows are read and overwritten with r + y, rows past T untouched
 *   gamma, eps, norm_kind   as in fused_proj_add_rmsnorm
 *   T               tokens of the whole batch (the same on every rank)
 *   microchunk_tokens  per rank, 0 = 1024, else 1..4096
 *   out             [T, H] bf16, the gathered normalised tensor (every rank)
 *   comm            this rank's handle (current device); stream: the caller's stream
 *
 * Every rank calls it with the same T, H and microchunk_tokens; the calls are
 * collective.  Asynchronous on `stream`; the communicator's second stream is
 * joined back before return.  Sequential use per communicator.  The norm is
 * computed from the fp32 sum, as in fused_proj_add_rmsnorm.  Errors:
 * FLN_ERR_INVALID_ARG (pointers, sizes, a communicator of another device),
 * FLN_ERR_COMM (a collective failed), FLN_ERR_CUDA.
 */
int fused_proj_rs_add_rmsnorm_ag(const fln_bf16* x, const fln_bf16* W, fln_bf16* residual_shard,
                                 const float* gamma, float eps, int norm_kind, int T, int K, int H,
                                 int microchunk_tokens, fln_bf16* out, fln_tp_comm* comm, fln_stream_t stream);

/* The UNFUSED path's split reduction (bf16 and FP8 operands): calls with at
 * most max_tokens tokens sum the split-K partials, add the residual and
 * normalise in the split-K GEMM's own tail (the last CTA to deliver a part of
 * a 128-row block of W reduces that block; after a grid-wide count every CTA
 * normalises a slice of the outputs: the grid is at most one CTA per SM, and
 * its bounded waits report FLN_ERR_DEVICE_TIMEOUT if other work keeps CTAs
 * from being resident together, as for the FUSED path);
 * larger calls use a separate reduce + add + norm kernel launched as the
 * GEMM's programmatic dependent.  0 (the default) = always the separate
 * kernel, which measured faster on the 70B decode shapes at 1-256 tokens; at
 * most 256.  Both give results within the parity tolerance of each other (the
 * summation order of the row statistics differs). */
int fln_set_splitk_tail_tokens(int max_tokens);

/* Test switch for failure reporting: with enable != 0, the next launch that
 * exchanges row statistics between CTAs (the FUSED path, the no-allocation
 * entry point, or the UNFUSED path's split-K tail) waits for a value that no
 * CTA publishes.  That bounded wait gives up after about two seconds, the
 * kernel unwinds without writing the affected outputs, and fln_device_status
 * returns FLN_ERR_DEVICE_TIMEOUT (and puts the tail's counters back to zero);
 * the device stays usable.  The switch clears itself after one launch.  No
 * fault, trap or unbounded wait is involved. */
int fln_debug_stall_next_call(int enable);

/* Library version: major * 10000 + minor * 100 + patch. */
int fln_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LIBFUSEDLN_H */
