// fln_internal.h -- types shared by the kernels and the host scheduler of
// libfusedln.  Not part of the public ABI (that is include/libfusedln.h).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fln {

// What the GEMM epilogue does with the fp32 accumulator tile.
enum EpilogueKind : int {
  // r = r0 + acc; per-row sum of squares over the full hidden size, combined
  // across the N-tiles of a row block through global partial sums and
  // per-tile release flags; out = r * rsqrt(ms + eps) * g.  Writes residual
  // (in place) and out, both bf16.
  EPI_FUSED_NORM = 0,
  // y (fp32) -> a pipeline slot [rows, ld]; the add + norm runs as a second
  // stage on another stream.
  EPI_STORE_F32 = 1,
  // Swapped operands (A = W, B = x) with a stream-K split of the K loop:
  // partial y^T tiles (fp32) go to a partial buffer, reduced by the
  // add + norm kernel.
  EPI_SPLITK_SWAP = 2,
  // The same split, with the reduction, residual add and norm in the GEMM's
  // own tail: the last CTA to deliver a partial of an m-tile sums the m-tile's
  // partial slots (fixed order), adds the residual, keeps fp32 r and each
  // token's sum of squares over the m-tile's 128 columns; once every m-tile
  // is reduced (a grid-wide count, bounded wait: the grid is at most one CTA
  // per SM, so every CTA is resident while the GPU runs nothing else), each
  // CTA normalises a slice of the [T, H] outputs.
  EPI_SPLITK_FUSED = 3,
};
__host__ __device__ constexpr bool is_splitk(int epi) { return epi == EPI_SPLITK_SWAP || epi == EPI_SPLITK_FUSED; }

struct GemmParams {
  int M;             // valid rows of the A operand in this launch
  int N;             // valid columns of the result (B rows)
  int K;             // reduction length
  int a_row0;        // TMA row coordinate of A's first row (chunk start)
  int num_m_tiles;   // ceil(M / 128)
  int num_n_tiles;   // ceil(N / BN)
  int num_k_blocks;  // ceil(K / 64)
  // fused-norm epilogue
  __nv_bfloat16* residual;  // [rows, ld] bf16, global row = a_row0 + local row
  __nv_bfloat16* out;       // [rows, ld] bf16
  const float* gamma;       // [ld] fp32
  float eps;
  int norm_kind;            // 0 standard, 1 Gemma (1 + gamma)
  int ld;                   // hidden size H (row stride in elements)
  float* psum;              // row partial sums of squares, [num_m_tiles, num_n_tiles, 128]: fp32 with
                            // separate flags (CTA kernel), or 64-bit {gen, value} words (pair kernel)
  unsigned int* flags;      // [num_m_tiles, num_n_tiles] publication flags (CTA kernel)
  unsigned int gen;         // value this launch writes into flags (never 0)
  int stall_rowstat;        // test switch: wait for a generation nobody publishes (bounded wait runs out)
  // store-f32 epilogue
  float* yout;              // [M, ld] fp32 slot, local rows
  // rank-major blocks of rows (store-f32 only; 0 = none): the launch's m-tiles
  // form blocks of blk_m_tiles tiles; block b reads x rows a_row0 + b *
  // blk_stride + local and stores slot rows b * blk_rows + local, local <
  // blk_rows (the TP region's slot: every rank's rows of one microchunk)
  int blk_m_tiles = 0;
  int blk_rows = 0;
  int blk_stride = 0;
  // split-K swap epilogue.  Each m-tile's first kb_static K-blocks are split
  // statically (stream-K over the grid); the remaining K-blocks form dyn_cpm
  // chunks of dyn_kc blocks, handed out at run time through an atomic counter.
  float* partial;           // [num_m_tiles * slot_stride, N, 128] fp32
  int max_split;            // static partial slots per m-tile (dynamic chunk i uses slot max_split + i)
  int slot_stride;          // partial slots per m-tile: max_split + dyn_cpm
  long long units_total;    // num_m_tiles * kb_static
  int kb_static;            // statically split K-blocks per m-tile
  int dyn_cpm;              // dynamic chunks per m-tile (0: none)
  int dyn_kc;               // K-blocks per dynamic chunk
  unsigned int* dyn_counter;  // chunk counter: zero before and after every launch
  // split-K with the fused tail: per m-tile {gen, deliveries} words, then
  // tiles_done[0] = {gen, m-tiles reduced} and tiles_done[1] = {gen, CTAs past
  // the wait} (each word is put back to zero by its last user, so graph
  // replays start from zero), and per-token sums of squares [N, num_m_tiles]
  // (the residual, out, gamma, eps and norm fields above hold the norm's
  // arguments; ld = M = H)
  unsigned long long* tile_arrivals;
  unsigned long long* tiles_done;
  float* rowstat;
  // FP8 (E4M3) operands: the accumulator of (token t, hidden h) is scaled by
  // x_scale[t * x_scale_stride] * w_scale[h * w_scale_stride] (stride 0: one
  // scale for the tensor); t is the global token row.  Unused for bf16.  The
  // split-K epilogue stores unscaled partials (the reducer scales the sum).
  const float* x_scale;
  int x_scale_stride;
  const float* w_scale;
  int w_scale_stride;
  // FP4 weights (split-K kernel of fln_gemm_w4.cu): block scales [M rows,
  // w4_nblk bytes], one per 16 (NVFP4) or 32 (MXFP4) elements of a row
  const uint8_t* w4_scales;
  int w4_nblk;
  // every path: the accumulator is multiplied by y_scale before anything
  // else (the NVFP4 tensor scale; 1 otherwise, an exact identity)
  float y_scale = 1.0f;
  unsigned int* err;        // device error word
  // pair kernel: the last split_tiles tiles of the launch are each computed
  // as two halves of their K-blocks on two pairs; the second half's fp32
  // accumulator goes through split_buf ([split_tiles, 2 CTAs, BN / 32, 8,
  // 128, 4]) and is announced by a {gen, 1} word per (tile, CTA, lane quarter)
  int split_tiles;
  float* split_buf;
  unsigned long long* split_flags;
  // pair kernel, slot mode: a grouped (MoE) GEMM when moe_off is set.  Rows
  // [moe_off[e], moe_off[e + 1]) of A times expert e's rows [e N, (e + 1) N)
  // of B, in row blocks of 256 that never cross an expert's end; y rows go to
  // their grouped positions in yout [M, ld].  The offsets are checked on the
  // device first: unless 0 = off[0] <= ... <= off[E] = M, nothing is written,
  // *moe_bad is set to 1 (else 0) and the device error word gets the
  // bad-index bit.  E <= 256.
  const int* moe_off = nullptr;
  int moe_E = 0;
  unsigned int* moe_bad = nullptr;
};

struct NormParams {
  const __nv_bfloat16* y_bf16;  // [T, H] bf16 addend (plain add_rmsnorm)
  const float* y_f32;           // [T, H] fp32 addend (pipeline slot), rows local to the launch
  const float* partial;         // split-K partials (layout of GemmParams::partial)
  int max_split;                // static slots per m-tile
  int slot_stride;              // slots per m-tile (static + dynamic)
  int dyn_cpm;                  // dynamic chunk slots per m-tile
  int num_k_blocks;             // statically split K-blocks per m-tile (to find contributing CTAs)
  int gemm_grid;
  long long units_total;

  __nv_bfloat16* residual;      // [T, H] in/out
  __nv_bfloat16* out;           // [T, H]
  const float* gamma;
  float eps;
  int norm_kind;
  int T;                        // rows in this launch
  int row0;                     // global row of local row 0 (residual/out/y_bf16)
  int H;
  int pdl;                      // launched as a programmatic dependent of the preceding kernel
  int out_local = 0;            // out rows are local to the launch (out + t * H), not row0 + t
  float y_scale = 1.0f;         // the addend is multiplied by this (1 = identity)
  // FP8 split-K: scale the summed partials by x_scale[(row0 + t) * stride] *
  // w_scale[h * stride] (null: no scaling)
  const float* x_scale;
  int x_scale_stride;
  const float* w_scale;
  int w_scale_stride;
};

// Operand element type of a projection: bf16 (K-blocks of 64 elements) or
// FP8 E4M3 (K-blocks of 128 elements); either way a K-block row is 128 bytes.
enum OperandType : int { OPERAND_BF16 = 0, OPERAND_E4M3 = 1 };
__host__ __device__ constexpr int kblock_elems(int f8) { return f8 ? 128 : 64; }

// launchers (return cudaError_t of the launch).  f8: E4M3 operands (epilogues
// STORE_F32 and SPLITK_SWAP only).
cudaError_t launch_gemm(EpilogueKind epi, int bn, int f8, const CUtensorMap& tmA, const CUtensorMap& tmB,
                        const GemmParams& p, int grid, cudaStream_t stream);
int gemm_smem_bytes(int bn);
int gemm_stages(int bn);
cudaError_t gemm_prepare(int bn, EpilogueKind epi, int f8);  // sets max dynamic smem attributes

// CTA-pair (cta_group::2) fused GEMM + add + RMSNorm for tile widths 128,
// 192, 224, 256 with four epilogue warps per CTA, or 224, 256 with eight.  prepare sets the shared-memory limit and reports how many pairs
// can be resident at once (the grid must not exceed it: the pairs exchange
// row statistics).  tmR maps the chunk's residual rows (read in 128 x 64
// boxes), tmRs / tmOs the chunk's residual and output rows in 32 x 64 boxes
// (stores).
// ew: epilogue warps per CTA, 4 (every tile width) or 8 (two groups of four on
// alternate tiles; tile widths 224, 256); ew = 0 runs the same kernel as the
// PIPELINED path's slot GEMM (tile widths 128, 256): the fp32 accumulator,
// scaled, to p.yout [M, ld] (launch-local rows), no residual, no norm, no
// split (tmR, tmRs, tmOs are not used).
cudaError_t pair_gemm_prepare(int bn, int f8, int ew, int* max_pairs);
cudaError_t launch_gemm_pair_fused(int bn, int f8, int ew, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                   const CUtensorMap& tmR, const CUtensorMap& tmRs, const CUtensorMap& tmOs,
                                   const GemmParams& p, int pairs, cudaStream_t stream);

// MoE region (fln_moe.cu): routing + grouping (two kernels), the grouped
// down projection into fp32 rows y [T * k, H], and the unpermute + add + norm.
// device error word bit for a device-resident MoE index (offsets, row_of, row_token) out of range; the
// bounded-wait bits sit beside the wait helpers
#define FLN_DEVERR_BAD_INDEX 0x20u
// device error word bit: the second K-half of a split tile never arrived at its owner (pair kernel)
#define FLN_DEVERR_TIMEOUT_SPLIT 0x40u
cudaError_t launch_moe_route(const float* logits, int T, int E, int k, int* ids, float* gates, int* offsets,
                             int* row_token, int* row_slot, int* row_of, cudaStream_t stream);
cudaError_t launch_moe_gather(const __nv_bfloat16* x, const int* row_token, int T, int k, int H, __nv_bfloat16* xg,
                              unsigned int* err, int sms, cudaStream_t stream);
cudaError_t moe_gemm_prepare();
cudaError_t launch_moe_grouped_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const int* offsets, int E, int R,
                                    int H, int K, float* y, unsigned int* err, unsigned int* bad_offsets, int grid,
                                    cudaStream_t stream);
cudaError_t launch_moe_combine_norm(const float* y, const int* row_of, const float* gates, __nv_bfloat16* residual,
                                    const float* gamma, float eps, int norm_kind, int T, int H, int k,
                                    __nv_bfloat16* out, unsigned int* err, const unsigned int* bad_offsets,
                                    cudaStream_t stream);

// FP4 weights (fmt 0 NVFP4: E4M3 scale per 16 elements; fmt 1 MXFP4: E8M0
// scale per 32): the split-K GEMM that dequantises W on the SM into tensor
// memory (fln_gemm_w4.cu; tokens on N: bn 16..256), and the conversion of a
// whole weight to bf16 (w = e2m1 * block scale, exact) for the paths with
// many tokens.  prepare sets the shared-memory limit.
cudaError_t w4_gemm_prepare(int bn, int fmt);
cudaError_t launch_w4_gemm_splitk(int bn, int fmt, const CUtensorMap& tmW, const CUtensorMap& tmX,
                                  const GemmParams& p, int grid, cudaStream_t stream);
cudaError_t launch_fp4_to_bf16(int fmt, const uint8_t* Wq, const uint8_t* S, __nv_bfloat16* out, int H, int K,
                               cudaStream_t stream);

enum NormSource : int { NORM_SRC_BF16 = 0, NORM_SRC_F32 = 1, NORM_SRC_SPLITK = 2 };
cudaError_t launch_add_rmsnorm(NormSource src, const NormParams& p, int grid_cap, cudaStream_t stream);

// Host helpers of the C ABI (fln_api.cu) that the TP region (fln_tp.cu) uses:
// the thread's last-error message, argument checks, tensor maps (bf16, 128-byte
// boxes with 128-byte swizzle), the launch counter and the library's lock.
int api_fail(int code, const char* fmt, ...);
int api_cuda_fail(cudaError_t e, const char* what);
int api_check_ptr(const char* name, const void* p);
int api_check_common(float eps, int kind, int T, int H);
bool api_overlaps(const void* a, size_t na, const void* b, size_t nb);
int api_make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);
void api_count_launch();
int api_device_error_word(unsigned int** word);  // the current device's workspace error word (created if needed)
void api_lock();
void api_unlock();

// split-K bookkeeping shared by the GEMM and the reducer: the CTA whose
// unit range [c*U/G, (c+1)*U/G) contains unit u.  32-bit arithmetic: the host
// only launches the split-K path when (U + 1) * G + U < 2^32.
__host__ __device__ inline int splitk_cta_of_unit(long long u, long long U, int G) {
  const uint32_t uu = static_cast<uint32_t>(u), UU = static_cast<uint32_t>(U), GG = static_cast<uint32_t>(G);
  return static_cast<int>(((uu + 1u) * GG + UU - 1u) / UU - 1u);
}

}  // namespace fln
