// fln_moe.cu -- the MoE region of the "TPSP Design" page (section 3 "Fusion
// regions": routing and expert reordering before the grouped GEMM, then
// unpermute and the add / next norm; section 5 "To-do": MoE), on one GPU:
//
//   routing    logits [T, E] -> the k experts of largest logit per token
//              (equal logits: smaller expert first) and softmax gates over
//              the chosen logits;
//   permute    the (token, slot) pairs grouped by expert, tokens ascending
//              within an expert: offsets [E + 1], row_token / row_slot per
//              grouped row, row_of per pair (the unpermute index);
//   grouped GEMM   y[r, :] = hg[r, :] . We[e(r)]^T for every grouped row
//              (tcgen05, bf16 operands, fp32 accumulate in TMEM);
//   combine + add + norm   r[t] += sum_j gate[t, j] * y[row_of[t, j]] (slot
//              order, fp32), out[t] = RMSNorm(r[t]).
#include <algorithm>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fln_internal.h"
#include "fln_ptx.cuh"

namespace fln {

namespace moe {

constexpr int MAX_E = 256;
constexpr int MAX_K = 8;

// ------------------------------------------------------------------ routing
// One warp per token.  Lane l holds the logits of experts l, l + 32, ...; for
// each of the k picks every lane proposes its best unchosen expert (larger
// logit, then smaller index) and a butterfly reduction agrees on the winner.
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int t, int E, int k,
                                            int* __restrict__ ids, float* __restrict__ gates) {
  const int lane = threadIdx.x & 31;
  const float* lt = logits + static_cast<size_t>(t) * E;
  float v[MAX_E / 32];
  unsigned taken = 0;
#pragma unroll
  for (int i = 0; i < MAX_E / 32; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? lt[e] : 0.f;
  }
  float sel[MAX_K];
#pragma unroll
  for (int j = 0; j < MAX_K; ++j) {
    if (j >= k) break;
    bool have = false;
    float bv = 0.f;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < MAX_E / 32; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (!have || v[i] > bv)) {
        have = true;
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const bool oh = __shfl_xor_sync(0xFFFFFFFFu, have, off);
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, off);
      if (oh && (!have || ov > bv || (ov == bv && oe < be))) {
        have = true;
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    sel[j] = bv;
    if (lane == 0) ids[static_cast<size_t>(t) * k + j] = be;
  }
  float denom = 0.f;
#pragma unroll
  for (int j = 0; j < MAX_K; ++j)
    if (j < k) denom += __expf(sel[j] - sel[0]);
#pragma unroll
  for (int j = 0; j < MAX_K; ++j)
    if (j < k && lane == j) gates[static_cast<size_t>(t) * k + j] = __expf(sel[j] - sel[0]) / denom;
}

__global__ void route_kernel(const float* __restrict__ logits, int T, int E, int k, int* __restrict__ ids,
                             float* __restrict__ gates) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t < T) route_token(logits, t, E, k, ids, gates);
}

// ------------------------------------------------------------------ permute
// One CTA of 1024 threads.  Pass 1 counts the pairs of each expert; the scan
// gives offsets; pass 2 walks the pairs in (token, slot) order in chunks of
// 1024: a pair's row is its expert's running cursor plus the number of
// earlier pairs of the same expert in the chunk (lanes of the same expert in
// its warp by __match_any_sync, earlier warps by their per-expert counts).
__device__ __forceinline__ void permute_block(const int* __restrict__ ids, int T, int E, int k,
                                              int* __restrict__ offsets, int* __restrict__ row_token,
                                              int* __restrict__ row_slot, int* __restrict__ row_of) {
  __shared__ int cnt[MAX_E];
  __shared__ int cursor[MAX_E];
  __shared__ int wcnt[32][MAX_E];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = T * k;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += blockDim.x) atomicAdd(&cnt[ids[p]], 1);
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      offsets[e] = run;
      cursor[e] = run;
      run += cnt[e];
    }
    offsets[E] = run;
  }
  __syncthreads();
  for (int base = 0; base < P; base += blockDim.x) {
    for (int i = tid; i < 32 * E; i += blockDim.x) wcnt[i / E][i % E] = 0;
    __syncthreads();
    const int p = base + tid;
    const bool valid = p < P;
    const int e = valid ? ids[p] : -1;
    const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
    const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
    if (valid && rank_in_warp == 0) wcnt[warp][e] = __popc(same);
    __syncthreads();
    if (valid) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += wcnt[w][e];
      const int row = cursor[e] + before + rank_in_warp;
      row_token[row] = p / k;
      row_slot[row] = p % k;
      row_of[p] = row;
    }
    __syncthreads();
    for (int x = tid; x < E; x += blockDim.x) {
      int add = 0;
      for (int w = 0; w < 32; ++w) add += wcnt[w][x];
      cursor[x] += add;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(1024, 1)
    permute_kernel(const int* __restrict__ ids, int T, int E, int k, int* __restrict__ offsets,
                   int* __restrict__ row_token, int* __restrict__ row_slot, int* __restrict__ row_of) {
  permute_block(ids, T, E, k, offsets, row_token, row_slot, row_of);
}

// T <= 32: both steps in one CTA (warp w routes token w), one launch instead of two
__global__ void __launch_bounds__(1024, 1)
    route_permute_kernel(const float* __restrict__ logits, int T, int E, int k, int* __restrict__ ids,
                         float* __restrict__ gates, int* __restrict__ offsets, int* __restrict__ row_token,
                         int* __restrict__ row_slot, int* __restrict__ row_of) {
  const int w = threadIdx.x >> 5;
  if (w < T) route_token(logits, w, E, k, ids, gates);
  __syncthreads();  // the block's global writes of ids are visible to the block after the barrier
  permute_block(ids, T, E, k, offsets, row_token, row_slot, row_of);
}

// ------------------------------------------------------------------ gather (permute)
// Grouped row r of xg is token row_token[r] of x: one 16-byte word (eight
// bf16) a thread, grid-stride over R * H / 8 words (H % 8 == 0).  A token
// index outside [0, T) leaves its row unwritten and raises the bad-index bit.
__global__ void gather_kernel(const uint4* __restrict__ x, const int* __restrict__ row_token, int T, int R, int W8,
                              uint4* __restrict__ xg, unsigned int* err) {
  const size_t n = static_cast<size_t>(R) * W8;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t r = i / W8;
    const int c = static_cast<int>(i - r * W8);
    const int t = row_token[r];
    if (static_cast<unsigned>(t) >= static_cast<unsigned>(T)) {
      if (c == 0) atomicOr(err, FLN_DEVERR_BAD_INDEX);
      continue;
    }
    xg[i] = x[static_cast<size_t>(t) * W8 + c];
  }
}

// ------------------------------------------------------------------ grouped GEMM
// Persistent, one CTA per SM.  Items are (expert, 256-column tile of H,
// 128-row tile of its rows), expert-major, row tiles fastest; CTA c takes
// items c, c + G, ...  A =
// 128 grouped rows of hg (rows past the expert's last belong to other experts
// or lie past the end and are never stored), B = 256 rows of We[e] viewed as
// [E * H, K] (rows past H are never stored).  Warps: 0 TMA producer, 1 TMEM
// owner + MMA issuer, 2-5 epilogue (fp32 rows of y).
constexpr int BM = 128, BN = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * 128, B_BYTES = BN * 128;
constexpr int THREADS = 192;
constexpr int SMEM = STAGES * (A_BYTES + B_BYTES) + 1024 + 1024;
constexpr int TMEM_COLS = 2 * BN;

struct Sched {
  const int* off;   // [E + 1] shared copy of the offsets
  const int* tb;    // [E + 1] items before expert e
  int E, NT;
  __device__ int total() const { return tb[E]; }
  // item -> (expert, first grouped row, rows of the tile, n tile)
  __device__ void decode(int item, int& e, int& row0, int& rows, int& n) const {
    int lo = 0, hi = E - 1;  // the last e with tb[e] <= item (experts without rows own no items)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tb[mid] <= item) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    const int local = item - tb[e];
    const int mt = (off[e + 1] - off[e] + BM - 1) / BM;  // row tiles of the expert, fastest: the CTAs of a
    n = local / mt;                                        // wave share the W tiles they stream
    const int m = local - n * mt;
    row0 = off[e] + m * BM;
    rows = min(BM, off[e + 1] - row0);
  }
};

__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const int* __restrict__ offsets, int E, int R, int H, int K, float* __restrict__ y,
                        unsigned int* err, unsigned int* bad_offsets) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain_bar = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  __shared__ int s_off[MAX_E + 1];
  __shared__ int s_tb[MAX_E + 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = (H + BN - 1) / BN;
  const int KB = (K + 63) / 64;
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = offsets[e];
  __syncthreads();
  // the offsets must describe a grouping of the R rows: 0 = off[0] <= off[1] <= ... <= off[E] = R; else no row
  // is written (every CTA leaves before it allocates TMEM or arms a barrier) and the verdict tells the combine
  // kernel that follows on the stream to write nothing either
  bool ok = threadIdx.x != 0 || (s_off[0] == 0 && s_off[E] == R);
  for (int e = threadIdx.x; e < E; e += blockDim.x) ok = ok && s_off[e] <= s_off[e + 1];
  ok = __syncthreads_and(ok);
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    *bad_offsets = ok ? 0u : 1u;
    if (!ok) atomicOr(err, FLN_DEVERR_BAD_INDEX);
  }
  if (!ok) return;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      s_tb[e] = run;
      run += (s_off[e + 1] - s_off[e] + BM - 1) / BM * NT;
    }
    s_tb[E] = run;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const Sched sch{s_off, s_tb, E, NT};
  const int total = sch.total();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_a = l2_policy_evict_last();
    // W tiles are read again by the expert's other row tiles when it has more than one
    const uint64_t pol_b_once = l2_policy_evict_first(), pol_b_again = l2_policy_evict_normal();
    int s = 0;
    uint32_t ph = 0, mask = 0, par = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      int e, row0, rows, n;
      sch.decode(item, e, row0, rows, n);
      const uint64_t pol_b = s_off[e + 1] - s_off[e] > BM ? pol_b_again : pol_b_once;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, err, FLN_DEVERR_TIMEOUT_EMPTY)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
        tma_load_2d(sA + s * A_BYTES, &tmA, &full[s], kb * 64, row0, pol_a);
        tma_load_2d(sB + s * B_BYTES, &tmB, &full[s], kb * 64, e * H + n * BN, pol_b);
        mask |= 1u << s;
        par = (par & ~(1u << s)) | (ph << s);
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {
      volatile int no_abort = 0;
      for (int i = 0; i < STAGES; ++i)
        if (mask & (1u << i)) mbar_wait(&full[i], (par >> i) & 1u, &no_abort, err, FLN_DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int s = 0, local = 0;
    uint32_t ph = 0;
    bool ok = true, issued_any = false;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x, ++local) {
      const int b = local & 1;
      if (!mbar_wait(&acc_empty[b], ((local >> 1) & 1) ^ 1u, abort_flag, err, FLN_DEVERR_TIMEOUT_ACC)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&full[s], ph, abort_flag, err, FLN_DEVERR_TIMEOUT_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sw128_kmajor_desc(smem_u32(sA + s * A_BYTES));
        const uint64_t bd = sw128_kmajor_desc(smem_u32(sB + s * B_BYTES));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(d_tmem, ad + static_cast<uint64_t>(kk * 2), bd + static_cast<uint64_t>(kk * 2), IDESC,
                   (kb > 0 || kk > 0) ? 1u : 0u);
        issued_any = true;
        mma_commit(&empty[s]);
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit(&acc_full[b]);
    }
    if (!ok && issued_any) {
      mma_commit(drain_bar);
      volatile int no_abort = 0;
      mbar_wait(drain_bar, 0, &no_abort, err, FLN_DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue: fp32 rows of y
    const int q = warp & 3;
    const int rl = q * 32 + lane;
    int local = 0;
    for (int item = blockIdx.x;; item += gridDim.x, ++local) {
      const bool have = item < total;
      const int b = local & 1;
      bool stop = !have;
      if (!stop && !mbar_wait(&acc_full[b], (local >> 1) & 1, abort_flag, err, FLN_DEVERR_TIMEOUT_ACC)) stop = true;
      if (named_bar_any(1, 128, stop)) break;
      tc_fence_after();
      int e, row0, rows, n;
      sch.decode(item, e, row0, rows, n);
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * BN);
      const int c_end = min(BN, H - n * BN);
      float* yrow = y + static_cast<size_t>(row0 + rl) * H + static_cast<size_t>(n) * BN;
#pragma unroll 1
      for (int c = 0; c < c_end; c += 32) {
        float v[32];
        tmem_ld32(tb + static_cast<uint32_t>(c), v);
        if (rl < rows) {
          if (c + 32 <= c_end) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(yrow + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          } else {
            for (int j = 0; j < c_end - c; ++j) yrow[c + j] = v[j];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------ combine + add + norm
// One CTA of 256 threads per token; each thread owns 8-column groups of H
// (H % 8 == 0).  z = sum_j gate_j * y[row_j] in slot order (fp32), r = r0 + z
// (fp32), sum r^2 over H, out = r * rsqrt(ms + eps) * g; residual and out
// written as bf16.
constexpr int CN_THREADS = 256;

// GROUPS 8-column groups a thread: H <= 256 * 8 * GROUPS (2: 4096, 4: 8192, 8: 16384); fewer groups keep
// fewer values in registers, so more CTAs share an SM
template <int GROUPS>
__global__ void __launch_bounds__(CN_THREADS)
    combine_norm_kernel(const float* __restrict__ y, const int* __restrict__ row_of, const float* __restrict__ gates,
                        __nv_bfloat16* __restrict__ residual, const float* __restrict__ gamma, float eps,
                        int norm_kind, int H, int k, __nv_bfloat16* __restrict__ out, unsigned int* err,
                        const unsigned int* __restrict__ bad_offsets) {
  if (*bad_offsets) return;  // the grouped GEMM refused the offsets and left y unwritten
  const int t = blockIdx.x;
  const int G = H / 8;
  const unsigned R = static_cast<unsigned>(gridDim.x) * k;
  __shared__ float red[CN_THREADS / 32];
  __shared__ float total;
  int rows[MAX_K];
  float gw[MAX_K];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < MAX_K; ++j) {
    rows[j] = j < k ? row_of[static_cast<size_t>(t) * k + j] : 0;
    gw[j] = j < k ? gates[static_cast<size_t>(t) * k + j] : 0.f;
    bad = bad || static_cast<unsigned>(rows[j]) >= R;
  }
  // the token's rows are the same for every thread of the block, so the whole block leaves together
  if (bad) {
    if (threadIdx.x == 0) atomicOr(err, FLN_DEVERR_BAD_INDEX);
    return;
  }
  float r[GROUPS][8];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < GROUPS; ++i) {
    const int g = threadIdx.x + i * CN_THREADS;
    if (g < G) {
      float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < MAX_K; ++j) {
        if (j < k) {
          const float4* yp = reinterpret_cast<const float4*>(y + static_cast<size_t>(rows[j]) * H + 8 * g);
          const float4 a = yp[0], c = yp[1];
          z[0] += gw[j] * a.x, z[1] += gw[j] * a.y, z[2] += gw[j] * a.z, z[3] += gw[j] * a.w;
          z[4] += gw[j] * c.x, z[5] += gw[j] * c.y, z[6] += gw[j] * c.z, z[7] += gw[j] * c.w;
        }
      }
      float r0[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(residual + static_cast<size_t>(t) * H + 8 * g), r0);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        r[i][c] = r0[c] + z[c];
        ss += r[i][c] * r[i][c];
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < CN_THREADS / 32; ++w) s += red[w];
    total = s;
  }
  __syncthreads();
  const float inv = rsqrtf(total / static_cast<float>(H) + eps);
#pragma unroll
  for (int i = 0; i < GROUPS; ++i) {
    const int g = threadIdx.x + i * CN_THREADS;
    if (g < G) {
      float o[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float gm = gamma[8 * g + c];
        o[c] = r[i][c] * inv * (norm_kind ? 1.0f + gm : gm);
      }
      *reinterpret_cast<uint4*>(residual + static_cast<size_t>(t) * H + 8 * g) = f32x8_to_bf16(r[i]);
      *reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H + 8 * g) = f32x8_to_bf16(o);
    }
  }
}

}  // namespace moe

cudaError_t launch_moe_route(const float* logits, int T, int E, int k, int* ids, float* gates, int* offsets,
                             int* row_token, int* row_slot, int* row_of, cudaStream_t stream) {
  if (T > 0 && T <= 32) {
    moe::route_permute_kernel<<<1, 1024, 0, stream>>>(logits, T, E, k, ids, gates, offsets, row_token, row_slot,
                                                       row_of);
    return cudaGetLastError();
  }
  if (T > 0) {
    moe::route_kernel<<<(T + 7) / 8, 256, 0, stream>>>(logits, T, E, k, ids, gates);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  moe::permute_kernel<<<1, 1024, 0, stream>>>(ids, T, E, k, offsets, row_token, row_slot, row_of);
  return cudaGetLastError();
}

cudaError_t launch_moe_gather(const __nv_bfloat16* x, const int* row_token, int T, int k, int H, __nv_bfloat16* xg,
                              unsigned int* err, int sms, cudaStream_t stream) {
  const int R = T * k;
  const size_t words = static_cast<size_t>(R) * (H / 8);
  const int grid = static_cast<int>(std::min<size_t>((words + 255) / 256, static_cast<size_t>(sms) * 8));
  if (grid > 0)
    moe::gather_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint4*>(x), row_token, T, R, H / 8,
                                                  reinterpret_cast<uint4*>(xg), err);
  return cudaGetLastError();
}

cudaError_t moe_gemm_prepare() {
  return cudaFuncSetAttribute(moe::grouped_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, moe::SMEM);
}

cudaError_t launch_moe_grouped_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const int* offsets, int E, int R,
                                    int H, int K, float* y, unsigned int* err, unsigned int* bad_offsets, int grid,
                                    cudaStream_t stream) {
  moe::grouped_gemm_kernel<<<grid, moe::THREADS, moe::SMEM, stream>>>(tmA, tmB, offsets, E, R, H, K, y, err,
                                                                       bad_offsets);
  return cudaGetLastError();
}

cudaError_t launch_moe_combine_norm(const float* y, const int* row_of, const float* gates, __nv_bfloat16* residual,
                                    const float* gamma, float eps, int norm_kind, int T, int H, int k,
                                    __nv_bfloat16* out, unsigned int* err, const unsigned int* bad_offsets,
                                    cudaStream_t stream) {
  const int groups = (H / 8 + moe::CN_THREADS - 1) / moe::CN_THREADS;
  if (groups <= 2)
    moe::combine_norm_kernel<2><<<T, moe::CN_THREADS, 0, stream>>>(y, row_of, gates, residual, gamma, eps, norm_kind,
                                                                   H, k, out, err, bad_offsets);
  else if (groups <= 4)
    moe::combine_norm_kernel<4><<<T, moe::CN_THREADS, 0, stream>>>(y, row_of, gates, residual, gamma, eps, norm_kind,
                                                                   H, k, out, err, bad_offsets);
  else
    moe::combine_norm_kernel<8><<<T, moe::CN_THREADS, 0, stream>>>(y, row_of, gates, residual, gamma, eps, norm_kind,
                                                                   H, k, out, err, bad_offsets);
  return cudaGetLastError();
}

}  // namespace fln
