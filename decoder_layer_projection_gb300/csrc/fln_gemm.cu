// fln_gemm.cu -- the projection GEMM y = x . W^T on sm_103a tensor cores
// (tcgen05 + TMEM + TMA), persistent and warp-specialised, with three
// epilogues: the fused residual add + RMSNorm, an fp32 slot store for the
// two-stream microchunk pipeline, and a stream-K split for the decode regime.
//
// What it computes follows the row-parallel projection of the vLLM "TPSP
// Design" page (section 1: local projection, then residual add and norm over
// the complete hidden size of each token; section 3 "Fusion regions":
// o_proj / down_proj followed by residual add + norm) with F.linear's layout
// (torch-spyre "Plugin Architecture", "Transposed linear weights": W is
// [out, in] = [H, K], used K-major with no transpose).
//
// CTA layout (192 threads, one CTA per SM):
//   warp 0      TMA producer (one lane): A and B tiles -> smem ring
//   warp 1      TMEM owner; one lane issues tcgen05.mma into a double-buffered
//               fp32 accumulator (2 x BN columns)
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, one TMEM lane (= one
//               result row) per thread
//
// Tiles: BM = 128 rows (MMA M), BN columns (MMA N), one 128-byte swizzle
// atom of K per row and stage (64 bf16 or, with FP8 E4M3 operands and
// kind::f8f6f4 MMAs, 128 elements).  Operands are K-major in shared memory
// with 128-byte swizzle, exactly as TMA writes them.  With FP8 operands the
// STORE_F32 epilogue applies the dequantisation scales; split-K partials stay
// unscaled (the reducer scales their sum).
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fln_internal.h"
#include "fln_ptx.cuh"

namespace fln {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int NUM_THREADS = 192;
constexpr int A_TILE_BYTES = BM * BK * 2;  // 16 KiB

__host__ __device__ constexpr int stage_bytes(int bn) { return A_TILE_BYTES + bn * BK * 2; }
// As many ring stages as fit in the 227 KiB a CTA may use (at most 16): the
// decode shapes stream W from HBM and need many bytes in flight per SM.
__host__ __device__ constexpr int stages_for(int bn) {
  return (232448 - 2560) / stage_bytes(bn) > 16 ? 16 : (232448 - 2560) / stage_bytes(bn);
}
__host__ __device__ constexpr int tmem_cols_for(int bn) {
  return (2 * bn) <= 32 ? 32 : (2 * bn) <= 64 ? 64 : (2 * bn) <= 128 ? 128 : (2 * bn) <= 256 ? 256 : 512;
}
// per-token 1 / rms of the fused split-K tail (up to 256 tokens)
constexpr int TAIL_SMEM = 1024;
__host__ __device__ constexpr int smem_bytes_for(int bn) {
  // ring + barriers/flags/work queue (512 B) + tail scratch + alignment slack for the 1024-byte swizzle base
  return stages_for(bn) * stage_bytes(bn) + 512 + TAIL_SMEM + 1024;
}

// One unit of work: an output tile and the K-block range it accumulates.
struct WorkItem {
  int m_tile, n_tile, kb_begin, kb_end, split;
};

// Static persistent schedule shared verbatim by the three roles, so that they
// agree on the sequence without communicating.  (The split-K mode appends
// dynamic chunks after it; those the producer hands to the others.)
// Dynamic chunk j of the split-K mode: m-tile j / dyn_cpm, K-blocks
// [kb_static + i * dyn_kc, ...) with i = j % dyn_cpm, partial slot max_split + i.
__device__ __forceinline__ WorkItem dyn_item(const GemmParams& p, int j) {
  WorkItem w;
  const int i = j % p.dyn_cpm;
  w.m_tile = j / p.dyn_cpm;
  w.n_tile = 0;
  w.kb_begin = p.kb_static + i * p.dyn_kc;
  w.kb_end = min(p.num_k_blocks, w.kb_begin + p.dyn_kc);
  w.split = p.max_split + i;
  return w;
}

// x row (TMA coordinate) of an m-tile's first row, and the slot row of its
// row rl: plain (a_row0 + tile * 128, tile * 128 + rl) or, with rank-major
// blocks, block b = tile / blk_m_tiles at x rows a_row0 + b * blk_stride and
// slot rows b * blk_rows (rows of a block past blk_rows are not stored)
__device__ __forceinline__ int a_row_of(const GemmParams& p, int m_tile) {
  if (p.blk_m_tiles > 0) {
    const int b = m_tile / p.blk_m_tiles;
    return p.a_row0 + b * p.blk_stride + (m_tile - b * p.blk_m_tiles) * BM;
  }
  return p.a_row0 + m_tile * BM;
}

template <int EPI>
struct Scheduler {
  const GemmParams& p;
  int next_tile;       // prefill: next tile index
  long long u, u_end;  // decode: stream-K unit cursor

  __device__ explicit Scheduler(const GemmParams& prm) : p(prm) {
    if (is_splitk(EPI)) {
      const long long U = p.units_total;
      u = U * blockIdx.x / gridDim.x;
      u_end = U * (blockIdx.x + 1) / gridDim.x;
      next_tile = 0;
    } else {
      next_tile = blockIdx.x;
      u = u_end = 0;
    }
  }

  __device__ bool next(WorkItem& w) {
    if (is_splitk(EPI)) {
      // static part: units (m-tile, K-block < kb_static) in m-major order
      if (u >= u_end) return false;
      const int KB = p.kb_static;
      w.m_tile = static_cast<int>(u / KB);
      w.n_tile = 0;
      w.kb_begin = static_cast<int>(u % KB);
      const long long left = u_end - u;
      w.kb_end = (KB - w.kb_begin) < left ? KB : w.kb_begin + static_cast<int>(left);
      const int c_first = splitk_cta_of_unit(static_cast<long long>(w.m_tile) * KB, p.units_total, gridDim.x);
      w.split = static_cast<int>(blockIdx.x) - c_first;
      u += w.kb_end - w.kb_begin;
      return true;
    } else {
      const int total = p.num_m_tiles * p.num_n_tiles;
      if (next_tile >= total) return false;
      w.m_tile = next_tile / p.num_n_tiles;  // row-block major: a row block's N-tiles run together
      w.n_tile = next_tile % p.num_n_tiles;
      w.kb_begin = 0;
      w.kb_end = p.num_k_blocks;
      w.split = 0;
      next_tile += gridDim.x;
      return true;
    }
  }
};

// The sequence of work items one role processes: the static schedule, then
// (split-K with dynamic chunks) the chunks the producer draws from a global
// counter and passes on through a 4-entry queue in shared memory.  Each CTA
// draws until it gets an id past the end, so one launch makes exactly
// (chunks + CTAs) draws; whoever makes the last one puts the counter back to
// zero, so every launch (a graph replay too) starts from zero.
template <int EPI>
struct WorkSource {
  Scheduler<EPI> sched;
  bool dyn = false;   // static part done
  bool done = false;  // this CTA has taken its id past the end
  int q = 0;
  __device__ explicit WorkSource(const GemmParams& prm) : sched(prm) {}

  __device__ bool has_dynamic() const { return is_splitk(EPI) && sched.p.dyn_cpm > 0; }

  // one draw; returns the chunk id or -1 past the end
  __device__ int draw() {
    const GemmParams& p = sched.p;
    const unsigned int nc = static_cast<unsigned int>(p.num_m_tiles * p.dyn_cpm);
    const unsigned int j = atomicAdd(p.dyn_counter, 1u);
    if (j < nc) return static_cast<int>(j);
    if (j == nc + gridDim.x - 1) atomicExch(p.dyn_counter, 0u);  // the launch's last draw
    done = true;
    return -1;
  }

  // producer: take the next chunk id and publish it; ok = false on a timeout
  __device__ bool next_producer(WorkItem& w, bool& ok, uint64_t* wq_full, uint64_t* wq_empty, volatile int* wq,
                                volatile int* abort_flag) {
    if (!dyn) {
      if (sched.next(w)) return true;
      if (!has_dynamic()) return false;
      dyn = true;
    }
    const GemmParams& p = sched.p;
    const int slot = q & 3;
    if (q >= 4 && !mbar_wait(&wq_empty[slot], static_cast<uint32_t>((q >> 2) - 1) & 1u, abort_flag, p.err,
                             FLN_DEVERR_TIMEOUT_EMPTY)) {
      ok = false;
      return false;
    }
    const int jj = draw();
    wq[slot] = jj;
    mbar_arrive(&wq_full[slot]);
    ++q;
    if (jj < 0) return false;
    w = dyn_item(p, jj);
    return true;
  }

  // unwinding after a timeout: keep drawing until past the end, so that the
  // launch still makes exactly (chunks + CTAs) draws and the counter returns
  // to zero
  __device__ void drain_ids() {
    if (!has_dynamic()) return;
    while (!done) draw();
  }

  // MMA issuer (one thread, whole_warp = false) / epilogue warps (all 32
  // lanes, lane 0 arrives): the next item; ok = false on a timeout
  __device__ bool next_consumer(WorkItem& w, bool& ok, uint64_t* wq_full, uint64_t* wq_empty, volatile int* wq,
                                volatile int* abort_flag, bool whole_warp) {
    if (!dyn) {
      if (sched.next(w)) return true;
      if (!has_dynamic()) return false;
      dyn = true;
    }
    const GemmParams& p = sched.p;
    const int slot = q & 3;
    if (!mbar_wait(&wq_full[slot], static_cast<uint32_t>(q >> 2) & 1u, abort_flag, p.err,
                   FLN_DEVERR_TIMEOUT_FULL)) {
      ok = false;
      return false;
    }
    const int jj = wq[slot];
    if (whole_warp) {
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&wq_empty[slot]);
    } else {
      mbar_arrive(&wq_empty[slot]);
    }
    ++q;
    if (jj < 0) return false;
    w = dyn_item(p, jj);
    return true;
  }
};


__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ fused split-K tail
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// {gen, count} word: add one delivery for launch generation gen; returns the
// count after it (a word left by another launch counts from zero).  Only the
// claim of a word that holds another generation is a compare-and-swap; once
// the word carries gen, every add is one hardware atomic (a swap loop with
// every CTA of the grid adding at once would retry once per CTA, each retry a
// round trip to L2).
__device__ __forceinline__ unsigned int tagged_add_one(unsigned long long* w, unsigned int gen) {
  unsigned long long cur = ld_relaxed_gpu_u64(w);
  while (static_cast<unsigned int>(cur >> 32) != gen) {
    const unsigned long long prev = atomicCAS(w, cur, (static_cast<unsigned long long>(gen) << 32) | 1ull);
    if (prev == cur) return 1u;
    cur = prev;  // someone else changed it: claimed it for gen (then add below) or added to it
  }
  return static_cast<unsigned int>(atomicAdd(w, 1ull)) + 1u;
}

// partial slots that deliver to m-tile m: the static split's CTAs, then the dynamic chunks
__device__ __forceinline__ int splitk_static_slots(const GemmParams& p, int m) {
  const long long KB = p.kb_static;
  const int a = splitk_cta_of_unit(static_cast<long long>(m) * KB, p.units_total, gridDim.x);
  const int b = splitk_cta_of_unit(static_cast<long long>(m + 1) * KB - 1, p.units_total, gridDim.x);
  return b - a + 1;
}

// The last delivery of m-tile m (128 epilogue threads): y = sum of its slots in
// slot order, scaled; r = r0 + y; bf16 r to the residual, fp32 r into slot 0
// (read back by the normalisation), the m-tile's sum of squares per token to
// rowstat[t, m].  Warp wid takes tokens wid, wid + 4, ...; a lane covers four
// consecutive hidden indices.
template <int F8>
__device__ void splitk_reduce_mtile(const GemmParams& p, int m, int ep_tid) {
  const int lane = ep_tid & 31, wid = ep_tid >> 5;
  const int n = splitk_static_slots(p, m);
  const int total = n + p.dyn_cpm;
  const int h0 = m * BM + lane * 4;
  const bool hv = h0 < p.M;  // M = H, a multiple of 8: the four columns are all valid or all not
  float sw[4] = {1.f, 1.f, 1.f, 1.f};
  if (F8 && hv) {
#pragma unroll
    for (int j = 0; j < 4; ++j) sw[j] = __ldg(p.w_scale + static_cast<size_t>(h0 + j) * p.w_scale_stride);
  }
  const size_t tile_base = static_cast<size_t>(m) * p.slot_stride * p.N * BM;
  const size_t slot_step = static_cast<size_t>(p.N) * BM;
  // four tokens per warp at a time (wid, wid + 4, wid + 8, wid + 12 of each group of 16), their
  // residual and slot loads all in flight together: one L2 round trip per four tokens
  constexpr int U = 4;
  for (int t0 = 0; t0 < p.N; t0 += 4 * U) {
    int tt[U];
    bool tv[U];
    uint2 u[U];
    float4 acc[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      tt[k] = t0 + wid + 4 * k;
      tv[k] = tt[k] < p.N;
      acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      u[k] = make_uint2(0u, 0u);
      if (tv[k] && hv) u[k] = *reinterpret_cast<const uint2*>(p.residual + static_cast<size_t>(tt[k]) * p.ld + h0);
    }
#pragma unroll 2
    for (int s = 0; s < total; ++s) {
      const int slot = s < n ? s : p.max_split + (s - n);
      const float* src = p.partial + tile_base + slot * slot_step + lane * 4;
#pragma unroll
      for (int k = 0; k < U; ++k) {
        if (tv[k]) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(tt[k]) * BM));
          acc[k].x += v.x;
          acc[k].y += v.y;
          acc[k].z += v.z;
          acc[k].w += v.w;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      if (!tv[k]) continue;  // warp-uniform
      const int t = tt[k];
      float ss = 0.f;
      if (hv) {
        float sx = p.y_scale;
        if (F8) sx *= __ldg(p.x_scale + static_cast<size_t>(t) * p.x_scale_stride);
        float r[4];
        r[0] = __uint_as_float(u[k].x << 16) + acc[k].x * (sx * sw[0]);
        r[1] = __uint_as_float(u[k].x & 0xFFFF0000u) + acc[k].y * (sx * sw[1]);
        r[2] = __uint_as_float(u[k].y << 16) + acc[k].z * (sx * sw[2]);
        r[3] = __uint_as_float(u[k].y & 0xFFFF0000u) + acc[k].w * (sx * sw[3]);
        *reinterpret_cast<uint2*>(p.residual + static_cast<size_t>(t) * p.ld + h0) =
            make_uint2(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]));
        __stcg(reinterpret_cast<float4*>(p.partial + tile_base + static_cast<size_t>(t) * BM + lane * 4),
               make_float4(r[0], r[1], r[2], r[3]));
#pragma unroll
        for (int j = 0; j < 4; ++j) ss = fmaf(r[j], r[j], ss);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) p.rowstat[static_cast<size_t>(t) * p.num_m_tiles + m] = ss;
    }
  }
}

// After every m-tile is reduced: this CTA's slice of the T x H outputs,
// out = r * rstd[t] * g, vectors of eight columns; rstd from the m-tiles'
// sums of squares of the token in a fixed order.
__device__ void splitk_normalise_slice(const GemmParams& p, int ep_tid, float* rstd_s) {
  const int H8 = p.M >> 3;
  const long long V = static_cast<long long>(p.N) * H8;
  const long long v0 = V * blockIdx.x / gridDim.x, v1 = V * (blockIdx.x + 1) / gridDim.x;
  const int ta = static_cast<int>(v0 / H8), tb = v1 > v0 ? static_cast<int>((v1 - 1) / H8) : ta - 1;
  const int lane = ep_tid & 31, wid = ep_tid >> 5;
  const size_t tile_step = static_cast<size_t>(p.slot_stride) * p.N * BM;
  // this thread's first vector: its r and gamma loads go out with the row statistics' loads
  float4 fa = make_float4(0.f, 0.f, 0.f, 0.f), fb = fa, fg0 = fa, fg1 = fa;
  const long long vf = v0 + ep_tid;
  if (vf < v1) {
    const int t = static_cast<int>(vf / H8);
    const int h = static_cast<int>(vf - static_cast<long long>(t) * H8) * 8;
    const float4* rp =
        reinterpret_cast<const float4*>(p.partial + (h >> 7) * tile_step + static_cast<size_t>(t) * BM + (h & 127));
    fa = __ldcg(rp);
    fb = __ldcg(rp + 1);
    fg0 = __ldg(reinterpret_cast<const float4*>(p.gamma + h));
    fg1 = __ldg(reinterpret_cast<const float4*>(p.gamma + h + 4));
  }
  for (int t = ta + wid; t <= tb; t += 4) {
    float ss = 0.f;
    for (int m = lane; m < p.num_m_tiles; m += 32) ss += __ldcg(p.rowstat + static_cast<size_t>(t) * p.num_m_tiles + m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) rstd_s[t - ta] = rsqrtf(ss / static_cast<float>(p.M) + p.eps);
  }
  named_bar_sync(1, 128);
  for (long long v = vf; v < v1; v += 128) {
    const int t = static_cast<int>(v / H8);
    const int h = static_cast<int>(v - static_cast<long long>(t) * H8) * 8;
    float4 a = fa, b = fb, g0 = fg0, g1 = fg1;
    if (v != vf) {
      const float4* rp =
          reinterpret_cast<const float4*>(p.partial + (h >> 7) * tile_step + static_cast<size_t>(t) * BM + (h & 127));
      a = __ldcg(rp);
      b = __ldcg(rp + 1);
      g0 = __ldg(reinterpret_cast<const float4*>(p.gamma + h));
      g1 = __ldg(reinterpret_cast<const float4*>(p.gamma + h + 4));
    }
    const float rs = rstd_s[t - ta];
    const float r[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = r[j] * rs * (p.norm_kind ? 1.0f + g[j] : g[j]);
    __stcs(reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * p.ld + h), f32x8_to_bf16(o));
  }
}

template <int BN, int EPI, int F8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fln_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p) {
  constexpr int STAGES = stages_for(BN);
  constexpr int STAGE_BYTES = stage_bytes(BN);
  constexpr int TMEM_COLS = tmem_cols_for(BN);
  constexpr uint32_t IDESC = F8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN);
  constexpr int KBE = kblock_elems(F8);  // elements of K per 128-byte K-block

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* acc_full = empty_bar + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain_bar = acc_empty + 2;
  uint64_t* wq_full = drain_bar + 1;   // dynamic split-K chunks: producer -> MMA and epilogue
  uint64_t* wq_empty = wq_full + 4;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(wq_empty + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* epi_abort = abort_flag + 1;
  volatile int* wq = epi_abort + 1;     // 4 queued chunk ids (-1 = no more)
  volatile int* tail_last = wq + 4;     // fused split-K tail: this delivery was the m-tile's last
  float* tail_rstd = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full_bar) + 512);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the split-K reducer may be scheduled right away: it waits for this grid to
  // finish before it reads anything
  if (is_splitk(EPI)) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&wq_full[i], 1);
      mbar_init(&wq_empty[i], 5);  // the MMA issuer and the four epilogue warps
    }
    *abort_flag = 0;
    *epi_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  // The producer lane initialised the barriers itself and needs no tensor
  // memory, so warp 0 only arrives at the start barrier and streams at once;
  // the other warps wait there for the barriers and the TMEM address.
  if (warp == 0) {
    __syncwarp();
    named_bar_arrive(2, NUM_THREADS);
  } else {
    tc_fence_before();
    named_bar_sync(2, NUM_THREADS);
    tc_fence_after();
  }
  const uint32_t tmem_base = warp == 0 ? 0u : *tmem_holder;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_a = is_splitk(EPI) ? l2_policy_evict_first() : l2_policy_evict_normal();
    const uint64_t pol_b = l2_policy_evict_last();
    WorkSource<EPI> src(p);
    WorkItem w;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0;     // stages with a load issued
    uint32_t issued_parity = 0;   // parity of that load's phase
    bool ok = true;
    while (ok && src.next_producer(w, ok, wq_full, wq_empty, wq, abort_flag)) {
      const int a_row = a_row_of(p, w.m_tile);
      const int b_row = w.n_tile * BN;
      for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_EMPTY)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + stage * STAGE_BYTES;
        uint8_t* sb = sa + A_TILE_BYTES;
        mbar_arrive_expect_tx(&full_bar[stage], STAGE_BYTES);
        tma_load_2d(sa, &tmA, &full_bar[stage], kb * KBE, a_row, pol_a);
        tma_load_2d(sb, &tmB, &full_bar[stage], kb * KBE, b_row, pol_b);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) src.drain_ids();
    if (!ok) {
      // unwinding: let every load already issued land before the CTA exits
      for (int s = 0; s < STAGES; ++s) {
        if (issued_mask & (1u << s)) {
          volatile int no_abort = 0;
          mbar_wait(&full_bar[s], (issued_parity >> s) & 1u, &no_abort, p.err, FLN_DEVERR_TIMEOUT_DRAIN);
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    WorkSource<EPI> src(p);
    WorkItem w;
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    bool issued_any = false;
    while (ok && src.next_consumer(w, ok, wq_full, wq_empty, wq, abort_flag, false)) {
      const int b = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait(&acc_empty[b], (use & 1u) ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_ACC)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
      for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
        if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.err, FLN_DEVERR_TIMEOUT_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t sb = sa + A_TILE_BYTES;
        const uint64_t adesc = sw128_kmajor_desc(sa);
        const uint64_t bdesc = sw128_kmajor_desc(sb);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // advance 32 bytes along K inside the swizzle atom (encoded >> 4):
          // 16 bf16 or 32 E4M3 elements per MMA
          if (F8)
            mma_e4m3(d_tmem, adesc + static_cast<uint64_t>(kk * 2), bdesc + static_cast<uint64_t>(kk * 2), IDESC,
                     (kb > w.kb_begin || kk > 0) ? 1u : 0u);
          else
            mma_bf16(d_tmem, adesc + static_cast<uint64_t>(kk * 2), bdesc + static_cast<uint64_t>(kk * 2), IDESC,
                     (kb > w.kb_begin || kk > 0) ? 1u : 0u);
        }
        issued_any = true;
        mma_commit(&empty_bar[stage]);  // frees the smem stage once these MMAs have read it
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit(&acc_full[b]);  // accumulator ready for the epilogue
      ++local;
    }
    if (!ok && issued_any) {
      // unwinding: wait until the tensor core has finished with TMEM and smem
      mma_commit(drain_bar);
      volatile int no_abort = 0;
      mbar_wait(drain_bar, 0, &no_abort, p.err, FLN_DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int rl = q * 32 + lane;      // row within the tile
    const int ep_tid = threadIdx.x - 64;
    WorkSource<EPI> src(p);
    WorkItem w;
    int local = 0;
    bool failed = false;  // a row-statistics wait of this CTA gave up
    for (;;) {
      bool okq = true;
      const bool have = src.next_consumer(w, okq, wq_full, wq_empty, wq, abort_flag, true);
      const int b = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      // All 128 epilogue threads decide together whether to continue: a thread
      // that leaves alone would strand the others at a named barrier.
      bool stop = !have || !okq || failed;
      if (!stop && !mbar_wait(&acc_full[b], use & 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_ACC)) stop = true;
      if (named_bar_any(1, 128, stop)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * BN);
      const int row = w.m_tile * BM + rl;  // local row of the launch (A operand)
      const bool vrow = row < p.M;

      if (EPI == EPI_FUSED_NORM) {
        const size_t grow = static_cast<size_t>(p.a_row0) + static_cast<size_t>(row);
        const __nv_bfloat16* rrow = p.residual + grow * static_cast<size_t>(p.ld);
        const int n0 = w.n_tile * BN;
        // phase 1: r = r0 + acc, partial sum of squares over this tile's columns
        float ss = 0.f;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          tmem_ld16(tb + static_cast<uint32_t>(c), v);
          if (vrow) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int col = n0 + c + 8 * h;
              if (col < p.N) {
                const uint4 u = *reinterpret_cast<const uint4*>(rrow + col);
                float f[8];
                bf16x8_to_f32(u, f);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float r = f[j] + v[8 * h + j];
                  ss = fmaf(r, r, ss);
                }
              }
            }
          }
        }
        // publish this tile's partial sums, then wait for the row block's others
        const int nN = p.num_n_tiles;
        float* ps = p.psum + (static_cast<size_t>(w.m_tile) * nN) * BM;
        ps[static_cast<size_t>(w.n_tile) * BM + rl] = ss;
        __threadfence();
        named_bar_sync(1, 128);
        if (ep_tid == 0) st_release_gpu(&p.flags[w.m_tile * nN + w.n_tile], p.gen);
        bool rs_fail = false;
        if (ep_tid < 32) {
          bool ok = true;
          for (int j = lane; j < nN; j += 32) {
            const unsigned int* f = &p.flags[w.m_tile * nN + j];
            // (the test switch makes flag 0 wait for a value nobody publishes)
            const unsigned int want = (p.stall_rowstat && j == 0) ? p.gen + 1u : p.gen;
            if (ld_acquire_gpu(f) != want) {
              const uint64_t t0 = globaltimer_ns();
              while (ld_acquire_gpu(f) != want) {
                if (*abort_flag || globaltimer_ns() - t0 > FLN_WAIT_TIMEOUT_NS) {
                  ok = false;
                  break;
                }
              }
            }
            if (!ok) break;
          }
          ok = __all_sync(0xffffffffu, ok);
          if (!ok && lane == 0) {
            if (!*abort_flag) atomicOr(p.err, FLN_DEVERR_TIMEOUT_ROWSTAT);
            *abort_flag = 1;
          }
          rs_fail = !ok;
        }
        const bool go = !named_bar_any(1, 128, rs_fail);
        if (!go) failed = true;
        // phase 2: normalise and store residual and out (bf16, 16-byte stores)
        float tot = 0.f;
        for (int j = 0; j < nN; ++j) tot += ld_cg_f32(&ps[static_cast<size_t>(j) * BM + rl]);
        const float rstd = rsqrtf(tot / static_cast<float>(p.ld) + p.eps);
        __nv_bfloat16* wrow = p.residual + grow * static_cast<size_t>(p.ld);
        __nv_bfloat16* orow = p.out + grow * static_cast<size_t>(p.ld);
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          tmem_ld16(tb + static_cast<uint32_t>(c), v);
          if (vrow && go) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int col = n0 + c + 8 * h;
              if (col < p.N) {
                const uint4 u = *reinterpret_cast<const uint4*>(rrow + col);
                float f[8];
                bf16x8_to_f32(u, f);
                const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.gamma + col));
                const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.gamma + col + 4));
                float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                float r[8], o[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  r[j] = f[j] + v[8 * h + j];
                  const float gj = p.norm_kind ? 1.0f + g[j] : g[j];
                  o[j] = r[j] * rstd * gj;
                }
                *reinterpret_cast<uint4*>(wrow + col) = f32x8_to_bf16(r);
                *reinterpret_cast<uint4*>(orow + col) = f32x8_to_bf16(o);
              }
            }
          }
        }
      } else if (EPI == EPI_STORE_F32) {
        const int n0 = w.n_tile * BN;
        int srow = row;  // slot row
        bool vslot = vrow;
        if (p.blk_m_tiles > 0) {
          const int blk = w.m_tile / p.blk_m_tiles;
          const int local = (w.m_tile - blk * p.blk_m_tiles) * BM + rl;
          srow = blk * p.blk_rows + local;
          vslot = local < p.blk_rows;
        }
        float* yrow = p.yout + static_cast<size_t>(srow) * static_cast<size_t>(p.ld);
        // FP8: this row's token scale (FP8 launches use no blocks)
        const float sxr =
            (F8 && vslot) ? __ldg(p.x_scale + static_cast<size_t>(p.a_row0 + row) * p.x_scale_stride) : 0.f;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          tmem_ld16(tb + static_cast<uint32_t>(c), v);
          if (vslot) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int col = n0 + c + 8 * h;
              if (F8) {
                float sw[8];
                load_scale8(p.w_scale, p.w_scale_stride, col, col < p.N, sw);
#pragma unroll
                for (int j = 0; j < 8; ++j) v[8 * h + j] *= sxr * sw[j];
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[8 * h + j] *= p.y_scale;  // NVFP4 tensor scale, else 1
              }
              if (col < p.N) {
                float4* d = reinterpret_cast<float4*>(yrow + col);
                d[0] = make_float4(v[8 * h + 0], v[8 * h + 1], v[8 * h + 2], v[8 * h + 3]);
                d[1] = make_float4(v[8 * h + 4], v[8 * h + 5], v[8 * h + 6], v[8 * h + 7]);
              }
            }
          }
        }
      } else {  // EPI_SPLITK_SWAP: TMEM lane = hidden index h, column = token t
        float* dst = p.partial +
                     static_cast<size_t>(w.m_tile * p.slot_stride + w.split) * static_cast<size_t>(p.N) * BM;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          tmem_ld16(tb + static_cast<uint32_t>(c), v);
          if (vrow) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int t = c + j;
              if (t < p.N) dst[static_cast<size_t>(t) * BM + rl] = v[j];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      ++local;
      if (EPI == EPI_SPLITK_FUSED) {
        // the partial is delivered; the m-tile's last delivery reduces the m-tile.  The CTA
        // barrier orders every thread's partial stores before thread 0's release fence, which
        // makes them visible before its count (and its acquire fence after the count makes the
        // other deliveries' partials visible to the threads after the next barrier).
        named_bar_sync(1, 128);
        if (ep_tid == 0) {
          fence_acq_rel_gpu();
          const unsigned int cnt = tagged_add_one(&p.tile_arrivals[w.m_tile], p.gen);
          fence_acq_rel_gpu();
          const bool last = cnt == static_cast<unsigned int>(splitk_static_slots(p, w.m_tile) + p.dyn_cpm);
          // the last delivery puts the word back to zero (a graph replay reuses the generation)
          if (last) st_relaxed_gpu_u64(&p.tile_arrivals[w.m_tile], 0ull);
          *tail_last = last ? 1 : 0;
        }
        named_bar_sync(1, 128);
        if (*tail_last) {
          splitk_reduce_mtile<F8>(p, w.m_tile, ep_tid);
          named_bar_sync(1, 128);
          if (ep_tid == 0) {
            fence_acq_rel_gpu();
            tagged_add_one(p.tiles_done, p.gen);
          }
        }
      }
    }
    if (EPI == EPI_SPLITK_FUSED) {
      // every m-tile reduced (a bounded wait), then this CTA's slice of the outputs
      bool ok = true;
      if (ep_tid == 0) {
        // (the test switch waits for one m-tile more than there are)
        const unsigned long long want = (static_cast<unsigned long long>(p.gen) << 32) |
                                        static_cast<unsigned int>(p.num_m_tiles + (p.stall_rowstat ? 1 : 0));
        if (*abort_flag) {
          ok = false;
        } else if (ld_acquire_u64(p.tiles_done) != want) {
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire_u64(p.tiles_done) != want) {
            if (*abort_flag || globaltimer_ns() - t0 > FLN_WAIT_TIMEOUT_NS) {
              ok = false;
              break;
            }
          }
          if (!ok && !*abort_flag) {
            atomicOr(p.err, FLN_DEVERR_TIMEOUT_ROWSTAT);
            *abort_flag = 1;
          }
        }
        if (ok && tagged_add_one(p.tiles_done + 1, p.gen) == gridDim.x) {
          // the last CTA past the wait: every CTA has read the count, put both words back to zero
          st_relaxed_gpu_u64(p.tiles_done, 0ull);
          st_relaxed_gpu_u64(p.tiles_done + 1, 0ull);
        }
        fence_acq_rel_gpu();
      }
      if (!named_bar_any(1, 128, !ok)) splitk_normalise_slice(p, ep_tid, tail_rstd);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------- host side
template <int BN, int EPI, int F8>
static cudaError_t prepare_one() {
  return cudaFuncSetAttribute(fln_gemm_kernel<BN, EPI, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem_bytes_for(BN));
}

template <int BN, int EPI, int F8>
static cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                              cudaStream_t stream) {
  fln_gemm_kernel<BN, EPI, F8><<<grid, NUM_THREADS, smem_bytes_for(BN), stream>>>(tmA, tmB, p);
  return cudaGetLastError();
}

int gemm_smem_bytes(int bn) {
  switch (bn) {
    case 16: return smem_bytes_for(16);
    case 32: return smem_bytes_for(32);
    case 64: return smem_bytes_for(64);
    case 128: return smem_bytes_for(128);
    case 256: return smem_bytes_for(256);
    default: return -1;
  }
}

int gemm_stages(int bn) { return stages_for(bn); }

#define FLN_BN_SWITCH(bn, EPI, F8, CALL)            \
  switch (bn) {                                     \
    case 16: return CALL<16, EPI, F8>();            \
    case 32: return CALL<32, EPI, F8>();            \
    case 64: return CALL<64, EPI, F8>();            \
    case 128: return CALL<128, EPI, F8>();          \
    case 256: return CALL<256, EPI, F8>();          \
    default: return cudaErrorInvalidValue;          \
  }

// FP8 operands exist for the pipelined (STORE_F32) and split-K epilogues.
cudaError_t gemm_prepare(int bn, EpilogueKind epi, int f8) {
  if (f8) {
    switch (epi) {
      case EPI_STORE_F32: FLN_BN_SWITCH(bn, EPI_STORE_F32, 1, prepare_one)
      case EPI_SPLITK_SWAP: FLN_BN_SWITCH(bn, EPI_SPLITK_SWAP, 1, prepare_one)
      case EPI_SPLITK_FUSED: FLN_BN_SWITCH(bn, EPI_SPLITK_FUSED, 1, prepare_one)
      default: return cudaErrorInvalidValue;
    }
  }
  switch (epi) {
    case EPI_FUSED_NORM: FLN_BN_SWITCH(bn, EPI_FUSED_NORM, 0, prepare_one)
    case EPI_STORE_F32: FLN_BN_SWITCH(bn, EPI_STORE_F32, 0, prepare_one)
    case EPI_SPLITK_SWAP: FLN_BN_SWITCH(bn, EPI_SPLITK_SWAP, 0, prepare_one)
    case EPI_SPLITK_FUSED: FLN_BN_SWITCH(bn, EPI_SPLITK_FUSED, 0, prepare_one)
  }
  return cudaErrorInvalidValue;
}

#undef FLN_BN_SWITCH
#define FLN_BN_LAUNCH(bn, EPI, F8)                                            \
  switch (bn) {                                                               \
    case 16: return launch_one<16, EPI, F8>(tmA, tmB, p, grid, stream);       \
    case 32: return launch_one<32, EPI, F8>(tmA, tmB, p, grid, stream);       \
    case 64: return launch_one<64, EPI, F8>(tmA, tmB, p, grid, stream);       \
    case 128: return launch_one<128, EPI, F8>(tmA, tmB, p, grid, stream);     \
    case 256: return launch_one<256, EPI, F8>(tmA, tmB, p, grid, stream);     \
    default: return cudaErrorInvalidValue;                                    \
  }

cudaError_t launch_gemm(EpilogueKind epi, int bn, int f8, const CUtensorMap& tmA, const CUtensorMap& tmB,
                        const GemmParams& p, int grid, cudaStream_t stream) {
  if (f8) {
    switch (epi) {
      case EPI_STORE_F32: FLN_BN_LAUNCH(bn, EPI_STORE_F32, 1)
      case EPI_SPLITK_SWAP: FLN_BN_LAUNCH(bn, EPI_SPLITK_SWAP, 1)
      case EPI_SPLITK_FUSED: FLN_BN_LAUNCH(bn, EPI_SPLITK_FUSED, 1)
      default: return cudaErrorInvalidValue;
    }
  }
  switch (epi) {
    case EPI_FUSED_NORM: FLN_BN_LAUNCH(bn, EPI_FUSED_NORM, 0)
    case EPI_STORE_F32: FLN_BN_LAUNCH(bn, EPI_STORE_F32, 0)
    case EPI_SPLITK_SWAP: FLN_BN_LAUNCH(bn, EPI_SPLITK_SWAP, 0)
    case EPI_SPLITK_FUSED: FLN_BN_LAUNCH(bn, EPI_SPLITK_FUSED, 0)
  }
  return cudaErrorInvalidValue;
}

}  // namespace fln
