// fln_gemm2.cu -- projection GEMM + residual add + RMSNorm on a CTA pair
// (tcgen05 cta_group::2) for the prefill regime.
//
// Computes, per 4096-token chunk, y = x . W^T (vLLM "TPSP Design", section 1:
// row-parallel projection; torch-spyre "Plugin Architecture", "Transposed
// linear weights": W is [H, K], used K-major) and fuses the residual add and
// the RMSNorm over the complete hidden size of each token ("TPSP Design",
// sections 1 and 3 "Fusion regions"; standard or Gemma (1 + gamma) weight).
//
// A cluster of two CTAs (on two SMs) computes a 256 x BN output tile with one
// MMA stream issued by the even CTA: each CTA loads its own 128 rows of x and
// half of the BN rows of W into its shared memory, the tensor cores read both
// halves, and each CTA's TMEM receives its own 128 rows.  Per SM this halves
// the W traffic of a 128 x BN tile.
//
// Epilogue (four warps per CTA, one TMEM lane = one row per thread; or two
// such groups taking alternate tiles): the residual streams through a ring of
// three 128-byte-swizzled 128 x 64 TMA boxes; with 16 KiB of output staging
// the epilogue holds 64 KiB of shared memory and the operand ring keeps 5
// stages at BN = 256.  Phase 1 forms r = r0 + acc in fp32 and the row's
// partial sum of squares; the row block's partial sums of all N-tiles are
// exchanged through global memory as 64-bit {launch generation, value} words
// (fixed summation order); phase 2 reads r back from TMEM, stages
// bf16(r * rstd * g) in shared memory and each warp writes its 32 rows back
// with TMA stores, rows past the chunk and columns past H clipped.
//
// Work units: the launch's tiles in row-block-major order, pair p taking
// units p, p + pairs, ...  When the last round of tiles would leave at least
// half of the pairs idle, each of its tiles becomes two units, one per half
// of the K-blocks: the first half's pair owns the tile (residual, norm,
// stores), the second half's pair writes its fp32 accumulator to global
// memory (L2) and announces it with a {launch generation, 1} word per lane
// quarter; the owner adds it to its own accumulator before the residual.
// With two epilogue groups the helper's half goes out before the helper
// takes the output-staging token, so it never waits for its pair's previous
// tile (the host then needs no guard on the round before).
//
// FP8 (E4M3) operands: the same kernel with kind::f8f6f4 MMAs over 128-byte
// K-blocks of 128 elements; phase 1 scales the accumulator by the token's and
// the column's dequantisation scales before the residual add.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fln_internal.h"
#include "fln_ptx.cuh"

namespace fln {

namespace pair {

constexpr int BM = 128;  // rows per CTA (256 per pair)
constexpr int BK = 64;
// warps: 0 producer, 1 MMA / TMEM, 2-5 epilogue, 6 residual loader, and with
// eight epilogue warps 7-10 as well
__host__ __device__ constexpr int threads_for(int ew) { return ew == 8 ? 352 : 224; }
constexpr int SMEM_LIMIT = 232448;  // 227 KiB opt-in per block
constexpr int BAR_BYTES = 512;

template <int BN>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;            // 16 KiB
  static constexpr int B_BYTES = (BN / 2) * BK * 2;      // this CTA's half of the W tile
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int GROUPS = (BN + 63) / 64;          // 64-column residual boxes per tile (last may be half used)
  static constexpr int BOX = BM * 64 * 2;                // one 128 x 64 bf16 box (16 KiB)
  static constexpr int NBOX = 3;                         // residual boxes in flight
  static constexpr int OSTAGE = 4 * 32 * 128;            // 32 rows x 64 bf16 output staging per warp
  static constexpr int E_BYTES = NBOX * BOX + OSTAGE;
  // the tile's gamma and weight scales in shared memory, [2 groups][2 tiles][2 vectors][BN] fp32:
  // where they fit beside the ring without costing a stage (every width but 256)
  static constexpr bool VEC = BN != 256 || false;
  static constexpr int VEC_BYTES = VEC ? 32 * BN : 0;
  static constexpr int RAW_STAGES = (SMEM_LIMIT - 1024 - BAR_BYTES - E_BYTES - VEC_BYTES) / STAGE;
  static constexpr int STAGES = RAW_STAGES > 8 ? 8 : RAW_STAGES;
  static constexpr int SMEM = STAGES * STAGE + E_BYTES + BAR_BYTES + VEC_BYTES + 1024;
  static constexpr int TMEM_COLS = (2 * BN) <= 256 ? 256 : 512;
  static_assert(BN % 32 == 0 && BN >= 128 && BN <= 256, "tile width");
  static_assert(STAGES >= 4, "pipeline depth");
  static_assert(SMEM <= SMEM_LIMIT, "shared memory");
};

enum UnitRole { UNIT_WHOLE = 0, UNIT_OWNER = 1, UNIT_HELPER = 2 };

struct Unit {
  int t;         // tile: row block t / nN, N-tile t % nN
  int kb0, kb1;  // K-blocks [kb0, kb1)
  int role;
  int j;         // split tiles: index among them
};

// unit u of a launch with `total` tiles whose last S are split (units: total + S)
__device__ __forceinline__ Unit unit_at(int u, int total, int S, int KB) {
  Unit w;
  const int D = total - S;
  if (u < D) {
    w.t = u;
    w.kb0 = 0;
    w.kb1 = KB;
    w.role = UNIT_WHOLE;
    w.j = 0;
  } else {
    const int v = u - D;
    const int h = v & 1;
    w.j = v >> 1;
    w.t = D + w.j;
    w.kb0 = h ? KB / 2 : 0;
    w.kb1 = h ? KB : KB / 2;
    w.role = h ? UNIT_HELPER : UNIT_OWNER;
  }
  return w;
}

__device__ __forceinline__ void st_release_gpu_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// wait (bounded) until the word at f carries generation gen
__device__ __forceinline__ bool wait_gen_word(const unsigned long long* f, unsigned int gen,
                                              volatile int* abort_flag) {
  if (static_cast<unsigned int>(ld_acquire_gpu_u64(f) >> 32) == gen) return true;
  const uint64_t t0 = globaltimer_ns();
  while (static_cast<unsigned int>(ld_acquire_gpu_u64(f) >> 32) != gen) {
    if (*abort_flag || globaltimer_ns() - t0 > FLN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

// byte offset of the 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled box
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// Where tile t of a launch lives: this CTA's first A row and B row, its
// first output row and the end of its valid rows, and the tile's first
// column.  Dense: row-pair block t / nN of the launch and N-tile t % nN.
// Grouped (slot mode with offsets): tiles of expert e are tb[e] ..
// tb[e + 1] - 1, row blocks fastest (the pairs of a round then stream the same
// W tiles), each row block starting at off[e] + 256 m.
struct TileAt {
  int a_row, b_row, out_row, row_end, n0;
};

template <int BN>
__device__ __forceinline__ TileAt tile_at(const GemmParams& p, int t, int nN, uint32_t rank, const int* g_off,
                                          const int* g_tb) {
  TileAt r;
  if (g_off == nullptr) {
    const int pm = t / nN, nt = t % nN;
    r.a_row = p.a_row0 + pm * 2 * BM + static_cast<int>(rank) * BM;
    r.b_row = nt * BN + static_cast<int>(rank) * (BN / 2);
    r.out_row = (pm * 2 + static_cast<int>(rank)) * BM;
    r.row_end = p.M;
    r.n0 = nt * BN;
    return r;
  }
  int lo = 0, hi = p.moe_E - 1;  // the last expert e with tb[e] <= t (experts without rows own no tiles)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (g_tb[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const int e = lo, local = t - g_tb[e];
  const int mb = (g_off[e + 1] - g_off[e] + 2 * BM - 1) / (2 * BM);  // row blocks of the expert
  const int nt = local / mb, m = local - nt * mb;
  r.a_row = g_off[e] + m * 2 * BM + static_cast<int>(rank) * BM;
  r.b_row = e * p.N + nt * BN + static_cast<int>(rank) * (BN / 2);
  r.out_row = r.a_row;
  r.row_end = g_off[e + 1];
  r.n0 = nt * BN;
  return r;
}

template <int BN, int F8, int EW>
__global__ void __launch_bounds__(threads_for(EW), 1)
    fln_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmRs,
                         const __grid_constant__ CUtensorMap tmOs, const GemmParams p) {
  using C = Cfg<BN>;
  // EW = 0: the PIPELINED path's slot GEMM -- the same mainloop, an epilogue
  // that writes the fp32 accumulator to the slot (no residual, no norm)
  constexpr bool SLOT = EW == 0;
  constexpr int STAGES = C::STAGES;
  constexpr uint32_t IDESC = F8 ? idesc_e4m3_f32(2 * BM, BN) : idesc_bf16_f32(2 * BM, BN);
  constexpr int KBE = kblock_elems(F8);  // elements of K per 128-byte K-block

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* sE = smem + STAGES * C::STAGE;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sE + C::E_BYTES);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* acc_full = empty_bar + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* e_full = acc_empty + 2;
  uint64_t* e_free = e_full + C::NBOX;
  uint64_t* drain_bar = e_free + C::NBOX;
  uint64_t* stg_done = drain_bar + 1;  // eight epilogue warps: per quarter, staging rows handed on
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(stg_done + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* epi_abort = abort_flag + 1;
  float* const svec = reinterpret_cast<float*>(sE + C::E_BYTES + BAR_BYTES);  // C::VEC only

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair_id = static_cast<int>(cluster_id_x());
  const int num_pairs = static_cast<int>(nclusters_x());
  const int nN = p.num_n_tiles;
  const int num_pm = (p.num_m_tiles + 1) / 2;
  // grouped slot GEMM: the offsets and the tiles before each expert, in the
  // residual boxes' space (slot mode has no residual); checked before any
  // barrier, TMEM or peer is touched, identically in both CTAs of a pair
  const bool grouped = SLOT && p.moe_off != nullptr;
  int* const g_off = grouped ? reinterpret_cast<int*>(sE) : nullptr;
  int* const g_tb = grouped ? g_off + 257 : nullptr;
  if (grouped) {
    const int E = p.moe_E;
    for (int e = threadIdx.x; e <= E; e += blockDim.x) g_off[e] = p.moe_off[e];
    __syncthreads();
    bool okg = threadIdx.x != 0 || (g_off[0] == 0 && g_off[E] == p.M);
    for (int e = threadIdx.x; e < E; e += blockDim.x) okg = okg && g_off[e] <= g_off[e + 1];
    okg = __syncthreads_and(okg);
    if (threadIdx.x == 0 && blockIdx.x == 0) {
      *p.moe_bad = okg ? 0u : 1u;
      if (!okg) atomicOr(p.err, FLN_DEVERR_BAD_INDEX);
    }
    if (!okg) return;
    if (threadIdx.x == 0) {
      int run = 0;
      for (int e = 0; e < E; ++e) {
        g_tb[e] = run;
        run += (g_off[e + 1] - g_off[e] + 2 * BM - 1) / (2 * BM) * nN;
      }
      g_tb[E] = run;
    }
    __syncthreads();
  }
  const int total = grouped ? g_tb[p.moe_E] : num_pm * nN;
  const int S = SLOT ? 0 : p.split_tiles;
  const int units = total + S;
  const int KB = p.num_k_blocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);  // the buffer's four epilogue warps in each CTA of the pair
    }
    for (int e = 0; e < C::NBOX; ++e) {
      mbar_init(&e_full[e], 1);
      mbar_init(&e_free[e], 4);  // one arrival per warp of the consuming group once it is done with the box
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&stg_done[i], 1);
    *abort_flag = 0;
    *epi_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (!SLOT) {
      tma_prefetch_desc(&tmR);
      tma_prefetch_desc(&tmRs);
    }
    if (!SLOT || p.moe_off == nullptr) tma_prefetch_desc(&tmOs);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    // W tiles are read again by every row block of the launch, x tiles only by
    // the N-tiles of their own row block (within the same round): W is kept in
    // L2 first (Llama-3-8B down_proj, 4096-token launches: 568 -> 553 us)
    const uint64_t pol_x = l2_policy_evict_normal();
    const uint64_t pol_w = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    bool ok = true;
    for (int u = pair_id; ok && u < units; u += num_pairs) {
      const Unit w = unit_at(u, total, S, KB);
      const TileAt ta = tile_at<BN>(p, w.t, nN, rank, g_off, g_tb);
      const int a_row = ta.a_row, b_row = ta.b_row;
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_EMPTY)) {
          ok = false;
          break;
        }
        uint8_t* sa = ring + stage * C::STAGE;
        uint8_t* sb = sa + C::A_BYTES;
        const uint32_t fb = map_to_cta(smem_u32(&full_bar[stage]), 0);
        if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * C::STAGE);
        tma_load_2d_pair(sa, &tmA, fb, kb * KBE, a_row, pol_x);
        tma_load_2d_pair(sb, &tmB, fb, kb * KBE, b_row, pol_w);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && leader) {
      for (int s = 0; s < STAGES; ++s) {
        if (issued_mask & (1u << s)) {
          volatile int no_abort = 0;
          mbar_wait(&full_bar[s], (issued_parity >> s) & 1u, &no_abort, p.err, FLN_DEVERR_TIMEOUT_DRAIN);
        }
      }
    }
  } else if (warp == 6 && lane == 0 && !SLOT) {
    // ------------------------------------------------------------ residual loader (both CTAs)
    // (a warp of its own: a lane spinning on a barrier would steal issue
    // slots from a producer or MMA lane of the same warp)
    // Box s of this CTA's sequence (buffer s % NBOX): the G boxes of each
    // unit that reads the residual, in unit order (a helper half reads none).
    constexpr int G = C::GROUPS;
    constexpr int NB = C::NBOX;
    const uint64_t pol_r = l2_policy_evict_normal();
    int s = 0;
    bool ok = true;
    for (int u = pair_id; ok && u < units; u += num_pairs) {
      const Unit w = unit_at(u, total, S, KB);
      if (w.role == UNIT_HELPER) continue;
      const int m0 = ((w.t / nN) * 2 + static_cast<int>(rank)) * BM;
      for (int g = 0; g < G; ++g, ++s) {
        if (s >= NB && !mbar_wait(&e_free[s % NB], static_cast<uint32_t>(s / NB - 1) & 1u, abort_flag, p.err,
                                  FLN_DEVERR_TIMEOUT_EMPTY)) {
          ok = false;
          break;
        }
        const int n0 = (w.t % nN) * BN + g * 64;
        mbar_arrive_expect_tx(&e_full[s % NB], C::BOX);
        tma_load_2d(sE + (s % NB) * C::BOX, &tmR, &e_full[s % NB], n0, m0, pol_r);
      }
    }
    // let the last boxes land before the CTA can exit (they may be unconsumed after an abort)
    for (int k = 1; k <= NB && s - k >= 0; ++k) {
      const int sb = s - k;
      volatile int no_abort = 0;
      mbar_wait(&e_full[sb % NB], static_cast<uint32_t>(sb / NB) & 1u, &no_abort, p.err, FLN_DEVERR_TIMEOUT_DRAIN);
    }
    (void)ok;
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true, issued_any = false;
    for (int u = pair_id; ok && u < units; u += num_pairs, ++local) {
      const Unit w = unit_at(u, total, S, KB);
      const int b = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait(&acc_empty[b], (use & 1u) ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_ACC)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.err, FLN_DEVERR_TIMEOUT_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(ring + stage * C::STAGE);
        const uint64_t adesc = sw128_kmajor_desc(sa);
        const uint64_t bdesc = sw128_kmajor_desc(sa + C::A_BYTES);
        // four MMAs of 32 bytes of K each (16 bf16 or 32 E4M3 elements)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if (F8)
            mma_e4m3_pair(d_tmem, adesc + static_cast<uint64_t>(kk * 2), bdesc + static_cast<uint64_t>(kk * 2),
                          IDESC, (kb > w.kb0 || kk > 0) ? 1u : 0u);
          else
            mma_bf16_pair(d_tmem, adesc + static_cast<uint64_t>(kk * 2), bdesc + static_cast<uint64_t>(kk * 2),
                          IDESC, (kb > w.kb0 || kk > 0) ? 1u : 0u);
        }
        issued_any = true;
        mma_commit_pair_mc(&empty_bar[stage], 0x3);  // frees the stage in both CTAs
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit_pair_mc(&acc_full[b], 0x3);  // accumulator ready in both CTAs
    }
    if (!ok && issued_any) {
      mma_commit_pair(drain_bar);
      volatile int no_abort = 0;
      mbar_wait(drain_bar, 0, &no_abort, p.err, FLN_DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp >= 2 && warp != 6) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // A group of four warps, one per quarter q = warp % 4 of the TMEM lanes
    // (32 rows), each warp covering all columns of its rows.  EW = 4: warps
    // 2-5 handle every tile of the pair.  EW = 8: warps 2-5 and 7-10 form two
    // groups that take alternate tiles, so that one group's wait for the row
    // statistics and its phase 2 overlap the other group's phase 1; the
    // pair's k-th tile uses TMEM buffer k % 2, i.e. always its group's.  The
    // groups share each quarter's output staging rows, passed on from tile to
    // tile in order through one mbarrier per quarter.
    constexpr int NG = SLOT ? 1 : EW / 4;  // epilogue groups
    const int q = warp & 3;       // TMEM lane quarter of this warp
    const int grp = warp >= 7 ? 1 : 0;
    const int rl = q * 32 + lane;  // row within this CTA's 128 rows
    const uint32_t acc_empty_leader = map_to_cta(smem_u32(&acc_empty[0]), 0);
    constexpr int G = C::GROUPS;
    constexpr int NB = C::NBOX;
    uint8_t* ostage = sE + C::NBOX * C::BOX + q * (32 * 128);  // the quarter's 32 output rows
    unsigned long long* psum = reinterpret_cast<unsigned long long*>(p.psum);
    const unsigned long long tag = static_cast<unsigned long long>(p.gen) << 32;
    int local = 0;        // k: the pair's k-th unit
    bool failed = false;  // a row-statistics or split wait of this warp gave up
    int sbox = 0;         // first residual box of the next unit that reads the residual
    for (int u = pair_id; u < units; u += num_pairs, ++local) {
      const Unit w = unit_at(u, total, S, KB);
      const int t = w.t;
      int s = sbox;  // this unit's first residual box
      if (w.role != UNIT_HELPER) sbox += G;
      if (NG == 2 && (local & 1) != grp) continue;  // the other group's tile
      const int b = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      const int mtile = (t / nN) * 2 + static_cast<int>(rank);  // 128-row block index in the launch
      const int nt = t % nN;
      const int n0 = nt * BN;
      const int col_end = min(p.N, n0 + BN);
      const int wrow0 = mtile * BM + q * 32;  // this warp's first row in the chunk
      // this tile's gamma [BN] and weight scales [BN] (C::VEC): the group's
      // tiles alternate between two slots, so a warp may fill the next slot
      // while the group's other warps still read this one; the group barrier
      // below orders the fill before every read
      float* const vslot = svec + ((grp * 2 + (NG == 2 ? (local >> 1) & 1 : local & 1)) * 2) * BN;
      // FP8: this row's token scale (rows past the chunk have a zero accumulator)
      float sxr = 0.f;
      if (F8 && !SLOT && w.role != UNIT_HELPER && wrow0 + lane < p.M)
        sxr = __ldg(p.x_scale + static_cast<size_t>(p.a_row0 + wrow0 + lane) * p.x_scale_stride);
      if (C::VEC && !SLOT && w.role != UNIT_HELPER) {
        for (int c = rl; c < BN; c += BM) {
          const int cc = n0 + c;
          const bool vc = cc < p.N;
          vslot[c] = vc ? __ldg(p.gamma + cc) : 0.f;
          if (F8) vslot[BN + c] = vc ? __ldg(p.w_scale + (p.w_scale_stride ? cc : 0)) : 0.f;
        }
      }
      // All epilogue threads decide together whether to continue: a thread
      // that leaves alone would strand the others at a named barrier.
      bool stop = failed;
      if (!stop && !mbar_wait(&acc_full[b], use & 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_ACC)) stop = true;
      // a split tile's owner: the other K-half of these 32 rows must have arrived
      const size_t split_slot = static_cast<size_t>(w.j) * 2 + rank;
      if (!stop && w.role == UNIT_OWNER && !wait_gen_word(p.split_flags + split_slot * 4 + q, p.gen, abort_flag)) {
        if (!*abort_flag) atomicOr(p.err, FLN_DEVERR_TIMEOUT_SPLIT);
        *abort_flag = 1;
        failed = true;
        stop = true;
      }
      if (named_bar_any(1 + grp, 128, stop)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * BN);
      // fp32 halves of split tiles: [chunk of 32 columns][quad i of 4 columns][row of this CTA][4], so
      // that each 16-byte access of a warp covers 512 contiguous bytes
      float* const half = p.split_buf + split_slot * (static_cast<size_t>(BN) * BM);
      if (SLOT) {
        // slot GEMM: y (scaled like the fused path) to the fp32 rows [M, ld]
        // (launch-local rows; grouped: rows at their grouped positions)
        const TileAt ta = tile_at<BN>(p, t, nN, rank, g_off, g_tb);
        const int row = ta.out_row + rl;
        const bool vrow = row < ta.row_end;
        const int n0 = ta.n0;
        float ysc = p.y_scale;
        if (F8 && vrow) ysc = __ldg(p.x_scale + static_cast<size_t>(p.a_row0 + row) * p.x_scale_stride);
        float* yrow = p.yout + static_cast<size_t>(row) * static_cast<size_t>(p.ld);
        if (!grouped) {
          // dense slot: each 32-column chunk of the warp's 32 rows goes out
          // through shared memory (two 4 KiB buffers a warp, in the residual
          // boxes' space) in one TMA store of whole 128-byte lines; the tensor
          // map clips rows past the chunk and columns past H
          uint8_t* const stg = sE + q * 8192;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_ld32(tb + static_cast<uint32_t>(c * 32), v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int col = n0 + c * 32 + 8 * i;
              float sc[8];
              if (F8) {
                load_scale8(p.w_scale, p.w_scale_stride, col, col < p.N, sc);
#pragma unroll
                for (int j = 0; j < 8; ++j) sc[j] *= ysc;
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) sc[j] = ysc;
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) v[8 * i + j] *= sc[j];
            }
            uint8_t* const buf = stg + (c & 1) * 4096;
            if (lane == 0 && c >= 2) bulk_wait_group_read<1>();  // the store of two chunks ago has read buf
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<float4*>(buf + swz(lane, k)) =
                  make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOs, buf, n0 + c * 32, ta.out_row + q * 32);
              bulk_commit_group();
            }
          }
          if (lane == 0) bulk_wait_group_read<0>();  // both buffers free for the warp's next tile
        } else {
          // grouped: rows stop at the expert's end, inside a box, so each lane stores its own row
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_ld32(tb + static_cast<uint32_t>(c * 32), v);
            if (vrow) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int col = n0 + c * 32 + 8 * i;
                if (col < p.N) {
                  float sc[8];
                  if (F8) {
                    load_scale8(p.w_scale, p.w_scale_stride, col, true, sc);
#pragma unroll
                    for (int j = 0; j < 8; ++j) sc[j] *= ysc;
                  } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) sc[j] = ysc;
                  }
                  float4* d = reinterpret_cast<float4*>(yrow + col);
                  d[0] = make_float4(v[8 * i] * sc[0], v[8 * i + 1] * sc[1], v[8 * i + 2] * sc[2], v[8 * i + 3] * sc[3]);
                  d[1] = make_float4(v[8 * i + 4] * sc[4], v[8 * i + 5] * sc[5], v[8 * i + 6] * sc[6],
                                     v[8 * i + 7] * sc[7]);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_leader + static_cast<uint32_t>(b * 8));
        continue;
      }
      if (w.role == UNIT_HELPER) {
        // second K-half: the raw accumulator goes to the owner (scales and the residual are the owner's)
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(tb + static_cast<uint32_t>(c * 32), v);
          float4* d4 = reinterpret_cast<float4*>(half) + static_cast<size_t>(c) * 8 * BM + rl;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            __stcg(d4 + i * BM, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_leader + static_cast<uint32_t>(b * 8));
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu_u64(p.split_flags + split_slot * 4 + q, tag | 1ull);
        if (NG == 2) {
          // two groups: hand the quarter's output staging on in unit order (this unit stores
          // nothing).  Taken only after the half is out, so the owner never waits for this
          // pair's previous tile, whose norm may need that very half.
          bool okh = true;
          if (lane == 0) {
            if (local >= 1)
              okh = mbar_wait(&stg_done[q], static_cast<uint32_t>(local - 1) & 1u, abort_flag, p.err,
                              FLN_DEVERR_TIMEOUT_ACC);
            if (okh) mbar_arrive(&stg_done[q]);
          }
          if (!__shfl_sync(0xffffffffu, okh ? 1 : 0, 0)) failed = true;
        }
        continue;
      }

      // phase 1: r = r0 + acc in fp32 and the row's partial sum of squares
      // over this tile.  The fp32 r replaces the accumulator in TMEM (phase 2
      // reads it back) and bf16(r) replaces r0 in the residual box, from where
      // each warp's 32 rows go out in one TMA store (rows past the chunk and
      // columns past H are clipped by the tensor map).  A half-used last box
      // (tile 224) is stored by the threads instead, so the next tile's
      // columns stay intact.  Rows past the chunk and columns past H read
      // zeros: acc and r0 are 0.
      float ss = 0.f;
      int pending = -1;  // box whose TMA store may still be reading it (freed one box later)
#pragma unroll 1
      for (int g = 0; g < G; ++g, ++s) {
        const int halves = (BN - g * 64) >= 64 ? 2 : 1;  // 32-column halves of this box inside the tile
        mbar_wait(&e_full[s % NB], static_cast<uint32_t>(s / NB) & 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_ACC);
        uint8_t* box = sE + (s % NB) * C::BOX;
#pragma unroll 1
        for (int c2 = 0; c2 < halves; ++c2) {
          float v[32];
          const uint32_t ta = tb + static_cast<uint32_t>(g * 64 + c2 * 32);
          // the residual rows and (FP8) the scales first: their latency then
          // overlaps the TMEM load's
          uint4 rin[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) rin[h] = *reinterpret_cast<const uint4*>(box + swz(rl, c2 * 4 + h));
          float scl[32];
          if (F8) {
            // dequantisation: y = acc * (sx[token] * sw[column])
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int cc = n0 + g * 64 + c2 * 32 + 8 * h;
              float sw[8];
              if (C::VEC) {
                const float4* sv = reinterpret_cast<const float4*>(vslot + BN + g * 64 + c2 * 32 + 8 * h);
                const float4 a = sv[0], bq = sv[1];
                sw[0] = a.x; sw[1] = a.y; sw[2] = a.z; sw[3] = a.w;
                sw[4] = bq.x; sw[5] = bq.y; sw[6] = bq.z; sw[7] = bq.w;
              } else {
                load_scale8(p.w_scale, p.w_scale_stride, cc, cc < p.N, sw);
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) scl[8 * h + j] = sxr * sw[j];
            }
          }
          tmem_ld32(ta, v);
          if (w.role == UNIT_OWNER) {
            // the other K-half of the accumulator (fixed order: this half + that half)
            const float4* h4 = reinterpret_cast<const float4*>(half) + static_cast<size_t>(g * 2 + c2) * 8 * BM + rl;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 a = __ldcg(h4 + i * BM);
              v[4 * i] += a.x;
              v[4 * i + 1] += a.y;
              v[4 * i + 2] += a.z;
              v[4 * i + 3] += a.w;
            }
          }
          if (F8) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= scl[j];
          } else {
            // a tensor scale of the weights (NVFP4 dequantised to bf16); 1 otherwise
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= p.y_scale;
          }
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            uint4* rp = reinterpret_cast<uint4*>(box + swz(rl, c2 * 4 + h));
            float f[8];
            bf16x8_to_f32(rin[h], f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float r = f[j] + v[8 * h + j];
              ss = fmaf(r, r, ss);
              v[8 * h + j] = r;
            }
            *rp = f32x8_to_bf16(&v[8 * h]);
          }
          tmem_st32(ta, v);
        }
        if (halves == 2) {
          fence_proxy_async_smem();  // the box rows are visible to the TMA store
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmRs, box + q * (32 * 128), n0 + g * 64, wrow0);
            bulk_commit_group();
            if (pending >= 0) {
              bulk_wait_group_read<1>();           // the previous box's store has read its rows
              mbar_arrive(&e_free[pending % NB]);  // this warp is done with that box
            }
          }
          pending = s;
          __syncwarp();
        } else {
          __syncwarp();
#pragma unroll 2
          for (int it = 0; it < 8; ++it) {
            const int rr = it * 4 + (lane >> 3);  // row within this warp's 32
            const int ch = lane & 7;
            const int lrow = wrow0 + rr;
            const int col = n0 + g * 64 + ch * 8;
            if (lrow < p.M && col < col_end) {
              const size_t off = (static_cast<size_t>(p.a_row0) + lrow) * static_cast<size_t>(p.ld) + col;
              *reinterpret_cast<uint4*>(p.residual + off) =
                  *reinterpret_cast<const uint4*>(box + swz(q * 32 + rr, ch));
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&e_free[s % NB]);  // this warp is done with box s
        }
      }
      if (lane == 0 && pending >= 0) {
        bulk_wait_group_read<0>();
        mbar_arrive(&e_free[pending % NB]);
      }
      // Row statistics across the row block's N-tiles: each row's partial sum
      // is published as one 64-bit word {generation of this launch, value}, so a
      // reader that sees this launch's generation also sees its value; no fence
      // or flag is needed.  The words are fetched eight at a time and added in
      // N-tile order.
      unsigned long long* prow = psum + static_cast<size_t>(mtile) * nN * BM + rl;
      st_relaxed_gpu_u64(prow + static_cast<size_t>(nt) * BM, tag | __float_as_uint(ss));
      const int nw = nN;
      float tot = 0.f;
      bool ok = true;
      for (int j0 = 0; j0 < nw && ok; j0 += 8) {
        unsigned long long v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          v[i] = (j0 + i < nw) ? ld_relaxed_gpu_u64(prow + static_cast<size_t>(j0 + i) * BM) : tag;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (j0 + i >= nw || !ok) continue;
          // (the test switch makes word 0 wait for a generation nobody publishes)
          const unsigned int want = (p.stall_rowstat && j0 + i == 0) ? p.gen + 1u : p.gen;
          if ((v[i] >> 32) != want) {
            const unsigned long long* f = prow + static_cast<size_t>(j0 + i) * BM;
            const uint64_t t0 = globaltimer_ns();
            while (((v[i] = ld_relaxed_gpu_u64(f)) >> 32) != want) {
              if (*abort_flag || globaltimer_ns() - t0 > FLN_WAIT_TIMEOUT_NS) {
                ok = false;
                break;
              }
            }
          }
          tot += __uint_as_float(static_cast<uint32_t>(v[i]));
        }
      }
      if (!ok) {
        if (!*abort_flag) atomicOr(p.err, FLN_DEVERR_TIMEOUT_ROWSTAT);
        *abort_flag = 1;
        failed = true;  // this warp; the next top-of-loop barrier stops all of them
      }
      bool go = __all_sync(0xffffffffu, ok);
      const float rstd = rsqrtf(tot / static_cast<float>(p.ld) + p.eps);
      // two groups: the quarter's staging rows are free once the previous
      // tile's phase 2 has handed them on
      if (NG == 2 && local >= 1 &&
          !mbar_wait(&stg_done[q], static_cast<uint32_t>(local - 1) & 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_ACC)) {
        go = false;
        failed = true;
      }

      // phase 2: out = r * rstd * g from the fp32 r in TMEM, staged in this
      // warp's 32 output rows and written by one TMA store per warp and box
      // (threads store a half-used last box themselves).
      tmem_wait_st();
#pragma unroll 1
      for (int g = 0; g < G; ++g) {
        const int halves = (BN - g * 64) >= 64 ? 2 : 1;
        uint4 ob[8];  // this box's bf16 outputs, computed before waiting for the staging rows
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          if (c2 < halves) {
            // gamma first: its latency then overlaps the TMEM load's
            float gw[32];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int cc = n0 + g * 64 + (c2 * 4 + h) * 8;
              if (C::VEC) {
                const float4* gv = reinterpret_cast<const float4*>(vslot + g * 64 + (c2 * 4 + h) * 8);
                const float4 g0 = gv[0], g1 = gv[1];
                gw[8 * h] = g0.x; gw[8 * h + 1] = g0.y; gw[8 * h + 2] = g0.z; gw[8 * h + 3] = g0.w;
                gw[8 * h + 4] = g1.x; gw[8 * h + 5] = g1.y; gw[8 * h + 6] = g1.z; gw[8 * h + 7] = g1.w;
              } else if (cc < p.N) {
                const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.gamma + cc));
                const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.gamma + cc + 4));
                gw[8 * h] = g0.x; gw[8 * h + 1] = g0.y; gw[8 * h + 2] = g0.z; gw[8 * h + 3] = g0.w;
                gw[8 * h + 4] = g1.x; gw[8 * h + 5] = g1.y; gw[8 * h + 6] = g1.z; gw[8 * h + 7] = g1.w;
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) gw[8 * h + j] = 0.f;
              }
            }
            float v[32];
            tmem_ld32(tb + static_cast<uint32_t>(g * 64 + c2 * 32), v);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              float o[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float gj = p.norm_kind ? 1.0f + gw[8 * h + j] : gw[8 * h + j];
                o[j] = v[8 * h + j] * rstd * gj;
              }
              ob[c2 * 4 + h] = f32x8_to_bf16(o);
            }
          }
        }
        if (lane == 0) bulk_wait_group_read<0>();  // the previous box's store has read the staging rows
        __syncwarp();
#pragma unroll
        for (int chunk = 0; chunk < 8; ++chunk)
          if (chunk < halves * 4) *reinterpret_cast<uint4*>(ostage + swz(lane, chunk)) = ob[chunk];
        if (halves == 2) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && go) {
            tma_store_2d(&tmOs, ostage, n0 + g * 64, wrow0);
            bulk_commit_group();
          }
          __syncwarp();
        } else {
          __syncwarp();
          if (go) {
#pragma unroll 2
            for (int it = 0; it < 8; ++it) {
              const int rr = it * 4 + (lane >> 3);
              const int ch = lane & 7;
              const int lrow = wrow0 + rr;
              const int col = n0 + g * 64 + ch * 8;
              if (lrow < p.M && col < col_end) {
                const size_t off = (static_cast<size_t>(p.a_row0) + lrow) * static_cast<size_t>(p.ld) + col;
                __stcs(reinterpret_cast<uint4*>(p.out + off), *reinterpret_cast<const uint4*>(ostage + swz(rr, ch)));
              }
            }
          }
          __syncwarp();
        }
      }
      if (NG == 2) {
        // hand the staging rows on once this tile's last store has read them
        if (lane == 0) {
          bulk_wait_group_read<0>();
          mbar_arrive(&stg_done[q]);
        }
        __syncwarp();
      }
      // TMEM reads of this tile are done: hand the accumulator back to the MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_leader + static_cast<uint32_t>(b * 8));
    }
    if (lane == 0) bulk_wait_group<0>();  // this warp's stores have completed before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its peer may still signal it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
}

template <int BN, int F8, int EW>
static cudaError_t launch_pair_bn(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmR,
                                  const CUtensorMap& tmRs, const CUtensorMap& tmOs, const GemmParams& p, int pairs,
                                  cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(threads_for(EW), 1, 1);
  cfg.dynamicSmemBytes = Cfg<BN>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fln_gemm_pair_kernel<BN, F8, EW>, tmA, tmB, tmR, tmRs, tmOs, p);
}

template <int BN, int F8, int EW>
static cudaError_t prepare_pair_bn(int* max_pairs) {
  cudaError_t e = cudaFuncSetAttribute(fln_gemm_pair_kernel<BN, F8, EW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<BN>::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(threads_for(EW), 1, 1);
  cfg.dynamicSmemBytes = Cfg<BN>::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_pairs, fln_gemm_pair_kernel<BN, F8, EW>, &cfg);
}

// The instantiated variants: every tile width with four epilogue warps, tile
// widths 224 and 256 also with eight; the slot GEMM (ew = 0) for 128 and 256.
struct PairArgs {
  const CUtensorMap *tmA, *tmB, *tmR, *tmRs, *tmOs;
  const GemmParams* p;
  int pairs;
  cudaStream_t stream;
  int* max_pairs;  // non-null: prepare instead of launch
};

template <int BN, int F8, int EW>
static cudaError_t run_variant(const PairArgs& a) {
  if (a.max_pairs) return prepare_pair_bn<BN, F8, EW>(a.max_pairs);
  return launch_pair_bn<BN, F8, EW>(*a.tmA, *a.tmB, *a.tmR, *a.tmRs, *a.tmOs, *a.p, a.pairs, a.stream);
}

template <int F8>
static cudaError_t dispatch_bn(int bn, int ew, const PairArgs& a) {
  if (ew == 0) {  // slot GEMM of the PIPELINED path
    switch (bn) {
      case 128: return run_variant<128, F8, 0>(a);
      case 256: return run_variant<256, F8, 0>(a);
    }
    return cudaErrorInvalidValue;
  }
  if (ew == 8) {
    switch (bn) {
      case 224: return run_variant<224, F8, 8>(a);
      case 256: return run_variant<256, F8, 8>(a);
    }
    return cudaErrorInvalidValue;
  }
  if (ew != 4) return cudaErrorInvalidValue;
  switch (bn) {
    case 128: return run_variant<128, F8, 4>(a);
    case 192: return run_variant<192, F8, 4>(a);
    case 224: return run_variant<224, F8, 4>(a);
    case 256: return run_variant<256, F8, 4>(a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pair

cudaError_t pair_gemm_prepare(int bn, int f8, int ew, int* max_pairs) {
  pair::PairArgs a{};
  a.max_pairs = max_pairs;
  return f8 ? pair::dispatch_bn<1>(bn, ew, a) : pair::dispatch_bn<0>(bn, ew, a);
}

cudaError_t launch_gemm_pair_fused(int bn, int f8, int ew, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                   const CUtensorMap& tmR, const CUtensorMap& tmRs, const CUtensorMap& tmOs,
                                   const GemmParams& p, int pairs, cudaStream_t stream) {
  pair::PairArgs a{&tmA, &tmB, &tmR, &tmRs, &tmOs, &p, pairs, stream, nullptr};
  return f8 ? pair::dispatch_bn<1>(bn, ew, a) : pair::dispatch_bn<0>(bn, ew, a);
}

}  // namespace fln
