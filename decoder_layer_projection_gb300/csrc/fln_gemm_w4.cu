// fln_gemm_w4.cu -- split-K projection GEMM for few tokens with NVFP4 or MXFP4 weights
// (the UNFUSED path of the "TPSP Design" page, section 3, for the page's
// section 5 to-do item "MXFP4 / NVFP4 dense": low-bit weight layouts and
// their scaling).
//
// W holds E2M1 codes packed two per byte along K (element 2j in the low
// nibble of byte j) with one E4M3 scale per 16 elements of a row (NVFP4) or
// one E8M0 scale per 32 (MXFP4, the OCP microscaling layout); x is bf16.
// Four K-blocks of 64 elements of 128 weight rows arrive packed (16 KiB,
// 128-byte swizzled) in one TMA load, their block scales by cp.async on the
// same barrier; eight dequantisation warps turn each row's 64 codes of a
// K-block into bf16 values e2m1 * scale -- exact, a product of at most six
// significant bits -- and store them, a W entry at a time, in tensor memory (row m = TMEM lane m,
// two values per column), where the MMA issuer's tcgen05.mma kind::f16 reads
// its A operand; x arrives as 64 x BN bf16 tiles in a ring of its own (from
// L2).  Keeping the dequantised weights out of shared memory leaves shared
// memory bandwidth to the packed stream.  The tensor scale of W is applied by
// the reducer.  So W costs 0.5625 bytes per element from HBM instead of 2,
// while the MMA and the partial tiles are those of the bf16 split-K kernel (H
// on the MMA's M side, tokens on N, a stream-K partition of the (m-tile,
// K-block) units over the grid, fp32 partial tiles summed by the add + norm
// kernel).
//
// Warps: 0 W producer (TMA + scale copies), 1 TMEM owner + MMA issuer, 2-5
// epilogue (partial tiles), 6-13 dequantisation (half a weight row of a
// K-block per thread), 14 x producer.
#include <algorithm>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fln_internal.h"
#include "fln_ptx.cuh"

namespace fln {

namespace w4 {

constexpr int BM = 128;
constexpr int DQW = 8;                       // dequantisation warps (two per TMEM lane quarter)
constexpr int XWARP = 6 + DQW;               // x producer
constexpr int THREADS = 32 * (XWARP + 1);
constexpr int KG = 4;                        // K-blocks per packed W entry
constexpr int W_BYTES = BM * 32 * KG;        // packed codes of KG K-blocks: 128 rows x 128 bytes, 128-byte swizzled
constexpr int S_BYTES = BM * 4 * KG;         // block scales of a W entry: 128 rows x 16 bytes
constexpr int TMEM_COLS = 512;
constexpr int A_COLS = 32 * KG;              // one dequantised W entry in TMEM: 4 x 64 bf16 per lane
constexpr int SMEM_LIMIT = 232448;
constexpr int BAR_BYTES = 2048;            // barriers, then (from byte 1024) the scale table

// Shared memory: packed W entries with their scales (the HBM stream: as many
// bytes in flight as fit) and the x ring (XK K-blocks a stage).  TMEM: NACC tiles of NSUB fp32
// accumulators of BN columns, then AS dequantised W entries.
template <int BN>
struct Cfg {
  static constexpr int X_BYTES = BN * 128;  // 64 x BN bf16 tile of x (one K-block)
  static constexpr int XK = BN <= 64 ? 4 : BN <= 128 ? 2 : 1;  // K-blocks per x stage (divides KG)
  static constexpr int XSTAGE = XK * X_BYTES;
  static constexpr int XS = BN <= 16 ? 4 : BN <= 32 ? 3 : BN <= 128 ? 2 : 3;
  static constexpr int RW_FIT = (SMEM_LIMIT - 1024 - BAR_BYTES - XS * XSTAGE) / (W_BYTES + S_BYTES);
  static constexpr int RW = RW_FIT > 10 ? 10 : RW_FIT;
  static constexpr int SMEM = RW * (W_BYTES + S_BYTES) + XS * XSTAGE + BAR_BYTES + 1024;
  // NSUB accumulators per tile take the K-steps in turn, so consecutive MMAs
  // do not wait on one another's result; the epilogue adds them up
  static constexpr int NSUB = BN <= 64 ? 4 : BN <= 128 ? 2 : 1;
  static constexpr int NACC = NSUB * BN * 2 + 2 * A_COLS <= TMEM_COLS ? 2 : 1;  // tiles in TMEM
  static constexpr int A_COL0 = NACC * NSUB * BN;
  static constexpr int AS_FIT = (TMEM_COLS - A_COL0) / A_COLS;
  static constexpr int AS = AS_FIT > 3 ? 3 : AS_FIT;  // dequantised entries in flight
  static_assert(KG % XK == 0, "x stages tile a W entry");
  static_assert(X_BYTES % 1024 == 0, "x tile alignment");
  static_assert(RW >= 4 && RW <= 16, "W ring depth");
  static_assert(SMEM <= SMEM_LIMIT, "shared memory");
  static_assert(AS >= 2, "tensor memory");
};

// byte offset of the 16-byte chunk c (0..7) of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// bf16 bit pattern of an E4M3 code (every E4M3 value is a bf16 value)
__device__ __forceinline__ uint32_t e4m3_to_bf16_bits(uint32_t code) {
  const uint32_t sgn = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  if (e != 0) return (sgn << 15) | ((e + 120u) << 7) | (m << 4);
  // subnormal: m * 2^-9, exact in fp32 and bf16
  const float v = static_cast<float>(m) * 0.001953125f;
  return (sgn << 15) | (__float_as_uint(v) >> 16);
}

// Eight E2M1 codes (code i in bits 4i..4i+3 of w) times a bf16 scale held in
// both halves of s2 -> eight bf16 values.  The magnitudes 0, .5, 1, 1.5, 2,
// 3, 4, 6 are bf16 patterns whose high and low bytes are looked up with byte
// permutes (four codes per permute); the sign bits are placed on the high
// bytes' top bits before the bytes are interleaved into bf16 pairs, and each
// pair is multiplied by the scale (exact).  About 2.5 instructions a weight.
__device__ __forceinline__ uint4 e2m1x8_to_bf16(uint32_t w, uint32_t s2) {
  constexpr uint32_t HI0 = 0x3F3F3F00u, HI1 = 0x40404040u;  // high bytes of magnitudes 0..7
  constexpr uint32_t LO0 = 0xC0800000u, LO1 = 0xC0804000u;  // low bytes of magnitudes 0..7
  const uint32_t mag = w & 0x77777777u;
  uint32_t hi03 = __byte_perm(HI0, HI1, mag & 0xFFFFu);
  const uint32_t lo03 = __byte_perm(LO0, LO1, mag & 0xFFFFu);
  uint32_t hi47 = __byte_perm(HI0, HI1, mag >> 16);
  const uint32_t lo47 = __byte_perm(LO0, LO1, mag >> 16);
  // sign bits: byte k of ev / od carries the sign of code 2k / 2k + 1 in its top bit
  const uint32_t ev = (w << 4) & 0x80808080u, od = w & 0x80808080u;
  hi03 |= __byte_perm(ev, od, 0x5140);
  hi47 |= __byte_perm(ev, od, 0x7362);
  const uint32_t p0 = __byte_perm(lo03, hi03, 0x5140);
  const uint32_t p1 = __byte_perm(lo03, hi03, 0x7362);
  const uint32_t p2 = __byte_perm(lo47, hi47, 0x5140);
  const uint32_t p3 = __byte_perm(lo47, hi47, 0x7362);
  const __nv_bfloat162 sc = *reinterpret_cast<const __nv_bfloat162*>(&s2);
  uint4 o;
  __nv_bfloat162 t;
  t = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&p0), sc);
  o.x = *reinterpret_cast<const uint32_t*>(&t);
  t = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&p1), sc);
  o.y = *reinterpret_cast<const uint32_t*>(&t);
  t = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&p2), sc);
  o.z = *reinterpret_cast<const uint32_t*>(&t);
  t = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&p3), sc);
  o.w = *reinterpret_cast<const uint32_t*>(&t);
  return o;
}

// prmt.b32 in its default mode: a selector nibble with its top bit set
// copies the sign bit of the selected byte into all eight bits of the result byte
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// bf16 bits of e4m3(code) * 2^118: a normal bf16 for every nonzero code (the
// exponent stays below 255), 0 for either zero
__device__ __forceinline__ uint32_t e4m3_to_bf16_bits_x2p118(uint32_t code) {
  const uint32_t b = e4m3_to_bf16_bits(code);
  return (b & 0x7FFFu) ? b + (118u << 7) : 0u;
}

// bf16 bits of the E8M0 scale code E: 2^(E - 127) (the code 0 is the bf16
// subnormal 2^-127), NaN for 255
__device__ __forceinline__ uint32_t e8m0_to_bf16_bits(uint32_t E) {
  return E == 255u ? 0x7FC0u : E == 0u ? 0x0040u : (E << 7);
}

// Eight E2M1 codes (code i in bits 4i..4i+3 of w) -> four bf16 pairs, codes
// 2j and 2j + 1 in the low and high half of word j, each e2m1 * 2^-126 times
// the bf16 in both halves of s2 (with UNBIAS, first times 2^126: then e2m1
// times s2, exact for any power-of-two scale whose product stays finite).  A code's three magnitude bits become the two
// lowest exponent bits and the top fraction bit of a bf16 and its sign the
// sign: that bf16 is e2m1 * 2^-126 exactly (the zero exponent, a subnormal,
// gives the code of 0.5 its value).  Byte j of ev / od holds code 2j / 2j + 1
// in its low nibble; a permute puts the two in bytes 0 and 2 with zero bytes
// (sign copies of a byte below 0x80) beside them, one multiply by 64 + 4096
// makes the shifted copies (magnitude at bit 6, sign at bit 15 of each half,
// no carries: the copies do not overlap) and a mask keeps those bits.  The
// product with s2 is exact when s2 holds a block scale times 2^118.
template <bool UNBIAS>
__device__ __forceinline__ uint4 e2m1x8_to_bf16_biased(uint32_t w, uint32_t s2) {
  const uint32_t ev = w & 0x0F0F0F0Fu, od = (w >> 4) & 0x0F0F0F0Fu;
  const __nv_bfloat162 sc = *reinterpret_cast<const __nv_bfloat162*>(&s2);
  constexpr uint32_t P126 = 0x7E807E80u;  // 2^126 in both halves
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t b = (prmt(ev, od, 0xC480u + 0x1111u * static_cast<uint32_t>(j)) * 4160u) & 0x81C081C0u;
    __nv_bfloat162 t = *reinterpret_cast<const __nv_bfloat162*>(&b);
    if (UNBIAS) t = __hmul2(t, *reinterpret_cast<const __nv_bfloat162*>(&P126));
    t = __hmul2(t, sc);
    o[j] = *reinterpret_cast<const uint32_t*>(&t);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The static stream-K schedule: units (m-tile, K-block) in m-major order, CTA
// c takes [U c / G, U (c + 1) / G); every role walks the same sequence.
struct Items {
  const GemmParams& p;
  long long u, u_end;
  __device__ explicit Items(const GemmParams& prm) : p(prm) {
    u = p.units_total * blockIdx.x / gridDim.x;
    u_end = p.units_total * (blockIdx.x + 1) / gridDim.x;
  }
  __device__ bool next(int& m_tile, int& kb_begin, int& kb_end, int& split) {
    if (u >= u_end) return false;
    const int KB = p.num_k_blocks;
    m_tile = static_cast<int>(u / KB);
    kb_begin = static_cast<int>(u % KB);
    const long long left = u_end - u;
    kb_end = (KB - kb_begin) < left ? KB : kb_begin + static_cast<int>(left);
    const int c_first = splitk_cta_of_unit(static_cast<long long>(m_tile) * KB, p.units_total, gridDim.x);
    split = static_cast<int>(blockIdx.x) - c_first;
    u += kb_end - kb_begin;
    return true;
  }
};

// FMT 0: NVFP4 (E4M3 scale per 16 elements, w carries 2^-8 for the reducer
// to undo); FMT 1: MXFP4 (E8M0 scale per 32 elements, w exact)
template <int BN, int FMT>
__global__ void __launch_bounds__(THREADS, 1)
    fln_gemm_w4_splitk_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                              const GemmParams p) {
  using C = Cfg<BN>;
  constexpr int RW = C::RW, XS = C::XS, NACC = C::NACC, AS = C::AS, NSUB = C::NSUB;
  constexpr int SPK = FMT ? 2 : 4;  // scale bytes per K-block of a row
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;                   // RW packed W entries
  uint8_t* sX = sW + RW * W_BYTES;      // XS x stages
  uint8_t* sS = sX + XS * C::XSTAGE;    // RW scale blocks, one per W entry
  uint64_t* w_full = reinterpret_cast<uint64_t*>(sS + RW * S_BYTES);
  uint64_t* w_empty = w_full + RW;
  uint64_t* a_full = w_empty + RW;
  uint64_t* a_empty = a_full + AS;
  uint64_t* x_full = a_empty + AS;
  uint64_t* x_empty = x_full + XS;
  uint64_t* acc_full = x_empty + XS;
  uint64_t* acc_empty = acc_full + NACC;
  uint64_t* drain_bar = acc_empty + NACC;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  // scale code -> the dequantisation's block-scale operand as bf16, in both halves: an E4M3 value
  // times 2^118 (NVFP4) or an E8M0 value (MXFP4)
  uint32_t* scale_lut = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(w_full) + 1024);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the reducer may be scheduled right away: it waits for this grid to finish before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    for (int i = 0; i < RW; ++i) {
      mbar_init(&w_full[i], 1 + 32);  // the TMA's transaction bytes, and the 32 scale-copying lanes
      mbar_init(&w_empty[i], DQW);    // every dequantisation warp is done with the entry
    }
    for (int i = 0; i < AS; ++i) {
      mbar_init(&a_full[i], DQW);
      mbar_init(&a_empty[i], 1);      // the MMA issuer's commit
    }
    for (int i = 0; i < XS; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 1);      // the MMA issuer's commit
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (threadIdx.x < 256) {
    const uint32_t b = FMT ? e8m0_to_bf16_bits(threadIdx.x) : e4m3_to_bf16_bits_x2p118(threadIdx.x);
    scale_lut[threadIdx.x] = b | (b << 16);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ W producer
    // per group of KG K-blocks of an item: one packed W entry (TMA, lane 0)
    // with its block scales (4-byte cp.async by all lanes: a row's scales sit
    // at any 4-byte offset, too loosely aligned for TMA)
    const uint64_t pol_w = l2_policy_evict_first();
    Items it(p);
    int m_tile, kb0, kb1, split;
    int rw = 0;
    uint32_t wph = 0;
    uint32_t w_mask = 0, w_par = 0;  // loads issued (lane 0), for unwinding
    bool ok = true;
    while (ok && it.next(m_tile, kb0, kb1, split)) {
      for (int g0 = kb0; g0 < kb1; g0 += KG) {
        const int g1 = min(kb1, g0 + KG);
        bool got = true;
        if (lane == 0) got = mbar_wait(&w_empty[rw], wph ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_EMPTY);
        if (!__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&w_full[rw], W_BYTES);
          tma_load_2d(sW + rw * W_BYTES, &tmW, &w_full[rw], g0 * 32, m_tile * BM, pol_w);  // 128 bytes = 4 K-blocks
          w_mask |= 1u << rw;
          w_par = (w_par & ~(1u << rw)) | (wph << rw);
        }
        // scales of K-blocks [g0, g1), SPK bytes a K-block: the 4-byte words covering them land
        // at r * 16 + 4 i (rows hold a multiple of 4 scale bytes, so no word crosses a row's end)
        const int b0 = (SPK * g0) & ~3, nw = ((SPK * g1 + 3) & ~3) - b0;
        const uint32_t sdst = smem_u32(sS + rw * S_BYTES);
#pragma unroll
        for (int i = 0; i < BM / 32; ++i) {
          const int r = lane + 32 * i;
          const int h = m_tile * BM + r;
          if (h < p.M) {
            const uint8_t* src = p.w4_scales + static_cast<size_t>(h) * static_cast<size_t>(p.w4_nblk) + b0;
            for (int o = 0; o < nw; o += 4) cp_async4(sdst + static_cast<uint32_t>(r * 16 + o), src + o);
          }
        }
        cp_async_mbar_arrive_noinc(&w_full[rw]);
        if (++rw == RW) {
          rw = 0;
          wph ^= 1u;
        }
      }
    }
    cp_async_wait_all();
    if (!ok && lane == 0) {
      volatile int no_abort = 0;
      for (int i = 0; i < RW; ++i)
        if (w_mask & (1u << i)) mbar_wait(&w_full[i], (w_par >> i) & 1u, &no_abort, p.err, FLN_DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp == XWARP) {
    // ------------------------------------------------------------ x producer
    if (lane == 0) {
      const uint64_t pol_x = l2_policy_evict_last();
      Items it(p);
      int m_tile, kb0, kb1, split;
      int xs = 0;
      uint32_t xph = 0, x_mask = 0, x_par = 0;
      bool ok = true;
      while (ok && it.next(m_tile, kb0, kb1, split)) {
        // x stages tile each W entry [g0, g0 + KG) of the item: XK K-blocks a stage
        for (int g = kb0; g < kb1; g += C::XK) {
          if (!mbar_wait(&x_empty[xs], xph ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_EMPTY)) {
            ok = false;
            break;
          }
          const int n = min(kb1 - g, C::XK);
          mbar_arrive_expect_tx(&x_full[xs], static_cast<uint32_t>(n * C::X_BYTES));
          for (int j = 0; j < n; ++j)  // 64 bf16 of every token per K-block
            tma_load_2d(sX + xs * C::XSTAGE + j * C::X_BYTES, &tmX, &x_full[xs], (g + j) * 64, 0, pol_x);
          x_mask |= 1u << xs;
          x_par = (x_par & ~(1u << xs)) | (xph << xs);
          if (++xs == XS) {
            xs = 0;
            xph ^= 1u;
          }
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        for (int i = 0; i < XS; ++i)
          if (x_mask & (1u << i)) mbar_wait(&x_full[i], (x_par >> i) & 1u, &no_abort, p.err, FLN_DEVERR_TIMEOUT_DRAIN);
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ dequantisation
    // warp w: TMEM lane quarter w % 4, i.e. weight row 32 (w % 4) + lane of each tile;
    // columns [32 half, 32 half + 32) of each K-block, half = (w - 6) / 4: per K-block 16
    // bytes of codes and two block scales in, 16 TMEM columns out.  One W entry (up to
    // four K-blocks) per round: its conversions are independent of one another, and the
    // waits, the TMEM store wait and the barrier arrivals are paid once per entry.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int half = (warp - 6) >> 2;
    const uint32_t a_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                            static_cast<uint32_t>(C::A_COL0 + 16 * half);
    uint32_t coff[KG];  // this thread's 16-byte chunk of K-block j in a swizzled entry: chunk 2 j + half
#pragma unroll
    for (int j = 0; j < KG; ++j) coff[j] = swz(row, 2 * j + half);
    Items it(p);
    int m_tile, kb0, kb1, split;
    int rw = 0, s = 0;
    uint32_t wph = 0, sph = 0;
    bool ok = true;
    while (ok && it.next(m_tile, kb0, kb1, split)) {
      const bool vrow = m_tile * BM + row < p.M;
      for (int g0 = kb0; g0 < kb1; g0 += KG) {
        const int nk = min(kb1 - g0, KG);
        // the warp decides together: tcgen05.st below is a warp-wide instruction
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&w_full[rw], wph, abort_flag, p.err, FLN_DEVERR_TIMEOUT_FULL))) {
          ok = false;
          break;
        }
        // this row's scale bytes of the entry (first byte at (SPK g0) % 4): NVFP4 K-block j's two for
        // this thread in word j, bytes 2 half and 2 half + 1; MXFP4 K-block j's one at byte 2 j + half
        const uint4 sc4 = *reinterpret_cast<const uint4*>(sS + rw * S_BYTES + row * 16);
        const uint32_t scw[KG] = {sc4.x, sc4.y, sc4.z, sc4.w};
        const int mx0 = ((SPK * g0) & 3) + half;  // MXFP4: byte of K-block 0
        const uint8_t* went = sW + rw * W_BYTES;
        uint32_t v[KG][16];
#pragma unroll
        for (int j = 0; j < KG; ++j) {
          if (j < nk) {
            // 16-byte chunk 2 j + half of this row in the swizzled entry
            const uint4 cq = *reinterpret_cast<const uint4*>(went + coff[j]);
            uint32_t s20, s21;
            if (FMT == 0) {
              // values w * 2^-8 (block scale times 2^118 on codes times 2^-126); the reducer multiplies by 2^8
              const uint32_t sc = vrow ? (scw[j] >> (16 * half)) : 0u;
              s20 = scale_lut[sc & 0xFFu];
              s21 = scale_lut[(sc >> 8) & 0xFFu];
            } else {
              const int bi = mx0 + 2 * j;
              const uint32_t wd = bi < 4 ? scw[0] : bi < 8 ? scw[1] : scw[2];
              s20 = s21 = vrow ? scale_lut[(wd >> (8 * (bi & 3))) & 0xFFu] : 0u;
            }
            const uint4 v0 = e2m1x8_to_bf16_biased<FMT == 1>(cq.x, s20);
            const uint4 v1 = e2m1x8_to_bf16_biased<FMT == 1>(cq.y, s20);
            const uint4 v2 = e2m1x8_to_bf16_biased<FMT == 1>(cq.z, s21);
            const uint4 v3 = e2m1x8_to_bf16_biased<FMT == 1>(cq.w, s21);
            v[j][0] = v0.x, v[j][1] = v0.y, v[j][2] = v0.z, v[j][3] = v0.w;
            v[j][4] = v1.x, v[j][5] = v1.y, v[j][6] = v1.z, v[j][7] = v1.w;
            v[j][8] = v2.x, v[j][9] = v2.y, v[j][10] = v2.z, v[j][11] = v2.w;
            v[j][12] = v3.x, v[j][13] = v3.y, v[j][14] = v3.z, v[j][15] = v3.w;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&w_empty[rw]);  // this warp has read its part of the entry
        if (++rw == RW) {
          rw = 0;
          wph ^= 1u;
        }
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&a_empty[s], sph ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_EMPTY))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < KG; ++j)
          if (j < nk) tmem_st16(a_lane + static_cast<uint32_t>(s * A_COLS + 32 * j), v[j]);
        tmem_wait_st();
        tc_fence_before();  // the MMA reads these columns after the barrier
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[s]);
        if (++s == AS) {
          s = 0;
          sph ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    Items it(p);
    int m_tile, kb0, kb1, split;
    int s = 0, xs = 0, local = 0;
    uint32_t sph = 0, xph = 0;
    bool ok = true, issued_any = false;
    while (ok && it.next(m_tile, kb0, kb1, split)) {
      const int b = local % NACC;
      const uint32_t use = static_cast<uint32_t>(local / NACC);
      if (!mbar_wait(&acc_empty[b], (use & 1u) ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_ACC)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * NSUB * BN);
      for (int g0 = kb0; ok && g0 < kb1; g0 += KG) {
        if (!mbar_wait(&a_full[s], sph, abort_flag, p.err, FLN_DEVERR_TIMEOUT_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(C::A_COL0 + s * A_COLS);
        // straight-line issue of the entry's (up to) 4 x 4 MMAs: j = K-block, kk = K-step
        const int nk = min(kb1 - g0, KG);
        const bool first = g0 == kb0;  // the item's first entry starts every accumulator afresh
        uint64_t bdesc0 = 0;
#pragma unroll
        for (int j = 0; j < KG; ++j) {
          if (j < nk) {
            constexpr int XK = C::XK;
            if (j % XK == 0) {
              if (!mbar_wait(&x_full[xs], xph, abort_flag, p.err, FLN_DEVERR_TIMEOUT_FULL)) {
                ok = false;
                break;
              }
              bdesc0 = sw128_kmajor_desc(smem_u32(sX + xs * C::XSTAGE));
            }
            const uint64_t bdesc = bdesc0 + static_cast<uint64_t>((j % XK) * (C::X_BYTES >> 4));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // 16 elements of K = 8 TMEM columns of A, 32 bytes of B's rows
              mma_bf16_ts(d_tmem + static_cast<uint32_t>((kk % NSUB) * BN),
                          a_tmem + static_cast<uint32_t>(32 * j + 8 * kk), bdesc + static_cast<uint64_t>(kk * 2),
                          IDESC, (first && j == 0 && kk < NSUB) ? 0u : 1u);
            issued_any = true;
            if (j % XK == XK - 1 || j == nk - 1) {
              mma_commit(&x_empty[xs]);  // the x stage is free once these MMAs have read it
              if (++xs == XS) {
                xs = 0;
                xph ^= 1u;
              }
            }
          }
        }
        if (!ok) break;
        mma_commit(&a_empty[s]);  // and the entry's TMEM columns once all of its MMAs have
        if (++s == AS) {
          s = 0;
          sph ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit(&acc_full[b]);
      ++local;
    }
    if (!ok && issued_any) {
      mma_commit(drain_bar);
      volatile int no_abort = 0;
      mbar_wait(drain_bar, 0, &no_abort, p.err, FLN_DEVERR_TIMEOUT_DRAIN);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ epilogue: fp32 partial tiles
    const int q = warp & 3;         // TMEM lane quarter
    const int rl = q * 32 + lane;   // weight row within the tile (TMEM lane)
    Items it(p);
    int m_tile, kb0, kb1, split;
    int local = 0;
    for (;;) {
      const bool have = it.next(m_tile, kb0, kb1, split);
      const int b = local % NACC;
      const uint32_t use = static_cast<uint32_t>(local / NACC);
      bool stop = !have;
      if (!stop && !mbar_wait(&acc_full[b], use & 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_ACC)) stop = true;
      if (named_bar_any(1, 128, stop)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * NSUB * BN);
      const bool vrow = m_tile * BM + rl < p.M;
      float* dst = p.partial + static_cast<size_t>(m_tile * p.slot_stride + split) * static_cast<size_t>(p.N) * BM;
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        tmem_ld16(tb + static_cast<uint32_t>(c), v);
#pragma unroll
        for (int sub = 1; sub < NSUB; ++sub) {
          float u[16];
          tmem_ld16(tb + static_cast<uint32_t>(sub * BN + c), u);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] += u[j];
        }
        if (vrow) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c + j < p.N) dst[static_cast<size_t>(c + j) * BM + rl] = v[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      ++local;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

template <int BN, int FMT>
static cudaError_t run_bn(const CUtensorMap* tmW, const CUtensorMap* tmX, const GemmParams* p, int grid,
                          cudaStream_t stream) {
  if (!tmW) {
    return cudaFuncSetAttribute(fln_gemm_w4_splitk_kernel<BN, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<BN>::SMEM);
  }
  fln_gemm_w4_splitk_kernel<BN, FMT><<<grid, THREADS, Cfg<BN>::SMEM, stream>>>(*tmW, *tmX, *p);
  return cudaGetLastError();
}

template <int FMT>
static cudaError_t dispatch_fmt(int bn, const CUtensorMap* tmW, const CUtensorMap* tmX, const GemmParams* p,
                                int grid, cudaStream_t stream) {
  switch (bn) {
    case 16: return run_bn<16, FMT>(tmW, tmX, p, grid, stream);
    case 32: return run_bn<32, FMT>(tmW, tmX, p, grid, stream);
    case 64: return run_bn<64, FMT>(tmW, tmX, p, grid, stream);
    case 128: return run_bn<128, FMT>(tmW, tmX, p, grid, stream);
    case 256: return run_bn<256, FMT>(tmW, tmX, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

static cudaError_t dispatch(int bn, int fmt, const CUtensorMap* tmW, const CUtensorMap* tmX, const GemmParams* p,
                            int grid, cudaStream_t stream) {
  return fmt ? dispatch_fmt<1>(bn, tmW, tmX, p, grid, stream) : dispatch_fmt<0>(bn, tmW, tmX, p, grid, stream);
}

// Whole weight to bf16 for the paths with many tokens: one thread per eight
// elements (one 32-bit word of codes), w = e2m1 * block scale (exact); the
// NVFP4 tensor scale stays with the GEMM.  K % 64 == 0.
template <int FMT>
__global__ void fp4_to_bf16_kernel(const uint32_t* __restrict__ Wq, const uint8_t* __restrict__ S,
                                   uint4* __restrict__ out, int H, int K) {
  const size_t words = static_cast<size_t>(H) * (K / 8);
  const int wpr = K / 8;                       // words per row
  const int nblk = FMT ? K / 32 : K / 16;      // scales per row
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < words;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t h = i / wpr;
    const int c = static_cast<int>(i - h * wpr);   // elements 8c .. 8c + 7 of the row
    const uint32_t code = S[h * nblk + (FMT ? (c >> 2) : (c >> 1))];
    const uint32_t sb = FMT ? e8m0_to_bf16_bits(code) : e4m3_to_bf16_bits(code);
    out[i] = e2m1x8_to_bf16(__ldg(Wq + i), sb | (sb << 16));
  }
}

}  // namespace w4

cudaError_t launch_fp4_to_bf16(int fmt, const uint8_t* Wq, const uint8_t* S, __nv_bfloat16* out, int H, int K,
                               cudaStream_t stream) {
  const size_t words = static_cast<size_t>(H) * (K / 8);
  const int grid = static_cast<int>(std::min<size_t>((words + 255) / 256, 152 * 16));
  if (fmt)
    w4::fp4_to_bf16_kernel<1><<<grid, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(Wq), S,
                                                        reinterpret_cast<uint4*>(out), H, K);
  else
    w4::fp4_to_bf16_kernel<0><<<grid, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(Wq), S,
                                                        reinterpret_cast<uint4*>(out), H, K);
  return cudaGetLastError();
}

cudaError_t w4_gemm_prepare(int bn, int fmt) { return w4::dispatch(bn, fmt, nullptr, nullptr, nullptr, 0, nullptr); }

cudaError_t launch_w4_gemm_splitk(int bn, int fmt, const CUtensorMap& tmW, const CUtensorMap& tmX,
                                  const GemmParams& p, int grid, cudaStream_t stream) {
  return w4::dispatch(bn, fmt, &tmW, &tmX, &p, grid, stream);
}

}  // namespace fln
