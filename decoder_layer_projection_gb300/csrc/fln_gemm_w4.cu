// fln_gemm_w4.cu -- split-K projection GEMM for few tokens with NVFP4 weights
// (the UNFUSED path of the "TPSP Design" page, section 3, for the page's
// section 5 to-do item "MXFP4 / NVFP4 dense": low-bit weight layouts and
// their scaling).
//
// W holds E2M1 codes packed two per byte along K (element 2j in the low
// nibble of byte j) with one E4M3 scale per 16 elements of a row; x is bf16.
// A K-block of 64 elements of 128 weight rows arrives packed (4 KiB) by TMA
// together with the 64 x BN bf16 tile of x; four dequantisation warps turn
// each row's 64 codes into bf16 values e2m1 * scale -- exact, a product of at
// most six significant bits -- written in the 128-byte-swizzled K-major
// layout the tensor core reads, and the MMA issuer runs the same
// tcgen05.mma kind::f16 as the bf16 path on them.  The tensor scale of W is
// applied by the reducer.  So W costs 0.5625 bytes per element from HBM
// instead of 2, while the MMA and the partial tiles are those of the bf16
// split-K kernel (H on the MMA's M side, tokens on N, a stream-K partition of
// the (m-tile, K-block) units over the grid, fp32 partial tiles summed by the
// add + norm kernel).
//
// Warps: 0 TMA producer, 1 TMEM owner + MMA issuer, 2-5 epilogue (partial
// tiles), 6-9 dequantisation (one weight row per thread).
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
constexpr int THREADS = 320;
constexpr int W_BYTES = BM * 32;   // packed codes of one K-block: 128 rows x 64 codes
constexpr int A_BYTES = BM * 128;  // the same K-block dequantised: 128 rows x 64 bf16
constexpr int AS = 4;              // dequantised stages
constexpr int SMEM_LIMIT = 232448;
constexpr int BAR_BYTES = 1024;

template <int BN>
struct Cfg {
  static constexpr int B_BYTES = BN * 128;         // 64 x BN bf16 tile of x
  static constexpr int RAW = W_BYTES + B_BYTES;    // one raw stage (a multiple of 1024 bytes)
  static constexpr int RAW_FIT = (SMEM_LIMIT - 1024 - BAR_BYTES - AS * A_BYTES) / RAW;
  static constexpr int RS = RAW_FIT > 24 ? 24 : RAW_FIT;  // raw stages: the bytes in flight from HBM
  static constexpr int SMEM = AS * A_BYTES + RS * RAW + BAR_BYTES + 1024;
  static constexpr int TMEM_COLS = (2 * BN) <= 32 ? 32 : (2 * BN) <= 64 ? 64 : (2 * BN) <= 128 ? 128
                                 : (2 * BN) <= 256 ? 256 : 512;
  static_assert(RAW % 1024 == 0, "raw stage alignment");
  static_assert(RS >= 4, "pipeline depth");
  static_assert(SMEM <= SMEM_LIMIT, "shared memory");
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
// permutes (four codes per permute), the sign bits are moved to bits 15 and
// 31 of each pair, and the pair is multiplied by the scale (exact).
__device__ __forceinline__ uint4 e2m1x8_to_bf16(uint32_t w, uint32_t s2) {
  constexpr uint32_t HI0 = 0x3F3F3F00u, HI1 = 0x40404040u;  // high bytes of magnitudes 0..7
  constexpr uint32_t LO0 = 0xC0800000u, LO1 = 0xC0804000u;  // low bytes of magnitudes 0..7
  const uint32_t mag = w & 0x77777777u;
  const uint32_t hi03 = __byte_perm(HI0, HI1, mag & 0xFFFFu);
  const uint32_t lo03 = __byte_perm(LO0, LO1, mag & 0xFFFFu);
  const uint32_t hi47 = __byte_perm(HI0, HI1, mag >> 16);
  const uint32_t lo47 = __byte_perm(LO0, LO1, mag >> 16);
  uint32_t p0 = __byte_perm(lo03, hi03, 0x5140);
  uint32_t p1 = __byte_perm(lo03, hi03, 0x7362);
  uint32_t p2 = __byte_perm(lo47, hi47, 0x5140);
  uint32_t p3 = __byte_perm(lo47, hi47, 0x7362);
  p0 |= ((w << 12) & 0x8000u) | ((w << 24) & 0x80000000u);
  p1 |= ((w << 4) & 0x8000u) | ((w << 16) & 0x80000000u);
  p2 |= ((w >> 4) & 0x8000u) | ((w << 8) & 0x80000000u);
  p3 |= ((w >> 12) & 0x8000u) | (w & 0x80000000u);
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

template <int BN>
__global__ void __launch_bounds__(THREADS, 1)
    fln_gemm_w4_splitk_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                              const GemmParams p) {
  using C = Cfg<BN>;
  constexpr int RS = C::RS;
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                    // AS dequantised stages
  uint8_t* sRaw = sA + AS * A_BYTES;     // RS raw stages: packed W, then the x tile
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(sRaw + RS * C::RAW);
  uint64_t* raw_empty = raw_full + RS;
  uint64_t* a_full = raw_empty + RS;
  uint64_t* a_empty = a_full + AS;
  uint64_t* acc_full = a_empty + AS;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain_bar = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the reducer may be scheduled right away: it waits for this grid to finish before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    for (int i = 0; i < RS; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], 1);  // the MMA issuer's commit: it read x after the dequantisers read W
    }
    for (int i = 0; i < AS; ++i) {
      mbar_init(&a_full[i], 4);     // the four dequantisation warps
      mbar_init(&a_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
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
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    Items it(p);
    int m_tile, kb0, kb1, split;
    int r = 0;
    uint32_t rph = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    bool ok = true;
    while (ok && it.next(m_tile, kb0, kb1, split)) {
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&raw_empty[r], rph ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_EMPTY)) {
          ok = false;
          break;
        }
        uint8_t* dst = sRaw + r * C::RAW;
        mbar_arrive_expect_tx(&raw_full[r], C::RAW);
        tma_load_2d(dst, &tmW, &raw_full[r], kb * 32, m_tile * BM, pol_w);             // 32 bytes = 64 codes
        tma_load_2d(dst + W_BYTES, &tmX, &raw_full[r], kb * 64, 0, pol_x);            // 64 bf16 of every token
        issued_mask |= 1u << r;
        issued_parity = (issued_parity & ~(1u << r)) | (rph << r);
        if (++r == RS) {
          r = 0;
          rph ^= 1u;
        }
      }
    }
    if (!ok) {
      for (int i = 0; i < RS; ++i) {
        if (issued_mask & (1u << i)) {
          volatile int no_abort = 0;
          mbar_wait(&raw_full[i], (issued_parity >> i) & 1u, &no_abort, p.err, FLN_DEVERR_TIMEOUT_DRAIN);
        }
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ dequantisation (row dq of each tile)
    const int dq = threadIdx.x - 192;
    Items it(p);
    int m_tile, kb0, kb1, split;
    int r = 0, s = 0;
    uint32_t rph = 0, sph = 0;
    bool ok = true;
    while (ok && it.next(m_tile, kb0, kb1, split)) {
      const int h = m_tile * BM + dq;  // weight row
      const bool vrow = h < p.M;
      const uint32_t* srow = reinterpret_cast<const uint32_t*>(p.w4_scales + (vrow ? static_cast<size_t>(h) : 0) *
                                                                                  static_cast<size_t>(p.w4_nblk));
      uint32_t sc_next = vrow ? __ldg(srow + kb0) : 0u;  // the four E4M3 scales of a K-block (K % 64 == 0)
      for (int kb = kb0; kb < kb1; ++kb) {
        const uint32_t sc = sc_next;
        if (kb + 1 < kb1) sc_next = vrow ? __ldg(srow + kb + 1) : 0u;
        if (!mbar_wait(&raw_full[r], rph, abort_flag, p.err, FLN_DEVERR_TIMEOUT_FULL) ||
            !mbar_wait(&a_empty[s], sph ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_EMPTY)) {
          ok = false;
          break;
        }
        const uint4* src = reinterpret_cast<const uint4*>(sRaw + r * C::RAW + dq * 32);
        const uint4 q0 = src[0], q1 = src[1];
        const uint32_t wv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint8_t* dst = sA + s * A_BYTES;
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // scale j covers elements 16j..16j+15 = chunks 2j, 2j+1
          const uint32_t sb = e4m3_to_bf16_bits((sc >> (8 * j)) & 0xFFu);
          const uint32_t s2 = sb | (sb << 16);
          *reinterpret_cast<uint4*>(dst + swz(dq, 2 * j)) = e2m1x8_to_bf16(wv[2 * j], s2);
          *reinterpret_cast<uint4*>(dst + swz(dq, 2 * j + 1)) = e2m1x8_to_bf16(wv[2 * j + 1], s2);
        }
        fence_proxy_async_smem();  // the tensor core reads what these threads wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[s]);
        if (++r == RS) {
          r = 0;
          rph ^= 1u;
        }
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
    int r = 0, s = 0, local = 0;
    uint32_t rph = 0, sph = 0;
    bool ok = true, issued_any = false;
    while (ok && it.next(m_tile, kb0, kb1, split)) {
      const int b = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait(&acc_empty[b], (use & 1u) ^ 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_ACC)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&a_full[s], sph, abort_flag, p.err, FLN_DEVERR_TIMEOUT_FULL) ||
            !mbar_wait(&raw_full[r], rph, abort_flag, p.err, FLN_DEVERR_TIMEOUT_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + s * A_BYTES));
        const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sRaw + r * C::RAW + W_BYTES));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(d_tmem, adesc + static_cast<uint64_t>(kk * 2), bdesc + static_cast<uint64_t>(kk * 2), IDESC,
                   (kb > kb0 || kk > 0) ? 1u : 0u);
        issued_any = true;
        mma_commit(&a_empty[s]);    // the dequantised stage is free once these MMAs have read it
        mma_commit(&raw_empty[r]);  // and so is the raw stage (x tile)
        if (++r == RS) {
          r = 0;
          rph ^= 1u;
        }
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
      const int b = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      bool stop = !have;
      if (!stop && !mbar_wait(&acc_full[b], use & 1u, abort_flag, p.err, FLN_DEVERR_TIMEOUT_ACC)) stop = true;
      if (named_bar_any(1, 128, stop)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * BN);
      const bool vrow = m_tile * BM + rl < p.M;
      float* dst = p.partial + static_cast<size_t>(m_tile * p.slot_stride + split) * static_cast<size_t>(p.N) * BM;
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        tmem_ld16(tb + static_cast<uint32_t>(c), v);
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
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

template <int BN>
static cudaError_t run_bn(const CUtensorMap* tmW, const CUtensorMap* tmX, const GemmParams* p, int grid,
                          cudaStream_t stream) {
  if (!tmW) {
    return cudaFuncSetAttribute(fln_gemm_w4_splitk_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<BN>::SMEM);
  }
  fln_gemm_w4_splitk_kernel<BN><<<grid, THREADS, Cfg<BN>::SMEM, stream>>>(*tmW, *tmX, *p);
  return cudaGetLastError();
}

static cudaError_t dispatch(int bn, const CUtensorMap* tmW, const CUtensorMap* tmX, const GemmParams* p, int grid,
                            cudaStream_t stream) {
  switch (bn) {
    case 16: return run_bn<16>(tmW, tmX, p, grid, stream);
    case 32: return run_bn<32>(tmW, tmX, p, grid, stream);
    case 64: return run_bn<64>(tmW, tmX, p, grid, stream);
    case 128: return run_bn<128>(tmW, tmX, p, grid, stream);
    case 256: return run_bn<256>(tmW, tmX, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

// Whole weight to bf16 for the paths with many tokens: one thread per eight
// elements (one 32-bit word of codes), w = e2m1 * block scale (exact); the
// tensor scale stays with the GEMM.  K % 64 == 0.
__global__ void nvfp4_to_bf16_kernel(const uint32_t* __restrict__ Wq, const uint8_t* __restrict__ S,
                                     uint4* __restrict__ out, int H, int K) {
  const size_t words = static_cast<size_t>(H) * (K / 8);
  const int wpr = K / 8;      // words per row
  const int nblk = K / 16;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < words;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t h = i / wpr;
    const int c = static_cast<int>(i - h * wpr);   // elements 8c .. 8c + 7 of the row
    const uint32_t sb = e4m3_to_bf16_bits(S[h * nblk + (c >> 1)]);
    out[i] = e2m1x8_to_bf16(__ldg(Wq + i), sb | (sb << 16));
  }
}

}  // namespace w4

cudaError_t launch_nvfp4_to_bf16(const uint8_t* Wq, const uint8_t* S, __nv_bfloat16* out, int H, int K,
                                 cudaStream_t stream) {
  const size_t words = static_cast<size_t>(H) * (K / 8);
  const int grid = static_cast<int>(std::min<size_t>((words + 255) / 256, 152 * 16));
  w4::nvfp4_to_bf16_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(Wq), S,
                                                     reinterpret_cast<uint4*>(out), H, K);
  return cudaGetLastError();
}

cudaError_t w4_gemm_prepare(int bn) { return w4::dispatch(bn, nullptr, nullptr, nullptr, 0, nullptr); }

cudaError_t launch_w4_gemm_splitk(int bn, const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmParams& p,
                                  int grid, cudaStream_t stream) {
  return w4::dispatch(bn, &tmW, &tmX, &p, grid, stream);
}

}  // namespace fln
