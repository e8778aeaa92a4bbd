// fln_norm.cu -- residual add + RMSNorm, memory bound, one token row per CTA
// iteration, 16-byte loads and stores, fp32 statistics.
//
//   r[t,:] = r0[t,:] + y[t,:]          (residual updated in place, bf16)
//   out[t,:] = r[t,:] * rsqrt(mean_h r^2 + eps) * g     g = gamma or 1 + gamma
//
// This is the add/norm step of the vLLM "TPSP Design" page (section 1: local
// residual add and norm over the complete hidden size of each token; section
// 3 "Microchunk pipeline": add/norm of a chunk on a second stream), with the
// norm forms of torch-spyre's "Plugin Architecture" page (RMSNorm with fp32
// statistics; GemmaRMSNorm's trailing fp32 (1 + gamma) multiply).
//
// The addend y comes from one of three sources:
//   BF16    a bf16 [T, H] tensor (the public add_rmsnorm call);
//   F32     an fp32 pipeline slot written by the projection GEMM;
//   SPLITK  the fp32 stream-K partials of the decode GEMM, summed here in a
//           fixed order (deterministic).
// Each thread keeps its VPT 8-element vectors of r in registers between the
// statistics pass and the normalisation pass, so every byte is read once.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fln_internal.h"
#include "fln_ptx.cuh"

namespace fln {

constexpr int NORM_THREADS = 256;

template <int SRC>
__device__ __forceinline__ void load_y8(const NormParams& p, int t, int h, float (&y)[8]) {
  if (SRC == NORM_SRC_BF16) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p.y_bf16 + (static_cast<size_t>(p.row0) + t) * p.H + h));
    bf16x8_to_f32(u, y);
  } else if (SRC == NORM_SRC_F32) {
    const float4* s = reinterpret_cast<const float4*>(p.y_f32 + static_cast<size_t>(t) * p.H + h);
    const float4 a = __ldcs(s);
    const float4 b = __ldcs(s + 1);
    y[0] = a.x; y[1] = a.y; y[2] = a.z; y[3] = a.w;
    y[4] = b.x; y[5] = b.y; y[6] = b.z; y[7] = b.w;
  } else {
    // split-K: the hidden index h lives in m-tile h / 128, lane h % 128; the
    // CTAs that touched m-tile m wrote partial slots 0 .. n-1 in unit order.
    const int m = h >> 7;
    const int hl = h & 127;
    const long long KB = p.num_k_blocks;
    const int c_first = splitk_cta_of_unit(static_cast<long long>(m) * KB, p.units_total, p.gemm_grid);
    const int c_last = splitk_cta_of_unit(static_cast<long long>(m + 1) * KB - 1, p.units_total, p.gemm_grid);
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = 0.f;
    for (int s = 0; s <= c_last - c_first; ++s) {
      const float4* src = reinterpret_cast<const float4*>(
          p.partial + (static_cast<size_t>(m * p.max_split + s) * p.T + t) * 128 + hl);
      const float4 a = __ldcs(src);
      const float4 b = __ldcs(src + 1);
      y[0] += a.x; y[1] += a.y; y[2] += a.z; y[3] += a.w;
      y[4] += b.x; y[5] += b.y; y[6] += b.z; y[7] += b.w;
    }
  }
}

template <int SRC, int VPT>
__global__ void __launch_bounds__(NORM_THREADS) fln_add_rmsnorm_kernel(const NormParams p) {
  __shared__ float warp_sums[NORM_THREADS / 32];
  __shared__ float row_total;
  const int tid = threadIdx.x;
  const int nvec = p.H >> 3;
  for (int t = blockIdx.x; t < p.T; t += gridDim.x) {
    const size_t grow = static_cast<size_t>(p.row0) + static_cast<size_t>(t);
    const __nv_bfloat16* r0 = p.residual + grow * p.H;
    float r[VPT][8];
    float ss = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int vi = v * NORM_THREADS + tid;
      if (vi < nvec) {
        const int h = vi << 3;
        float y[8], f[8];
        load_y8<SRC>(p, t, h, y);
        const uint4 u = *reinterpret_cast<const uint4*>(r0 + h);
        bf16x8_to_f32(u, f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          r[v][j] = f[j] + y[j];
          ss = fmaf(r[v][j], r[v][j], ss);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) warp_sums[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < NORM_THREADS / 32; ++w) tot += warp_sums[w];
      row_total = tot;
    }
    __syncthreads();
    const float rstd = rsqrtf(row_total / static_cast<float>(p.H) + p.eps);
    __nv_bfloat16* rw = p.residual + grow * p.H;
    __nv_bfloat16* ow = p.out + grow * p.H;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int vi = v * NORM_THREADS + tid;
      if (vi < nvec) {
        const int h = vi << 3;
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.gamma + h));
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.gamma + h + 4));
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        float o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float gj = p.norm_kind ? 1.0f + g[j] : g[j];
          o[j] = r[v][j] * rstd * gj;
        }
        *reinterpret_cast<uint4*>(rw + h) = f32x8_to_bf16(r[v]);
        __stcs(reinterpret_cast<uint4*>(ow + h), f32x8_to_bf16(o));
      }
    }
    __syncthreads();  // warp_sums / row_total reuse on the next row
  }
}

template <int SRC>
static cudaError_t launch_src(const NormParams& p, int grid, cudaStream_t s) {
  const int nvec = p.H / 8;
  const int vpt = (nvec + NORM_THREADS - 1) / NORM_THREADS;
  if (vpt <= 1) fln_add_rmsnorm_kernel<SRC, 1><<<grid, NORM_THREADS, 0, s>>>(p);
  else if (vpt <= 2) fln_add_rmsnorm_kernel<SRC, 2><<<grid, NORM_THREADS, 0, s>>>(p);
  else if (vpt <= 4) fln_add_rmsnorm_kernel<SRC, 4><<<grid, NORM_THREADS, 0, s>>>(p);
  else if (vpt <= 8) fln_add_rmsnorm_kernel<SRC, 8><<<grid, NORM_THREADS, 0, s>>>(p);
  else if (vpt <= 16) fln_add_rmsnorm_kernel<SRC, 16><<<grid, NORM_THREADS, 0, s>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_add_rmsnorm(NormSource src, const NormParams& p, int grid_cap, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  int grid = p.T;
  if (grid_cap > 0 && grid > grid_cap) grid = grid_cap;
  switch (src) {
    case NORM_SRC_BF16: return launch_src<NORM_SRC_BF16>(p, grid, stream);
    case NORM_SRC_F32: return launch_src<NORM_SRC_F32>(p, grid, stream);
    case NORM_SRC_SPLITK: return launch_src<NORM_SRC_SPLITK>(p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fln
