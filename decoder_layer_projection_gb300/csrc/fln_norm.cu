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
//           fixed order (deterministic); with FP8 operands the sum is scaled
//           by the token's and the column's dequantisation scales.
// Each thread keeps its VPT 8-element vectors of r in registers between the
// statistics pass and the normalisation pass, so every byte is read once.  All
// loads of a thread are independent and issued before their first use (the
// split-K sum is unrolled to a compile-time bound of splits), so a row costs
// about one memory latency, not one per split.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fln_internal.h"
#include "fln_ptx.cuh"

namespace fln {

// split-K: the hidden index h lives in m-tile h / 128, lane h % 128; the
// CTAs that touched m-tile m in the static split wrote partial slots
// 0 .. n-1 in unit order, the dynamic chunks slots max_split .. max_split +
// dyn_cpm - 1; the slots are summed in that fixed order (at most MAXS).
template <int MAXS>
__device__ __forceinline__ void load_splitk8(const NormParams& p, int t, int h, float (&y)[8]) {
  const int m = h >> 7;
  const int hl = h & 127;
  const long long KB = p.num_k_blocks;
  const int c_first = splitk_cta_of_unit(static_cast<long long>(m) * KB, p.units_total, p.gemm_grid);
  const int c_last = splitk_cta_of_unit(static_cast<long long>(m + 1) * KB - 1, p.units_total, p.gemm_grid);
  const int n = c_last - c_first + 1;
  const int total = n + p.dyn_cpm;
  float4 a[MAXS], b[MAXS];
#pragma unroll
  for (int s = 0; s < MAXS; ++s) {
    if (s < total) {
      const int slot = s < n ? s : p.max_split + (s - n);
      const float4* src = reinterpret_cast<const float4*>(
          p.partial + (static_cast<size_t>(m * p.slot_stride + slot) * p.T + t) * 128 + hl);
      a[s] = __ldcs(src);
      b[s] = __ldcs(src + 1);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) y[j] = 0.f;
#pragma unroll
  for (int s = 0; s < MAXS; ++s) {
    if (s < total) {
      y[0] += a[s].x; y[1] += a[s].y; y[2] += a[s].z; y[3] += a[s].w;
      y[4] += b[s].x; y[5] += b[s].y; y[6] += b[s].z; y[7] += b[s].w;
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) y[j] *= p.y_scale;  // NVFP4 tensor scale, else 1
  if (p.w_scale) {
    // FP8 operands: y = sum * (sx[token] * sw[column])
    const float sx = __ldg(p.x_scale + static_cast<size_t>(p.row0 + t) * p.x_scale_stride);
    float sw[8];
    load_scale8(p.w_scale, p.w_scale_stride, h, true, sw);
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] *= sx * sw[j];
  }
}

template <int SRC, int MAXS>
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
    load_splitk8<MAXS>(p, t, h, y);
  }
}

template <int SRC, int VPT, int NT, int MAXS>
__global__ void __launch_bounds__(NT) fln_add_rmsnorm_kernel(const NormParams p) {
  __shared__ float warp_sums[NT / 32];
  __shared__ float row_total;
  const int tid = threadIdx.x;
  const int nvec = p.H >> 3;
  // When launched as a programmatic dependent, wait until the producing
  // kernel has finished and its writes are visible (a no-op otherwise).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int t = blockIdx.x; t < p.T; t += gridDim.x) {
    const size_t grow = static_cast<size_t>(p.row0) + static_cast<size_t>(t);
    const __nv_bfloat16* r0 = p.residual + grow * p.H;
    float r[VPT][8];
    float ss = 0.f;
    // all loads first
    uint4 u[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int vi = v * NT + tid;
      if (vi < nvec) {
        load_y8<SRC, MAXS>(p, t, vi << 3, r[v]);
        u[v] = *reinterpret_cast<const uint4*>(r0 + (vi << 3));
      }
    }
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int vi = v * NT + tid;
      if (vi < nvec) {
        float f[8];
        bf16x8_to_f32(u[v], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          r[v][j] += f[j];
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
      for (int w = 0; w < NT / 32; ++w) tot += warp_sums[w];
      row_total = tot;
    }
    __syncthreads();
    const float rstd = rsqrtf(row_total / static_cast<float>(p.H) + p.eps);
    __nv_bfloat16* rw = p.residual + grow * p.H;
    __nv_bfloat16* ow = p.out + (p.out_local ? static_cast<size_t>(t) : grow) * p.H;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int vi = v * NT + tid;
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

template <int SRC, int VPT, int NT, int MAXS>
static cudaError_t launch_k(const NormParams& p, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fln_add_rmsnorm_kernel<SRC, VPT, NT, MAXS>, p);
}

template <int SRC, int NT, int MAXS>
static cudaError_t launch_nt(const NormParams& p, int grid, cudaStream_t s) {
  const int nvec = p.H / 8;
  const int vpt = (nvec + NT - 1) / NT;
  if (vpt <= 1) return launch_k<SRC, 1, NT, MAXS>(p, grid, s);
  if (vpt <= 2) return launch_k<SRC, 2, NT, MAXS>(p, grid, s);
  if (vpt <= 4) return launch_k<SRC, 4, NT, MAXS>(p, grid, s);
  if (vpt <= 8) return launch_k<SRC, 8, NT, MAXS>(p, grid, s);
  if (vpt <= 16) return launch_k<SRC, 16, NT, MAXS>(p, grid, s);
  return cudaErrorInvalidValue;
}

// Few rows: each row is split over a cluster of CL CTAs (one slice of H/CL
// columns each, one 8-column vector per thread), so a row's loads come from
// CL SMs at once.  Each CTA writes its slice's sum of squares into every
// CTA of the cluster (distributed shared memory), one cluster barrier later
// every CTA adds the CL sums in rank order (the same float in all of them).
// Residual and gamma are read before waiting for the addend: no kernel that
// this one depends on programmatically writes them.
template <int SRC, int CL, int MAXS>
__global__ void __launch_bounds__(256) fln_add_rmsnorm_cluster_kernel(const NormParams p) {
  __shared__ float warp_sums[8];
  __shared__ float slice_ss[CL];
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  const int t = static_cast<int>(cluster_id_x());
  const int slice = p.H / CL;             // columns of this CTA
  const int nvec = slice >> 3;
  const int vi = tid;
  const bool active = vi < nvec;
  const int h = static_cast<int>(rank) * slice + (vi << 3);
  const size_t grow = static_cast<size_t>(p.row0) + static_cast<size_t>(t);
  uint4 u = make_uint4(0u, 0u, 0u, 0u);
  float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;
  if (active) {
    u = *reinterpret_cast<const uint4*>(p.residual + grow * p.H + h);
    g0 = __ldg(reinterpret_cast<const float4*>(p.gamma + h));
    g1 = __ldg(reinterpret_cast<const float4*>(p.gamma + h + 4));
  }
  // when launched as a programmatic dependent, wait for the producing kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float r[8];
  float ss = 0.f;
  if (active) {
    load_y8<SRC, MAXS>(p, t, h, r);
    float f[8];
    bf16x8_to_f32(u, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      r[j] += f[j];
      ss = fmaf(r[j], r[j], ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) warp_sums[tid >> 5] = ss;
  __syncthreads();
  if (tid < CL) {
    // thread k sends this slice's sum to CTA k
    float tot = 0.f;
    for (int w = 0; w < (blockDim.x + 31) / 32; ++w) tot += warp_sums[w];
    const uint32_t a = map_to_cta(smem_u32(&slice_ss[rank]), static_cast<uint32_t>(tid));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(tot) : "memory");
  }
  cluster_sync();  // all CL slice sums are in this CTA's shared memory; no remote access follows
  if (active) {
    float tot = 0.f;
#pragma unroll
    for (int k = 0; k < CL; ++k) tot += slice_ss[k];
    const float rstd = rsqrtf(tot / static_cast<float>(p.H) + p.eps);
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = r[j] * rstd * (p.norm_kind ? 1.0f + g[j] : g[j]);
    *reinterpret_cast<uint4*>(p.residual + grow * p.H + h) = f32x8_to_bf16(r);
    __stcs(reinterpret_cast<uint4*>(p.out + (p.out_local ? static_cast<size_t>(t) : grow) * p.H + h),
           f32x8_to_bf16(o));
  }
}

template <int SRC, int CL, int MAXS>
static cudaError_t launch_cluster(const NormParams& p, cudaStream_t s) {
  const int nvec = p.H / CL / 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.T * CL, 1, 1);
  cfg.blockDim = dim3(((nvec + 31) / 32) * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, fln_add_rmsnorm_cluster_kernel<SRC, CL, MAXS>, p);
}

// Block size: 512 threads when there are few rows (a row's loads spread over
// more threads, so more of them are in flight), 256 otherwise.
template <int SRC, int MAXS>
static cudaError_t launch_src(const NormParams& p, int grid, cudaStream_t s) {
  const bool wide = p.T <= 64 && p.H >= 8192;
  return wide ? launch_nt<SRC, 512, MAXS>(p, grid, s) : launch_nt<SRC, 256, MAXS>(p, grid, s);
}

cudaError_t launch_add_rmsnorm(NormSource src, const NormParams& p, int grid_cap, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  int grid = p.T;
  if (grid_cap > 0 && grid > grid_cap) grid = grid_cap;
  // few long rows: one 8-CTA cluster per row (slices of H/8 columns, at most
  // 256 vectors of 8 per CTA)
  if (p.T <= 64 && p.H % 64 == 0 && p.H / 64 <= 256 && p.H >= 2048 && grid_cap == 0) {
    switch (src) {
      case NORM_SRC_BF16: return launch_cluster<NORM_SRC_BF16, 8, 1>(p, stream);
      case NORM_SRC_F32: return launch_cluster<NORM_SRC_F32, 8, 1>(p, stream);
      case NORM_SRC_SPLITK:
        if (p.max_split + p.dyn_cpm <= 4) return launch_cluster<NORM_SRC_SPLITK, 8, 4>(p, stream);
        if (p.max_split + p.dyn_cpm <= 8) return launch_cluster<NORM_SRC_SPLITK, 8, 8>(p, stream);
        if (p.max_split + p.dyn_cpm <= 12) return launch_cluster<NORM_SRC_SPLITK, 8, 12>(p, stream);
        break;
    }
  }
  switch (src) {
    case NORM_SRC_BF16: return launch_src<NORM_SRC_BF16, 1>(p, grid, stream);
    case NORM_SRC_F32: return launch_src<NORM_SRC_F32, 1>(p, grid, stream);
    case NORM_SRC_SPLITK:
      if (p.max_split + p.dyn_cpm <= 4) return launch_src<NORM_SRC_SPLITK, 4>(p, grid, stream);
      if (p.max_split + p.dyn_cpm <= 8) return launch_src<NORM_SRC_SPLITK, 8>(p, grid, stream);
      if (p.max_split + p.dyn_cpm <= 16) return launch_src<NORM_SRC_SPLITK, 16>(p, grid, stream);
      return cudaErrorInvalidValue;
  }
  return cudaErrorInvalidValue;
}

}  // namespace fln
