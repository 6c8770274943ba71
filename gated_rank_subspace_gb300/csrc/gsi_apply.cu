// Apply kernel: the fast path y = M g and the slow path y = W x in one launch.
//
// "Gated Subspace Inference for Transformer Acceleration", §2.2: fast tokens
// (rho < eps) read only the cached image M (d_out x k); slow tokens read the
// full W (d_out x d).  The gate's decision stays on the device: this kernel
// reads the fast / slow counts and the stable index lists the gate kernel
// wrote, so the host never waits for the flags.
//
// Work is split into units of about 8 KB of weights, each handled by one
// warp: a fast unit is 16 / vplm rows of M, a slow unit one or more rows of W.
// Fast units come first, then slow units; the persistent grid's warps stride
// over them, so a call with both kinds of tokens streams M and W at once and
// a call with one kind streams only that matrix.  Weights are read with
// 16-byte non-allocating loads, each row once per block of tokens; the
// projections g of fast tokens and the slow tokens' x are staged in shared
// memory when they fit.  Row sums use warp shuffles (a butterfly that reduces
// 16 rows in 16 shuffles for the fast path).  Fixed summation order:
// results are bitwise reproducible.

#include "gsi_common.cuh"
#include "gsi_plan.h"
#include "gsi_kernels.h"

namespace gsi {

template <class E, int VPLM>
__device__ __forceinline__ void fast_unit(const ApplyArgs& a, int64_t u, int n_fast, int ngs,
                                          const float* gst, int lane) {
  constexpr int RM = 16 / VPLM;
  constexpr int PV = E::kPerVec;
  const int k = a.k;
  const int nvm = k * E::kBytes / 16;
  const int64_t row0 = u * RM;
  const char* mbase = reinterpret_cast<const char*>(a.M);
  uint4 mv[RM][VPLM];
#pragma unroll
  for (int r = 0; r < RM; ++r)
#pragma unroll
    for (int j = 0; j < VPLM; ++j) {
      const int vv = lane + 32 * j;
      const int64_t row = row0 + r;
      mv[r][j] = (row < a.d_out && vv < nvm)
                     ? ld_weight_v4(mbase + row * k * E::kBytes + int64_t(vv) * 16)
                     : make_uint4(0u, 0u, 0u, 0u);
    }
  for (int f = 0; f < n_fast; ++f) {
    const int tok = __ldcg(&a.idx[f]);
    float gv[VPLM][PV];
#pragma unroll
    for (int j = 0; j < VPLM; ++j) {
      const int vv = lane + 32 * j;
      if (vv < nvm) {
        const float* src = f < ngs ? gst + int64_t(f) * k + vv * PV : nullptr;
#pragma unroll
        for (int e4 = 0; e4 < PV / 4; ++e4) {
          float4 g4 = src ? reinterpret_cast<const float4*>(src)[e4]
                          : __ldcg(reinterpret_cast<const float4*>(a.G + int64_t(tok) * k + vv * PV) + e4);
          gv[j][e4 * 4 + 0] = g4.x;
          gv[j][e4 * 4 + 1] = g4.y;
          gv[j][e4 * 4 + 2] = g4.z;
          gv[j][e4 * 4 + 3] = g4.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < PV; ++e) gv[j][e] = 0.f;
      }
    }
    float part[RM];
#pragma unroll
    for (int r = 0; r < RM; ++r) {
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < VPLM; ++j) {
        float w[PV];
        E::unpack(mv[r][j], w);
#pragma unroll
        for (int e = 0; e < PV; ++e) s = fmaf(w[e], gv[j][e], s);
      }
      part[r] = s;
    }
    const float s = warp_reduce_multi<RM>(part, lane);
    const int r = row_of_lane<RM>(lane);
    if ((lane & (32 / RM - 1)) == 0 && row0 + r < a.d_out)
      a.Y[int64_t(tok) * a.d_out + row0 + r] = s;
  }
}

template <class E>
__device__ __forceinline__ void slow_unit(const ApplyArgs& a, int64_t u, int n_slow, int nxs,
                                          const unsigned char* xst, int lane) {
  constexpr int PV = E::kPerVec;
  constexpr int CH = 8;   // 16-byte vectors per lane in flight per chunk
  constexpr int TB = 4;   // tokens per pass over a row
  const int64_t nvw = a.d * E::kBytes / 16;
  const int64_t xrow_b = a.d * E::kBytes;
  for (int rr = 0; rr < a.rows_slow; ++rr) {
    const int64_t row = u * a.rows_slow + rr;
    if (row >= a.d_out) return;
    const char* wrow = reinterpret_cast<const char*>(a.W) + row * xrow_b;
    for (int s0 = 0; s0 < n_slow; s0 += TB) {
      const int tb = min(TB, n_slow - s0);
      int tok[TB];
#pragma unroll
      for (int i = 0; i < TB; ++i) tok[i] = i < tb ? __ldcg(&a.idx[a.T + s0 + i]) : 0;
      float acc[TB];
#pragma unroll
      for (int i = 0; i < TB; ++i) acc[i] = 0.f;
      for (int64_t c0 = 0; c0 < nvw; c0 += 32 * CH) {
        uint4 wv[CH];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const int64_t vv = c0 + lane + 32 * j;
          wv[j] = vv < nvw ? ld_weight_v4(wrow + vv * 16) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const int64_t vv = c0 + lane + 32 * j;
          if (vv < nvw) {
            float w[PV];
            E::unpack(wv[j], w);
#pragma unroll
            for (int i = 0; i < TB; ++i) {
              if (i < tb) {
                const int si = s0 + i;
                const uint4 xv =
                    si < nxs ? reinterpret_cast<const uint4*>(xst + int64_t(si) * xrow_b)[vv]
                             : ld_cg_v4(reinterpret_cast<const char*>(a.X) + int64_t(tok[i]) * xrow_b + vv * 16);
                float xf[PV];
                E::unpack(xv, xf);
#pragma unroll
                for (int e = 0; e < PV; ++e) acc[i] = fmaf(w[e], xf[e], acc[i]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < TB; ++i) {
        const float s = warp_sum(acc[i]);
        if (i < tb && lane == 0) a.Y[int64_t(tok[i]) * a.d_out + row] = s;
      }
    }
  }
}

template <class E, int VPLM>
__global__ void __launch_bounds__(kApplyThreads) apply_kernel(ApplyArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* xst = smem_raw;                                  // [nxs][d] raw elements
  float* gst = reinterpret_cast<float*>(smem_raw + kApplyXStage);  // [ngs][k]
  pdl_launch_dependents();
  pdl_wait();
  const int n_fast = __ldcg(&a.ctrl->counts[0]);
  const int n_slow = __ldcg(&a.ctrl->counts[1]);
  const int nxs = min(n_slow, a.x_stage_max);
  const int ngs = min(n_fast, a.g_stage_max);
  const int64_t xrow_v = a.d * E::kBytes / 16;
  for (int64_t e = threadIdx.x; e < int64_t(nxs) * xrow_v; e += blockDim.x) {
    const int j = int(e / xrow_v);
    const int64_t vv = e - int64_t(j) * xrow_v;
    const int tok = __ldcg(&a.idx[a.T + j]);
    reinterpret_cast<uint4*>(xst)[e] =
        ld_cg_v4(reinterpret_cast<const char*>(a.X) + int64_t(tok) * a.d * E::kBytes + vv * 16);
  }
  const int kv4 = a.k / 4;
  for (int e = threadIdx.x; e < ngs * kv4; e += blockDim.x) {
    const int j = e / kv4, vv = e - (e / kv4) * kv4;
    const int tok = __ldcg(&a.idx[j]);
    reinterpret_cast<float4*>(gst)[e] = __ldcg(reinterpret_cast<const float4*>(a.G + int64_t(tok) * a.k) + vv);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t uf = n_fast > 0 ? a.fast_units : 0;
  const int64_t us = n_slow > 0 ? a.slow_units : 0;
  const int64_t wpb = blockDim.x >> 5;
  const int64_t nwarps = int64_t(gridDim.x) * wpb;
  for (int64_t u = int64_t(blockIdx.x) * wpb + warp; u < uf + us; u += nwarps) {
    if (u < uf)
      fast_unit<E, VPLM>(a, u, n_fast, ngs, gst, lane);
    else
      slow_unit<E>(a, u - uf, n_slow, nxs, xst, lane);
  }
}

template <class E, int VPLM>
static cudaError_t launch_apply_t(const ApplyArgs& a, const ApplyPlan& p, int nsm, cudaStream_t s,
                                  bool pdl) {
  auto kern = apply_kernel<E, VPLM>;
  // One persistent wave: as many CTAs as fit on the device at once.
  static int per_sm = 0;
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(p.smem));
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kApplyThreads, p.smem);
    if (e != cudaSuccess) return e;
    per_sm = n > 0 ? n : 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(nsm * per_sm));
  cfg.blockDim = dim3(kApplyThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <class E>
static cudaError_t launch_apply_e(const ApplyArgs& a, const ApplyPlan& p, int nsm, cudaStream_t s,
                                  bool pdl) {
  switch (p.vplm) {
    case 1: return launch_apply_t<E, 1>(a, p, nsm, s, pdl);
    case 2: return launch_apply_t<E, 2>(a, p, nsm, s, pdl);
    default: return launch_apply_t<E, 4>(a, p, nsm, s, pdl);
  }
}

cudaError_t launch_apply(const ApplyArgs& a, const ApplyPlan& p, gsi_dtype dt, int nsm,
                         cudaStream_t s, bool pdl) {
  return dt == GSI_BF16 ? launch_apply_e<BF16>(a, p, nsm, s, pdl)
                        : launch_apply_e<F32>(a, p, nsm, s, pdl);
}

}  // namespace gsi
