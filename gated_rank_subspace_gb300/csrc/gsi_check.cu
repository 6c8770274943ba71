// Explicit-residual check of the gate ("Gated Subspace Inference for
// Transformer Acceleration", §2.1 core decomposition: x = V_k g + r with
// g = V_k^T x; §2.2 gated residual step: rho = ||r|| / ||x||).
//
// The gate kernels never form the residual: they evaluate
// ||r||^2 = ||x||^2 - 2||g||^2 + g^T (V_k^T V_k) g from three sums, so that V_k
// is read once per call.  This pass forms r_t = x_t - V_k g_t itself, from the
// same projections g_t, with a second pass over V_k, and reports
//   rho_x[t] = ||r_t|| / ||x_t||     and     max_t |rho[t]^2 - rho_x[t]^2|
// over the tokens whose two values are finite.  It is a validation mode: the
// gated map does not depend on it.
//
// residual_partial_kernel: CTA (s, c) takes rows [s R, (s + 1) R) of V_k and
//   tokens [c TC, (c + 1) TC).  Warp w takes rows w, w + 8, ... of the slab;
//   for each row, lane l multiplies columns l, l + 32, ... of V_k with the
//   same columns of the TC projections, one butterfly reduces the TC dot
//   products, and the lane that holds token t's dot adds (x_ti - dot)^2 and
//   x_ti^2 to its sums.  The warps' sums are added in warp order:
//   part[s][t] = {sum of r_i^2, sum of x_i^2} over the slab's rows.
// residual_finish_kernel: one CTA; thread u takes tokens u, u + 256, ... and
//   adds their slabs' partials in slab order, in double; the largest deviation
//   is a block max.  Every sum has one fixed order: the results are bitwise
//   reproducible.

#include "gsi_common.cuh"
#include "gsi_kernels.h"

namespace gsi {

constexpr int kCheckThreads = 256;
constexpr int kCheckWarps = kCheckThreads / 32;
constexpr int kCheckTokens = 8;                  // TC
constexpr int kCheckRowsPerWarp = 8;
constexpr int kCheckRows = kCheckWarps * kCheckRowsPerWarp;  // R

template <class E>
__global__ void __launch_bounds__(kCheckThreads) residual_partial_kernel(const void* X, const void* V, const float* G,
                                                                         int64_t d, int k, int64_t T,
                                                                         float2* part) {
  extern __shared__ __align__(16) float gs[];  // [TC][k] projections, then [NW][TC] sums
  __shared__ float2 wsum[kCheckWarps][kCheckTokens];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t t0 = int64_t(blockIdx.y) * kCheckTokens;
  const int64_t i0 = int64_t(blockIdx.x) * kCheckRows;
  for (int e = tid; e < kCheckTokens * k; e += kCheckThreads) {
    const int64_t t = t0 + e / k;
    gs[e] = t < T ? G[t * k + e % k] : 0.f;
  }
  __syncthreads();
  // after the butterfly, lane l holds the dot product of token tl
  const int tl = row_of_lane<kCheckTokens>(lane);
  const bool owner = (lane & (32 / kCheckTokens - 1)) == 0 && t0 + tl < T;
  float r2 = 0.f, x2 = 0.f;
  for (int rr = 0; rr < kCheckRowsPerWarp; ++rr) {
    const int64_t i = i0 + warp + int64_t(rr) * kCheckWarps;
    if (i >= d) break;  // warp-uniform
    float dot[kCheckTokens];
#pragma unroll
    for (int t = 0; t < kCheckTokens; ++t) dot[t] = 0.f;
    for (int j = lane; j < k; j += 32) {
      const float v = E::load1(V, i * k + j);
#pragma unroll
      for (int t = 0; t < kCheckTokens; ++t) dot[t] = fmaf(v, gs[t * k + j], dot[t]);
    }
    const float s = warp_reduce_multi<kCheckTokens>(dot, lane);
    if (owner) {
      const float x = E::load1(X, (t0 + tl) * d + i);
      const float r = x - s;
      r2 = fmaf(r, r, r2);
      x2 = fmaf(x, x, x2);
    }
  }
  if (owner) wsum[warp][tl] = make_float2(r2, x2);
  __syncthreads();
  if (tid < kCheckTokens && t0 + tid < T) {
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int w = 0; w < kCheckWarps; ++w) {
      const bool has = i0 + w < d;  // warp w held at least one row
      a += has ? wsum[w][tid].x : 0.f;
      b += has ? wsum[w][tid].y : 0.f;
    }
    part[int64_t(blockIdx.x) * T + t0 + tid] = make_float2(a, b);
  }
}

__global__ void __launch_bounds__(kCheckThreads) residual_finish_kernel(const float2* part, int n_slabs, int64_t T,
                                                                        const float* rho, float* rho_x,
                                                                        float* max_dev) {
  __shared__ float red[kCheckWarps];
  float worst = 0.f;
  for (int64_t t = threadIdx.x; t < T; t += kCheckThreads) {
    double rr = 0.0, xx = 0.0;
    for (int s = 0; s < n_slabs; ++s) {
      const float2 p = part[int64_t(s) * T + t];
      rr += p.x;
      xx += p.y;
    }
    const float rx = xx == 0.0 ? 0.f : float(sqrt(rr / xx));
    rho_x[t] = rx;
    const float rg = rho[t];
    const float dev = fabsf(rg * rg - rx * rx);
    if (isfinite(dev)) worst = fmaxf(worst, dev);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = worst;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < kCheckWarps; ++w) m = fmaxf(m, red[w]);
    *max_dev = m;
  }
}

size_t residual_check_work_bytes(int64_t d, int64_t T) {
  return size_t((d + kCheckRows - 1) / kCheckRows) * size_t(T) * sizeof(float2);
}

cudaError_t launch_residual_check(const void* X, const void* V, const float* G, const float* rho, int64_t d, int k,
                                  int64_t T, gsi_dtype dt, float* rho_x, float* max_dev, void* work,
                                  cudaStream_t s) {
  const int n_slabs = int((d + kCheckRows - 1) / kCheckRows);
  const int64_t n_chunks = (T + kCheckTokens - 1) / kCheckTokens;
  if (n_chunks > 65535) return cudaErrorInvalidValue;
  float2* part = static_cast<float2*>(work);
  const dim3 grid{unsigned(n_slabs), unsigned(n_chunks), 1u};
  const size_t smem = size_t(kCheckTokens) * k * sizeof(float);
  if (dt == GSI_BF16)
    residual_partial_kernel<BF16><<<grid, kCheckThreads, smem, s>>>(X, V, G, d, k, T, part);
  else
    residual_partial_kernel<F32><<<grid, kCheckThreads, smem, s>>>(X, V, G, d, k, T, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  residual_finish_kernel<<<1, kCheckThreads, 0, s>>>(part, n_slabs, T, rho, rho_x, max_dev);
  return cudaGetLastError();
}

}  // namespace gsi
