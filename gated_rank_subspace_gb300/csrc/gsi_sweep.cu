// Threshold sweep: what each eps would cost and how far it would move the
// output ("Gated Subspace Inference for Transformer Acceleration", §2.2 gated
// residual step and its Theorem 4 bound; §4 static-projection control).
//
// path_norms_kernel: per token t, err_t = ||y_fast_t - y_slow_t|| and
//   ynorm_t = ||y_slow_t|| from the two candidate outputs (the fast path's
//   M g_t and the slow path's W x_t), one CTA per token.
// sweep_kernel: per threshold eps, one CTA: the slow tokens (!(rho < eps),
//   so ties and NaN go slow), the calls (blocks of tokens_per_call tokens)
//   that hold one and so read W, and the relative output error
//   sqrt(sum over fast tokens of err^2) / sqrt(sum of ynorm^2).
// Sums are accumulated in double and reduced in a fixed order: the results
// are bitwise reproducible.

#include "gsi_common.cuh"
#include "gsi_kernels.h"

namespace gsi {

constexpr int kSweepThreads = 256;

// Block sum in a fixed order (warp butterflies, then warp 0 over the warps).
__device__ __forceinline__ double block_sum(double v, double* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double s = 0.0;
  if (warp == 0) {
    s = lane < kSweepThreads / 32 ? red[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  }
  __syncthreads();
  return s;  // valid in warp 0
}

__global__ void __launch_bounds__(kSweepThreads) path_norms_kernel(const float* Yf, const float* Ys, int64_t d_out,
                                                                   float* err, float* ynorm) {
  __shared__ double red[kSweepThreads / 32];
  const int64_t t = blockIdx.x;
  const float* f = Yf + t * d_out;
  const float* s = Ys + t * d_out;
  double e2 = 0.0, y2 = 0.0;
  for (int64_t i = threadIdx.x; i < d_out; i += kSweepThreads) {
    const double a = f[i], b = s[i];
    e2 += (a - b) * (a - b);
    y2 += b * b;
  }
  e2 = block_sum(e2, red);
  y2 = block_sum(y2, red);
  if (threadIdx.x == 0) {
    err[t] = float(sqrt(e2));
    ynorm[t] = float(sqrt(y2));
  }
}

__global__ void __launch_bounds__(kSweepThreads) sweep_kernel(const float* rho, const float* err, const float* ynorm,
                                                              int64_t T, const float* eps, int64_t tokens_per_call,
                                                              int32_t* n_slow, int32_t* n_slow_calls,
                                                              float* rel_err) {
  __shared__ double red[kSweepThreads / 32];
  const float e = eps[blockIdx.x];
  double ns = 0.0, e2 = 0.0, y2 = 0.0, nc = 0.0;
  for (int64_t t = threadIdx.x; t < T; t += kSweepThreads) {
    const bool slow = !(rho[t] < e);
    const double yn = ynorm[t];
    y2 += yn * yn;
    if (slow) {
      ns += 1.0;
    } else {
      const double er = err[t];
      e2 += er * er;
    }
  }
  const int64_t n_calls = (T + tokens_per_call - 1) / tokens_per_call;
  for (int64_t c = threadIdx.x; c < n_calls; c += kSweepThreads) {
    const int64_t t1 = (c + 1) * tokens_per_call < T ? (c + 1) * tokens_per_call : T;
    bool any = false;
    for (int64_t t = c * tokens_per_call; t < t1; ++t) any = any || !(rho[t] < e);
    nc += any ? 1.0 : 0.0;
  }
  ns = block_sum(ns, red);
  nc = block_sum(nc, red);
  e2 = block_sum(e2, red);
  y2 = block_sum(y2, red);
  if (threadIdx.x == 0) {
    n_slow[blockIdx.x] = int32_t(ns);
    n_slow_calls[blockIdx.x] = int32_t(nc);
    rel_err[blockIdx.x] = y2 > 0.0 ? float(sqrt(e2 / y2)) : 0.f;
  }
}

cudaError_t launch_path_norms(const float* Yf, const float* Ys, int64_t T, int64_t d_out, float* err, float* ynorm,
                              cudaStream_t s) {
  path_norms_kernel<<<unsigned(T), kSweepThreads, 0, s>>>(Yf, Ys, d_out, err, ynorm);
  return cudaGetLastError();
}

cudaError_t launch_sweep(const float* rho, const float* err, const float* ynorm, int64_t T, const float* eps,
                         int64_t n_eps, int64_t tokens_per_call, int32_t* n_slow, int32_t* n_slow_calls,
                         float* rel_err, cudaStream_t s) {
  sweep_kernel<<<unsigned(n_eps), kSweepThreads, 0, s>>>(rho, err, ynorm, T, eps, tokens_per_call, n_slow,
                                                         n_slow_calls, rel_err);
  return cudaGetLastError();
}

}  // namespace gsi
