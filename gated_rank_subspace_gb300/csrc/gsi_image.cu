// Image build: M = W V_k and the Gram matrix V_k^T V_k (one-off per map).
//
// "Gated Subspace Inference for Transformer Acceleration", §2.1: M = W V_k is
// the low-rank weight image that is precomputed and cached.  The Gram matrix
// is the library's own cached artefact: it lets the gate evaluate
// ||x - V_k g|| exactly for a basis that rounding has made slightly
// non-orthonormal.
//
// A plain shared-memory tiled contraction on the CUDA cores with float32
// accumulation, 64 x 64 output tiles, 16-deep k-steps and a 4 x 4 register
// block per thread.  Operands are addressed through (row, column) strides so
// the same kernel forms W V (both row-major) and V^T V (V read transposed).
// Each output is summed in one fixed order: bitwise reproducible.

#include "gsi_common.cuh"
#include "gsi_kernels.h"

namespace gsi {

constexpr int kTM = 64, kTN = 64, kTK = 16;

template <class EA, class EB>
__global__ void __launch_bounds__(256) contract_kernel(const void* A, int64_t sam, int64_t sak,
                                                       const void* B, int64_t sbk, int64_t sbn,
                                                       void* C, int c_bf16, int64_t ldc,
                                                       int64_t Md, int64_t Nd, int64_t Kd) {
  __shared__ float As[kTK][kTM + 4];
  __shared__ float Bs[kTK][kTN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int64_t m0 = int64_t(blockIdx.y) * kTM, n0 = int64_t(blockIdx.x) * kTN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  // Pick the fastest-varying index of each tile load so that consecutive
  // threads touch consecutive addresses.
  const bool a_k_fast = sak == 1;
  const bool b_n_fast = sbn == 1;
  for (int64_t k0 = 0; k0 < Kd; k0 += kTK) {
    for (int e = tid; e < kTM * kTK; e += 256) {
      const int mm = a_k_fast ? e / kTK : e % kTM;
      const int kk = a_k_fast ? e % kTK : e / kTM;
      const int64_t m = m0 + mm, kx = k0 + kk;
      As[kk][mm] = (m < Md && kx < Kd) ? EA::load1(A, m * sam + kx * sak) : 0.f;
    }
    for (int e = tid; e < kTN * kTK; e += 256) {
      const int nn = b_n_fast ? e % kTN : e / kTK;
      const int kk = b_n_fast ? e / kTN : e % kTK;
      const int64_t n = n0 + nn, kx = k0 + kk;
      Bs[kk][nn] = (n < Nd && kx < Kd) ? EB::load1(B, kx * sbk + n * sbn) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < Md && n < Nd) {
        if (c_bf16)
          BF16::store1(C, m * ldc + n, acc[i][j]);
        else
          F32::store1(C, m * ldc + n, acc[i][j]);
      }
    }
}

template <class EA, class EB = EA>
static cudaError_t contract(const void* A, int64_t sam, int64_t sak, const void* B, int64_t sbk,
                            int64_t sbn, void* C, int c_bf16, int64_t ldc, int64_t Md, int64_t Nd,
                            int64_t Kd, cudaStream_t s) {
  dim3 grid(unsigned(cdiv(Nd, kTN)), unsigned(cdiv(Md, kTM)));
  contract_kernel<EA, EB><<<grid, 256, 0, s>>>(A, sam, sak, B, sbk, sbn, C, c_bf16, ldc, Md, Nd, Kd);
  return cudaGetLastError();
}

// C (float32, Md x Nd, row stride ldc) = A (Md x Kd) B (Kd x Nd) through
// element strides; A of element type adt, B of bdt.
cudaError_t launch_contract(const void* A, gsi_dtype adt, int64_t sam, int64_t sak, const void* B, gsi_dtype bdt,
                            int64_t sbk, int64_t sbn, float* C, int64_t ldc, int64_t Md, int64_t Nd, int64_t Kd,
                            cudaStream_t s) {
  if (adt == GSI_BF16 && bdt == GSI_F32)
    return contract<BF16, F32>(A, sam, sak, B, sbk, sbn, C, 0, ldc, Md, Nd, Kd, s);
  if (adt == GSI_F32 && bdt == GSI_BF16)
    return contract<F32, BF16>(A, sam, sak, B, sbk, sbn, C, 0, ldc, Md, Nd, Kd, s);
  if (adt == GSI_BF16) return contract<BF16>(A, sam, sak, B, sbk, sbn, C, 0, ldc, Md, Nd, Kd, s);
  return contract<F32>(A, sam, sak, B, sbk, sbn, C, 0, ldc, Md, Nd, Kd, s);
}

cudaError_t launch_image(const void* W, const void* V, void* M, float* gram, int64_t d,
                         int64_t d_out, int64_t k, gsi_dtype dt, cudaStream_t s) {
  const int out_bf16 = dt == GSI_BF16;
  cudaError_t e;
  // M[o][j] = sum_i W[o][i] V[i][j]
  if (dt == GSI_BF16)
    e = contract<BF16>(W, d, 1, V, k, 1, M, out_bf16, k, d_out, k, d, s);
  else
    e = contract<F32>(W, d, 1, V, k, 1, M, out_bf16, k, d_out, k, d, s);
  if (e != cudaSuccess || !gram) return e;
  return launch_gram(V, gram, d, k, dt, s);
}

// Gram[a][b] = sum_i V[i][a] V[i][b], float32 FMA chains in one fixed order.
// The Gram matrix V_k^T V_k (k x k, float32) of a d x k basis: one 32 x 32
// tile of the output per CTA, so a k = 256 basis spreads over 64 CTAs (the
// 64 x 64 tiles of the general contraction gave it 16, ~0.7 ms at d = 4096);
// 32 rows of V staged at a time.  Every output is one float32 sum over the
// rows of V in row order -- the same sums, in the same order, as the general
// contraction.
constexpr int kGT = 32;

template <class E>
__global__ void __launch_bounds__(256) gram_kernel(const void* V, float* G, int64_t d, int64_t k) {
  __shared__ float A[kGT][kGT + 1];  // [row of V][column m0 + i]
  __shared__ float B[kGT][kGT + 1];  // [row of V][column n0 + j]
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int64_t m0 = int64_t(blockIdx.y) * kGT, n0 = int64_t(blockIdx.x) * kGT;
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  for (int64_t r0 = 0; r0 < d; r0 += kGT) {
    for (int e = tid; e < kGT * kGT; e += 256) {
      const int rr = e / kGT, cc = e % kGT;  // consecutive threads: consecutive columns of a row
      const int64_t r = r0 + rr;
      A[rr][cc] = (r < d && m0 + cc < k) ? E::load1(V, r * k + m0 + cc) : 0.f;
      B[rr][cc] = (r < d && n0 + cc < k) ? E::load1(V, r * k + n0 + cc) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int rr = 0; rr < kGT; ++rr) {
      const float a0 = A[rr][ty * 2], a1 = A[rr][ty * 2 + 1];
      const float b0 = B[rr][tx * 2], b1 = B[rr][tx * 2 + 1];
      acc[0][0] = fmaf(a0, b0, acc[0][0]);
      acc[0][1] = fmaf(a0, b1, acc[0][1]);
      acc[1][0] = fmaf(a1, b0, acc[1][0]);
      acc[1][1] = fmaf(a1, b1, acc[1][1]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int64_t m = m0 + ty * 2 + i, n = n0 + tx * 2 + j;
      if (m < k && n < k) G[m * k + n] = acc[i][j];
    }
}

cudaError_t launch_gram(const void* V, float* gram, int64_t d, int64_t k, gsi_dtype dt, cudaStream_t s) {
  const dim3 grid(unsigned(cdiv(k, kGT)), unsigned(cdiv(k, kGT)));
  if (dt == GSI_BF16)
    gram_kernel<BF16><<<grid, 256, 0, s>>>(V, gram, d, k);
  else
    gram_kernel<F32><<<grid, 256, 0, s>>>(V, gram, d, k);
  return cudaGetLastError();
}

}  // namespace gsi
