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
cudaError_t launch_gram(const void* V, float* gram, int64_t d, int64_t k, gsi_dtype dt, cudaStream_t s) {
  if (dt == GSI_BF16) return contract<BF16>(V, 1, k, V, k, 1, gram, 0, k, k, k, d, s);
  return contract<F32>(V, 1, k, V, k, 1, gram, 0, k, k, k, d, s);
}

}  // namespace gsi
