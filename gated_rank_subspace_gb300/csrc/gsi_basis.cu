// Basis construction: DGKS Gram-Schmidt, subspace coherence, export.
//
// "Gated Subspace Inference for Transformer Acceleration", §2.3 depth
// cascade and calibration: a layer's basis starts from the previous layer's
// and is corrected by rank-1 updates kept orthogonal by DGKS
// re-orthogonalisation.  The correction step of the library is
// V <- orthonormalise((X^T X) V) for a calibration block X; this file holds
// the orthonormalisation (classical Gram-Schmidt column by column, projected
// a second time when the norm after a projection falls below 1/sqrt(2) of the
// norm before it -- the Daniel-Gragg-Kaufman-Stewart test), the coherence of
// two bases and the export of a basis to a map's row-major layout.
//
// dgks_kernel: one cluster of 8 CTAs.  The basis is held transposed, Qt
// (k x d float32, row i = basis vector i), in global memory (it fits in L2);
// CTA r owns columns [r * rs, (r + 1) * rs) of Qt, i.e. the same slice of
// every basis vector, so its global reads and writes touch only its own
// slice.  Per basis vector j: the dot products with vectors 0 .. j-1 and the
// squared norms are summed over the CTA's slice, pushed into every CTA's
// shared memory and added in rank order after a cluster barrier, so every CTA
// holds the same bits and takes the same re-orthogonalisation decision.
// Cluster barriers have no timeout, and every CTA reaches each of them.

#include "gsi_common.cuh"
#include "gsi_kernels.h"

namespace gsi {

constexpr int kBasisCS = 8;
constexpr int kBasisThreads = 512;
constexpr int kBasisWarps = kBasisThreads / 32;
constexpr float kDgksEta = 0.70710678118654752f;  // 1 / sqrt(2)

__global__ void __cluster_dims__(kBasisCS, 1, 1) __launch_bounds__(kBasisThreads, 1)
    dgks_kernel(float* Qt, int64_t d, int k, int32_t* n_reorth) {
  // shared: h_in[CS][k] pushed partial dot products, n_in[CS] partial norms,
  // h[k] the summed dot products, hp[k] this CTA's partials
  extern __shared__ __align__(16) float sm[];
  float* h_in = sm;
  float* n_in = h_in + kBasisCS * k;
  float* h = n_in + kBasisCS;
  float* hp = h + k;
  float* red = hp + k;  // [kBasisWarps]
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = int(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t rs = (d + kBasisCS - 1) / kBasisCS;
  const int64_t r0 = int64_t(rank) * rs;
  const int64_t nr = r0 >= d ? 0 : (d - r0 < rs ? d - r0 : rs);
  int reorth = 0;

  // sum of squares of the slice of vector j, summed over the cluster (same
  // bits in every CTA)
  auto cluster_norm2 = [&](const float* z) -> float {
    float s = 0.f;
    for (int64_t r = tid; r < nr; r += kBasisThreads) s = fmaf(z[r], z[r], s);
    s = warp_sum(s);
    if (lane == 0) red[warp] = s;
    __syncthreads();
    if (tid < kBasisCS) {
      float t = 0.f;
      for (int w = 0; w < kBasisWarps; ++w) t += red[w];
      cluster.map_shared_rank(n_in, tid)[rank] = t;
    }
    cluster.sync();
    float n2 = 0.f;
    for (int q = 0; q < kBasisCS; ++q) n2 += n_in[q];
    cluster.sync();  // n_in is read before the next push
    return n2;
  };

  for (int j = 0; j < k; ++j) {
    float* z = Qt + int64_t(j) * d + r0;  // this CTA's slice of vector j
    const float before = cluster_norm2(z);
    float after = before;
    for (int pass = 0; pass < 2 && j > 0; ++pass) {
      // h_i = <q_i, z> for i < j: warp w takes i = w, w + 16, ...
      for (int i = warp; i < j; i += kBasisWarps) {
        const float* q = Qt + int64_t(i) * d + r0;
        float s = 0.f;
        for (int64_t r = lane; r < nr; r += 32) s = fmaf(q[r], z[r], s);
        s = warp_sum(s);
        if (lane == 0) hp[i] = s;
      }
      __syncthreads();
      for (int e = tid; e < kBasisCS * j; e += kBasisThreads) {
        const int q = e / j, i = e - (e / j) * j;
        cluster.map_shared_rank(h_in, q)[rank * k + i] = hp[i];
      }
      cluster.sync();
      for (int i = tid; i < j; i += kBasisThreads) {
        float s = 0.f;
        for (int q = 0; q < kBasisCS; ++q) s += h_in[q * k + i];
        h[i] = s;
      }
      __syncthreads();
      // z <- z - sum_i h_i q_i (each thread its own entries of the slice)
      for (int64_t r = tid; r < nr; r += kBasisThreads) {
        float v = z[r];
        for (int i = 0; i < j; ++i) v = fmaf(-h[i], Qt[int64_t(i) * d + r0 + r], v);
        z[r] = v;
      }
      __syncthreads();
      after = cluster_norm2(z);
      if (after >= kDgksEta * kDgksEta * before) break;  // ||z|| >= eta * ||a||
      if (pass == 0) ++reorth;
    }
    const float inv = 1.f / sqrtf(after);
    for (int64_t r = tid; r < nr; r += kBasisThreads) z[r] *= inv;
    __syncthreads();
  }
  if (n_reorth && rank == 0 && tid == 0) *n_reorth = reorth;
}

// out = scale * sum of S[i]^2 over n entries (one CTA, fixed order, double).
__global__ void __launch_bounds__(256) sumsq_kernel(const float* S, int64_t n, float scale, float* out) {
  __shared__ double red[8];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += 256) s += double(S[i]) * double(S[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < 8; ++w) t += red[w];
    *out = float(t * double(scale));
  }
}

// V (d x k, row-major, dtype) = Qt^T, rounded to nearest even for bf16;
// 32 x 32 tiles through shared memory.
template <class E>
__global__ void __launch_bounds__(256) transpose_cast_kernel(const float* Qt, int64_t k, int64_t d, void* V) {
  __shared__ float tile[32][33];
  const int64_t i0 = int64_t(blockIdx.y) * 32, r0 = int64_t(blockIdx.x) * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int yy = ty; yy < 32; yy += 8) {
    const int64_t i = i0 + yy, r = r0 + tx;
    tile[yy][tx] = (i < k && r < d) ? Qt[i * d + r] : 0.f;
  }
  __syncthreads();
  for (int yy = ty; yy < 32; yy += 8) {
    const int64_t r = r0 + yy, i = i0 + tx;
    if (r < d && i < k) E::store1(V, r * k + i, tile[tx][yy]);
  }
}

cudaError_t launch_dgks(float* Qt, int64_t d, int k, int32_t* n_reorth, cudaStream_t s) {
  const size_t smem = (size_t(kBasisCS) * k + kBasisCS + 2 * size_t(k) + kBasisWarps) * sizeof(float);
  cudaError_t e = set_kernel_smem(dgks_kernel, smem);
  if (e != cudaSuccess) return e;
  dgks_kernel<<<kBasisCS, kBasisThreads, smem, s>>>(Qt, d, k, n_reorth);
  return cudaGetLastError();
}

cudaError_t launch_sumsq(const float* S, int64_t n, float scale, float* out, cudaStream_t s) {
  sumsq_kernel<<<1, 256, 0, s>>>(S, n, scale, out);
  return cudaGetLastError();
}

cudaError_t launch_transpose_cast(const float* Qt, int64_t k, int64_t d, void* V, gsi_dtype dt, cudaStream_t s) {
  dim3 grid(unsigned((d + 31) / 32), unsigned((k + 31) / 32));
  if (dt == GSI_BF16)
    transpose_cast_kernel<BF16><<<grid, 256, 0, s>>>(Qt, k, d, V);
  else
    transpose_cast_kernel<F32><<<grid, 256, 0, s>>>(Qt, k, d, V);
  return cudaGetLastError();
}

}  // namespace gsi
