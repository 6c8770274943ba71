// Gate kernel: projection, norms, residual ratio, per-token flag, compaction.
//
// "Gated Subspace Inference for Transformer Acceleration", §2.1 (g = V_k^T x,
// r = x - V_k g) and §2.2 (rho = ||r|| / ||x||, slow when rho >= eps).
//
// Layout of the work.  V (d x k, row-major) is cut into slabs of rs
// consecutive rows, one slab per CTA, so every CTA streams one contiguous
// block of V with 16-byte loads.  A CTA computes its slab's partial
// projections sum_i x_t[i] V[i, :] for all tokens plus the partial ||x_t||^2.
// The 8 CTAs of a thread-block cluster add their partials through
// distributed shared memory (fixed rank order), so each cluster writes one
// partial per token to global memory.  The last cluster to finish (an atomic
// ticket) finalises: it adds the cluster partials in cluster order, forms
//   ||x - V g||^2 = ||x||^2 - 2 ||g||^2 + g^T (V^T V) g
// (exact for any basis, so a bf16-rounded V needs no re-orthonormalisation
// and no second pass over V), then rho, the flag, and the stable fast / slow
// index lists.  Every sum runs in a fixed order: results are bitwise
// reproducible run to run, and no float atomics are used.
//
// Before waiting on the previous kernel of the stream (programmatic dependent
// launch) the CTA already holds its V slab in registers and has asked L2 for
// its share of the image M, so weight traffic overlaps the previous kernel.

#include "gsi_common.cuh"
#include "gsi_plan.h"
#include "gsi_kernels.h"

namespace gsi {

// One warp: stable compaction of T flags into fast / slow index lists
// (fast list at idx[0..), slow list at idx[T..)) and their counts.
__device__ void compact_warp(const uint8_t* flags, int T, int32_t* idx, int32_t* counts,
                             int lane) {
  int nf = 0, ns = 0;
  for (int base = 0; base < T; base += 32) {
    const int t = base + lane;
    const bool valid = t < T;
    const bool slow = valid && ld_cg_u8(flags + t) != 0;
    const unsigned ms = __ballot_sync(0xffffffffu, slow);
    const unsigned mf = __ballot_sync(0xffffffffu, valid && !slow);
    const unsigned lt = (1u << lane) - 1u;
    if (valid && idx) {
      if (slow)
        idx[T + ns + __popc(ms & lt)] = t;
      else
        idx[nf + __popc(mf & lt)] = t;
    }
    nf += __popc(mf);
    ns += __popc(ms);
  }
  if (lane == 0 && counts) {
    counts[0] = nf;
    counts[1] = ns;
  }
}

__global__ void __launch_bounds__(32) compact_kernel(const uint8_t* flags, int T, int32_t* idx,
                                                     int32_t* counts) {
  compact_warp(flags, T, idx, counts, threadIdx.x);
}

template <class E, int TC>
__global__ void __cluster_dims__(kClusterSize, 1, 1) __launch_bounds__(kGateThreads)
    gate_kernel(GateArgs a) {
  extern __shared__ __align__(16) float smem[];
  __shared__ int s_last;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = int(cluster.block_rank());
  const int cid = int(blockIdx.x) / kClusterSize;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k, rs = a.rs, nv = a.nv, nrg = a.nrg, T = a.T, ks = a.ks;
  const int64_t d = a.d;
  const int64_t r0 = int64_t(blockIdx.x) * rs;
  const int64_t rows_left = d - r0;
  const int rows = rows_left <= 0 ? 0 : (rows_left < rs ? int(rows_left) : rs);
  constexpr int PV = E::kPerVec;

  // ---- prologue: read-only weights only (may overlap the previous kernel)
  pdl_launch_dependents();
  if (a.gram_share && tid == 32) {
    // The finalising cluster reads the whole Gram: stage it in L2 now.
    const uint64_t off = uint64_t(blockIdx.x) * a.gram_share;
    const uint64_t total = uint64_t(k) * k * 4;
    if (off < total) {
      const uint64_t rem = total - off;
      prefetch_l2(reinterpret_cast<const char*>(a.gram) + off, uint32_t(rem < a.gram_share ? rem : a.gram_share));
    }
  }
  if (a.pf_share && tid == 0) {
    const uint64_t off = uint64_t(blockIdx.x) * a.pf_share;
    if (off < a.pf_total) {
      const uint64_t rem = a.pf_total - off;
      const uint64_t n = rem < a.pf_share ? rem : a.pf_share;
      prefetch_l2(a.pf_base + off, uint32_t(n));
    }
  }
  const int rg = tid / nv, v = tid - (tid / nv) * nv;
  const bool active = rg < nrg;
  uint4 vreg[kGateMaxRowsPerThread];
#pragma unroll
  for (int j = 0; j < kGateMaxRowsPerThread; ++j) {
    const int i = rg + j * nrg;
    vreg[j] = (active && i < rows)
                  ? ld_weight_v4(reinterpret_cast<const char*>(a.V) +
                                 ((r0 + i) * k * E::kBytes) + v * 16)
                  : make_uint4(0u, 0u, 0u, 0u);
  }
  // ---- tokens may come from the previous kernel: wait for it
  pdl_wait();

  float* xs = smem;                     // [TC][rs]
  float* red = xs + TC * rs;            // [nrg][TC][k]
  float* pg = red + nrg * TC * k;       // [TC][k]
  float* px = pg + TC * k;              // [TC]
  const int c0 = rank * ks;
  const int c1 = min(k, c0 + ks);

  for (int t0 = 0; t0 < T; t0 += TC) {
    const int tc = min(TC, T - t0);
    for (int e = tid; e < TC * rs; e += kGateThreads) {
      const int t = e / rs, i = e - (e / rs) * rs;
      xs[e] = (t < tc && i < rows) ? E::load1_cg(a.X, int64_t(t0 + t) * d + r0 + i) : 0.f;
    }
    __syncthreads();
    if (warp < TC) {
      float s = 0.f;
      for (int i = lane; i < rs; i += 32) {
        const float xv = xs[warp * rs + i];
        s += xv * xv;
      }
      s = warp_sum(s);
      if (lane == 0) px[warp] = s;
    }
    if (active) {
      float acc[TC][PV];
#pragma unroll
      for (int t = 0; t < TC; ++t)
#pragma unroll
        for (int e = 0; e < PV; ++e) acc[t][e] = 0.f;
#pragma unroll
      for (int j = 0; j < kGateMaxRowsPerThread; ++j) {
        const int i = rg + j * nrg;
        if (i < rows) {
          float w[PV];
          E::unpack(vreg[j], w);
#pragma unroll
          for (int t = 0; t < TC; ++t) {
            const float xv = xs[t * rs + i];
#pragma unroll
            for (int e = 0; e < PV; ++e) acc[t][e] = fmaf(xv, w[e], acc[t][e]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TC; ++t)
#pragma unroll
        for (int e = 0; e < PV; ++e) red[(rg * TC + t) * k + v * PV + e] = acc[t][e];
    }
    __syncthreads();
    for (int e = tid; e < TC * k; e += kGateThreads) {
      float s = 0.f;
      for (int g = 0; g < nrg; ++g) s += red[g * TC * k + e];
      pg[e] = s;
    }
    cluster.sync();
    // cluster reduction: this CTA owns columns [c0, c1) of every token
    for (int e = tid; e < TC * ks; e += kGateThreads) {
      const int t = e / ks, col = c0 + (e - (e / ks) * ks);
      if (t < tc && col < c1) {
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < kClusterSize; ++q) s += cluster.map_shared_rank(pg, q)[t * k + col];
        a.part_g[(int64_t(cid) * T + t0 + t) * k + col] = s;
      }
    }
    if (rank == 0 && tid < tc) {
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < kClusterSize; ++q) s += cluster.map_shared_rank(px, q)[tid];
      a.part_x[int64_t(cid) * T + t0 + tid] = s;
    }
    cluster.sync();
  }

  // ---- arrival ticket: the last cluster finalises
  __threadfence();
  cluster.sync();
  if (rank == 0 && tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&a.ctrl->ticket, 1u);
    const int last = old == unsigned(a.n_clusters - 1);
    __threadfence();
#pragma unroll
    for (int q = 0; q < kClusterSize; ++q) *cluster.map_shared_rank(&s_last, q) = last;
  }
  cluster.sync();
  if (!s_last) return;
  __threadfence();

  float* gsl = red;                            // [TC][ks]   this CTA's slice of g
  float* gfull = gsl + ((TC * ks + 3) & ~3);   // [TC][k]    the whole g (16-byte aligned)
  float* qw = gfull + TC * k;                  // [8][TC]    per-warp g^T Gram g partials
  float* nw = qw + 8 * TC;                     // [8][TC]    per-warp ||g||^2 partials
  float* qc = nw + 8 * TC;                     // [TC]       per-CTA partials
  float* nc = qc + TC;                         // [TC]
  float* nx2 = nc + TC;                        // [TC]       ||x||^2 (rank 0)
  const int nclu = a.n_clusters;
  const int64_t cstride = int64_t(T) * k;      // distance between clusters' partials

  // Sums over the clusters' partials are split over groups of `grp` adjacent
  // lanes (lane g of a group adds clusters g, g + grp, ...), so every thread
  // has its loads in flight together; the group then combines in a fixed
  // butterfly order (bitwise reproducible).
  const int ne = TC * ks;
  const int grp = kGateThreads / ne >= 8 ? 8 : kGateThreads / ne >= 4 ? 4 : kGateThreads / ne >= 2 ? 2 : 1;

  for (int t0 = 0; t0 < T; t0 += TC) {
    const int tc = min(TC, T - t0);
    for (int base = 0; base < ne * grp; base += kGateThreads) {
      const int id = base + tid;
      const int e = id / grp, g = id - (id / grp) * grp;
      const int t = e / ks, col = c0 + (e - (e / ks) * ks);
      const bool valid = e < ne && t < tc && col < c1;
      float s = 0.f;
      if (valid) {
        const float* src = a.part_g + int64_t(t0 + t) * k + col;
        int cl = g;
        for (; cl + 3 * grp < nclu; cl += 4 * grp) {
          const float v0 = __ldcg(src + cl * cstride), v1 = __ldcg(src + (cl + grp) * cstride);
          const float v2 = __ldcg(src + (cl + 2 * grp) * cstride), v3 = __ldcg(src + (cl + 3 * grp) * cstride);
          s += v0;
          s += v1;
          s += v2;
          s += v3;
        }
        for (; cl < nclu; cl += grp) s += __ldcg(src + cl * cstride);
      }
      for (int o = 1; o < grp; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (g == 0 && e < ne) {
        if (valid) a.G[int64_t(t0 + t) * k + col] = s;
        gsl[e] = valid ? s : 0.f;
      }
    }
    if (rank == 0 && warp == 0) {
      // ||x||^2: token (lane / 4) summed over clusters by 4 lanes
      const int t = lane >> 2, g = lane & 3;
      float s = 0.f;
      if (t < tc)
        for (int cl = g; cl < nclu; cl += 4) s += __ldcg(&a.part_x[int64_t(cl) * T + t0 + t]);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (g == 0 && t < TC) nx2[t] = s;
    }
    cluster.sync();
    for (int e = tid; e < TC * k; e += kGateThreads) {
      const int t = e / k, col = e - (e / k) * k;
      const int q = col / ks;
      gfull[e] = cluster.map_shared_rank(gsl, q)[t * ks + (col - q * ks)];
    }
    __syncthreads();
    // g^T Gram g and ||g||^2 over this CTA's Gram rows [c0, c1): the slice is
    // read as 16-byte vectors, eight per thread in flight at once.
    float qa[TC], na[TC];
#pragma unroll
    for (int t = 0; t < TC; ++t) qa[t] = na[t] = 0.f;
    for (int i = c0 + tid; i < c1; i += kGateThreads) {
#pragma unroll
      for (int t = 0; t < TC; ++t) na[t] = fmaf(gfull[t * k + i], gfull[t * k + i], na[t]);
    }
    if (a.gram && c1 > c0) {
      const int k4 = k >> 2;
      const int nvec = (c1 - c0) * k4;
      for (int v0 = 0; v0 < nvec; v0 += 8 * kGateThreads) {
        float4 gv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * kGateThreads + tid;
          gv[u] = v < nvec ? __ldg(reinterpret_cast<const float4*>(a.gram + int64_t(c0 + v / k4) * k) + (v % k4))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * kGateThreads + tid;
          if (v < nvec) {
            const int i = c0 + v / k4, j = 4 * (v % k4);
#pragma unroll
            for (int t = 0; t < TC; ++t) {
              const float4 gj = *reinterpret_cast<const float4*>(gfull + t * k + j);
              float h = gv[u].x * gj.x;
              h = fmaf(gv[u].y, gj.y, h);
              h = fmaf(gv[u].z, gj.z, h);
              h = fmaf(gv[u].w, gj.w, h);
              qa[t] = fmaf(gfull[t * k + i], h, qa[t]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TC; ++t) {
      const float q = warp_sum(qa[t]);
      const float n = warp_sum(na[t]);
      if (lane == 0) {
        qw[warp * TC + t] = q;
        nw[warp * TC + t] = n;
      }
    }
    __syncthreads();
    if (tid < TC) {
      float q = 0.f, n = 0.f;
      for (int w = 0; w < kGateThreads / 32; ++w) {
        q += qw[w * TC + tid];
        n += nw[w * TC + tid];
      }
      qc[tid] = q;
      nc[tid] = n;
    }
    cluster.sync();
    if (rank == 0 && tid < tc) {
      float q = 0.f, n = 0.f;
#pragma unroll
      for (int r = 0; r < kClusterSize; ++r) {
        q += cluster.map_shared_rank(qc, r)[tid];
        n += cluster.map_shared_rank(nc, r)[tid];
      }
      if (!a.gram) q = n;  // orthonormal basis: ||V g||^2 = ||g||^2
      const float xx = nx2[tid];
      float rr = xx - 2.f * n + q;
      rr = rr < 0.f ? 0.f : rr;          // keeps NaN
      const float rho = xx == 0.f ? 0.f : sqrtf(rr / xx);
      const int t = t0 + tid;
      if (a.rho) a.rho[t] = rho;
      a.flags[t] = (rho < a.eps) ? uint8_t(0) : uint8_t(1);
    }
    cluster.sync();
  }

  if (rank == 0) {
    __threadfence();
    __syncthreads();
    if (warp == 0) compact_warp(a.flags, T, a.idx, a.idx ? a.ctrl->counts : nullptr, lane);
    if (tid == 0) a.ctrl->ticket = 0u;
  }
}

template <class E, int TC>
static cudaError_t launch_gate_t(const GateArgs& a, const GatePlan& p, cudaStream_t s, bool pdl) {
  auto kern = gate_kernel<E, TC>;
  static size_t smem_set = 0;  // raise the opt-in limit only when a plan needs more
  if (p.smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(p.smem));
    if (e != cudaSuccess) return e;
    smem_set = p.smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_slabs);
  cfg.blockDim = dim3(kGateThreads);
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
static cudaError_t launch_gate_e(const GateArgs& a, const GatePlan& p, cudaStream_t s, bool pdl) {
  switch (p.tc) {
    case 1: return launch_gate_t<E, 1>(a, p, s, pdl);
    case 2: return launch_gate_t<E, 2>(a, p, s, pdl);
    case 4: return launch_gate_t<E, 4>(a, p, s, pdl);
    default: return launch_gate_t<E, 8>(a, p, s, pdl);
  }
}

cudaError_t launch_gate(const GateArgs& a, const GatePlan& p, gsi_dtype dt, cudaStream_t s,
                        bool pdl) {
  return dt == GSI_BF16 ? launch_gate_e<BF16>(a, p, s, pdl) : launch_gate_e<F32>(a, p, s, pdl);
}

cudaError_t launch_compact(const uint8_t* flags, int T, int32_t* idx, int32_t* counts,
                           cudaStream_t s) {
  compact_kernel<<<1, 32, 0, s>>>(flags, T, idx, counts);
  return cudaGetLastError();
}

}  // namespace gsi
