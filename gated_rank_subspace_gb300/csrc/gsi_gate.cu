// Projection kernel: g = V_k^T x and ||x||^2, reduced per thread-block cluster.
//
// "Gated Subspace Inference for Transformer Acceleration", §2.1: the
// projection g = V_k^T x of the core decomposition.  V (d x k, row-major) is
// cut into slabs of rs consecutive rows, one slab per CTA, so every CTA
// streams one contiguous block of V with 16-byte loads; it holds its slab in
// registers before waiting on the previous kernel of the stream
// (programmatic dependent launch), so the weight traffic overlaps that
// kernel.  A CTA forms its slab's partial projections sum_i x_t[i] V[i, :]
// and the partial ||x_t||^2; the 8 CTAs of a cluster add theirs through
// distributed shared memory in rank order and write one partial per cluster.
// The decide-and-apply kernel finishes the sums.  No atomics, fixed order:
// bitwise reproducible.

#include "gsi_common.cuh"
#include "gsi_plan.h"
#include "gsi_kernels.h"

namespace gsi {

// Stable compaction by one 1024-thread CTA: per chunk of 4096 flags, thread
// i takes flags 4i .. 4i + 3 (loaded together), a block scan of the per-thread
// fast / slow counts gives each thread its output positions, and chunks
// follow one another with running totals.  Token order is kept in both lists.
constexpr int kCompactThreads = 1024;
constexpr int kCompactPer = 4;

__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const uint8_t* flags, int T, int32_t* idx,
                                                                  int32_t* counts) {
  __shared__ int wf[kCompactThreads / 32], wsl[kCompactThreads / 32];
  __shared__ int tot[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int base_f = 0, base_s = 0;
  for (int c0 = 0; c0 < T; c0 += kCompactThreads * kCompactPer) {
    int kind[kCompactPer];  // 0: none, 1: fast, 2: slow
    int nf = 0, ns = 0;
#pragma unroll
    for (int u = 0; u < kCompactPer; ++u) {
      const int t = c0 + tid * kCompactPer + u;
      kind[u] = t < T ? (ld_cg_u8(flags + t) != 0 ? 2 : 1) : 0;
      nf += kind[u] == 1;
      ns += kind[u] == 2;
    }
    // inclusive scans inside the warp, then over the warps' totals
    int xf = nf, xs = ns;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yf = __shfl_up_sync(0xffffffffu, xf, o), ys = __shfl_up_sync(0xffffffffu, xs, o);
      if (lane >= o) {
        xf += yf;
        xs += ys;
      }
    }
    if (lane == 31) {
      wf[warp] = xf;
      wsl[warp] = xs;
    }
    __syncthreads();
    if (warp == 0) {
      int a = wf[lane], b = wsl[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) {
          a += ya;
          b += yb;
        }
      }
      wf[lane] = a - wf[lane];  // exclusive
      wsl[lane] = b - wsl[lane];
      if (lane == 31) {
        tot[0] = a;
        tot[1] = b;
      }
    }
    __syncthreads();
    int of = base_f + wf[warp] + xf - nf, os = base_s + wsl[warp] + xs - ns;
    if (idx) {
#pragma unroll
      for (int u = 0; u < kCompactPer; ++u) {
        const int t = c0 + tid * kCompactPer + u;
        if (kind[u] == 1) idx[of++] = t;
        if (kind[u] == 2) idx[T + os++] = t;
      }
    }
    base_f += tot[0];
    base_s += tot[1];
    __syncthreads();  // wf / wsl / tot are rewritten by the next chunk
  }
  if (tid == 0 && counts) {
    counts[0] = base_f;
    counts[1] = base_s;
  }
}

template <class E, int TC>
__global__ void __cluster_dims__(kClusterSize, 1, 1) __launch_bounds__(kGateThreads, 4)
    project_kernel(GateArgs a) {
  extern __shared__ __align__(16) float smem[];
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
  if (tid == 0 || tid == 32) {
    // this CTA's share of M (thread 0) or of the Gram (thread 32), into L2
    const char* base = tid == 0 ? a.pf_m : a.pf_g;
    const uint64_t total = tid == 0 ? a.pf_m_bytes : a.pf_g_bytes;
    if (base && total) {
      const uint64_t share = ((total + gridDim.x - 1) / gridDim.x + 15) / 16 * 16;
      const uint64_t off = uint64_t(blockIdx.x) * share;
      if (off < total) {
        const uint64_t rem = total - off;
        prefetch_l2(base + off, uint32_t(rem < share ? rem : share));
      }
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
  cluster_arrive_relaxed();
  // ---- tokens may come from the previous kernel: wait for it
  pdl_wait();

  float* xs = smem;                     // [TC][rs]
  float* red = xs + TC * rs;            // [nrg][TC][k]
  float* pg = red + nrg * TC * k;       // [TC][k]
  float* px = pg + TC * k;              // [TC]
  float* inbox = px + TC;               // [8 ranks][TC][ks]  slices pushed by the peers
  float* inbox_x = inbox + kClusterSize * TC * ks;  // [8 ranks][TC]
  const int c0 = rank * ks;
  const int c1 = min(k, c0 + ks);
  bool started = false;

  for (int t0 = 0; t0 < T; t0 += TC) {
    const int tc = min(TC, T - t0);
    for (int e = tid; e < TC * rs; e += kGateThreads) {
      const int t = e / rs, i = e - (e / rs) * rs;
      xs[e] = (t < tc && i < rows) ? E::load1_cg(a.X, int64_t(t0 + t) * d + r0 + i) : 0.f;
    }
    __syncthreads();
    for (int t = warp; t < TC; t += kGateThreads / 32) {
      float s = 0.f;
      for (int i = lane; i < rs; i += 32) {
        const float xv = xs[t * rs + i];
        s += xv * xv;
      }
      s = warp_sum(s);
      if (lane == 0) px[t] = s;
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
    if (!started) {
      cluster_wait();  // every CTA of the cluster is running: peers' shared memory is live
      started = true;
    }
    // push: column col of the CTA partial goes to the rank owning col's slice
    for (int e = tid; e < TC * k; e += kGateThreads) {
      float s = 0.f;
      for (int g = 0; g < nrg; ++g) s += red[g * TC * k + e];
      const int t = e / k, col = e - (e / k) * k;
      const int q = col / ks;
      cluster.map_shared_rank(inbox, q)[(rank * TC + t) * ks + (col - q * ks)] = s;
    }
    if (tid < TC) cluster.map_shared_rank(inbox_x, 0)[rank * TC + tid] = px[tid];
    cluster.sync();
    // this CTA owns columns [c0, c1): add the eight ranks' slices in rank order
    for (int e = tid; e < TC * ks; e += kGateThreads) {
      const int t = e / ks, j = e - (e / ks) * ks, col = c0 + j;
      if (t < tc && col < c1) {
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < kClusterSize; ++q) s += inbox[(q * TC + t) * ks + j];
        a.part_g[(int64_t(cid) * T + t0 + t) * k + col] = s;
      }
    }
    if (rank == 0 && tid < tc) {
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < kClusterSize; ++q) s += inbox_x[q * TC + tid];
      a.part_x[int64_t(cid) * T + t0 + tid] = s;
    }
    if (t0 + TC < T) cluster.sync();  // the inboxes are read before the next chunk refills them
  }
  if (!started) cluster_wait();

}

template <class E, int TC>
static cudaError_t launch_gate_t(const GateArgs& a, const GatePlan& p, cudaStream_t s, bool pdl) {
  auto kern = project_kernel<E, TC>;
  static size_t smem_set = 0;  // raise the opt-in limit only when a plan needs more
  if (p.smem > smem_set) {
    cudaError_t e = set_kernel_smem(kern, p.smem);
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
  compact_kernel<<<1, kCompactThreads, 0, s>>>(flags, T, idx, counts);
  return cudaGetLastError();
}

}  // namespace gsi
