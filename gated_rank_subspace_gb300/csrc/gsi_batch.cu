// Small-batch decode kernel: the whole gated map for 2 to 16 tokens of a
// bf16 map in one launch.
//
// "Gated Subspace Inference for Transformer Acceleration", §2.1-§2.2: for
// each token x_t, g_t = V_k^T x_t and rho_t = ||x_t - V_k g_t|| / ||x_t||;
// rho_t < eps takes y_t = M g_t (M = W V_k, the cached image), rho_t >= eps
// the exact y_t = W x_t.  With several tokens a call, the three products
// (X V_k, G M^T, X W^T) carry up to 16 token columns each -- more multiply-
// adds per weight byte than the CUDA cores sustain at HBM rate once a few
// tokens are slow -- so they run as warp-level tensor-core products
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation) on 128-byte
// swizzled tiles that TMA copies into shared memory.  Everything else is
// fp32 on the CUDA cores.
//
//   prologue  the copy warp (the ninth) issues the TMA copies of the CTA's
//             V_k slab and the bulk copy of its rank's Gram slice (weight
//             traffic, before the dependency wait on the previous kernel of
//             the stream), and the M rows once the V_k slab has landed;
//             three threads stage the next map's weights and tokens in L2.
//   project   CTA b multiplies its token slab [16 x vr] by its V_k slab
//             [vr x k] (grid projection); warp w takes the 8-column tiles
//             w, w + 8, ... of g.  The fp32 accumulators go to shared memory
//             by column slice; lane q of warp 0 sends slice q to rank q with
//             one bulk copy into its shared memory (completion on its
//             mbarrier), and the slab's ||x_t||^2 to rank 0.
//   reduce    rank q adds its 16 inboxes in rank order and publishes its
//             slice of the cluster's sum as epoch-tagged 64-bit words; it
//             polls every cluster's words of that slice, adds them in
//             cluster order and sends the final slice to every rank of its
//             cluster, one bulk copy per token, landing in token order (rank
//             0 does the same for the norms).  Every CTA ends with the same
//             bits of G [T][k] and of ||x_t||^2.
//   decide    warp w takes tokens w and w + 8 over all of the rank's Gram
//             slice: their shares of g^T (V_k^T V_k) g and of ||g||^2 go to
//             every rank; every CTA adds the ranks' shares in rank order, so
//             every CTA takes the same flags.
//   fast      while the shares are in flight, G is rounded to bf16 as a high
//             and a low part (their sum is g to about 2^-16 relative) and
//             M G = M hi + M lo is formed for the CTA's rows and every token
//             (one warp per 16 x 8 output tile, kept in registers); fast
//             tokens' rows are written once the flags are known.
//   slow      when some token is slow, the copy warp streams the CTA's rows
//             of W, with the matching 128 columns of X, through a ring of
//             stages that takes the scratch and M space; warp w multiplies
//             the columns [16 w, 16 w + 16) of every stage for all row tiles
//             and tokens into registers; the warps' partial sums meet in the
//             ring's space, are added in warp order, and the slow tokens'
//             rows are written.
//
// Every wait is bounded (~2 s of clock, ~1 ms once a wait of the thread has
// given up): on expiry the workspace error word is set and the kernel goes
// on, waits (bounded) for its own copies in flight and leaves.  No float
// atomics: every sum has one fixed order, so results are reproducible.

#include <cuda.h>

#include "gsi_async.cuh"
#include "gsi_common.cuh"
#include "gsi_kernels.h"
#include "gsi_plan.h"

namespace gsi {

namespace {

// Low byte of the small-batch kernel's epochs: the single-token and stack
// kernels use 1 .. kStackMaxMaps there, so no epoch of another kernel's
// words can ever match one of this kernel's.
constexpr uint32_t kBatchEpochTag = 0xB0u;

struct BatchParams {
  CUtensorMap tv;  // V_k (d x k): boxes of vr rows x 64 columns
  CUtensorMap tm;  // M (d_out x k): boxes of rpc rows x 64 columns
  CUtensorMap tw;  // W (d_out x d): boxes of rpc rows x 64 columns
  CUtensorMap tx;  // X (T x d): boxes of T rows x 64 columns
  BatchCall c;
  BatchPlan p;
};

__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          sa(dst)),
      "l"(map), "r"(x), "r"(y), "r"(sa(bar))
      : "memory");
}

// ldmatrix: four (two) 8 x 8 bf16 matrices; lane l gives the row address of
// matrix l / 8.  Volatile: the same addresses are read again after a ring
// slot has been refilled.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// c += a b for a 16 x 16 bf16 tile a (row-major fragments) and a 16 x 8 bf16
// tile b (column-major fragments), fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void st_async_v2(uint32_t raddr, float a, float b, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(raddr),
               "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(rbar)
               : "memory");
}

// Bulk copy of this CTA's shared memory into a peer's (16-byte aligned,
// multiple of 16 bytes), completing on the peer's mbarrier; the issuing
// thread tracks it in its bulk async-group.
__device__ __forceinline__ void bulk_s2c(uint32_t dst_cluster, const void* src, uint32_t bytes, uint32_t bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_cluster),
               "r"(sa(src)), "r"(bytes), "r"(bar_cluster)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The sources of this thread's bulk copies have been read.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// The eight compute warps only (named barrier 1).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Byte offset of the 16-byte chunk `ch` (0..7) of row `row` in a box of
// 128-byte rows written by TMA with 128-byte swizzle (1024-byte aligned).
__device__ __forceinline__ uint32_t swz(int row, int ch) { return uint32_t(row * 128 + ((ch ^ (row & 7)) << 4)); }

__device__ __forceinline__ uint32_t bf16_bits(float v) {
  return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

}  // namespace

template <int NT>
__global__ void __launch_bounds__(kBatchThreads, 1) batch_decode_kernel(const __grid_constant__ BatchParams a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  constexpr int CS = kBatchCluster;
  constexpr int NW = kBatchWarps;
  constexpr int NC = kBatchWarps * 32;  // compute threads
  constexpr unsigned FULL = 0xffffffffu;
  const BatchCall& c = a.c;
  const BatchPlan& p = a.p;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (gridDim.x % CS != 0 || gridDim.x / CS > kBatchMaxClusters) {
    if (tid == 0) atomicOr(c.err, kErrTimeout | kErrLaunchShape);
    return;  // before any barrier, copy or access to another CTA
  }
  unsigned char* smem = smem_raw + ((1024u - (sa(smem_raw) & 1023u)) & 1023u);

  // ---- geometry
  const int T = c.T, k = c.k, ks = p.ks, kb = p.kb, S = p.stages;
  const int64_t d = c.d, d_out = c.d_out;
  const int rank = int(cg::this_cluster().block_rank());
  const int cl = int(blockIdx.x) / CS, ncl = int(gridDim.x) / CS;
  const int64_t v0 = int64_t(blockIdx.x) * p.vr;   // this CTA's rows of V_k
  const bool has_v = v0 < d;
  const int64_t r0 = int64_t(blockIdx.x) * p.rpc;  // this CTA's output rows
  const int nrows = r0 >= d_out ? 0 : int(d_out - r0 < p.rpc ? d_out - r0 : p.rpc);
  const int n_mt = (nrows + 15) >> 4;
  const int c0 = rank * ks;  // this rank's columns of g and rows of the Gram slice
  const int g_ = lane >> 2, t4 = lane & 3;  // fragment coordinates of this lane

  // ---- shared memory
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* vbar = bars + 0;   // V slab
  uint64_t* mbar = bars + 1;   // M rows
  uint64_t* gbar = bars + 2;   // Gram slice
  uint64_t* xbar = bars + 3;   // partial-g and norm inboxes
  uint64_t* gxbar = bars + 4;  // gathered g and norms
  uint64_t* qbar = bars + 5;   // share inbox
  uint64_t* full = bars + 8;   // [kBatchMaxStages] ring stage landed
  uint64_t* empty = full + kBatchMaxStages;  // [kBatchMaxStages] ring stage consumed (8 warps)
  uint32_t* words = reinterpret_cast<uint32_t*>(smem + 512);
  unsigned char* gbf = smem + p.off_gbf;  // [2][16][gbf_pitch]: g in bf16, high then low part
  uint32_t* dflag = reinterpret_cast<uint32_t*>(smem + p.off_dec);  // [16]
  float* drho = reinterpret_cast<float*>(smem + p.off_dec) + kBatchMaxT;  // [16]
  float* wsh = reinterpret_cast<float*>(smem + p.off_wsh);  // [16][2] the rank's shares of each token
  unsigned char* vs = smem + p.off_v;                       // kb boxes of [vr][128 B]
  unsigned char* xs = smem + p.off_xs;                      // [16][xs_pitch] token slab
  float* inbox = reinterpret_cast<float*>(smem + p.off_in);  // [CS][T][ks]
  float* nin = reinterpret_cast<float*>(smem + p.off_nin);   // [CS][16]
  float* g32 = reinterpret_cast<float*>(smem + p.off_g32);   // [T][k]: g by token
  float* gnx = g32 + T * k;                                  // [16] ||x_t||^2
  float* gt = g32;
  float* pg = reinterpret_cast<float*>(gbf);                 // [CS][T][ks]: this CTA's partial g
  float* fs = reinterpret_cast<float*>(smem + p.off_fs);     // [T][ks] this rank's final slice, then 16 norms
  float* nxs = reinterpret_cast<float*>(smem + p.off_nx);    // [16] the slab's ||x_t||^2
  float2* qin = reinterpret_cast<float2*>(smem + p.off_qin);  // [CS][16]
  const float* gram_s = reinterpret_cast<const float*>(smem + p.off_gram);  // [ks][k]
  unsigned char* ms = smem + p.off_m;                       // kb boxes of [rpc][128 B]
  unsigned char* ring = smem + p.off_scr;                   // S stages, once the flags are known

  uint32_t* err = c.err;
  bool ok = true;
  long long lim = kSpinCycles;
  auto note = [&](bool r) {
    if (!r) {
      ok = false;
      lim = kSpinCyclesAfterError;
    }
  };

  // ---- prologue: barriers, the call's epoch, weight copies
  if (tid == 0) {
    words[0] = ((uint32_t(atomicAdd(c.ticket, 1ull) / gridDim.x) + 1u) << 8) | kBatchEpochTag;
    bar_init(vbar, 1);
    bar_init(mbar, 1);
    bar_init(gbar, 1);
    bar_init(xbar, 1);
    bar_init(gxbar, 1);
    bar_init(qbar, 1);
    for (int s = 0; s < kBatchMaxStages; ++s) {
      bar_init(&full[s], 1);
      bar_init(&empty[s], NW);
    }
    // the exchanges' byte counts (each expect_tx is its barrier's one arrival)
    bar_expect_tx(xbar, uint32_t(CS * T * ks * 4 + (rank == 0 ? CS * kBatchMaxT * 4 : 0)));
    bar_expect_tx(gxbar, uint32_t(T * k * 4 + kBatchMaxT * 4));
    bar_expect_tx(qbar, uint32_t(CS * T * 8));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_launch_dependents();
  if (warp == NW && lane == 0) {
    if (has_v) {
      bar_expect_tx(vbar, uint32_t(kb * p.vr * 128));
      for (int b = 0; b < kb; ++b) tma2d(vs + b * p.vr * 128, &a.tv, vbar, b * 64, int(v0));
    }
    const uint32_t gb = uint32_t(ks) * uint32_t(k) * 4u;
    bar_expect_tx(gbar, gb);
    bulk_g2s(smem + p.off_gram, c.gram + int64_t(c0) * k, gb, gbar);
  }
  if (tid == 64 || tid == 96 || tid == 128 || tid == 160) {
    // this CTA's share of the next map's weights and tokens, into L2
    const char* base = tid == 64 ? c.next_v : tid == 96 ? c.next_m : tid == 128 ? c.next_gram : c.next_x;
    const uint64_t total = tid == 64    ? c.next_v_bytes
                           : tid == 96  ? c.next_m_bytes
                           : tid == 128 ? c.next_gram_bytes
                                        : c.next_x_bytes;
    if (base && total) {
      const uint64_t share = ((total + gridDim.x - 1) / gridDim.x + 15) / 16 * 16;
      const uint64_t off = uint64_t(blockIdx.x) * share;
      if (off < total) prefetch_l2(base + off, uint32_t(total - off < share ? total - off : share));
    }
  }
  cluster_arrive_relaxed();
  pdl_wait();

  // ---- the tokens' elements of this CTA's slab: [16][vr] bf16 (zeros past T and d)
  {
    const int vpt = p.vr / 8;  // 16-byte vectors of a token's slab
#pragma unroll 1
    for (int e = tid; e < kBatchMaxT * vpt; e += kBatchThreads) {
      const int t = e / vpt, j = e - t * vpt;
      const int64_t col = v0 + 8 * j;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (t < T && col < d) v = ld_cg_v4(static_cast<const char*>(c.X) + (int64_t(t) * d + col) * 2);
      *reinterpret_cast<uint4*>(xs + t * p.xs_pitch + j * 16) = v;
    }
  }
  __syncthreads();
  if (warp == NW && lane == 0 && nrows > 0) {
    // the M rows once the V slab has landed: the projection waits for V, the
    // fast products only several exchanges later
    if (has_v) note(bar_wait(vbar, 0, err, lim, kWaitV));
    bar_expect_tx(mbar, uint32_t(kb * p.rpc * 128));
    for (int b = 0; b < kb; ++b) tma2d(ms + b * p.rpc * 128, &a.tm, mbar, b * 64, int(r0));
  }

  // ---- projection: this warp's 8-column tiles of g over the slab
  constexpr int kNtW = kBatchMaxK / 8 / NW;  // tiles a warp (k <= kBatchMaxK)
  const int n_nt = k / 8;
  float pacc[kNtW][4];
#pragma unroll
  for (int j = 0; j < kNtW; ++j) pacc[j][0] = pacc[j][1] = pacc[j][2] = pacc[j][3] = 0.f;
  float nx0 = 0.f, nx1 = 0.f;
  if (warp < NW) {
    if (has_v) {
      note(__all_sync(FULL, bar_wait(vbar, 0, err, lim, kWaitV)));
      const uint32_t xs_a = sa(xs), vs_a = sa(vs);
      for (int kk = 0; kk < p.vr / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(xs_a + (lane & 15) * p.xs_pitch + (kk * 2 + (lane >> 4)) * 16, a0, a1, a2, a3);
        const int row = kk * 16 + (lane & 15);
#pragma unroll
        for (int j = 0; j < kNtW; ++j) {
          const int nt = warp + j * NW;
          if (nt < n_nt) {
            uint32_t b0, b1;
            ldsm_x2_t(vs_a + (nt >> 3) * p.vr * 128 + swz(row, nt & 7), b0, b1);
            mma16816(pacc[j], a0, a1, a2, a3, b0, b1);
          }
        }
      }
    }
    // ||x_t||^2 over the slab for tokens warp and warp + 8 (exact squares, fp32 sums)
    const uint16_t* x0 = reinterpret_cast<const uint16_t*>(xs + warp * p.xs_pitch);
    const uint16_t* x1 = reinterpret_cast<const uint16_t*>(xs + (warp + NW) * p.xs_pitch);
    for (int j = lane; j < p.vr; j += 32) {
      const float u = __uint_as_float(uint32_t(x0[j]) << 16), w = __uint_as_float(uint32_t(x1[j]) << 16);
      nx0 = fmaf(u, u, nx0);
      nx1 = fmaf(w, w, nx1);
    }
    nx0 = warp_sum(nx0);
    nx1 = warp_sum(nx1);
    // the accumulators by column slice (the slice of rank q contiguous), the
    // norms beside them, for the bulk copies of the reduce-scatter
#pragma unroll
    for (int j = 0; j < kNtW; ++j) {
      const int nt = warp + j * NW;
      if (nt < n_nt) {
        const int col = nt * 8 + 2 * t4;
        const int q = col / ks, cc = col - q * ks;
        if (g_ < T) *reinterpret_cast<float2*>(pg + (q * T + g_) * ks + cc) = make_float2(pacc[j][0], pacc[j][1]);
        if (g_ + 8 < T)
          *reinterpret_cast<float2*>(pg + (q * T + g_ + 8) * ks + cc) = make_float2(pacc[j][2], pacc[j][3]);
      }
    }
    if (lane == 0) {
      nxs[warp] = nx0;
      nxs[warp + NW] = nx1;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    compute_sync();
  }
  // The cluster shape, checked before the first access to another CTA (read
  // here, off the path to the token load).  Without it this CTA waits
  // (bounded) for its own copies and leaves.
  if (!cluster_shape_ok(CS)) {
    if (warp == NW && lane == 0) {
      if (nrows > 0) bar_wait(mbar, 0, err, kSpinCyclesAfterError, kWaitM);
      bar_wait(gbar, 0, err, kSpinCyclesAfterError, kWaitGram);
    }
    if (tid == 0) atomicOr(err, kErrTimeout | kErrLaunchShape);
    return;
  }
  cluster_wait();  // every CTA of the cluster runs and has initialised its barriers

  if (warp < NW) {
    // ---- reduce-scatter: rank q receives every rank's slice q, and rank 0
    //      every rank's norms, by one bulk copy each
    if (tid < CS) {  // lane q of warp 0 sends slice q (lane 0: the norms too)
      const int q = tid;
      bulk_s2c(map_rank(sa(inbox + rank * T * ks), q), pg + q * T * ks, uint32_t(T * ks * 4), map_rank(sa(xbar), q));
      if (q == 0) bulk_s2c(map_rank(sa(nin + rank * kBatchMaxT), 0), nxs, kBatchMaxT * 4, map_rank(sa(xbar), 0));
      bulk_commit();
    }
    note(bar_wait_cluster(xbar, 0, err, lim, kWaitPartials));

    // ---- this rank's slice of g (rank 0: also the norms), summed over the
    //      ranks, then over the clusters through epoch-tagged words, and
    //      pushed to every rank of the cluster.  Item = two adjacent values.
    const uint32_t epoch = words[0];
    const int gi = T * (ks / 2), ni = rank == 0 ? kBatchMaxT / 2 : 0;
    for (int it = tid; it < gi + ni; it += NC) {
      const bool gitem = it < gi;
      const int t = gitem ? it / (ks / 2) : 0;
      const int cc = gitem ? (it - t * (ks / 2)) * 2 : 0;
      const int tn = gitem ? 0 : (it - gi) * 2;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int r = 0; r < CS; ++r) {
        const float2 v = gitem ? *reinterpret_cast<const float2*>(inbox + (r * T + t) * ks + cc)
                               : *reinterpret_cast<const float2*>(nin + r * kBatchMaxT + tn);
        s0 += v.x;
        s1 += v.y;
      }
      unsigned long long* wsrc = gitem ? c.part_g + (int64_t(t) * k + c0 + cc) : c.part_x + tn;
      const int64_t cstride = gitem ? int64_t(T) * k : kBatchMaxT;
      const unsigned long long tag = uint64_t(epoch) << 32;
      if (!(c.dbg_withhold && cl == 0)) {
        st_relaxed_u64(wsrc + cl * cstride, tag | __float_as_uint(s0));
        st_relaxed_u64(wsrc + cl * cstride + 1, tag | __float_as_uint(s1));
      }
      float v0s[kBatchMaxClusters], v1s[kBatchMaxClusters];
      uint32_t pending = (1u << ncl) - 1u;
      const long long plim = c.poll_cycles > 0 ? c.poll_cycles : lim;
      const long long tw0 = clock64();
      while (pending) {
        unsigned long long w0[kBatchMaxClusters], w1[kBatchMaxClusters];  // all loads in flight, then the checks
#pragma unroll
        for (int q = 0; q < kBatchMaxClusters; ++q) {
          const bool on = (pending >> q) & 1u;
          w0[q] = on ? ld_relaxed_u64(wsrc + q * cstride) : 0ull;
          w1[q] = on ? ld_relaxed_u64(wsrc + q * cstride + 1) : 0ull;
        }
#pragma unroll
        for (int q = 0; q < kBatchMaxClusters; ++q)
          if (((pending >> q) & 1u) && uint32_t(w0[q] >> 32) == epoch && uint32_t(w1[q] >> 32) == epoch) {
            v0s[q] = __uint_as_float(uint32_t(w0[q]));
            v1s[q] = __uint_as_float(uint32_t(w1[q]));
            pending &= ~(1u << q);
          }
        if (pending && clock64() - tw0 > plim) {
          atomicOr(err, kErrTimeout | kWaitSlices);
          note(false);
          break;
        }
      }
      s0 = s1 = 0.f;
#pragma unroll
      for (int q = 0; q < kBatchMaxClusters; ++q)
        if (q < ncl && !((pending >> q) & 1u)) {
          s0 += v0s[q];
          s1 += v1s[q];
        }
      *reinterpret_cast<float2*>(gitem ? fs + t * ks + cc : fs + T * ks + tn) = make_float2(s0, s1);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    compute_sync();
    // ---- all-gather: thread 16 t + q sends token t of this rank's final
    //      slice to rank q, where it lands in token order (rank 0: the norms
    //      too), so the products below read consecutive columns of a token
    if (tid < T * CS) {
      const int t = tid >> 4, q = tid & (CS - 1);
      bulk_s2c(map_rank(sa(g32 + t * k + rank * ks), q), fs + t * ks, uint32_t(ks * 4), map_rank(sa(gxbar), q));
      if (rank == 0 && t == 0) bulk_s2c(map_rank(sa(gnx), q), fs + T * ks, kBatchMaxT * 4, map_rank(sa(gxbar), q));
      bulk_commit();
    }
    note(bar_wait_cluster(gxbar, 0, err, lim, kWaitGathered));
    if (tid < CS) bulk_wait_read();  // the partial g's space is about to hold g in bf16

    // ---- shares of the Gram form: warp w takes tokens w and w + 8 over all of
    //      the rank's Gram rows i (columns c0 + i of g); lane l owns the column
    //      groups l, l + 32, ... (float4): u_j = sum_i g_i Gram[i][j] over the
    //      rows in order, then the token's share sum_j g_j u_j (a butterfly
    //      over the lanes) and its share of ||g||^2 over the rank's columns
    {
      note(__all_sync(FULL, bar_wait(gbar, 0, err, lim, kWaitGram)));
      constexpr int NG = kBatchMaxK / 4 / 32;  // float4 groups of a row a lane
      const int nf4 = k >> 2;
      const int t_a = warp, t_b = warp + NW;
      const float* ga_row = gt + (t_a < T ? t_a : 0) * k;
      const float* gb_row = gt + (t_b < T ? t_b : 0) * k;
      float4 ua[NG], ub[NG];
#pragma unroll
      for (int u = 0; u < NG; ++u) ua[u] = ub[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      // the rows four at a time (ks is a multiple of 4), their loads first
#pragma unroll 1
      for (int i0 = 0; i0 < ks; i0 += 4) {
        float4 gr[4][NG];
        float ca[4], cb[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
#pragma unroll
          for (int u = 0; u < NG; ++u) {
            const int jg = lane + 32 * u;
            gr[r][u] = jg < nf4 ? reinterpret_cast<const float4*>(gram_s + (i0 + r) * k)[jg]
                                : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          ca[r] = ga_row[c0 + i0 + r];
          cb[r] = gb_row[c0 + i0 + r];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int u = 0; u < NG; ++u) {
            ua[u].x = fmaf(ca[r], gr[r][u].x, ua[u].x);
            ua[u].y = fmaf(ca[r], gr[r][u].y, ua[u].y);
            ua[u].z = fmaf(ca[r], gr[r][u].z, ua[u].z);
            ua[u].w = fmaf(ca[r], gr[r][u].w, ua[u].w);
            ub[u].x = fmaf(cb[r], gr[r][u].x, ub[u].x);
            ub[u].y = fmaf(cb[r], gr[r][u].y, ub[u].y);
            ub[u].z = fmaf(cb[r], gr[r][u].z, ub[u].z);
            ub[u].w = fmaf(cb[r], gr[r][u].w, ub[u].w);
          }
      }
      float qa = 0.f, qb = 0.f;
#pragma unroll
      for (int u = 0; u < NG; ++u) {
        const int jg = lane + 32 * u;
        if (jg < nf4) {
          const float4 a = reinterpret_cast<const float4*>(ga_row)[jg], b = reinterpret_cast<const float4*>(gb_row)[jg];
          qa = fmaf(a.x, ua[u].x, qa);
          qa = fmaf(a.y, ua[u].y, qa);
          qa = fmaf(a.z, ua[u].z, qa);
          qa = fmaf(a.w, ua[u].w, qa);
          qb = fmaf(b.x, ub[u].x, qb);
          qb = fmaf(b.y, ub[u].y, qb);
          qb = fmaf(b.z, ub[u].z, qb);
          qb = fmaf(b.w, ub[u].w, qb);
        }
      }
      // ||g||^2 over the rank's columns: lane l takes column c0 + l (ks <= 32)
      const float ea = lane < ks ? ga_row[c0 + lane] : 0.f, eb = lane < ks ? gb_row[c0 + lane] : 0.f;
      float na = ea * ea, nb = eb * eb;
      qa = warp_sum(qa);
      qb = warp_sum(qb);
      na = warp_sum(na);
      nb = warp_sum(nb);
      if (lane == 0) {
        wsh[t_a * 2] = qa;
        wsh[t_a * 2 + 1] = na;
        wsh[t_b * 2] = qb;
        wsh[t_b * 2 + 1] = nb;
      }
    }
    compute_sync();
    // thread 16 t + r sends the rank's pair of token t to rank r
    if (tid < T * CS) {
      const int t = tid >> 4, r = tid & (CS - 1);
      st_async_v2(map_rank(sa(qin + rank * kBatchMaxT + t), r), wsh[t * 2], wsh[t * 2 + 1], map_rank(sa(qbar), r));
    }
  }
  cluster_arrive_relaxed();  // this CTA's last push into a peer is issued

  // ---- fast path for every token: M G = M hi + M lo, 16 x 8 tiles in
  //      registers.  (Spreading the tiles over the copy warp too measured
  //      slower: the tensor pipes are per SM sub-partition, and a ninth warp
  //      puts three warps' tiles on one of them.)
  constexpr int kUnits = (kBatchMaxMt * NT + NW - 1) / NW;
  float facc[kUnits][4];
#pragma unroll
  for (int j = 0; j < kUnits; ++j) facc[j][0] = facc[j][1] = facc[j][2] = facc[j][3] = 0.f;
  const int gp = p.gbf_pitch;
  if (warp < NW) {
    // warp w: tokens w and w + 8, lanes over column pairs
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = warp + h * NW;
#pragma unroll 1
      for (int col = 2 * lane; col < k; col += 64) {
        const float2 x = t < T ? *reinterpret_cast<const float2*>(gt + t * k + col) : make_float2(0.f, 0.f);
        const uint32_t h0 = bf16_bits(x.x), h1 = bf16_bits(x.y);
        const uint32_t l0 = bf16_bits(x.x - __uint_as_float(h0 << 16)), l1 = bf16_bits(x.y - __uint_as_float(h1 << 16));
        *reinterpret_cast<uint32_t*>(gbf + t * gp + col * 2) = h0 | (h1 << 16);
        *reinterpret_cast<uint32_t*>(gbf + (kBatchMaxT + t) * gp + col * 2) = l0 | (l1 << 16);
      }
    }
    compute_sync();  // g in bf16 is in place
    if (nrows > 0) {
      note(__all_sync(FULL, bar_wait(mbar, 0, err, lim, kWaitM)));
      const uint32_t ms_a = sa(ms), gh_a = sa(gbf), gl_a = sa(gbf + kBatchMaxT * gp);
      // k steps outside, the warp's tiles inside: independent accumulators
      // (high and low part apart) keep the tensor pipe busy
      float flo[kUnits][4];
#pragma unroll
      for (int j = 0; j < kUnits; ++j) flo[j][0] = flo[j][1] = flo[j][2] = flo[j][3] = 0.f;
      const int nu = n_mt * NT;
#pragma unroll 2
      for (int kk = 0; kk < k / 16; ++kk) {
        const int ch = kk * 2 + (lane >> 4);
        const uint32_t bch = uint32_t((kk * 2 + ((lane >> 3) & 1)) * 16);
#pragma unroll
        for (int j = 0; j < kUnits; ++j) {
          const int u = warp + j * NW;
          if (u < nu) {
            const int mt = u / NT, nt = u - mt * NT;
            const int row = mt * 16 + (lane & 15);
            const uint32_t boff = uint32_t((nt * 8 + (lane & 7)) * gp) + bch;
            uint32_t a0, a1, a2, a3, b0, b1, c0r, c1r;
            ldsm_x4(ms_a + (ch >> 3) * p.rpc * 128 + swz(row, ch & 7), a0, a1, a2, a3);
            ldsm_x2(gh_a + boff, b0, b1);
            ldsm_x2(gl_a + boff, c0r, c1r);
            mma16816(facc[j], a0, a1, a2, a3, b0, b1);
            mma16816(flo[j], a0, a1, a2, a3, c0r, c1r);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kUnits; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) facc[j][e] += flo[j][e];
    }

    // ---- the decision (warp 0), from the ranks' shares in rank order
    if (warp == 0) {
      note(bar_wait_cluster(qbar, 0, err, lim, kWaitShares));
      if (lane < T) {
        float Q = 0.f, N = 0.f;
#pragma unroll
        for (int r = 0; r < CS; ++r) {
          const float2 v = qin[r * kBatchMaxT + lane];
          Q += v.x;
          N += v.y;
        }
        if (!c.gram) Q = N;  // orthonormal basis: ||V g||^2 = ||g||^2
        const float xx = gnx[lane];
        float rr = xx - 2.f * N + Q;
        rr = rr < 0.f ? 0.f : rr;  // keeps NaN
        const float rho = xx == 0.f ? 0.f : sqrtf(rr / xx);
        const bool slow = !(rho < c.eps);
        dflag[lane] = slow ? 1u : 0u;
        drho[lane] = rho;
        if (blockIdx.x == 0) {
          if (c.rho) c.rho[lane] = rho;
          c.flags[lane] = uint8_t(slow ? 1 : 0);
        }
      }
    }
  }
  __syncthreads();
  uint32_t slow_mask = 0;
  for (int t = 0; t < T; ++t) slow_mask |= dflag[t] << t;
  const uint32_t fast_mask = ~slow_mask & ((1u << T) - 1u);

  // ---- fast tokens' rows, from the registers
  if (warp < NW && nrows > 0 && fast_mask) {
#pragma unroll
    for (int j = 0; j < kUnits; ++j) {
      const int u = warp + j * NW;
      if (u < n_mt * NT) {
        const int mt = u / NT, nt = u - mt * NT;
        const int ra = mt * 16 + g_, rb2 = ra + 8;
        const int ta = nt * 8 + 2 * t4, tb = ta + 1;
        if ((fast_mask >> ta) & 1u) {
          if (ra < nrows) c.Y[int64_t(ta) * d_out + r0 + ra] = facc[j][0];
          if (rb2 < nrows) c.Y[int64_t(ta) * d_out + r0 + rb2] = facc[j][2];
        }
        if ((fast_mask >> tb) & 1u) {
          if (ra < nrows) c.Y[int64_t(tb) * d_out + r0 + ra] = facc[j][1];
          if (rb2 < nrows) c.Y[int64_t(tb) * d_out + r0 + rb2] = facc[j][3];
        }
      }
    }
  }

  // ---- slow tokens: W streamed through the ring
  const int nch = int((d + kBatchKC - 1) / kBatchKC);
  const bool stream = slow_mask != 0 && nrows > 0;
  const uint32_t stage_tx = uint32_t(2 * p.rpc * 128 + 2 * T * 128);
  if (stream && warp == NW) {
    if (lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      for (int j = 0; j < nch; ++j) {
        const int s = j % S;
        if (j >= S) note(bar_wait(&empty[s], uint32_t((j / S) - 1) & 1u, err, lim, kWaitRing));
        unsigned char* st = ring + s * p.stage_bytes;
        bar_expect_tx(&full[s], stage_tx);
        tma2d(st, &a.tw, &full[s], j * kBatchKC, int(r0));
        tma2d(st + p.rpc * 128, &a.tw, &full[s], j * kBatchKC + 64, int(r0));
        tma2d(st + 2 * p.rpc * 128, &a.tx, &full[s], j * kBatchKC, 0);
        tma2d(st + 2 * p.rpc * 128 + kBatchMaxT * 128, &a.tx, &full[s], j * kBatchKC + 64, 0);
      }
    }
  } else if (stream) {
    float acc[kBatchMaxMt][NT][4];
#pragma unroll
    for (int mt = 0; mt < kBatchMaxMt; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
    const int box = warp >> 2, ch0 = (warp & 3) * 2;  // this warp's 16 columns of a stage
    const uint32_t ring_a = sa(ring);
    for (int j = 0; j < nch; ++j) {
      const int s = j % S;
      note(__all_sync(FULL, bar_wait(&full[s], uint32_t(j / S) & 1u, err, lim, kWaitRing)));
      const uint32_t st = ring_a + uint32_t(s * p.stage_bytes);
      const uint32_t xb = st + uint32_t(2 * p.rpc * 128 + box * kBatchMaxT * 128);
      uint32_t b[NT][2];
      if (NT == 2) {
        const int tok = (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4(xb + swz(tok, ch0 + ((lane >> 3) & 1)), b[0][0], b[0][1], b[NT - 1][0], b[NT - 1][1]);
      } else {
        const int tok = lane & 7;
        ldsm_x2(xb + swz(tok, ch0 + ((lane >> 3) & 1)), b[0][0], b[0][1]);
      }
      const uint32_t wb = st + uint32_t(box * p.rpc * 128);
#pragma unroll
      for (int mt = 0; mt < kBatchMaxMt; ++mt) {
        if (mt < n_mt) {
          const int row = mt * 16 + (lane & 15);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(wb + swz(row, ch0 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(acc[mt][nt], a0, a1, a2, a3, b[nt][0], b[nt][1]);
        }
      }
      __syncwarp();
      if (lane == 0) bar_arrive(&empty[s]);
    }
    compute_sync();  // every warp is done with the ring: its space takes the partial sums
    float* red = reinterpret_cast<float*>(ring);  // [NW][16][rpc]
#pragma unroll
    for (int mt = 0; mt < kBatchMaxMt; ++mt) {
      if (mt < n_mt) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int ra = mt * 16 + g_, ta = nt * 8 + 2 * t4;
          red[(warp * kBatchMaxT + ta) * p.rpc + ra] = acc[mt][nt][0];
          red[(warp * kBatchMaxT + ta + 1) * p.rpc + ra] = acc[mt][nt][1];
          red[(warp * kBatchMaxT + ta) * p.rpc + ra + 8] = acc[mt][nt][2];
          red[(warp * kBatchMaxT + ta + 1) * p.rpc + ra + 8] = acc[mt][nt][3];
        }
      }
    }
    compute_sync();
    for (int e = tid; e < T * nrows; e += NC) {
      const int t = e / nrows, r = e - t * nrows;
      if ((slow_mask >> t) & 1u) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) s += red[(w * kBatchMaxT + t) * p.rpc + r];
        c.Y[int64_t(t) * d_out + r0 + r] = s;
      }
    }
  }

  // ---- this CTA's copies in flight land before it leaves (no-op waits
  //      unless a wait expired somewhere)
  if (warp == NW && lane == 0) {
    const long long l2 = kSpinCyclesAfterError;
    if (has_v) bar_wait(vbar, 0, err, l2, kWaitV);
    if (nrows > 0) bar_wait(mbar, 0, err, l2, kWaitM);
    bar_wait(gbar, 0, err, l2, kWaitGram);
  }
  if (warp == NW && lane == 0 && stream) {
    // the last use of every slot (a no-op wait when the consumers saw it land)
    for (int j = nch - S > 0 ? nch - S : 0; j < nch; ++j)
      bar_wait(&full[j % S], uint32_t(j / S) & 1u, err, ok ? lim : kSpinCyclesAfterError, kWaitRing);
  }
  if (tid < T * CS) bulk_wait_read();  // the all-gather's source
  // No CTA leaves while a peer of its cluster may still push into it.
  cluster_wait();
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFnB)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFnB batch_encode_fn() {
  static EncodeTiledFnB fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnB>(ptr);
  }
  return fn;
}

// bf16 row-major (rows x cols) matrix, boxes of box_rows x 64 columns,
// 128-byte swizzle, zero fill outside the matrix.
static cudaError_t batch_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  EncodeTiledFnB fn = batch_encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  cuuint32_t box[2] = {64u, cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int NT>
static cudaError_t launch_batch_t(const BatchParams& a, cudaStream_t s) {
  auto kern = batch_decode_kernel<NT>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_kernel_smem(kern, 232448);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(a.p.ncta));
  cfg.blockDim = dim3(kBatchThreads);
  cfg.dynamicSmemBytes = a.p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr_l[3];
  attr_l[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr_l[0].val.programmaticStreamSerializationAllowed = 1;
  attr_l[1].id = cudaLaunchAttributeClusterDimension;
  attr_l[1].val.clusterDim.x = kBatchCluster;
  attr_l[1].val.clusterDim.y = 1;
  attr_l[1].val.clusterDim.z = 1;
  // the CTAs poll other clusters' words: co-resident launch
  static int no_coop = 0;
  return launch_maybe_coop(cfg, attr_l, 2, true, &no_coop, kern, a);
}

cudaError_t launch_batch_decode(const BatchCall& c, const BatchPlan& p, cudaStream_t s) {
  static thread_local BatchParams a;
  a = BatchParams{};
  cudaError_t e;
  if ((e = batch_map(&a.tv, c.V, c.d, c.k, p.vr)) != cudaSuccess) return e;
  if ((e = batch_map(&a.tm, c.M, c.d_out, c.k, p.rpc)) != cudaSuccess) return e;
  if ((e = batch_map(&a.tw, c.W, c.d_out, c.d, p.rpc)) != cudaSuccess) return e;
  if ((e = batch_map(&a.tx, c.X, c.T, c.d, c.T)) != cudaSuccess) return e;
  a.c = c;
  a.p = p;
  return c.T <= 8 ? launch_batch_t<1>(a, s) : launch_batch_t<2>(a, s);
}

int batch_max_clusters(size_t smem) {
  auto kern = batch_decode_kernel<2>;
  if (set_kernel_smem(kern, 232448) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kBatchCluster * 64);
  cfg.blockDim = dim3(kBatchThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kBatchCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n > kBatchMaxClusters ? kBatchMaxClusters : n;
}

}  // namespace gsi
