// Decide-and-apply kernel: residual ratio, gate, and the fast / slow paths.
//
// "Gated Subspace Inference for Transformer Acceleration", §2.2: per token,
// rho = ||x - V_k g|| / ||x||; fast tokens (rho < eps) take y = M g (the
// cached image, d_out x k), slow tokens the exact y = W x (d_out x d).
//
// Input: partial sums of g = V_k^T x and ||x||^2 -- either the projection
// kernel's cluster partials (two-launch path) or, in the single-launch form
// (FUSED), the partials every CTA of this grid publishes after projecting x
// on its own slab of V_k, behind a grid barrier on the workspace's ticket
// counter.  Every 8-CTA cluster then finishes the gate on its own: CTA r adds
// the partials of its slice of g's columns (coalesced loads, one fixed
// order), the slices are pushed into every CTA's shared memory by st.async
// (completion on the receiver's mbarrier), CTA r forms its share of
// g^T (V_k^T V_k) g from the Gram slice it copied into shared memory before
// the dependency wait, and the shares are pushed the same way and added in
// rank order.  All clusters do the same arithmetic on the same data in the
// same order, so they reach the same bits, and every CTA knows every token's
// flag without a host round trip.
//
// Each CTA owns a contiguous block of output rows.  Before the dependency
// wait it copies its rows of M into shared memory (TMA bulk copy); a
// decide-and-apply call computes y = M g for its tokens while the decision's
// last exchange is in flight and keeps the rows of the fast ones.  Slow tokens
// stream the CTA's rows of W: each of the eight warps owns rows warp,
// warp + 8, ... and pulls them in 4 KB segments through a private ring of bulk
// copies completed on mbarriers; a row's sum is one warp's, in lane order.
// Every wait on an mbarrier is bounded: on expiry the kernel sets the
// workspace error word, drains its own copies (bounded) and returns.
//
// Modes: decide and apply (gsi_linear), decide only (gsi_gate: writes G,
// rho, flags and the compaction), apply a stored decision (gsi_apply), and
// decide and apply the fast tokens only, with the compaction (bf16 maps on
// the two-launch path: the slow rows follow as a tensor-core contraction).

#include "gsi_common.cuh"
#include "gsi_async.cuh"
#include "gsi_kernels.h"
#include "gsi_plan.h"

namespace gsi {

// ------------------------------------------------------------------ kernel
// FUSED: the grid computes g = V_k^T x itself (one launch per call, T <= 2):
// every CTA projects its own slab of V_k and the partials meet at a grid
// barrier; otherwise g comes from the projection kernel's cluster partials.
// CS: CTAs per cluster (8; 16 for the cluster projection), set at launch.
template <class E, int TC, int GRV, bool FUSED, int CS>
__global__ void __maxnreg__(168) decide_apply_kernel(DecideArgs a) {
  constexpr int PV = E::kPerVec;
  constexpr int NCW = 8;  // consumer warps
  extern __shared__ __align__(128) unsigned char smem[];
  if (!cluster_shape_ok(CS)) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrTimeout | kErrLaunchShape);
    return;  // before any barrier, copy or access to another CTA
  }
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = int(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k, T = a.T, ks = a.ks;
  const int64_t d = a.d, d_out = a.d_out;
  const int64_t r0 = int64_t(blockIdx.x) * a.rows_per_cta;
  const int nrows = int(r0 >= d_out ? 0 : (d_out - r0 < a.rows_per_cta ? d_out - r0 : a.rows_per_cta));
  const int64_t row_b = d * E::kBytes;      // bytes of a W row
  const int mrow_b = k * E::kBytes;         // bytes of an M row
  const int c0 = rank * ks, c1 = min(k, c0 + ks);

  // shared-memory carve-up (offsets computed on the host, see plan_decide)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);          // [8 warps][wstages]
  uint64_t* mfull = full + (kApplyThreads / 32) * a.wstages;   // [1]
  uint64_t* gfull_bar = mfull + 1;                             // [1] Gram slice copy
  const float* gram_s = reinterpret_cast<const float*>(smem + a.off_gram);
  unsigned char* Ms = smem + a.off_m;                          // staged M rows / W rings
  unsigned char* xst = smem + a.off_x;                         // staged x of slow tokens
  float* gfull = reinterpret_cast<float*>(smem + a.off_g);     // [TC][k]
  float* gsl = gfull + TC * k;                                 // [TC][ks]
  float* qw = gsl + TC * ks;                                   // [8][TC]
  float* nw = qw + 8 * TC;                                     // [8][TC]
  float* qin = nw + 8 * TC;                                    // [CS ranks][TC] pushed shares
  float* nin = qin + CS * TC;                                  // [CS ranks][TC]
  float* nx2 = nin + CS * TC;                                  // [TC]
  float* rowpart = nx2 + TC;                                   // [8 warps][4]
  int* sflag = reinterpret_cast<int*>(rowpart + 8 * 4);        // [TC]
  int* slist = sflag + TC;                                     // [TC] slow tokens of the chunk
  int* flist = slist + TC;                                     // [TC] fast tokens of the chunk
  int* scount = flist + TC;                                    // [2]
  float* red3 = reinterpret_cast<float*>(scount + 4);          // [kApplyThreads] partial-sum scratch
  // fused decode only: V slab, token slice, partial sums
  uint64_t* vbar = gfull_bar + 1;                              // [1] V slab copy
  uint64_t* gx_bar = gfull_bar + 2;                            // [1] peers' slices of g received
  uint64_t* qn_bar = gfull_bar + 3;                            // [1] peers' Gram / norm shares received
  const unsigned char* Vs = smem + a.off_v;                    // [v_rows][k] elements
  float* xsl = reinterpret_cast<float*>(smem + a.off_xs);      // [TC][v_rows]
  float* red2 = xsl + TC * ((a.v_rows + 3) & ~3);              // [ngrp][TC][k], 16-byte aligned
  float* xsq = red2 + a.ngrp * TC * k;                         // [TC]
  // cluster projection only: this CTA's partial g and the all-to-all inboxes
  float* pg = xsq + 8;                                         // [TC][k]; xsq is 16-byte aligned, TC <= 8
  float* inbox = pg + TC * k;                                  // [CS][TC][k]
  float* inbox_x = inbox + CS * TC * k;                        // [CS][TC]

  // ---- prologue: only weights (may overlap the projection kernel)
  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < (kApplyThreads / 32) * a.wstages; ++s) bar_init(&full[s], 1);
    bar_init(mfull, 1);
    bar_init(gfull_bar, 1);
    bar_init(gfull_bar + 1, 1);
    bar_init(gfull_bar + 2, 1);
    bar_init(gfull_bar + 3, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool stage_m = a.stage_m && a.mode != 1 && nrows > 0;
  // (with the cluster projection the M rows take the V slice's place once it
  // has been read, so their copy is issued after the projection)
  if (tid == kApplyThreads - 32 && stage_m && !(FUSED && a.cproj)) {
    const uint32_t bytes = uint32_t(nrows) * mrow_b;
    bar_expect_tx(mfull, bytes);
    bulk_g2s(Ms, static_cast<const char*>(a.M) + r0 * mrow_b, bytes, mfull);
  }
  // Gram slice rows [c0, c1) into shared memory (bulk copy, overlaps the wait)
  const int k4_ = k >> 2;
  const int gvec_ = (c1 > c0) ? (c1 - c0) * k4_ : 0;
  const bool gram_smem = a.off_gram != 0 && a.gram && a.mode != 2 && gvec_ > 0;
  if (gram_smem && tid == kApplyThreads - 32) {
    const uint32_t bytes = uint32_t(gvec_) * 16u;
    bar_expect_tx(gfull_bar, bytes);
    bulk_g2s(smem + a.off_gram, a.gram + int64_t(c0) * k, bytes, gfull_bar);
  }
  bool gram_waited = false;
  // fused decode: this CTA's slab of V (rows [v0, v0 + vn)), one bulk copy
  const int64_t v0 = int64_t(FUSED && a.cproj ? rank : int(blockIdx.x)) * a.v_rows;
  const int vn = FUSED ? int(v0 >= d ? 0 : (d - v0 < a.v_rows ? d - v0 : a.v_rows)) : 0;
  if (FUSED && a.mode != 2 && vn > 0 && tid == kApplyThreads - 32) {
    const uint32_t bytes = uint32_t(vn) * uint32_t(mrow_b);
    bar_expect_tx(vbar, bytes);
    bulk_g2s(smem + a.off_v, static_cast<const char*>(a.V) + v0 * mrow_b, bytes, vbar);
  }
  bool v_waited = !(FUSED && a.mode != 2 && vn > 0);
  // weights of the next map of a stack, into L2 (this CTA's share)
  if (tid == 64 || tid == 96 || tid == 128) {
    const char* base = tid == 64 ? a.next_v : tid == 96 ? a.next_m : a.next_gram;
    const uint64_t total = tid == 64 ? a.next_v_bytes : tid == 96 ? a.next_m_bytes : a.next_gram_bytes;
    if (base && total) {
      const uint64_t share = ((total + gridDim.x - 1) / gridDim.x + 15) / 16 * 16;
      const uint64_t off = uint64_t(blockIdx.x) * share;
      if (off < total) {
        const uint64_t rem = total - off;
        prefetch_l2(base + off, uint32_t(rem < share ? rem : share));
      }
    }
  }
  // (alternative when the slice does not fit: GRV float4 registers per thread)
  float4 gr[GRV > 0 ? GRV : 1];
  const int k4 = k >> 2;
  const int gvec = (c1 > c0) ? (c1 - c0) * k4 : 0;
  if (GRV > 0 && a.gram && a.mode != 2 && tid < 256) {
#pragma unroll
    for (int u = 0; u < (GRV > 0 ? GRV : 1); ++u) {
      const int v = u * 256 + tid;
      // volatile loads: issued here, before the dependency wait, not sunk to their use
      uint4 raw = v < gvec ? ld_weight_v4(a.gram + (int64_t(c0 + v / k4) * k + 4 * (v % k4)))
                           : make_uint4(0u, 0u, 0u, 0u);
      gr[u] = make_float4(__uint_as_float(raw.x), __uint_as_float(raw.y), __uint_as_float(raw.z),
                          __uint_as_float(raw.w));
    }
  }
  if (GRV == 0 && !gram_smem && a.gram && a.mode != 2 && tid == 0 && gvec > 0)
    prefetch_l2(a.gram + int64_t(c0) * k, uint32_t(gvec) * 16u);  // read after the wait
  cluster_arrive_relaxed();
  pdl_wait();
  bool started = false;

  bool ok = true;
  bool m_live = stage_m;  // staged M rows still in shared memory (the W ring reuses it)
  bool m_waited = false;  // the M copy has been waited for
  int wuse = 0;           // this warp's ring items used so far (running count over token chunks)
  const int E_ = TC * ks;
  int grp = 1;  // threads that share one column of g when its partials are added
  while (grp < 32 && E_ * grp * 2 <= kApplyThreads) grp *= 2;
  const int64_t cstride = int64_t(T) * k;

  float* ybuf = reinterpret_cast<float*>(smem + a.off_y);  // [TC][rows_per_cta]
  // y[t][r] = M[r0 + r] . g_t for the tokens tok_of(0 .. ntok), each result
  // handed to emit(t, r, value); warp w takes row blocks of RB rows, RB the
  // smallest block that gives all NCW warps rows (few rows per CTA still use
  // every warp)
  auto fast_apply = [&](int ntok, auto tok_of, auto emit) {
    const unsigned char* mrows = m_live ? Ms : static_cast<const unsigned char*>(a.M) + r0 * mrow_b;
    const int nvm = mrow_b / 16;
    // A block of RB rows at a time: the lane's vectors of those rows are
    // read once (NL = 1 or 2 vectors a lane) and multiplied with every
    // token's g, instead of re-reading the rows per token; each product sum
    // keeps its order (the lane's vectors in order, then the butterfly).
    auto fast_rows = [&](auto rb_c, auto nl_c) {
      constexpr int RB = decltype(rb_c)::value;
      constexpr int NL = decltype(nl_c)::value;
      for (int rb = warp * RB; rb < nrows; rb += NCW * RB) {
        uint4 mv[RB][NL];
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
          for (int j = 0; j < NL; ++j) {
            const int vv = lane + 32 * j;
            mv[r][j] = (rb + r < nrows && vv < nvm)
                           ? *reinterpret_cast<const uint4*>(mrows + int64_t(rb + r) * mrow_b + vv * 16)
                           : make_uint4(0u, 0u, 0u, 0u);
          }
        for (int f = 0; f < ntok; ++f) {
          const int t = tok_of(f);
          float part[RB];
#pragma unroll
          for (int r = 0; r < RB; ++r) part[r] = 0.f;
#pragma unroll
          for (int j = 0; j < NL; ++j) {
            const int vv = lane + 32 * j;
            if (vv < nvm) {
              float gv[PV];
#pragma unroll
              for (int e4 = 0; e4 < PV / 4; ++e4) {
                const float4 g4 = *reinterpret_cast<const float4*>(gfull + t * k + vv * PV + 4 * e4);
                gv[4 * e4] = g4.x;
                gv[4 * e4 + 1] = g4.y;
                gv[4 * e4 + 2] = g4.z;
                gv[4 * e4 + 3] = g4.w;
              }
#pragma unroll
              for (int r = 0; r < RB; ++r) {
                float w[PV];
                E::unpack(mv[r][j], w);
#pragma unroll
                for (int e = 0; e < PV; ++e) part[r] = fmaf(w[e], gv[e], part[r]);
              }
            }
          }
          const float sum = warp_reduce_multi<RB>(part, lane);
          const int r = row_of_lane<RB>(lane);
          if ((lane & (32 / RB - 1)) == 0 && rb + r < nrows) emit(t, rb + r, sum);
        }
      }
    };
    // (at most 8 rows a block: the rows' vectors stay in registers)
    if (nvm > 32) {  // rows over 512 bytes: two vectors a lane
      if (nrows <= NCW * 4)
        fast_rows(IntC<4>{}, IntC<2>{});
      else
        fast_rows(IntC<8>{}, IntC<2>{});
    } else if (nrows <= NCW * 4) {
      fast_rows(IntC<4>{}, IntC<1>{});
    } else {
      fast_rows(IntC<8>{}, IntC<1>{});
    }
  };
  // decide-and-apply calls compute the fast outputs before the decision ends
  const bool yspec = (a.mode == 0 || a.mode == 3) && nrows > 0;

  for (int t0 = 0; t0 < T; t0 += TC) {
    const int tc = min(TC, T - t0);
    if (a.mode != 2 && FUSED) {
      // -- g from the grid's own slabs of V: CTA b projects rows
      //    [v0, v0 + vn) of V and publishes its partials for all clusters
      for (int e = tid; e < TC * a.v_rows; e += blockDim.x) {
        const int t = e / a.v_rows, i = e - (e / a.v_rows) * a.v_rows;
        xsl[e] = (t < tc && i < vn) ? E::load1_cg(a.X, int64_t(t0 + t) * d + v0 + i) : 0.f;
      }
      if (!v_waited) {
        if (!__all_sync(0xffffffffu, bar_wait(vbar, 0, a.err))) ok = false;
        v_waited = true;
      }
      __syncthreads();
      if (warp < TC) {
        float sq = 0.f;
        for (int i = lane; i < vn; i += 32) sq = fmaf(xsl[warp * a.v_rows + i], xsl[warp * a.v_rows + i], sq);
        sq = warp_sum(sq);
        if (lane == 0) xsq[warp] = sq;
      }
      {
        // thread (group g, vector w): 16-byte vector w of rows g, g + ngrp, ...
        const int vecs = mrow_b / 16;
        const int grp_id = tid / vecs, w = tid - (tid / vecs) * vecs;
        if (ok && grp_id < a.ngrp) {
          float acc[TC][PV];
#pragma unroll
          for (int t = 0; t < TC; ++t)
#pragma unroll
            for (int e = 0; e < PV; ++e) acc[t][e] = 0.f;
          int i = grp_id;
          for (; i + a.ngrp < vn; i += 2 * a.ngrp) {
            const uint4 u0 = *reinterpret_cast<const uint4*>(Vs + int64_t(i) * mrow_b + 16 * w);
            const uint4 u1 = *reinterpret_cast<const uint4*>(Vs + int64_t(i + a.ngrp) * mrow_b + 16 * w);
#pragma unroll
            for (int t = 0; t < TC; ++t) {
              E::axpy(u0, xsl[t * a.v_rows + i], acc[t]);  // rows i, then i + ngrp
              E::axpy(u1, xsl[t * a.v_rows + i + a.ngrp], acc[t]);
            }
          }
          if (i < vn) {
            const uint4 u0 = *reinterpret_cast<const uint4*>(Vs + int64_t(i) * mrow_b + 16 * w);
#pragma unroll
            for (int t = 0; t < TC; ++t) E::axpy(u0, xsl[t * a.v_rows + i], acc[t]);
          }
#pragma unroll
          for (int t = 0; t < TC; ++t)
#pragma unroll
            for (int e = 0; e < PV; e += 4)
              *reinterpret_cast<float4*>(&red2[(grp_id * TC + t) * k + w * PV + e]) =
                  make_float4(acc[t][e], acc[t][e + 1], acc[t][e + 2], acc[t][e + 3]);
        }
      }
      __syncthreads();
      if (a.cproj) {
        // The V slice has been read: the M rows take its place (bulk copy,
        // from L2 when the previous call staged them there).
        if (stage_m && tid == kApplyThreads - 32) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          const uint32_t bytes = uint32_t(nrows) * mrow_b;
          bar_expect_tx(mfull, bytes);
          bulk_g2s(Ms, static_cast<const char*>(a.M) + r0 * mrow_b, bytes, mfull);
        }
        // this CTA's partial g (rows [v0, v0 + vn) of V), then an all-to-all
        // inside the cluster: every CTA receives every rank's partial g and
        // ||x||^2 slice (st.async, completion on its own mbarrier) and adds
        // them in rank order -- the full g, the same bits in every CTA and,
        // as every cluster does the same arithmetic, in every cluster
        for (int e = tid; e < TC * k; e += blockDim.x) {
          float s2 = 0.f;
          for (int g = 0; g < a.ngrp; ++g) s2 += red2[g * TC * k + e];
          pg[e] = s2;
        }
        if (!started) {
          cluster_wait();  // every CTA of the cluster is running: peers' shared memory is live
          started = true;
        }
        __syncthreads();
        const uint32_t aph = uint32_t(t0 / TC) & 1u;
        if (tid == 0) bar_expect_tx(gx_bar, uint32_t(CS * TC * (k + 1) * 4));
        const int n4 = TC * k / 4;
        for (int e = tid; e < CS * n4; e += blockDim.x) {
          const int q = e / n4, f4 = e - (e / n4) * n4;
          st_async_v4(map_rank(sa(inbox + rank * TC * k + 4 * f4), q),
                      *reinterpret_cast<const float4*>(pg + 4 * f4), map_rank(sa(gx_bar), q));
        }
        if (tid < TC * CS) {
          const int t = tid % TC, q = tid / TC;
          st_async_f32(map_rank(sa(inbox_x + rank * TC + t), q), xsq[t], map_rank(sa(gx_bar), q));
        }
        if (!__all_sync(0xffffffffu, bar_wait_cluster(gx_bar, aph, a.err))) ok = false;
        for (int e = tid; e < TC * k; e += blockDim.x) {
          float s2 = 0.f;
#pragma unroll
          for (int r = 0; r < CS; ++r) s2 += inbox[r * TC * k + e];
          gfull[e] = e / k < tc ? s2 : 0.f;
        }
        if (tid < TC) {
          float s2 = 0.f;
#pragma unroll
          for (int r = 0; r < CS; ++r) s2 += inbox_x[r * TC + tid];
          nx2[tid] = s2;
        }
        ok = __syncthreads_and(ok) != 0;
      } else {
      // this CTA's partials to the workspace, laid out like the projection
      // kernel's cluster partials (one "cluster" per CTA)
      for (int e = tid; e < TC * k; e += blockDim.x) {
        if (e / k < tc) {
          float s2 = 0.f;
          for (int g = 0; g < a.ngrp; ++g) s2 += red2[g * TC * k + e];
          a.fpart_g[(int64_t(blockIdx.x) * T + t0) * k + e] = s2;
        }
      }
      if (tid < tc) a.fpart_x[int64_t(blockIdx.x) * T + t0 + tid] = xsq[tid];
      __syncthreads();
      // every CTA's partials of this chunk are published
      if (tid == 0 && !grid_barrier(a.ticket, gridDim.x, a.err)) ok = false;
      ok = __syncthreads_and(ok) != 0;
      }
    }
    // the cluster projection already holds the full g
    const bool have_g = FUSED && a.cproj;
    if (a.mode != 2 && !have_g) {
      // -- g: this CTA's column slice summed over the published partials
      //    (the projection clusters', or every CTA's of a fused grid) in one
      //    fixed order.  Thread (g, e) takes column e (consecutive threads:
      //    consecutive columns, so a warp's loads are contiguous) and adds
      //    partials g, g + grp, ... (16 loads in flight); the grp sums of a
      //    column are then added in g order.  Every cluster gets the same bits.
      // decode chunks: warp 0 issues its loads of the ||x||^2 partials first,
      // so they are in flight together with the loads of g's partials
      constexpr bool kXEarly = TC <= 2;
      float xpart[kXEarly ? TC : 1][8];
      const bool x_early = kXEarly && a.nclu <= 256;
      if (kXEarly && x_early && warp == 0) {
#pragma unroll
        for (int t = 0; t < (kXEarly ? TC : 1); ++t)
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int cl = lane + 32 * u;
            xpart[t][u] = (t < tc && cl < a.nclu) ? __ldcg(&a.part_x[int64_t(cl) * T + t0 + t]) : 0.f;
          }
      }
      if (grp > 1) {
        if (tid < E_ * grp) {
          const int g = tid / E_, e = tid - (tid / E_) * E_;
          const int t = e / ks, col = c0 + (e - (e / ks) * ks);
          float s = 0.f;
          if (t < tc && col < c1) {
            const float* src = a.part_g + int64_t(t0 + t) * k + col;
            for (int cb = g; cb < a.nclu; cb += 16 * grp) {
              float v[16];
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const int cl = cb + u * grp;
                v[u] = cl < a.nclu ? __ldcg(src + int64_t(cl) * cstride) : 0.f;
              }
#pragma unroll
              for (int u = 0; u < 16; ++u) s += v[u];
            }
          }
          red3[tid] = s;
        }
        __syncthreads();
        if (tid < E_) {
          float s = 0.f;
          for (int g = 0; g < grp; ++g) s += red3[g * E_ + tid];
          const int t = tid / ks, col = c0 + (tid - (tid / ks) * ks);
          gsl[tid] = (t < tc && col < c1) ? s : 0.f;
        }
      } else {
        for (int e = tid; e < E_; e += kApplyThreads) {
          const int t = e / ks, col = c0 + (e - (e / ks) * ks);
          float s = 0.f;
          if (t < tc && col < c1) {
            const float* src = a.part_g + int64_t(t0 + t) * k + col;
            for (int cb = 0; cb < a.nclu; cb += 16) {
              float v[16];
#pragma unroll
              for (int u = 0; u < 16; ++u) v[u] = cb + u < a.nclu ? __ldcg(src + int64_t(cb + u) * cstride) : 0.f;
#pragma unroll
              for (int u = 0; u < 16; ++u) s += v[u];
            }
          }
          gsl[e] = (t < tc && col < c1) ? s : 0.f;
        }
      }
      if (warp == 0) {
        // ||x||^2: lane l adds partials l, l + 32, ... (8 in flight), then
        // the warp adds the lanes in a fixed order
#pragma unroll
        for (int t = 0; t < TC; ++t) {
          float s = 0.f;
          if (kXEarly && x_early) {
#pragma unroll
            for (int u = 0; u < 8; ++u) s += xpart[kXEarly ? t : 0][u];
          } else if (t < tc)
            for (int cb = lane; cb < a.nclu; cb += 32 * 8) {
              float v[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int cl = cb + 32 * u;
                v[u] = cl < a.nclu ? __ldcg(&a.part_x[int64_t(cl) * T + t0 + t]) : 0.f;
              }
#pragma unroll
              for (int u = 0; u < 8; ++u) s += v[u];
            }
          s = warp_sum(s);
          if (lane == 0) nx2[t] = s;
        }
      }
    }
    if (a.mode != 2) {
      if (!started) {
        cluster_wait();  // every CTA of the cluster is running
        started = true;
      }
      __syncthreads();
      // push this CTA's slice of g into every CTA's full copy; each CTA
      // receives TC x k floats per chunk (the slices partition [0, k)).
      // (The cluster projection already has the full g in every CTA.)
      const uint32_t xph = uint32_t(t0 / TC) & 1u;
      if (!have_g) {
        if (tid == 0) bar_expect_tx(gx_bar, uint32_t(TC * k * 4));
        for (int e = tid; e < E_ * CS; e += blockDim.x) {
          const int q = e / E_, f = e - (e / E_) * E_;
          const int t = f / ks, col = c0 + (f - (f / ks) * ks);
          if (col < c1) st_async_f32(map_rank(sa(gfull + t * k + col), q), gsl[f], map_rank(sa(gx_bar), q));
        }
        if (!__all_sync(0xffffffffu, bar_wait_cluster(gx_bar, xph, a.err))) ok = false;
      }
      // -- ||g||^2 and g^T Gram g over this CTA's Gram rows
      float qa[TC], na[TC];
#pragma unroll
      for (int t = 0; t < TC; ++t) qa[t] = na[t] = 0.f;
      if (tid < 256) {
        for (int i = c0 + tid; i < c1; i += 256) {
#pragma unroll
          for (int t = 0; t < TC; ++t) na[t] = fmaf(gfull[t * k + i], gfull[t * k + i], na[t]);
        }
        if (a.gram && gram_smem) {
          if (!gram_waited && !bar_wait(gfull_bar, 0, a.err)) ok = false;
          gram_waited = true;
          for (int v = tid; v < gvec; v += 256) {
            const float4 gv = reinterpret_cast<const float4*>(gram_s)[v];
            const int i = c0 + v / k4, j = 4 * (v % k4);
#pragma unroll
            for (int t = 0; t < TC; ++t) {
              const float4 gj = *reinterpret_cast<const float4*>(gfull + t * k + j);
              float h = gv.x * gj.x;
              h = fmaf(gv.y, gj.y, h);
              h = fmaf(gv.z, gj.z, h);
              h = fmaf(gv.w, gj.w, h);
              qa[t] = fmaf(gfull[t * k + i], h, qa[t]);
            }
          }
        } else if (a.gram) {
          if (GRV > 0) {
#pragma unroll
            for (int u = 0; u < (GRV > 0 ? GRV : 1); ++u) {
              const int v = u * 256 + tid;
              if (v < gvec) {
                const int i = c0 + v / k4, j = 4 * (v % k4);
#pragma unroll
                for (int t = 0; t < TC; ++t) {
                  const float4 gj = *reinterpret_cast<const float4*>(gfull + t * k + j);
                  float h = gr[u].x * gj.x;
                  h = fmaf(gr[u].y, gj.y, h);
                  h = fmaf(gr[u].z, gj.z, h);
                  h = fmaf(gr[u].w, gj.w, h);
                  qa[t] = fmaf(gfull[t * k + i], h, qa[t]);
                }
              }
            }
          } else {
            for (int v = tid; v < gvec; v += 256) {
              const float4 gv = __ldg(reinterpret_cast<const float4*>(a.gram + int64_t(c0 + v / k4) * k) + (v % k4));
              const int i = c0 + v / k4, j = 4 * (v % k4);
#pragma unroll
              for (int t = 0; t < TC; ++t) {
                const float4 gj = *reinterpret_cast<const float4*>(gfull + t * k + j);
                float h = gv.x * gj.x;
                h = fmaf(gv.y, gj.y, h);
                h = fmaf(gv.z, gj.z, h);
                h = fmaf(gv.w, gj.w, h);
                qa[t] = fmaf(gfull[t * k + i], h, qa[t]);
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
      }
      __syncthreads();
      if (tid == 0) bar_expect_tx(qn_bar, uint32_t(CS * TC * 8));
      if (tid < TC * CS) {
        // this CTA's share of g^T Gram g and ||g||^2, pushed to every CTA
        const int t = tid % TC, dst = tid / TC;
        float q = 0.f, n = 0.f;
        for (int w = 0; w < 8; ++w) {
          q += qw[w * TC + t];
          n += nw[w * TC + t];
        }
        const uint32_t rb = map_rank(sa(qn_bar), dst);
        st_async_f32(map_rank(sa(qin + rank * TC + t), dst), q, rb);
        st_async_f32(map_rank(sa(nin + rank * TC + t), dst), n, rb);
      }
      // decide-and-apply: y = M g for every token of the chunk while the
      // shares travel (the decision only picks which rows are kept)
      if (yspec) {
        if (m_live && !m_waited && !bar_wait(mfull, 0, a.err)) ok = false;
        m_waited = m_waited || m_live;
        if (ok)
          fast_apply(tc, [](int f) { return f; }, [&](int t, int r, float v) { ybuf[t * a.rows_per_cta + r] = v; });
      }
      // warp 0 decides (the shares of all CS ranks have landed)
      if (warp == 0 && !__all_sync(0xffffffffu, bar_wait_cluster(qn_bar, xph, a.err))) ok = false;
      if (tid < TC) {
        int slow = 0;
        if (tid < tc) {
          float q = 0.f, n = 0.f;
#pragma unroll
          for (int r = 0; r < CS; ++r) {
            q += qin[r * TC + tid];
            n += nin[r * TC + tid];
          }
          if (!a.gram) q = n;  // orthonormal basis: ||V g||^2 = ||g||^2
          const float xx = nx2[tid];
          float rr = xx - 2.f * n + q;
          rr = rr < 0.f ? 0.f : rr;  // keeps NaN
          const float rho = xx == 0.f ? 0.f : sqrtf(rr / xx);
          slow = rho < a.eps ? 0 : 1;
          if (blockIdx.x == 0) {
            if (a.rho) a.rho[t0 + tid] = rho;
            a.flags[t0 + tid] = uint8_t(slow);
            if (a.flags_user) a.flags_user[t0 + tid] = uint8_t(slow);
          }
        }
        sflag[tid] = slow;
      }
      if (blockIdx.x == 0 && a.G) {
        for (int e = tid; e < tc * k; e += blockDim.x) a.G[int64_t(t0) * k + e] = gfull[e];
      }

    } else {
      // stored decision (gsi_apply): flags and g from the preceding gate
      for (int e = tid; e < TC * k; e += blockDim.x) {
        const int t = e / k;
        gfull[e] = t < tc ? __ldcg(&a.Gin[int64_t(t0) * k + e]) : 0.f;
      }
      if (tid < TC) sflag[tid] = tid < tc ? int(ld_cg_u8(a.flags_in + t0 + tid) != 0) : 0;
      __syncthreads();
    }
    // -- per-chunk token lists (every thread reads the same smem flags);
    //    decide-only calls apply nothing
    __syncwarp();  // warp 0's lanes wrote the chunk's flags
    if (tid == 0) {
      int nf = 0, ns = 0;
      for (int t = 0; t < tc; ++t) {
        if (a.mode == 1) break;
        if (sflag[t])
          slist[ns++] = t;
        else
          flist[nf++] = t;
      }
      scount[0] = ok ? nf : 0;
      scount[1] = ok ? ns : 0;
    }
    __syncthreads();
    // (mode 3 leaves the slow rows to the tensor-core contraction that follows)
    const int nf = scount[0], ns = a.mode == 3 ? 0 : scount[1];

    // -- fast tokens: y = M g.  Decide-and-apply calls computed it for every
    //    token of the chunk while the decision's last exchange was in flight
    //    (yspec): copy the fast tokens' rows out; otherwise compute it now.
    if (nf > 0 && nrows > 0) {
      if (yspec) {
        for (int f = 0; f < nf; ++f) {
          const int t = flist[f];
          for (int r = tid; r < nrows; r += blockDim.x) a.Y[int64_t(t0 + t) * d_out + r0 + r] = ybuf[t * a.rows_per_cta + r];
        }
      } else {
        if (m_live && !m_waited && !bar_wait(mfull, 0, a.err)) ok = false;
        if (ok)
          fast_apply(nf, [&](int f) { return flist[f]; },
                     [&](int t, int r, float v) { a.Y[int64_t(t0 + t) * d_out + r0 + r] = v; });
      }
    }

    ok = __syncthreads_and(ok) != 0;
    if (nf > 0 && nrows > 0) m_waited = m_waited || m_live;
    // -- slow tokens: every warp streams its own rows of W (rows warp,
    //    warp + 8, ...) in segments through a private ring of bulk copies.
    //    The ring shares shared memory with the staged M rows: wait for that
    //    copy and retire the staged rows before the first segment lands.
    if (ns > 0 && nrows > 0 && ok) {
      const int nxs = min(ns, a.x_stage_max);
      if (m_live) {
        if (tid == 0 && !m_waited && !bar_wait(mfull, 0, a.err)) ok = false;
        m_live = false;
        m_waited = true;
      }
      // the staged M rows are retired: the rings may overwrite them
      const bool ring_ok = __syncthreads_and(ok) != 0;
      const int nwarp = kApplyThreads / 32;
      const int seg_b = a.seg_bytes;
      const int SW = a.wstages;
      const int nseg = int((row_b + seg_b - 1) / seg_b);
      const int my_rows = warp < nrows ? (nrows - warp + nwarp - 1) / nwarp : 0;
      const int items = ring_ok ? my_rows * nseg : 0;
      unsigned char* wring = Ms + int64_t(warp) * SW * seg_b;
      uint64_t* wfull = full + warp * SW;
      const char* wbase = static_cast<const char*>(a.W) + r0 * row_b;
      // Item q of this warp is segment q % nseg of its row q / nseg (CTA row
      // warp + (q / nseg) * nwarp), in ring slot (wuse + q) % SW.  The copy
      // issuer (lane 0) and the consumer step through the items with
      // counters, so the loop does no integer division.
      int q_row = 0, q_seg = 0, q_slot = wuse % SW;  // next item to issue (lane 0)
      auto issue_next = [&]() {
        const int64_t offq = int64_t(q_seg) * seg_b;
        const uint32_t bytes = uint32_t(min(int64_t(seg_b), row_b - offq));
        bar_expect_tx(&wfull[q_slot], bytes);
        bulk_g2s(wring + q_slot * seg_b, wbase + (int64_t(warp) + int64_t(q_row) * nwarp) * row_b + offq, bytes,
                 &wfull[q_slot]);
        if (++q_seg == nseg) {
          q_seg = 0;
          ++q_row;
        }
        if (++q_slot == SW) q_slot = 0;
      };
      int issued = min(items, SW);  // warp-uniform
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        for (int q = 0; q < issued; ++q) issue_next();
      }
      // the slow tokens' x is staged while the first segments of W are in flight
      const int64_t xv = row_b / 16;
      for (int64_t e = tid; e < int64_t(nxs) * xv; e += blockDim.x) {
        const int j = int(e / xv);
        const int64_t v = e - int64_t(j) * xv;
        reinterpret_cast<uint4*>(xst)[e] =
            ld_cg_v4(static_cast<const char*>(a.X) + int64_t(t0 + slist[j]) * row_b + v * 16);
      }
      __syncthreads();
      // two partial sums per token, added at the row's end
      float acc[TC][2];
#pragma unroll
      for (int t = 0; t < TC; ++t) acc[t][0] = acc[t][1] = 0.f;
      int c_slot = wuse % SW, c_row = 0, c_seg = 0;
      uint32_t c_ph = uint32_t(wuse / SW) & 1u;
      int i = 0;
      for (; i < items; ++i) {
        if (!__all_sync(0xffffffffu, bar_wait(&wfull[c_slot], c_ph, a.err))) {
          ok = false;
          break;
        }
        const int64_t off = int64_t(c_seg) * seg_b;
        const int nvec = int(min(int64_t(seg_b), row_b - off) / 16);
        const unsigned char* segp = wring + c_slot * seg_b;
        // lane l takes 16-byte vectors l, l + 32, ... of the segment.  They
        // are copied to registers and the slot is refilled at once, so the
        // ring keeps SW segments in flight while the warp multiplies.
        const bool full_seg = nvec == kSegVecs * 32;
        uint4 wq[kSegVecs];
        if (full_seg) {
#pragma unroll
          for (int u = 0; u < kSegVecs; ++u) wq[u] = *reinterpret_cast<const uint4*>(segp + (u * 32 + lane) * 16);
        } else {
#pragma unroll
          for (int u = 0; u < kSegVecs; ++u) {
            const int v = u * 32 + lane;
            wq[u] = v < nvec ? *reinterpret_cast<const uint4*>(segp + v * 16) : make_uint4(0u, 0u, 0u, 0u);
          }
        }
        // the loaded values are in registers before the slot is handed back
        uint32_t dep = 0;
#pragma unroll
        for (int u = 0; u < kSegVecs; ++u) dep ^= wq[u].x;
        asm volatile("" ::"r"(dep) : "memory");
        __syncwarp();
        if (issued < items) {
          if (lane == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_next();
          }
          ++issued;
        }
        // x of each slow token: a batch of loads, then the multiplies
        auto dot = [&](auto full_c) {
          constexpr bool FULL = decltype(full_c)::value;
#pragma unroll
          for (int t = 0; t < TC; ++t) {
            if (t < ns) {
              uint4 xq[kSegVecs];
              if (t < nxs) {
                const unsigned char* xs = xst + int64_t(t) * row_b + off;
#pragma unroll
                for (int u = 0; u < kSegVecs; ++u) {
                  const int v = u * 32 + lane;
                  xq[u] = (FULL || v < nvec) ? *reinterpret_cast<const uint4*>(xs + v * 16) : make_uint4(0u, 0u, 0u, 0u);
                }
              } else {
                const char* xg = static_cast<const char*>(a.X) + int64_t(t0 + slist[t]) * row_b + off;
#pragma unroll
                for (int u = 0; u < kSegVecs; ++u) {
                  const int v = u * 32 + lane;
                  xq[u] = (FULL || v < nvec) ? ld_cg_v4(xg + v * 16) : make_uint4(0u, 0u, 0u, 0u);
                }
              }
#pragma unroll
              for (int u = 0; u < kSegVecs; ++u) E::dot_acc(wq[u], xq[u], acc[t][0], acc[t][1]);
            }
          }
        };
        if (full_seg)
          dot(BoolC<true>{});
        else
          dot(BoolC<false>{});
        if (++c_slot == SW) {
          c_slot = 0;
          c_ph ^= 1u;
        }
        if (++c_seg == nseg) {
#pragma unroll
          for (int t = 0; t < TC; ++t) {
            if (t < ns) {
              const float sum = warp_sum(acc[t][0] + acc[t][1]);
              if (lane == 0) a.Y[int64_t(t0 + slist[t]) * d_out + r0 + warp + int64_t(c_row) * nwarp] = sum;
            }
            acc[t][0] = acc[t][1] = 0.f;
          }
          c_seg = 0;
          ++c_row;
        }
      }
      // after an error: wait (bounded) for this warp's copies still in flight
      if (lane == 0)
        for (int q = i; q < issued; ++q) {
          bar_wait(&wfull[c_slot], c_ph, a.err);
          if (++c_slot == SW) {
            c_slot = 0;
            c_ph ^= 1u;
          }
        }
      wuse += issued;
    }
    // another chunk follows: stop applying if any CTA has met an error
    // (the last chunk skips this read of the error word, an L2 round trip)
    if (t0 + TC < T) ok = __syncthreads_and(ok && *reinterpret_cast<volatile uint32_t*>(a.err) == 0) != 0;
    // every CTA of the cluster is done with this chunk's g copy and shares
    // before the next chunk's pushes; after an error the remaining chunks
    // only pass through their barriers (a CTA leaving early would strand the
    // cluster's other CTAs at a barrier)
    if (t0 + TC < T) cluster.sync();
  }

  if ((a.mode == 1 || a.mode == 3) && blockIdx.x == 0) {
    __threadfence();
    __syncthreads();
    if (warp == 0) compact_warp(a.flags, T, a.idx, a.counts, lane);
  }
  if (!started) cluster_wait();
  if (gram_smem && tid < 256 && !gram_waited) bar_wait(gfull_bar, 0, a.err);
  if (!v_waited && tid == 0) bar_wait(vbar, 0, a.err);
  // bounded drain of the M copy if it was never waited for
  if (stage_m && !m_waited && tid == 0) bar_wait(mfull, 0, a.err);
}

template <class E, int TC, bool FUSED, int CS>
static cudaError_t launch_da_t(const DecideArgs& a, const DecidePlan& p, cudaStream_t s) {
  auto kern = decide_apply_kernel<E, TC, 0, FUSED, CS>;
  static size_t smem_set = 0;
  if (p.smem > smem_set) {
    cudaError_t e = set_kernel_smem(kern, p.smem);
    if (e != cudaSuccess) return e;
    if (CS > 8 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
      return e;
    smem_set = p.smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(p.ncta));
  cfg.blockDim = dim3(kApplyThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CS;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  // the fused form without the cluster projection meets at a grid barrier
  static int no_coop = 0;
  return launch_maybe_coop(cfg, attr, 2, FUSED && !a.cproj, &no_coop, kern, a);
}

template <class E, bool FUSED, int CS>
static cudaError_t launch_da_f(const DecideArgs& a, const DecidePlan& p, cudaStream_t s) {
  switch (p.tc) {
    case 1: return launch_da_t<E, 1, FUSED, CS>(a, p, s);
    case 2: return launch_da_t<E, 2, FUSED, CS>(a, p, s);
    case 4: return launch_da_t<E, 4, FUSED, CS>(a, p, s);
    default: return launch_da_t<E, 8, FUSED, CS>(a, p, s);
  }
}

template <class E>
static cudaError_t launch_da_e(const DecideArgs& a, const DecidePlan& p, cudaStream_t s) {
  if (!p.fused) return launch_da_f<E, false, 8>(a, p, s);
  if (p.tc > 2) return cudaErrorInvalidValue;  // the fused decode handles one chunk of at most 2 tokens
  if (p.cs == 16) return p.tc == 1 ? launch_da_t<E, 1, true, 16>(a, p, s) : launch_da_t<E, 2, true, 16>(a, p, s);
  return p.tc == 1 ? launch_da_t<E, 1, true, 8>(a, p, s) : launch_da_t<E, 2, true, 8>(a, p, s);
}

cudaError_t launch_decide_apply(const DecideArgs& a, const DecidePlan& p, gsi_dtype dt, cudaStream_t s) {
  return dt == GSI_BF16 ? launch_da_e<BF16>(a, p, s) : launch_da_e<F32>(a, p, s);
}

// Co-resident clusters of cs CTAs of the decide-and-apply kernel with `smem`
// bytes of shared memory each (the grid size of a plan); 0 if not possible.
template <class E, bool FUSED, int CS>
static int max_clusters_t(size_t smem) {
  auto kern = decide_apply_kernel<E, 1, 0, FUSED, CS>;
  if (set_kernel_smem(kern, smem) != cudaSuccess) return 0;
  if (CS > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS * 64);
  cfg.blockDim = dim3(kApplyThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int decide_apply_max_clusters(size_t smem, gsi_dtype dt, bool fused, int cs) {
  if (dt == GSI_BF16) {
    if (!fused) return max_clusters_t<BF16, false, 8>(smem);
    return cs == 16 ? max_clusters_t<BF16, true, 16>(smem) : max_clusters_t<BF16, true, 8>(smem);
  }
  if (!fused) return max_clusters_t<F32, false, 8>(smem);
  return cs == 16 ? max_clusters_t<F32, true, 16>(smem) : max_clusters_t<F32, true, 8>(smem);
}

}  // namespace gsi
