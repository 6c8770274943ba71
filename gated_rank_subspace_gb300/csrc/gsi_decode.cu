// Single-token decode kernel: the whole gated map for one token in one launch.
//
// "Gated Subspace Inference for Transformer Acceleration", §2.1-§2.2: for a
// token x, g = V_k^T x, rho = ||x - V_k g|| / ||x||; rho < eps takes the fast
// path y = M g (M = W V_k, the cached image), rho >= eps the exact y = W x.
//
// This is the batch-1 decode form.  Where the basis fits a cluster, each
// cluster of 16 CTAs holds all of V_k in shared memory and finds g on its
// own (cluster projection: no CTA waits on another cluster).  Larger bases
// are split over the whole grid (grid projection): each cluster reduces its
// CTAs' partials by a reduce-scatter in distributed shared memory and every
// rank publishes its slice of columns as epoch-tagged 64-bit words; rank q
// of every cluster polls the clusters' words of its slice until they carry
// the call's epoch, adds them in cluster order and gathers g inside its
// cluster.  No grid-wide barrier: the epoch comes from a ticket each CTA
// takes in its prologue.  Both forms give every CTA the same bits of g.
//
//   prologue   each warp bulk-copies its own rows of the rank's V slab (one
//              mbarrier per warp); the Gram slice and the CTA's M rows follow.
//              All of this is weight traffic, issued before the dependency
//              wait on the previous kernel of the stream.
//   project    lane l of warp w loads token element v0 + w*rw + l and
//              leaves it in the warp's slot of shared memory; the warp walks
//              its V rows in batches of eight (four when a lane holds two
//              vectors; vectors and elements loaded first) and keeps one
//              16-byte column group of g per lane (two for rows longer than
//              512 bytes); ||x||^2 is a warp sum.  Each warp leaves its
//              partial in the space of its own, consumed, V rows.
//   exchange   thread c adds the eight warps' partials of column c and
//              pushes the sum to the rank that owns the column (a
//              reduce-scatter by st.async, completion on the receiver's
//              mbarrier); each rank adds its 16 inboxes in rank order and
//              pushes its slice of g to every rank (an all-gather) -- the
//              same bits in every CTA of every cluster.
//   decide     warp w takes Gram rows c0 + w, c0 + w + 8, ... of the rank's
//              slice: its share of g^T (V_k^T V_k) g and of ||g||^2 goes to
//              every rank at once, and the warp goes on to y = M g for its
//              own groups of 4, 8 or 16 output rows.  Every warp then adds all
//              ranks' shares in one fixed order, so all warps of all CTAs
//              reach the same rho = sqrt(||x||^2 - 2||g||^2 + g^T G g) / ||x||
//              and flag with no block-wide barrier.
//   apply      fast: each warp writes its own y rows.  Slow: the eight
//              warps stream the CTA's W rows (warp w: rows w, w + 8, ...)
//              through per-warp rings of bulk copies that reuse the V and M
//              space (as deep as shared memory allows, up to six 4 KB
//              slots a warp), with the token staged in shared memory.  (An
//              L2 prefetch of the segments ahead of the rings was measured
//              slower at every distance tried.)
//
// The persistent stack kernel runs this call for each map of a list in one
// launch (the maps of a layer, or of several layers), with a grid barrier
// between consecutive maps; a CTA sets up the next map's barriers and weight
// copies while the rest of the grid finishes the current map.
//
// Every wait is bounded (~2 s of clock): on expiry the workspace error word
// is set and the kernel carries on to its end without further waits on that
// barrier.  There are no float atomics; every sum has one fixed order.

#include "gsi_async.cuh"
#include "gsi_common.cuh"
#include "gsi_kernels.h"
#include "gsi_plan.h"

namespace gsi {

// One map's call, split so that a kernel can run one call (decode_kernel) or
// a list of calls (stack_decode_kernel):
//   decode_init_bars    mbarriers and the exchanges' byte counts;
//   decode_issue_copies the weight copies (V slab rows, Gram slice, M rows);
//   decode_prefetch_l2  this CTA's share of another map's weights into L2;
//   decode_run          everything after the dependency wait.
// NV: 16-byte vectors of a V / M row per lane (1: a row of at most 512 bytes,
// 2: up to 1 KB, e.g. k = 320 or 512 in bf16).

struct DecodeBars {
  uint64_t* vbar;   // [NW] V rows of warp w
  uint64_t* gbar;   // Gram slice
  uint64_t* mbar;   // M rows
  uint64_t* xbar;   // every rank's partial g and ||x||^2
  uint64_t* qbar;   // every rank's Gram and norm shares
  uint64_t* gxbar;  // g and ||x||^2 gathered from the ranks
  uint64_t* ring;   // [NW][sw] W segments
  uint32_t* words;  // [kDecodeCtaWords] CTA words
  __device__ __forceinline__ explicit DecodeBars(unsigned char* smem) {
    constexpr int NW = kApplyThreads / 32;
    vbar = reinterpret_cast<uint64_t*>(smem);
    gbar = vbar + NW;
    mbar = vbar + NW + 1;
    xbar = vbar + NW + 2;
    qbar = vbar + NW + 3;
    gxbar = vbar + NW + 4;
    ring = vbar + NW + kDecodeBars;
    words = reinterpret_cast<uint32_t*>(smem + kDecodeWordsOff);
  }
};

// One barrier per thread; the exchanges' byte counts are known now: every
// rank pushes the receiver's columns of its partial g and its ||x||^2, and
// two shares per warp; the gathered g and ||x||^2 are k + 1 floats.  The
// caller synchronises the block before any barrier is used.  `reinit`: the
// barriers of the previous call (quiescent: every copy and push into them
// has completed) are invalidated first.
__device__ __forceinline__ void decode_init_bars(const DecodeMap& m, unsigned char* smem, int tid, int rank,
                                                 bool reinit = false) {
  constexpr int NW = kApplyThreads / 32;
  constexpr int CS = kDecodeCluster;
  const DecodeBars b(smem);
  const int c0 = rank * m.ks, c1 = min(m.k, c0 + m.ks);
  if (tid < NW + kDecodeBars + NW * kDecodeMaxStages) {
    if (reinit) bar_inval(&b.vbar[tid]);
    bar_init(&b.vbar[tid], 1);
    if (tid == NW + 2) bar_expect_tx(b.xbar, uint32_t(CS * ((c1 > c0 ? c1 - c0 : 0) + 1) * 4));
    if (tid == NW + 3) bar_expect_tx(b.qbar, uint32_t(CS * NW * 2 * 4));
    if (tid == NW + 4) bar_expect_tx(b.gxbar, uint32_t((m.k + 1) * 4));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
}

// Weight copies of one call (after decode_init_bars and a block barrier):
// each warp its own rows of the rank's V slab, then the Gram slice and the
// CTA's M rows (unless they wait for the consumed V slab: m_late).
template <class E>
__device__ __forceinline__ void decode_issue_copies(const DecodeMap& m, unsigned char* smem, int tid, int lane,
                                                    int warp, int rank) {
  const DecodeBars b(smem);
  const int mrow_b = m.k * E::kBytes;
  const int64_t r0 = int64_t(blockIdx.x) * m.rpc;
  const int nrows = r0 >= m.d_out ? 0 : int(m.d_out - r0 < m.rpc ? m.d_out - r0 : m.rpc);
  const int64_t v0 = int64_t(m.grid ? int(blockIdx.x) : rank) * m.vr;
  const int vn = v0 >= m.d ? 0 : int(m.d - v0 < m.vr ? m.d - v0 : m.vr);
  const int wr0 = warp * m.rw;
  const int wrn = vn - wr0 < 0 ? 0 : (vn - wr0 < m.rw ? vn - wr0 : m.rw);
  const int c0 = rank * m.ks, c1 = min(m.k, c0 + m.ks);
  if (lane == 0 && wrn > 0) {
    const uint32_t bytes = uint32_t(wrn) * uint32_t(mrow_b);
    bar_expect_tx(&b.vbar[warp], bytes);
    bulk_g2s(smem + m.off_v + int64_t(wr0) * mrow_b, static_cast<const char*>(m.V) + (v0 + wr0) * mrow_b, bytes,
             &b.vbar[warp]);
  }
  if (tid == kApplyThreads - 32) {
    if (m.gram != nullptr && c1 > c0) {
      const uint32_t bytes = uint32_t(c1 - c0) * uint32_t(m.k) * 4u;
      bar_expect_tx(b.gbar, bytes);
      bulk_g2s(smem + m.off_gram, m.gram + int64_t(c0) * m.k, bytes, b.gbar);
    }
    if (nrows > 0 && !m.m_late) {
      const uint32_t bytes = uint32_t(nrows) * uint32_t(mrow_b);
      bar_expect_tx(b.mbar, bytes);
      bulk_g2s(smem + m.off_m, static_cast<const char*>(m.M) + r0 * mrow_b, bytes, b.mbar);
    }
  }
}

// This CTA's share of another map's V, M and Gram, into L2.
__device__ __forceinline__ void decode_prefetch_l2(const char* v, uint64_t vb, const char* mm, uint64_t mb,
                                                   const char* g, uint64_t gb, int tid) {
  if (tid == 64 || tid == 96 || tid == 128) {
    const char* base = tid == 64 ? v : tid == 96 ? mm : g;
    const uint64_t total = tid == 64 ? vb : tid == 96 ? mb : gb;
    if (base && total) {
      const uint64_t share = ((total + gridDim.x - 1) / gridDim.x + 15) / 16 * 16;
      const uint64_t off = uint64_t(blockIdx.x) * share;
      if (off < total) {
        const uint64_t rem = total - off;
        prefetch_l2(base + off, uint32_t(rem < share ? rem : share));
      }
    }
  }
}

// A call's geometry for this CTA and warp, from the map's plan alone: the
// kernels compute it before the dependency wait on the previous kernel, so
// none of this arithmetic sits between that wait and the token load.
struct DecodeGeom {
  int64_t r0;   // this CTA's output rows [r0, r0 + nrows)
  int64_t v0;   // this CTA's V rows [v0, v0 + vn)
  int nrows, vn;
  int wr0, wrn;  // this warp's rows of the slab
  int c0, c1;    // this rank's Gram rows
};

__device__ __forceinline__ DecodeGeom decode_geom(const DecodeMap& m, int rank, int warp) {
  DecodeGeom g;
  g.r0 = int64_t(blockIdx.x) * m.rpc;
  g.nrows = g.r0 >= m.d_out ? 0 : int(m.d_out - g.r0 < m.rpc ? m.d_out - g.r0 : m.rpc);
  g.v0 = int64_t(m.grid ? int(blockIdx.x) : rank) * m.vr;
  g.vn = g.v0 >= m.d ? 0 : int(m.d - g.v0 < m.vr ? m.d - g.v0 : m.vr);
  g.wr0 = warp * m.rw;
  g.wrn = g.vn - g.wr0 < 0 ? 0 : (g.vn - g.wr0 < m.rw ? g.vn - g.wr0 : m.rw);
  g.c0 = rank * m.ks;
  g.c1 = min(m.k, g.c0 + m.ks);
  return g;
}

// Everything of one call after the dependency wait: projection, exchanges,
// decision, apply.  `epoch` tags the grid projection's published words;
// `lim` bounds every wait (kSpinCycles, or the short limit after an error).
// Returns with every warp done with its shared memory and its copies.
template <class E, int NV>
__device__ __forceinline__ void decode_run(const DecodeMap& m, const DecodeGeom& geo, float eps, float* part_g_ws,
                                           float* part_x_ws, uint32_t epoch, uint32_t* err, long long lim,
                                           int withhold, long long poll_cycles, unsigned char* smem) {
  constexpr int PV = E::kPerVec;
  constexpr int CS = kDecodeCluster;
  constexpr int NW = kApplyThreads / 32;
  constexpr unsigned FULL = 0xffffffffu;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = int(cg::this_cluster().block_rank());
  // one instantiation for both projection forms: the four maps of a layer
  // then run the same code, which stays in the instruction cache
  const bool grid_proj = m.grid != 0;
  const int k = m.k;
  const int64_t d = m.d;
  const int mrow_b = k * E::kBytes;  // bytes of a V / M row
  const int nvec = mrow_b / 16;      // 16-byte vectors of such a row (<= 32 NV)
  const int nf4 = k >> 2;            // float4 groups of g
  const int64_t row_b = d * E::kBytes;

  const int64_t r0 = geo.r0, v0 = geo.v0;
  const int nrows = geo.nrows, wr0 = geo.wr0, wrn = geo.wrn, c0 = geo.c0, c1 = geo.c1;

  const DecodeBars b(smem);
  uint64_t* vbar = b.vbar;
  uint64_t* gbar = b.gbar;
  uint64_t* mbar = b.mbar;
  uint64_t* xbar = b.xbar;
  uint64_t* qbar = b.qbar;
  uint64_t* gxbar = b.gxbar;
  uint64_t* ring = b.ring;
  float* gfull = reinterpret_cast<float*>(smem + m.off_g);  // [k]
  float* inx = gfull + k;                                   // [CS] ||x||^2 partials
  float* qin = inx + CS;                                    // [CS][NW] g^T G g shares
  float* nin = qin + CS * NW;                               // [CS][NW] ||g||^2 shares
  float* nx2 = nin + CS * NW;                               // [1]
  float* xw = nx2 + 4;                                      // [NW][32] token elements of each warp
  float* ybuf = reinterpret_cast<float*>(smem + m.off_y);   // [rpc] y = M g
  float* inbox = reinterpret_cast<float*>(smem + m.off_in); // [CS][ks] partial-g slices; later the slow token
  const float* gram_s = reinterpret_cast<const float*>(smem + m.off_gram);  // [ks][k]
  unsigned char* Vs = smem + m.off_v;                       // V slab, then the W rings
  unsigned char* Ms = smem + m.off_m;                       // M rows
  float* red = reinterpret_cast<float*>(smem + m.off_red);  // warp w's partial at w * red_stride

  // ---- projection of this warp's rows
  const float xv = lane < wrn ? E::load1_cg(m.X, v0 + wr0 + lane) : 0.f;
  float* xme = xw + warp * 32;
  xme[lane] = xv;
  __syncwarp();
  const float xsq = warp_sum(xv * xv);
  // lane l owns column groups l and (NV = 2) l + 32 of g
  bool on[NV];
  int vl[NV];  // the lane's vectors, clamped to vector 0 where a row has fewer
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    on[v] = lane + 32 * v < nvec;
    vl[v] = on[v] ? lane + 32 * v : 0;
  }
  float acc[NV][PV];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int e = 0; e < PV; ++e) acc[v][e] = 0.f;
  if (wrn > 0) {
    __all_sync(FULL, bar_wait(&vbar[warp], 0, err, lim, kWaitV));
    // rows in batches of 8 / NV: the vectors and token elements are loaded
    // first, then multiplied in row order
    constexpr int RBT = 8 / NV;
    const unsigned char* vrows = Vs + int64_t(wr0) * mrow_b;
    int i = 0;
    for (; i + RBT <= wrn; i += RBT) {
      uint4 u[RBT][NV];
      float xi[RBT];
#pragma unroll
      for (int j = 0; j < RBT; ++j) {
#pragma unroll
        for (int v = 0; v < NV; ++v)
          u[j][v] = on[v] ? *reinterpret_cast<const uint4*>(vrows + int64_t(i + j) * mrow_b + vl[v] * 16)
                          : make_uint4(0u, 0u, 0u, 0u);
        xi[j] = xme[i + j];
      }
#pragma unroll
      for (int j = 0; j < RBT; ++j)
#pragma unroll
        for (int v = 0; v < NV; ++v) E::axpy(u[j][v], xi[j], acc[v]);
    }
    for (; i < wrn; ++i) {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const uint4 u = on[v] ? *reinterpret_cast<const uint4*>(vrows + int64_t(i) * mrow_b + vl[v] * 16)
                              : make_uint4(0u, 0u, 0u, 0u);
        E::axpy(u, xme[i], acc[v]);
      }
    }
  }
  __syncwarp();
  {
    float* mine = red + warp * m.red_stride;  // this warp's own (consumed) V rows, or a separate slot
#pragma unroll
    for (int v = 0; v < NV; ++v)
      if (on[v]) {
#pragma unroll
        for (int e = 0; e < PV; e += 4)
          *reinterpret_cast<float4*>(mine + vl[v] * PV + e) =
              make_float4(acc[v][e], acc[v][e + 1], acc[v][e + 2], acc[v][e + 3]);
      }
    if (lane == 0) mine[k] = xsq;
  }
  __syncthreads();
  if (m.m_late && nrows > 0 && tid == kApplyThreads - 32) {
    // the V slab is consumed: the M rows take its place
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t bytes = uint32_t(nrows) * uint32_t(mrow_b);
    bar_expect_tx(mbar, bytes);
    bulk_g2s(Ms, static_cast<const char*>(m.M) + r0 * mrow_b, bytes, mbar);
  }

  cluster_wait();  // every CTA of the cluster runs and has initialised its barriers
  // ---- reduce-scatter inside the cluster: rank q gets every rank's columns
  //      [q ks, (q + 1) ks) of the partial g, and every rank's ||x||^2
  const int ks = m.ks;
  for (int c = tid; c < k; c += kApplyThreads) {
    float s = red[c];
#pragma unroll
    for (int w = 1; w < NW; ++w) s += red[w * m.red_stride + c];
    const int q = c / ks;
    st_async_f32(map_rank(sa(inbox + rank * ks + (c - q * ks)), q), s, map_rank(sa(xbar), q));
  }
  if (tid < CS) {
    float s = red[k];
#pragma unroll
    for (int w = 1; w < NW; ++w) s += red[w * m.red_stride + k];
    st_async_f32(map_rank(sa(inx + rank), tid), s, map_rank(sa(xbar), tid));
  }
  __all_sync(FULL, bar_wait_cluster(xbar, 0, err, lim, kWaitPartials));
  // ---- this rank's slice of g (rank 0: also ||x||^2), summed over the ranks
  //      in rank order -- grid projection: then over the clusters, through
  //      epoch-tagged words -- and pushed to every rank of the cluster
  const bool xlane = tid == ks && rank == 0;
  if (tid < c1 - c0 || xlane) {
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < CS; ++r) s += xlane ? inx[r] : inbox[r * ks + tid];
    if (grid_proj) {
      const int cl = int(blockIdx.x) / CS, ncl = int(gridDim.x) / CS;
      unsigned long long* src = xlane ? reinterpret_cast<unsigned long long*>(part_x_ws)
                                      : reinterpret_cast<unsigned long long*>(part_g_ws) + c0 + tid;
      const int64_t stride = xlane ? 1 : k;  // [ncl][k] slices, [ncl] norms
      if (!(withhold && cl == 0)) st_relaxed_u64(src + cl * stride, (uint64_t(epoch) << 32) | __float_as_uint(s));
      // every cluster's word, polled until it carries this call's epoch
      // (bounded), added in cluster order
      float v[kDecodeMaxClusters];
      uint32_t pending = (1u << ncl) - 1u;
      const long long plim = poll_cycles > 0 ? poll_cycles : lim;
      const long long t0 = clock64();
      while (pending) {
        unsigned long long w[kDecodeMaxClusters];  // all loads in flight, then the checks
#pragma unroll
        for (int c = 0; c < kDecodeMaxClusters; ++c)
          w[c] = ((pending >> c) & 1u) ? ld_relaxed_u64(src + c * stride) : 0ull;
#pragma unroll
        for (int c = 0; c < kDecodeMaxClusters; ++c)
          if (((pending >> c) & 1u) && uint32_t(w[c] >> 32) == epoch) {
            v[c] = __uint_as_float(uint32_t(w[c]));
            pending &= ~(1u << c);
          }
        if (pending && clock64() - t0 > plim) {
          atomicOr(err, kErrTimeout | kWaitSlices);
          break;
        }
      }
      s = 0.f;
#pragma unroll
      for (int c = 0; c < kDecodeMaxClusters; ++c)
        if (c < ncl) s += ((pending >> c) & 1u) ? 0.f : v[c];
    }
    const uint32_t dst = sa(xlane ? nx2 : gfull + c0 + tid), bar = sa(gxbar);
    for (int q = 0; q < CS; ++q) st_async_f32(map_rank(dst, q), s, map_rank(bar, q));
  }
  __all_sync(FULL, bar_wait_cluster(gxbar, 0, err, lim, kWaitGathered));

  // ---- every warp: its share of the Gram form (Gram rows c0 + warp,
  //      c0 + warp + NW, ...) and of ||g||^2, pushed to every rank, then
  //      y = M g for its rows (groups of RB rows: RB warp, RB warp + RB NW, ...)
  const bool have_gram = m.gram != nullptr && c1 > c0;
  {
    float q = 0.f, n = 0.f;
    if (have_gram) {
      __all_sync(FULL, bar_wait(gbar, 0, err, lim, kWaitGram));
      // lane l takes column groups l, l + 32, ... (clamped loads, masked)
      constexpr int NG = 2 * NV;  // float4 groups of a Gram row per lane (k <= 256 NV)
      const float4* g4 = reinterpret_cast<const float4*>(gfull);
      bool og[NG];
      int jg[NG];
      float4 gq[NG];
#pragma unroll
      for (int u = 0; u < NG; ++u) {
        og[u] = lane + 32 * u < nf4;
        jg[u] = og[u] ? lane + 32 * u : 0;
        gq[u] = g4[jg[u]];
      }
      for (int i = c0 + warp; i < c1; i += NW) {
        const float4* grow = reinterpret_cast<const float4*>(gram_s) + (i - c0) * nf4;
        float4 vg[NG];
#pragma unroll
        for (int u = 0; u < NG; ++u) vg[u] = grow[jg[u]];
        const float gi = gfull[i];
        float h = 0.f;
#pragma unroll
        for (int u = 0; u < NG; ++u) {
          float hu = vg[u].x * gq[u].x;
          hu = fmaf(vg[u].y, gq[u].y, hu);
          hu = fmaf(vg[u].z, gq[u].z, hu);
          hu = fmaf(vg[u].w, gq[u].w, hu);
          h += og[u] ? hu : 0.f;
        }
        q = fmaf(gi, h, q);
      }
    }
    for (int i = c0 + warp; i < c1; i += NW) n = fmaf(gfull[i], gfull[i], n);
    q = warp_sum(q);
    if (lane < CS) {
      const uint32_t rb = map_rank(sa(qbar), lane);
      st_async_f32(map_rank(sa(qin + rank * NW + warp), lane), q, rb);
      st_async_f32(map_rank(sa(nin + rank * NW + warp), lane), n, rb);
    }
  }
  if (nrows > 0) {
    __all_sync(FULL, bar_wait(mbar, 0, err, lim, kWaitM));
    // lane l multiplies column group l of RB rows at a time; the row loads
    // are unconditional (rows past the CTA's last repeat it, lanes past the
    // row's vectors repeat vector 0) and masked afterwards, so all RB are in
    // flight together
    float gv[NV][PV];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int e = 0; e < PV; ++e) gv[v][e] = gfull[vl[v] * PV + e];
    auto apply_rows = [&](auto rb_c) {
      constexpr int RB = decltype(rb_c)::value;
      for (int rb = warp * RB; rb < nrows; rb += NW * RB) {
        uint4 u[RB][NV];
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
          for (int v = 0; v < NV; ++v)
            u[r][v] = *reinterpret_cast<const uint4*>(Ms + int64_t(min(rb + r, nrows - 1)) * mrow_b + vl[v] * 16);
        float part[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          part[r] = 0.f;
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            const float p = E::dot_vec(u[r][v], gv[v]);
            part[r] += on[v] ? p : 0.f;
          }
        }
        const float sum = warp_reduce_multi<RB>(part, lane);
        const int r = row_of_lane<RB>(lane);
        if ((lane & (32 / RB - 1)) == 0 && rb + r < nrows) ybuf[rb + r] = sum;
      }
    };
    if (nrows <= NW * 4)
      apply_rows(IntC<4>{});
    else if (nrows <= NW * 8 || NV > 1)  // (16 rows of two vectors: too many registers)
      apply_rows(IntC<8>{});
    else
      apply_rows(IntC<16 / NV>{});
  }
  // ---- the decision, taken by every warp from the same shares in the same
  //      order (lane l adds shares 4l .. 4l + 3 of the rank-major list, then
  //      a butterfly over the lanes)
  __all_sync(FULL, bar_wait_cluster(qbar, 0, err, lim, kWaitShares));
  static_assert(CS * NW == 4 * 32, "four shares per lane");
  const float4 q4 = reinterpret_cast<const float4*>(qin)[lane];
  const float4 n4 = reinterpret_cast<const float4*>(nin)[lane];
  const float Qr = (q4.x + q4.y) + (q4.z + q4.w);
  const float Nr = (n4.x + n4.y) + (n4.z + n4.w);
  float Q = warp_sum(Qr);
  const float N = warp_sum(Nr);
  if (!m.gram) Q = N;  // orthonormal basis: ||V g||^2 = ||g||^2
  const float xx = *nx2;
  float rr = xx - 2.f * N + Q;
  rr = rr < 0.f ? 0.f : rr;  // keeps NaN
  const float rho = xx == 0.f ? 0.f : sqrtf(rr / xx);
  const bool slow = !(rho < eps);
  if (blockIdx.x == 0 && tid == 0) {
    if (m.rho) m.rho[0] = rho;
    m.flags[0] = uint8_t(slow ? 1 : 0);
  }

  // ---- apply
  if (!slow) {
    // this warp's rows of y (the row groups it computed), from its own lanes
    __syncwarp();
    const int rbw = nrows <= NW * 4 ? 4 : (nrows <= NW * 8 || NV > 1) ? 8 : 16;
    for (int rb = warp * rbw; rb < nrows; rb += NW * rbw)
      if (lane < rbw && rb + lane < nrows) m.Y[r0 + rb + lane] = ybuf[rb + lane];
    return;
  }
  if (nrows == 0) return;
  // Slow token: the V slab, the partials and the M rows are consumed, so the
  // W rings take their space; the token goes where the inboxes were.
  const int seg_b = m.seg_bytes, SW = m.sw;
  const int nseg = int((row_b + seg_b - 1) / seg_b);
  const int my_rows = warp < nrows ? (nrows - warp + NW - 1) / NW : 0;
  const int items = my_rows * nseg;
  unsigned char* wring = Vs + int64_t(warp) * SW * seg_b;
  uint64_t* wfull = ring + warp * SW;
  const char* wbase = static_cast<const char*>(m.W) + r0 * row_b;
  // item q of this warp: segment q % nseg of its row q / nseg (CTA row
  // warp + (q / nseg) * NW), in ring slot q % SW; issuer and consumer step
  // through the items with counters
  int q_row = 0, q_seg = 0, q_slot = 0;
  auto issue_next = [&]() {
    const int64_t offq = int64_t(q_seg) * seg_b;
    const uint32_t bytes = uint32_t(min(int64_t(seg_b), row_b - offq));
    bar_expect_tx(&wfull[q_slot], bytes);
    bulk_g2s(wring + q_slot * seg_b, wbase + (int64_t(warp) + int64_t(q_row) * NW) * row_b + offq, bytes,
             &wfull[q_slot]);
    if (++q_seg == nseg) {
      q_seg = 0;
      ++q_row;
    }
    if (++q_slot == SW) q_slot = 0;
  };
  int issued = min(items, SW);
  __syncthreads();  // every warp is done with the V slab and the M rows
  if (lane == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int q = 0; q < issued; ++q) issue_next();
  }
  unsigned char* xst = reinterpret_cast<unsigned char*>(inbox);
  for (int64_t e = tid; e < row_b / 16; e += kApplyThreads)
    reinterpret_cast<uint4*>(xst)[e] = ld_cg_v4(static_cast<const char*>(m.X) + e * 16);
  __syncthreads();
  float acc0 = 0.f, acc1 = 0.f;
  int c_slot = 0, c_seg = 0, c_row = 0;
  uint32_t c_ph = 0;
  int i = 0;
  for (; i < items; ++i) {
    if (!__all_sync(FULL, bar_wait(&wfull[c_slot], c_ph, err, lim, kWaitRing))) break;
    const int64_t off = int64_t(c_seg) * seg_b;
    const int nv = int(min(int64_t(seg_b), row_b - off) / 16);
    const unsigned char* segp = wring + c_slot * seg_b;
    uint4 wq[kSegVecs];
#pragma unroll
    for (int u = 0; u < kSegVecs; ++u) {
      const int v = u * 32 + lane;
      wq[u] = v < nv ? *reinterpret_cast<const uint4*>(segp + v * 16) : make_uint4(0u, 0u, 0u, 0u);
    }
    // the segment is in registers before its slot is refilled
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
    const unsigned char* xs = xst + off;
#pragma unroll
    for (int u = 0; u < kSegVecs; ++u) {
      const int v = u * 32 + lane;
      const uint4 xq = v < nv ? *reinterpret_cast<const uint4*>(xs + v * 16) : make_uint4(0u, 0u, 0u, 0u);
      E::dot_acc(wq[u], xq, acc0, acc1);
    }
    if (++c_slot == SW) {
      c_slot = 0;
      c_ph ^= 1u;
    }
    if (++c_seg == nseg) {
      const float sum = warp_sum(acc0 + acc1);
      if (lane == 0) m.Y[r0 + warp + int64_t(c_row) * NW] = sum;
      acc0 = acc1 = 0.f;
      c_seg = 0;
      ++c_row;
    }
  }
  // after an expired wait: wait (bounded) for this warp's copies still in flight
  if (lane == 0)
    for (int q = i; q < issued; ++q) {
      bar_wait(&wfull[c_slot], c_ph, err, lim, kWaitRing);
      if (++c_slot == SW) {
        c_slot = 0;
        c_ph ^= 1u;
      }
    }
}

// The single-token call as its own kernel body: the same steps and the same
// arithmetic as decode_run (so the results are bitwise those of a stack
// launch), written out with every piece of geometry and every shared-memory
// address formed before the prologue (measured ~0.1 us a call faster than the
// shared function).
template <class E, int NV>
__global__ void __launch_bounds__(kApplyThreads, 1) decode_kernel(DecodeArgs a) {
  constexpr int PV = E::kPerVec;
  constexpr int CS = kDecodeCluster;
  constexpr int NW = kApplyThreads / 32;
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // (No launch-shape check here: reading the cluster size costs ~0.15 us on
  // a call's path.  Profilers that relaunch kernels must run with
  // GSI_COOPERATIVE=0, see the header.)
  const int rank = int(cg::this_cluster().block_rank());
  // one instantiation for both projection forms: the four maps of a layer
  // then run the same code, which stays in the instruction cache
  const bool grid_proj = a.m.grid != 0;
  const int k = a.m.k;
  const int64_t d = a.m.d, d_out = a.m.d_out;
  const int mrow_b = k * E::kBytes;  // bytes of a V / M row
  const int nvec = mrow_b / 16;      // 16-byte vectors of such a row (<= 32 NV)
  const int nf4 = k >> 2;            // float4 groups of g
  const int64_t row_b = d * E::kBytes;

  const int64_t r0 = int64_t(blockIdx.x) * a.m.rpc;  // this CTA's output rows
  const int nrows = r0 >= d_out ? 0 : int(d_out - r0 < a.m.rpc ? d_out - r0 : a.m.rpc);
  const int64_t v0 = int64_t(grid_proj ? int(blockIdx.x) : rank) * a.m.vr;  // this CTA's V rows
  const int vn = v0 >= d ? 0 : int(d - v0 < a.m.vr ? d - v0 : a.m.vr);
  const int wr0 = warp * a.m.rw;                     // this warp's rows of the slab
  const int wrn = vn - wr0 < 0 ? 0 : (vn - wr0 < a.m.rw ? vn - wr0 : a.m.rw);
  const int c0 = rank * a.m.ks, c1 = min(k, c0 + a.m.ks);  // this rank's Gram rows

  uint64_t* vbar = reinterpret_cast<uint64_t*>(smem);  // [NW] V rows of warp w
  uint64_t* gbar = vbar + NW;                          // Gram slice
  uint64_t* mbar = vbar + NW + 1;                      // M rows
  uint64_t* xbar = vbar + NW + 2;                      // every rank's partial g and ||x||^2
  uint64_t* qbar = vbar + NW + 3;                      // every rank's Gram and norm shares
  uint64_t* gxbar = vbar + NW + 4;                     // g and ||x||^2 gathered from the ranks
  uint64_t* ring = vbar + NW + kDecodeBars;            // [NW][sw] W segments
  float* gfull = reinterpret_cast<float*>(smem + a.m.off_g);  // [k]
  float* inx = gfull + k;                                   // [CS] ||x||^2 partials
  float* qin = inx + CS;                                    // [CS][NW] g^T G g shares
  float* nin = qin + CS * NW;                               // [CS][NW] ||g||^2 shares
  float* nx2 = nin + CS * NW;                               // [1]
  uint32_t* sepoch = reinterpret_cast<uint32_t*>(nx2 + 1);  // [1] grid projection: this call's epoch
  float* xw = nx2 + 4;                                      // [NW][32] token elements of each warp
  float* ybuf = reinterpret_cast<float*>(smem + a.m.off_y);   // [rpc] y = M g
  float* inbox = reinterpret_cast<float*>(smem + a.m.off_in); // [CS][ks] partial-g slices; later the slow token
  const float* gram_s = reinterpret_cast<const float*>(smem + a.m.off_gram);  // [ks][k]
  unsigned char* Vs = smem + a.m.off_v;                       // V slab, then the W rings
  unsigned char* Ms = smem + a.m.off_m;                       // M rows
  float* red = reinterpret_cast<float*>(smem + a.m.off_red);  // warp w's partial at w * red_stride

  // ---- prologue: weights only (may overlap the previous kernel's tail)
  // Grid projection: this CTA's ticket, taken before the next kernel of the
  // stream may start, numbers the call: every CTA of call e takes one of the
  // tickets [(e - 1) n, e n), n = the grid size, so epoch e = ticket / n + 1
  // is known to all of them without a barrier.
  // (The word carries the call number in its upper 24 bits and the map's
  // place in a launch, here 1, in the lower 8, as the persistent stack
  // kernel's do: the two kernels share the ticket counter and the words.)
  if (grid_proj && tid == 0) *sepoch = ((uint32_t(atomicAdd(a.ticket, 1ull) / gridDim.x) + 1u) << 8) | 1u;
  // one barrier per thread; the exchanges' byte counts are known now: every
  // rank pushes the receiver's columns of its partial g and its ||x||^2, and
  // two shares per warp; the gathered g and ||x||^2 are k + 1 floats
  if (tid < NW + kDecodeBars + NW * a.m.sw) {
    bar_init(&vbar[tid], 1);
    if (tid == NW + 2) bar_expect_tx(xbar, uint32_t(CS * ((c1 > c0 ? c1 - c0 : 0) + 1) * 4));
    if (tid == NW + 3) bar_expect_tx(qbar, uint32_t(CS * NW * 2 * 4));
    if (tid == NW + 4) bar_expect_tx(gxbar, uint32_t((k + 1) * 4));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_launch_dependents();
  if (lane == 0 && wrn > 0) {
    const uint32_t bytes = uint32_t(wrn) * uint32_t(mrow_b);
    bar_expect_tx(&vbar[warp], bytes);
    bulk_g2s(Vs + int64_t(wr0) * mrow_b, static_cast<const char*>(a.m.V) + (v0 + wr0) * mrow_b, bytes, &vbar[warp]);
  }
  const bool have_gram = a.m.gram != nullptr && c1 > c0;
  if (tid == kApplyThreads - 32) {
    if (have_gram) {
      const uint32_t bytes = uint32_t(c1 - c0) * uint32_t(k) * 4u;
      bar_expect_tx(gbar, bytes);
      bulk_g2s(smem + a.m.off_gram, a.m.gram + int64_t(c0) * k, bytes, gbar);
    }
    if (nrows > 0 && !a.m.m_late) {
      const uint32_t bytes = uint32_t(nrows) * uint32_t(mrow_b);
      bar_expect_tx(mbar, bytes);
      bulk_g2s(Ms, static_cast<const char*>(a.m.M) + r0 * mrow_b, bytes, mbar);
    }
  }
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
  cluster_arrive_relaxed();
  pdl_wait();

  // ---- projection of this warp's rows
  const float xv = lane < wrn ? E::load1_cg(a.m.X, v0 + wr0 + lane) : 0.f;
  float* xme = xw + warp * 32;
  xme[lane] = xv;
  __syncwarp();
  const float xsq = warp_sum(xv * xv);
  // lane l owns column groups l and (NV = 2) l + 32 of g
  bool on[NV];
  int vl[NV];  // the lane's vectors, clamped to vector 0 where a row has fewer
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    on[v] = lane + 32 * v < nvec;
    vl[v] = on[v] ? lane + 32 * v : 0;
  }
  float acc[NV][PV];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int e = 0; e < PV; ++e) acc[v][e] = 0.f;
  if (wrn > 0) {
    __all_sync(FULL, bar_wait(&vbar[warp], 0, a.err, kSpinCycles, kWaitV));
    // rows in batches of 8 / NV: the vectors and token elements are loaded
    // first, then multiplied in row order
    constexpr int RBT = 8 / NV;
    const unsigned char* vrows = Vs + int64_t(wr0) * mrow_b;
    int i = 0;
    for (; i + RBT <= wrn; i += RBT) {
      uint4 u[RBT][NV];
      float xi[RBT];
#pragma unroll
      for (int j = 0; j < RBT; ++j) {
#pragma unroll
        for (int v = 0; v < NV; ++v)
          u[j][v] = on[v] ? *reinterpret_cast<const uint4*>(vrows + int64_t(i + j) * mrow_b + vl[v] * 16)
                          : make_uint4(0u, 0u, 0u, 0u);
        xi[j] = xme[i + j];
      }
#pragma unroll
      for (int j = 0; j < RBT; ++j)
#pragma unroll
        for (int v = 0; v < NV; ++v) E::axpy(u[j][v], xi[j], acc[v]);
    }
    for (; i < wrn; ++i) {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const uint4 u = on[v] ? *reinterpret_cast<const uint4*>(vrows + int64_t(i) * mrow_b + vl[v] * 16)
                              : make_uint4(0u, 0u, 0u, 0u);
        E::axpy(u, xme[i], acc[v]);
      }
    }
  }
  __syncwarp();
  {
    float* mine = red + warp * a.m.red_stride;  // this warp's own (consumed) V rows, or a separate slot
#pragma unroll
    for (int v = 0; v < NV; ++v)
      if (on[v]) {
#pragma unroll
        for (int e = 0; e < PV; e += 4)
          *reinterpret_cast<float4*>(mine + vl[v] * PV + e) =
              make_float4(acc[v][e], acc[v][e + 1], acc[v][e + 2], acc[v][e + 3]);
      }
    if (lane == 0) mine[k] = xsq;
  }
  __syncthreads();
  if (a.m.m_late && nrows > 0 && tid == kApplyThreads - 32) {
    // the V slab is consumed: the M rows take its place
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t bytes = uint32_t(nrows) * uint32_t(mrow_b);
    bar_expect_tx(mbar, bytes);
    bulk_g2s(Ms, static_cast<const char*>(a.m.M) + r0 * mrow_b, bytes, mbar);
  }
  cluster_wait();  // every CTA of the cluster runs and has initialised its barriers
  // ---- reduce-scatter inside the cluster: rank q gets every rank's columns
  //      [q ks, (q + 1) ks) of the partial g, and every rank's ||x||^2
  const int ks = a.m.ks;
  for (int c = tid; c < k; c += kApplyThreads) {
    float s = red[c];
#pragma unroll
    for (int w = 1; w < NW; ++w) s += red[w * a.m.red_stride + c];
    const int q = c / ks;
    st_async_f32(map_rank(sa(inbox + rank * ks + (c - q * ks)), q), s, map_rank(sa(xbar), q));
  }
  if (tid < CS) {
    float s = red[k];
#pragma unroll
    for (int w = 1; w < NW; ++w) s += red[w * a.m.red_stride + k];
    st_async_f32(map_rank(sa(inx + rank), tid), s, map_rank(sa(xbar), tid));
  }
  __all_sync(FULL, bar_wait_cluster(xbar, 0, a.err, kSpinCycles, kWaitPartials));
  // ---- this rank's slice of g (rank 0: also ||x||^2), summed over the ranks
  //      in rank order -- grid projection: then over the clusters, through
  //      epoch-tagged words -- and pushed to every rank of the cluster
  const bool xlane = tid == ks && rank == 0;
  if (tid < c1 - c0 || xlane) {
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < CS; ++r) s += xlane ? inx[r] : inbox[r * ks + tid];
    if (grid_proj) {
      const int cl = int(blockIdx.x) / CS, ncl = int(gridDim.x) / CS;
      const uint32_t epoch = *sepoch;
      unsigned long long* src = xlane ? reinterpret_cast<unsigned long long*>(a.part_x)
                                      : reinterpret_cast<unsigned long long*>(a.part_g) + c0 + tid;
      const int64_t stride = xlane ? 1 : k;  // [ncl][k] slices, [ncl] norms
      if (!(a.dbg_withhold && cl == 0)) st_relaxed_u64(src + cl * stride, (uint64_t(epoch) << 32) | __float_as_uint(s));
      // every cluster's word, polled until it carries this call's epoch
      // (bounded), added in cluster order
      float v[kDecodeMaxClusters];
      uint32_t pending = (1u << ncl) - 1u;
      const long long plim = a.poll_cycles > 0 ? a.poll_cycles : kSpinCycles;
      const long long t0 = clock64();
      while (pending) {
        unsigned long long w[kDecodeMaxClusters];  // all loads in flight, then the checks
#pragma unroll
        for (int c = 0; c < kDecodeMaxClusters; ++c)
          w[c] = ((pending >> c) & 1u) ? ld_relaxed_u64(src + c * stride) : 0ull;
#pragma unroll
        for (int c = 0; c < kDecodeMaxClusters; ++c)
          if (((pending >> c) & 1u) && uint32_t(w[c] >> 32) == epoch) {
            v[c] = __uint_as_float(uint32_t(w[c]));
            pending &= ~(1u << c);
          }
        if (pending && clock64() - t0 > plim) {
          atomicOr(a.err, kErrTimeout | kWaitSlices);
          break;
        }
      }
      s = 0.f;
#pragma unroll
      for (int c = 0; c < kDecodeMaxClusters; ++c)
        if (c < ncl) s += ((pending >> c) & 1u) ? 0.f : v[c];
    }
    const uint32_t dst = sa(xlane ? nx2 : gfull + c0 + tid), bar = sa(gxbar);
    for (int q = 0; q < CS; ++q) st_async_f32(map_rank(dst, q), s, map_rank(bar, q));
  }
  __all_sync(FULL, bar_wait_cluster(gxbar, 0, a.err, kSpinCycles, kWaitGathered));

  // ---- every warp: its share of the Gram form (Gram rows c0 + warp,
  //      c0 + warp + NW, ...) and of ||g||^2, pushed to every rank, then
  //      y = M g for its rows (groups of RB rows: RB warp, RB warp + RB NW, ...)
  {
    float q = 0.f, n = 0.f;
    if (have_gram) {
      __all_sync(FULL, bar_wait(gbar, 0, a.err, kSpinCycles, kWaitGram));
      // lane l takes column groups l, l + 32, ... (clamped loads, masked)
      constexpr int NG = 2 * NV;  // float4 groups of a Gram row per lane (k <= 256 NV)
      const float4* g4 = reinterpret_cast<const float4*>(gfull);
      bool og[NG];
      int jg[NG];
      float4 gq[NG];
#pragma unroll
      for (int u = 0; u < NG; ++u) {
        og[u] = lane + 32 * u < nf4;
        jg[u] = og[u] ? lane + 32 * u : 0;
        gq[u] = g4[jg[u]];
      }
      for (int i = c0 + warp; i < c1; i += NW) {
        const float4* grow = reinterpret_cast<const float4*>(gram_s) + (i - c0) * nf4;
        float4 vg[NG];
#pragma unroll
        for (int u = 0; u < NG; ++u) vg[u] = grow[jg[u]];
        const float gi = gfull[i];
        float h = 0.f;
#pragma unroll
        for (int u = 0; u < NG; ++u) {
          float hu = vg[u].x * gq[u].x;
          hu = fmaf(vg[u].y, gq[u].y, hu);
          hu = fmaf(vg[u].z, gq[u].z, hu);
          hu = fmaf(vg[u].w, gq[u].w, hu);
          h += og[u] ? hu : 0.f;
        }
        q = fmaf(gi, h, q);
      }
    }
    for (int i = c0 + warp; i < c1; i += NW) n = fmaf(gfull[i], gfull[i], n);
    q = warp_sum(q);
    if (lane < CS) {
      const uint32_t rb = map_rank(sa(qbar), lane);
      st_async_f32(map_rank(sa(qin + rank * NW + warp), lane), q, rb);
      st_async_f32(map_rank(sa(nin + rank * NW + warp), lane), n, rb);
    }
  }
  if (nrows > 0) {
    __all_sync(FULL, bar_wait(mbar, 0, a.err, kSpinCycles, kWaitM));
    // lane l multiplies column group l of RB rows at a time; the row loads
    // are unconditional (rows past the CTA's last repeat it, lanes past the
    // row's vectors repeat vector 0) and masked afterwards, so all RB are in
    // flight together
    float gv[NV][PV];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int e = 0; e < PV; ++e) gv[v][e] = gfull[vl[v] * PV + e];
    auto apply_rows = [&](auto rb_c) {
      constexpr int RB = decltype(rb_c)::value;
      for (int rb = warp * RB; rb < nrows; rb += NW * RB) {
        uint4 u[RB][NV];
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
          for (int v = 0; v < NV; ++v)
            u[r][v] = *reinterpret_cast<const uint4*>(Ms + int64_t(min(rb + r, nrows - 1)) * mrow_b + vl[v] * 16);
        float part[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          part[r] = 0.f;
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            const float p = E::dot_vec(u[r][v], gv[v]);
            part[r] += on[v] ? p : 0.f;
          }
        }
        const float sum = warp_reduce_multi<RB>(part, lane);
        const int r = row_of_lane<RB>(lane);
        if ((lane & (32 / RB - 1)) == 0 && rb + r < nrows) ybuf[rb + r] = sum;
      }
    };
    if (nrows <= NW * 4)
      apply_rows(IntC<4>{});
    else if (nrows <= NW * 8 || NV > 1)  // (16 rows of two vectors: too many registers)
      apply_rows(IntC<8>{});
    else
      apply_rows(IntC<16 / NV>{});
  }
  // ---- the decision, taken by every warp from the same shares in the same
  //      order (lane l adds shares 4l .. 4l + 3 of the rank-major list, then
  //      a butterfly over the lanes)
  __all_sync(FULL, bar_wait_cluster(qbar, 0, a.err, kSpinCycles, kWaitShares));
  static_assert(CS * NW == 4 * 32, "four shares per lane");
  const float4 q4 = reinterpret_cast<const float4*>(qin)[lane];
  const float4 n4 = reinterpret_cast<const float4*>(nin)[lane];
  const float Qr = (q4.x + q4.y) + (q4.z + q4.w);
  const float Nr = (n4.x + n4.y) + (n4.z + n4.w);
  float Q = warp_sum(Qr);
  const float N = warp_sum(Nr);
  if (!a.m.gram) Q = N;  // orthonormal basis: ||V g||^2 = ||g||^2
  const float xx = *nx2;
  float rr = xx - 2.f * N + Q;
  rr = rr < 0.f ? 0.f : rr;  // keeps NaN
  const float rho = xx == 0.f ? 0.f : sqrtf(rr / xx);
  const bool slow = !(rho < a.eps);
  if (blockIdx.x == 0 && tid == 0) {
    if (a.m.rho) a.m.rho[0] = rho;
    a.m.flags[0] = uint8_t(slow ? 1 : 0);
  }

  // ---- apply
  if (!slow) {
    // this warp's rows of y (the row groups it computed), from its own lanes
    __syncwarp();
    const int rbw = nrows <= NW * 4 ? 4 : (nrows <= NW * 8 || NV > 1) ? 8 : 16;
    for (int rb = warp * rbw; rb < nrows; rb += NW * rbw)
      if (lane < rbw && rb + lane < nrows) a.m.Y[r0 + rb + lane] = ybuf[rb + lane];
    return;
  }
  if (nrows == 0) return;
  // Slow token: the V slab, the partials and the M rows are consumed, so the
  // W rings take their space; the token goes where the inboxes were.
  const int seg_b = a.m.seg_bytes, SW = a.m.sw;
  const int nseg = int((row_b + seg_b - 1) / seg_b);
  const int my_rows = warp < nrows ? (nrows - warp + NW - 1) / NW : 0;
  const int items = my_rows * nseg;
  unsigned char* wring = Vs + int64_t(warp) * SW * seg_b;
  uint64_t* wfull = ring + warp * SW;
  const char* wbase = static_cast<const char*>(a.m.W) + r0 * row_b;
  // item q of this warp: segment q % nseg of its row q / nseg (CTA row
  // warp + (q / nseg) * NW), in ring slot q % SW; issuer and consumer step
  // through the items with counters
  int q_row = 0, q_seg = 0, q_slot = 0;
  auto issue_next = [&]() {
    const int64_t offq = int64_t(q_seg) * seg_b;
    const uint32_t bytes = uint32_t(min(int64_t(seg_b), row_b - offq));
    bar_expect_tx(&wfull[q_slot], bytes);
    bulk_g2s(wring + q_slot * seg_b, wbase + (int64_t(warp) + int64_t(q_row) * NW) * row_b + offq, bytes,
             &wfull[q_slot]);
    if (++q_seg == nseg) {
      q_seg = 0;
      ++q_row;
    }
    if (++q_slot == SW) q_slot = 0;
  };
  int issued = min(items, SW);
  __syncthreads();  // every warp is done with the V slab and the M rows
  if (lane == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int q = 0; q < issued; ++q) issue_next();
  }
  unsigned char* xst = reinterpret_cast<unsigned char*>(inbox);
  for (int64_t e = tid; e < row_b / 16; e += kApplyThreads)
    reinterpret_cast<uint4*>(xst)[e] = ld_cg_v4(static_cast<const char*>(a.m.X) + e * 16);
  __syncthreads();
  float acc0 = 0.f, acc1 = 0.f;
  int c_slot = 0, c_seg = 0, c_row = 0;
  uint32_t c_ph = 0;
  int i = 0;
  for (; i < items; ++i) {
    if (!__all_sync(FULL, bar_wait(&wfull[c_slot], c_ph, a.err, kSpinCycles, kWaitRing))) break;
    const int64_t off = int64_t(c_seg) * seg_b;
    const int nv = int(min(int64_t(seg_b), row_b - off) / 16);
    const unsigned char* segp = wring + c_slot * seg_b;
    uint4 wq[kSegVecs];
#pragma unroll
    for (int u = 0; u < kSegVecs; ++u) {
      const int v = u * 32 + lane;
      wq[u] = v < nv ? *reinterpret_cast<const uint4*>(segp + v * 16) : make_uint4(0u, 0u, 0u, 0u);
    }
    // the segment is in registers before its slot is refilled
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
    const unsigned char* xs = xst + off;
#pragma unroll
    for (int u = 0; u < kSegVecs; ++u) {
      const int v = u * 32 + lane;
      const uint4 xq = v < nv ? *reinterpret_cast<const uint4*>(xs + v * 16) : make_uint4(0u, 0u, 0u, 0u);
      E::dot_acc(wq[u], xq, acc0, acc1);
    }
    if (++c_slot == SW) {
      c_slot = 0;
      c_ph ^= 1u;
    }
    if (++c_seg == nseg) {
      const float sum = warp_sum(acc0 + acc1);
      if (lane == 0) a.m.Y[r0 + warp + int64_t(c_row) * NW] = sum;
      acc0 = acc1 = 0.f;
      c_seg = 0;
      ++c_row;
    }
  }
  // after an expired wait: wait (bounded) for this warp's copies still in flight
  if (lane == 0)
    for (int q = i; q < issued; ++q) {
      bar_wait(&wfull[c_slot], c_ph, a.err, kSpinCycles, kWaitRing);
      if (++c_slot == SW) {
        c_slot = 0;
        c_ph ^= 1u;
      }
    }
}

// The persistent stack kernel: the calls of a list of maps in order, in one
// launch.  Map i + 1's barriers and weight copies are set up as soon as the
// CTA has finished map i (while the other CTAs finish theirs), and the CTAs
// then meet at a grid barrier on the workspace's arrival counter before
// map i + 1 reads its token.  The counter only grows: an episode is the n
// arrivals after a multiple of n (n the grid size), and a CTA's returning
// add tells it the episode's target.  Episodes cannot overlap: a CTA
// arrives for map i + 1 only after the episode of map i is complete, and a
// launch's first arrival comes after its dependency wait on the previous
// kernel of the stream.  The launch number (from the ticket the single-token
// kernel also draws, so that grid-projection epochs never repeat) and the
// map's place give each grid-projection call its epoch.  After a wait has
// given up anywhere in the grid (the error word, read after each barrier),
// the remaining waits use a short limit.
template <class E, int NV>
__global__ void __launch_bounds__(kApplyThreads, 1) stack_decode_kernel(const __grid_constant__ StackDecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (!cluster_shape_ok(kDecodeCluster) || gridDim.x % kDecodeCluster != 0 ||
      gridDim.x / kDecodeCluster > kDecodeMaxClusters) {
    if (tid == 0) atomicOr(a.err, kErrTimeout | kErrLaunchShape);
    return;  // before any barrier, copy or access to another CTA
  }
  const int rank = int(cg::this_cluster().block_rank());
  const DecodeBars b(smem);
  const int n = a.n_maps;
  if (tid == 0) {
    b.words[0] = uint32_t(atomicAdd(a.ticket, 1ull) / gridDim.x) + 1u;  // launch number
    b.words[1] = 0u;                                                     // error seen
  }
  decode_init_bars(a.maps[0], smem, tid, rank);
  __syncthreads();
  const uint32_t launch = b.words[0];
  decode_issue_copies<E>(a.maps[0], smem, tid, lane, warp, rank);
  if (n > 1) {
    const DecodeMap& nx = a.maps[1];
    decode_prefetch_l2(static_cast<const char*>(nx.V), uint64_t(nx.d) * nx.k * E::kBytes,
                       static_cast<const char*>(nx.M), uint64_t(nx.d_out) * nx.k * E::kBytes,
                       reinterpret_cast<const char*>(nx.gram), nx.gram ? uint64_t(nx.k) * nx.k * 4 : 0, tid);
  }
  cluster_arrive_relaxed();
  if (n == 1) pdl_launch_dependents();
  pdl_wait();
  long long lim = kSpinCycles;
  for (int i = 0; i < n; ++i) {
    const DecodeMap m = a.maps[i];  // a register copy: the table is indexed at run time
    decode_run<E, NV>(m, decode_geom(m, rank, warp), a.eps, a.part_g, a.part_x, (launch << 8) | uint32_t(i + 1),
                      a.err, lim, 0, 0, smem);
    if (i + 1 == n) break;
    // every warp has written its rows of map i and is done with shared
    // memory; its generic writes are ordered before the next map's copies
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    // map i + 1: barriers; then the last thread arrives for map i (its
    // returning add is an L2 round trip) while the others issue the weight
    // copies and the L2 prefetch of map i + 2
    const DecodeMap& m1 = a.maps[i + 1];
    decode_init_bars(m1, smem, tid, rank, true);
    __syncthreads();
    constexpr int kArrive = kApplyThreads - 1;  // no copy, prefetch or barrier duty
    unsigned long long target = 0;
    if (tid == kArrive) {
      __threadfence();
      const unsigned long long mine = atomicAdd(a.arrive, 1ull);
      target = (mine / gridDim.x + 1) * gridDim.x;
    }
    decode_issue_copies<E>(m1, smem, tid, lane, warp, rank);
    if (i + 2 < n) {
      const DecodeMap& nx = a.maps[i + 2];
      decode_prefetch_l2(static_cast<const char*>(nx.V), uint64_t(nx.d) * nx.k * E::kBytes,
                         static_cast<const char*>(nx.M), uint64_t(nx.d_out) * nx.k * E::kBytes,
                         reinterpret_cast<const char*>(nx.gram), nx.gram ? uint64_t(nx.k) * nx.k * 4 : 0, tid);
    }
    cluster_arrive_relaxed();
    if (tid == kArrive) {
      // every CTA has finished map i (bounded); then the grid's error word
      if (ld_acquire_gpu(a.arrive) < target) {
        const long long t0 = clock64();
        while (ld_acquire_gpu(a.arrive) < target) {
          if (clock64() - t0 > lim) {
            atomicOr(a.err, kErrTimeout | kWaitGrid);
            break;
          }
        }
      }
      b.words[1] = *reinterpret_cast<volatile uint32_t*>(a.err);
    }
    if (i + 2 == n) pdl_launch_dependents();
    __syncthreads();
    if (b.words[1] != 0u) lim = kSpinCyclesAfterError;
  }
  // No CTA leaves while a peer of its cluster may still push into its shared
  // memory: after a wait has given up, the CTAs of a cluster can be at
  // different steps of the last call.
  cluster_arrive_relaxed();
  cluster_wait();
}

template <class E, int NV>
static cudaError_t launch_decode_t(const DecodeArgs& a, const DecodePlan& p, cudaStream_t s) {
  auto kern = decode_kernel<E, NV>;
  static size_t smem_set = 0;
  if (p.smem > smem_set) {
    cudaError_t e = set_kernel_smem(kern, p.smem);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess) return e;
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
  attr[1].val.clusterDim.x = kDecodeCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  // the grid projection's CTAs poll other clusters' words: co-resident launch
  static int no_coop = 0;
  return launch_maybe_coop(cfg, attr, 2, a.m.grid != 0, &no_coop, kern, a);
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& p, gsi_dtype dt, cudaStream_t s) {
  const bool two = a.m.k * (dt == GSI_BF16 ? 2 : 4) > 512;  // two 16-byte vectors of a row per lane
  if (dt == GSI_BF16) return two ? launch_decode_t<BF16, 2>(a, p, s) : launch_decode_t<BF16, 1>(a, p, s);
  return two ? launch_decode_t<F32, 2>(a, p, s) : launch_decode_t<F32, 1>(a, p, s);
}

template <class E, int NV>
static cudaError_t launch_stack_t(const StackDecodeArgs& a, size_t smem, int ncta, cudaStream_t s) {
  auto kern = stack_decode_kernel<E, NV>;
  static size_t smem_set = 0;
  if (smem > smem_set) {
    cudaError_t e = set_kernel_smem(kern, smem);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess) return e;
    smem_set = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(ncta));
  cfg.blockDim = dim3(kApplyThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kDecodeCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  // the CTAs meet at grid barriers between maps: co-resident launch
  static int no_coop = 0;
  return launch_maybe_coop(cfg, attr, 2, true, &no_coop, kern, a);
}

cudaError_t launch_stack_decode(const StackDecodeArgs& a, size_t smem, int ncta, int nv, gsi_dtype dt,
                                cudaStream_t s) {
  if (dt == GSI_BF16) return nv == 2 ? launch_stack_t<BF16, 2>(a, smem, ncta, s) : launch_stack_t<BF16, 1>(a, smem, ncta, s);
  return nv == 2 ? launch_stack_t<F32, 2>(a, smem, ncta, s) : launch_stack_t<F32, 1>(a, smem, ncta, s);
}

template <class K>
static int max_clusters_of(K kern, size_t smem) {
  if (set_kernel_smem(kern, smem) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kDecodeCluster * 64);
  cfg.blockDim = dim3(kApplyThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kDecodeCluster;
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

int decode_max_clusters(size_t smem, gsi_dtype dt) {
  return dt == GSI_BF16 ? max_clusters_of(decode_kernel<BF16, 1>, smem) : max_clusters_of(decode_kernel<F32, 1>, smem);
}

int stack_max_clusters(size_t smem, gsi_dtype dt, int nv) {
  if (dt == GSI_BF16)
    return nv == 2 ? max_clusters_of(stack_decode_kernel<BF16, 2>, smem) : max_clusters_of(stack_decode_kernel<BF16, 1>, smem);
  return nv == 2 ? max_clusters_of(stack_decode_kernel<F32, 2>, smem) : max_clusters_of(stack_decode_kernel<F32, 1>, smem);
}

}  // namespace gsi
