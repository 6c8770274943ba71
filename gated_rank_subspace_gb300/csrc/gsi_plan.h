// Host-side launch plans shared by the C ABI and the kernels' launchers.
// Pure integer arithmetic: the workspace size of a call depends only on the
// map's shape and T, never on the device, so it can be queried without a GPU.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace gsi {

constexpr int kClusterSize = 8;     // CTAs per cluster in the gate kernel
constexpr int kGateThreads = 128;  // small enough to share an SM with a decide-and-apply CTA
// 8 warps: with at most 168 registers a thread, two warps of a decide CTA on
// each SM sub-partition leave room for one warp of a projection CTA, so the
// two kernels of consecutive calls can share an SM and overlap.
constexpr int kApplyThreads = 256;
constexpr int kGateMaxRowsPerThread = 8;
constexpr int kGateTargetSlabs = 256;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t rup(int64_t a, int64_t b) { return cdiv(a, b) * b; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Gate kernel geometry.  V (d x k) is cut into slabs of `rs` consecutive rows,
// one slab per CTA; inside a CTA each of `nrg` row groups of `nv` threads
// (one 16-byte vector of a V row each) walks rows rg, rg + nrg, ...
struct GatePlan {
  int nv;          // 16-byte vectors per V row
  int nrg;         // row groups per CTA
  int rs;          // rows per slab
  int n_slabs;     // CTAs (multiple of the cluster size)
  int n_clusters;
  int tc;          // tokens per chunk (register-blocked)
  int ks;          // columns of g owned by each CTA of a cluster in reductions
  size_t smem;     // dynamic shared memory bytes
};

inline GatePlan plan_gate(int64_t d, int64_t k, int elem_bytes, int64_t T) {
  GatePlan p{};
  p.nv = int(k * elem_bytes / 16);
  p.nrg = kGateThreads / p.nv;
  int64_t max_rs = int64_t(kGateMaxRowsPerThread) * p.nrg;
  max_rs = max_rs / 8 * 8;
  int64_t rs = rup(cdiv(d, kGateTargetSlabs), 8);
  if (rs < 8) rs = 8;
  if (rs > max_rs) rs = max_rs;
  p.rs = int(rs);
  p.n_slabs = int(rup(cdiv(d, rs), kClusterSize));
  p.n_clusters = p.n_slabs / kClusterSize;
  p.tc = T >= 8 ? 8 : T >= 4 ? 4 : T >= 2 ? 2 : 1;
  p.ks = int(cdiv(k, kClusterSize));
  // main loop:  xs[tc][rs] + red[nrg][tc][k] + pg[tc][k] + px[tc]
  // finalizer (aliases red): gsl[tc][ks] + gfull[tc][k] + q/ng partials
  size_t main_b = size_t(p.tc) * p.rs * 4 + size_t(p.nrg) * p.tc * k * 4 +
                  size_t(p.tc) * k * 4 + size_t(p.tc) * 4 +
                  size_t(kClusterSize) * p.tc * (p.ks + 1) * 4;
  size_t fin_b = size_t(p.tc) * p.rs * 4 + size_t(p.tc) * p.ks * 4 + 16 + size_t(p.tc) * k * 4 +
                 size_t(p.tc) * k * 4 + size_t(p.tc) * 4 + 2 * 8 * size_t(p.tc) * 4 + 64;
  p.smem = (main_b > fin_b ? main_b : fin_b) + 64;
  return p;
}

// Workspace layout of one stream-path call (offsets in bytes, 256-aligned).
struct StreamLayout {
  size_t ctrl, part_g, part_x, g, idx, flags, xslow, total;
};

inline StreamLayout layout_stream(int64_t d, int64_t k, int elem_bytes, int64_t T) {
  GatePlan p = plan_gate(d, k, elem_bytes, T);
  StreamLayout L{};
  size_t off = 0;
  L.ctrl = off;    off += 256;
  L.part_g = off;  off += align256(size_t(p.n_clusters) * T * k * 4);
  L.part_x = off;  off += align256(size_t(p.n_clusters) * T * 4);
  L.g = off;       off += align256(size_t(T) * k * 4);
  L.idx = off;     off += align256(size_t(2) * T * 4);
  L.flags = off;   off += align256(size_t(T));
  L.xslow = off;   off += elem_bytes == 2 ? align256(size_t(T) * d * 2) : 0;  // slow tokens' x (bf16)
  L.total = off;
  return L;
}

// Workspace layout of one fused-decode call: every CTA of the grid (at most
// kFusedMaxCtas) publishes its partial g and ||x||^2 for the grid's barrier.
constexpr int kFusedMaxCtas = 256;

struct FusedLayout {
  size_t ctrl, part_g, part_x, total;
};

inline FusedLayout layout_fused(int64_t k, int64_t T) {
  FusedLayout L{};
  size_t off = 0;
  L.ctrl = off;    off += 256;
  L.part_g = off;  off += align256(size_t(kFusedMaxCtas) * T * k * 4);
  L.part_x = off;  off += align256(size_t(kFusedMaxCtas) * T * 4);
  L.total = off;
  return L;
}

// Workspace layout of one tensor-core-path call.
struct TensorLayout {
  size_t ctrl, vt, g, gbf, gfast, xslow, idx, gt, norms, total;
};

// Token count of a prefill-sized call: the tensor path's slow-token
// contraction takes 256 token rows per CTA from here on.
constexpr int64_t kTensorMinT = 128;

// Split-K slices of the tensor path's projection contraction G = X V_k: 8 at
// prefill-sized T, 16 below it (few token rows: more CTAs, shorter chains).
constexpr int kGSplitMax = 16;
inline int g_split(int64_t T) { return T < kTensorMinT ? 16 : 8; }

// The tensor path's finalize (rho, flags, bf16 g) runs as two kernels: a
// per-token pass (kNormThreads threads a token: split-K sum of g, ||g||^2,
// ||x||^2) and the Gram form, which takes tokens in chunks of kFinTok and
// cuts the Gram rows into fin_blocks(T, k) blocks, one thread-block cluster
// a chunk, so that every T gives about three CTAs an SM of a GB300 (456) or
// more: at most kFinMaxBlocks blocks (a portable cluster) and at least 32
// Gram rows a block.  A CTA of the Gram form has kFinThreads compute threads
// (two token octets x 64 column quads of a kFinCols-column pass) and one
// copy warp, and streams its Gram rows through kFinStages shared-memory
// stages of kFinStageBytes.
constexpr int kFinTok = 16;
constexpr int kNormThreads = 64;
constexpr int kFinThreads = 128;
constexpr int kFinCols = 256;
constexpr int kFinStages = 3;
constexpr int64_t kFinStageBytes = 12288;
constexpr int kFinMaxBlocks = 8;
inline int fin_blocks(int64_t T, int64_t k) {
  const int64_t chunks = cdiv(T, kFinTok);
  int64_t nb = cdiv(456, chunks);
  int64_t cap = k / 32 < kFinMaxBlocks ? k / 32 : kFinMaxBlocks;
  if (cap < 1) cap = 1;
  if (nb > cap) nb = cap;
  return int(nb < 1 ? 1 : nb);
}
inline size_t fin_smem(int64_t k) {
  return size_t(kFinStages) * kFinStageBytes + size_t(kFinTok) * k * 4 + 4 * kFinTok * 4;
}

inline TensorLayout layout_tensor(int64_t d, int64_t k, int64_t T) {
  TensorLayout L{};
  size_t off = 0;
  L.ctrl = off;   off += 256;
  L.vt = off;     off += align256(size_t(k) * d * 2);
  L.g = off;      off += align256(size_t(g_split(T)) * T * k * 4);  // split-K partial projections
  L.gbf = off;    off += align256(size_t(T) * k * 2);
  L.gfast = off;  off += align256(size_t(T) * k * 2);
  L.xslow = off;  off += align256(size_t(T) * d * 2);
  L.idx = off;    off += align256(size_t(2) * T * 4);
  L.gt = off;     off += align256(size_t(cdiv(T, kFinTok)) * kFinTok * k * 4);  // g by chunk, column, token slot
  L.norms = off;  off += align256(size_t(T) * 8);                                  // (||g||^2, ||x||^2)
  L.total = off;
  return L;
}
// Token count from which GSI_PATH_AUTO uses the tensor cores for bf16 maps.
// Measured per call on the 13B maps (d = 5120, k = 320) without slow tokens:
// 40-46 us on the tensor path from T = 2 to 16; 16-38 us on the streaming
// kernels up to T = 8 (one chunk of 8 tokens), 67-74 us at T = 12-16 (two
// chunks).  Slow rows take the tensor cores on both paths (bf16).
constexpr int64_t kTensorAutoMinT = 9;

// Decide-and-apply kernel geometry (see gsi_apply.cu).  The device part
// (how many CTAs are co-resident) comes in as ncta; everything else is
// arithmetic on the shapes.  Each CTA owns rows_per_cta contiguous output
// rows.  Its eight warps stream their own W rows in seg_bytes segments through
// private rings of wstages slots; the rings share one shared-memory region
// with the staged M rows (a call's fast rows are computed before its slow
// rows stream).
struct DecidePlan {
  int tc, grv, ncta, rows_per_cta, seg_bytes, wstages, x_stage_max, stage_m;
  int off_m, off_x, off_g, off_gram;  // off_gram = 0: Gram slice read from global
  int off_y;                          // [tc][rows_per_cta] fast outputs computed before the decision
  bool fused;  // single-launch decode: the grid projects x itself
  bool cproj;  // fused, and each cluster projects x on all of V (no grid barrier)
  int cs;      // CTAs per cluster
  int ks;      // columns of g owned by each rank
  int v_rows, ngrp, off_v, off_xs;
  size_t smem;
  bool ok;
};

constexpr int kSegBytes = 4096;
constexpr int kSegVecs = kSegBytes / (32 * 16);  // 16-byte vectors per lane in one segment
constexpr int kWarpStages = 4;
constexpr int kXStage = 16 * 1024;

inline DecidePlan plan_decide(int64_t d, int64_t d_out, int64_t k, int es, int64_t T, int ncta,
                              size_t smem_budget, bool fused = false, int cs = kClusterSize, bool cproj = false) {
  DecidePlan p{};
  p.ok = true;
  p.fused = fused;
  p.cproj = fused && cproj;
  p.cs = cs;
  p.tc = T >= 8 ? 8 : T >= 4 ? 4 : T >= 2 ? 2 : 1;
  const int64_t ks = cdiv(k, cs);
  p.ks = int(ks);
  p.grv = 0;
  const int64_t row_b = d * es;
  const int64_t mrow_b = k * es;
  p.seg_bytes = int(row_b < kSegBytes ? row_b : kSegBytes);
  p.wstages = kWarpStages;
  const size_t ring = size_t(kApplyThreads / 32) * p.wstages * p.seg_bytes;
  const int64_t xs = fused ? 0 : kXStage / row_b;
  p.x_stage_max = int(xs < p.tc ? xs : p.tc);
  size_t g_area = (size_t(p.tc) * k + size_t(p.tc) * ks + 8 * 2 * size_t(p.tc) + 2 * size_t(cs) * p.tc +
                   6 * size_t(p.tc) + 40 + kApplyThreads + 4) * 4;
  const size_t bars = size_t(kApplyThreads / 32) * p.wstages * 8 + 40;  // + M, Gram, V, two exchanges
  size_t off = (bars + 127) & ~size_t(127);
  const size_t gram_b = size_t(ks) * k * 4;
  p.off_gram = 0;
  if (gram_b <= 40 * 1024) {
    p.off_gram = int(off);
    off += (gram_b + 127) & ~size_t(127);
  }
  p.off_x = int(off);
  off += size_t(p.x_stage_max) * row_b;
  off = (off + 127) & ~size_t(127);
  p.off_g = int(off);
  off += g_area;
  off = (off + 127) & ~size_t(127);
  p.off_y = int(off);
  off += size_t(p.tc) * size_t(cdiv(d_out, ncta)) * 4;
  off = (off + 127) & ~size_t(127);
  p.v_rows = 0;
  p.ngrp = 0;
  p.off_xs = 0;
  if (fused) {
    // CTA b (grid projection) or cluster rank r (cluster projection)
    // projects rows [b * v_rows, ...) or [r * v_rows, ...) of V: its token
    // slice, the row groups' partial sums and its slice of ||x||^2; the
    // cluster projection adds this CTA's partial g [tc][k] and the inboxes
    // of the all-to-all, [cs][tc][k] and [cs][tc]
    p.v_rows = int(cdiv(d, p.cproj ? cs : ncta));
    const int vecs = int(mrow_b / 16);  // 16-byte vectors per V row
    p.ngrp = kApplyThreads / vecs >= 1 ? kApplyThreads / vecs : 1;
    p.off_xs = int(off);
    // (xsq takes 8 floats when the cluster projection's 16-byte aligned pg follows it)
    off += (size_t(p.tc) * rup(p.v_rows, 4) + size_t(p.ngrp) * p.tc * k + size_t(p.tc) + 8) * 4;
    if (p.cproj) off += (size_t(p.tc) * k + size_t(cs) * p.tc * k + size_t(cs) * p.tc + 8) * 4;
    off = (off + 127) & ~size_t(127);
  }
  p.off_m = int(off);
  p.ncta = ncta;
  p.rows_per_cta = int(cdiv(d_out, ncta));
  const size_t m_bytes = (size_t(p.rows_per_cta) * mrow_b + 127) & ~size_t(127);
  const size_t v_bytes = fused ? size_t(p.v_rows) * mrow_b : 0;
  // region after off_m: [M rows | V slice] before the decision, W rings after
  // it; with the cluster projection the M rows replace the V slice once it
  // is consumed (copied after the projection)
  size_t need_mv = p.cproj ? (m_bytes > v_bytes ? m_bytes : v_bytes) : m_bytes + v_bytes;
  p.stage_m = off + (need_mv > ring ? need_mv : ring) <= smem_budget ? 1 : 0;
  if (fused && !p.stage_m) {
    need_mv = v_bytes;  // M then comes from global (L2) after the decision
  }
  p.off_v = int(off + (p.stage_m && !p.cproj ? m_bytes : 0));
  const size_t region = (p.stage_m || fused) ? (need_mv > ring ? need_mv : ring) : ring;
  p.smem = off + region;
  p.ok = p.smem <= smem_budget;
  // shared memory left over stages more slow tokens' x (up to the chunk)
  if (p.ok && p.x_stage_max < p.tc) {
    const int64_t more = int64_t(smem_budget - p.smem) / row_b;
    const int64_t grow = more < p.tc - p.x_stage_max ? more : p.tc - p.x_stage_max;
    const size_t shift = (size_t(grow) * row_b + 127) & ~size_t(127);
    if (grow > 0 && p.smem + shift <= smem_budget) {
      p.x_stage_max += int(grow);
      p.off_g += int(shift);
      p.off_y += int(shift);
      if (fused) p.off_xs += int(shift);
      p.off_m += int(shift);
      p.off_v += int(shift);
      p.smem += shift;
    }
  }
  return p;
}

// Single-token decode kernel geometry (see gsi_decode.cu).  Clusters of
// kDecodeCluster CTAs.  Cluster projection: cluster rank r projects V rows
// [r * vr, (r + 1) * vr), so every cluster holds all of V.  Grid projection
// (bases too large for that): CTA b projects rows [b * vr, (b + 1) * vr).
// Warp w takes rows [w * rw, (w + 1) * rw) of the CTA's slab, at most 32, one
// per lane.  CTA b applies output rows [b * rpc, (b + 1) * rpc).  Shared
// memory: mbarriers | g, exchange inboxes, token elements | fast outputs |
// partial-g inbox (then the slow token's x) | Gram slice | V slab | M rows.
// The W rings of a slow token reuse the V slab and M rows (and the space
// after them) once the decision is taken.  When V and M do not fit side by
// side, the M rows are copied over the V slab after the projection (m_late)
// and the warps' partial sums get their own region.
constexpr int kDecodeCluster = 16;
constexpr int kDecodeMaxStages = 6;
constexpr int kDecodeBars = 5;  // Gram, M, partials, shares, gathered g
constexpr int kDecodeMaxClusters = 16;  // grid projection: clusters whose slices are polled
constexpr int kDecodeCtaWords = 2;      // 32-bit words after the mbarriers
// byte offset of those words
constexpr int kDecodeWordsOff = (kApplyThreads / 32 + kDecodeBars + kApplyThreads / 32 * kDecodeMaxStages) * 8;

struct DecodePlan {
  int vr, rw, rpc, ks, seg_bytes, sw, red_stride, m_late, grid;
  int off_g, off_y, off_in, off_gram, off_red, off_v, off_m;
  int ncta;
  size_t smem;
  bool ok;
};

inline DecodePlan plan_decode(int64_t d, int64_t d_out, int64_t k, int es, int ncta, size_t smem_budget,
                              bool grid) {
  DecodePlan p{};
  p.ok = false;
  const int64_t mrow_b = k * es, row_b = d * es;
  const int nw = kApplyThreads / 32;
  if (ncta < kDecodeCluster || ncta % kDecodeCluster || k % 4 || mrow_b % 16 || row_b % 16) return p;
  if (mrow_b / 16 > 64) return p;             // at most two 16-byte vectors of a V / M row per lane
  if (grid && k % kDecodeCluster) return p;  // equal column slices for the reduce-scatter
  if (grid && ncta > kDecodeCluster * kDecodeMaxClusters) return p;
  p.ncta = ncta;
  p.grid = grid ? 1 : 0;
  p.vr = int(cdiv(d, grid ? ncta : kDecodeCluster));
  p.rw = int(cdiv(p.vr, nw));
  if (p.rw > 32) return p;  // one token element per lane
  p.rpc = int(cdiv(d_out, ncta));
  p.ks = int(cdiv(k, kDecodeCluster));
  p.seg_bytes = int(row_b < kSegBytes ? row_b : kSegBytes);
  // mbarriers, then two CTA words (the call's epoch or the launch number, and
  // the persistent kernel's error flag) at a fixed offset for every map
  const size_t bars = size_t(nw + kDecodeBars + nw * kDecodeMaxStages) * 8 + kDecodeCtaWords * 4;
  size_t off = (bars + 127) & ~size_t(127);
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = (off + bytes + 127) & ~size_t(127);
    return int(at);
  };
  p.off_g = take(size_t(k + kDecodeCluster + 2 * kDecodeCluster * nw + 4 + nw * 32) * 4);
  p.off_y = take(size_t(p.rpc) * 4);
  const size_t inbox = size_t(kDecodeCluster) * p.ks * 4;  // partial-g slices of every rank
  p.off_in = take(inbox > size_t(row_b) ? inbox : size_t(row_b));
  p.off_gram = take(size_t(p.ks) * k * 4);
  const size_t v_bytes = size_t(nw) * p.rw * mrow_b;
  const size_t m_bytes = size_t(p.rpc) * mrow_b;
  const size_t red_b = size_t(k + 4) * 4;  // a warp's partial g and its ||x||^2
  const size_t rest = off;
  for (int late = 0; late < 2; ++late) {
    off = rest;
    const bool alias = !late && size_t(p.rw) * mrow_b >= red_b;
    p.off_red = alias ? 0 : take(size_t(nw) * red_b);
    p.red_stride = int(alias ? size_t(p.rw) * mrow_b / 4 : red_b / 4);
    p.off_v = int(off);
    if (alias) p.off_red = p.off_v;
    p.off_m = late ? p.off_v : int(off + v_bytes);
    const size_t need = late ? (v_bytes > m_bytes ? v_bytes : m_bytes) : v_bytes + m_bytes;
    // the deepest W ring (at least 2 slots a warp) that fits
    for (int sw = kDecodeMaxStages; sw >= 2; --sw) {
      const size_t ring = size_t(nw) * sw * p.seg_bytes;
      const size_t region = ring > need ? ring : need;
      if (size_t(p.off_v) + region <= smem_budget) {
        p.sw = sw;
        p.m_late = late;
        p.smem = size_t(p.off_v) + region;
        p.ok = true;
        return p;
      }
    }
  }
  return p;
}

// Small-batch decode kernel geometry (see gsi_batch.cu): 2 <= T <= 16
// tokens of a bf16 map in one launch, clusters of kBatchCluster CTAs with
// eight compute warps and one copy warp each.  CTA b projects rows
// [b * vr, (b + 1) * vr) of V_k and applies output rows [b * rpc, (b + 1) *
// rpc); both are multiples of 16 (one tensor-core tile).  Shared memory
// (offsets from a 1024-byte aligned base): mbarriers and words | g in bf16,
// high and low halves, [2][16][k] (before that, the CTA's partial g by
// column slice) | the decision | per-warp shares | the rank's final slice of
// g and the norms | the slab norms | then the call's scratch: V slab (128-byte swizzled boxes of 64 columns), the
// token slab, partial-g inbox, norm inbox, gathered g, share inbox, Gram
// slice | M rows (swizzled boxes).  Once the flags are known (the fast
// outputs are then in registers) the W ring -- stages of rpc x 128 columns
// of W plus T x 128 of X -- takes the space from the scratch on, M rows
// included; its stages end up holding the warps' partial sums for the final
// reduction.
constexpr int kBatchThreads = 288;
constexpr int kBatchWarps = 8;  // compute warps (the ninth issues copies)
constexpr int kBatchMaxT = 16;
constexpr int kBatchMinT = 2;
constexpr int kBatchCluster = 16;
constexpr int kBatchMaxClusters = 16;
constexpr int kBatchMaxMt = 10;   // output rows a CTA: at most 10 tiles of 16
constexpr int kBatchKC = 128;     // W columns per ring stage (8 steps of 16)
constexpr int kBatchMaxStages = 6;
constexpr int kBatchMaxK = 384;
constexpr int kBatchSmemSlack = 1024;  // the kernel aligns its base to 1024 bytes

struct BatchPlan {
  int T, ncta, vr, rpc, ks, kb, stages, stage_bytes;
  int gbf_pitch, xs_pitch;
  int off_gbf, off_dec, off_wsh, off_fs, off_nx, off_scr, off_v, off_xs, off_in, off_nin, off_g32, off_qin, off_gram,
      off_m;
  size_t smem;  // dynamic shared memory to request (alignment slack included)
  bool ok;
};

inline BatchPlan plan_batch(int64_t d, int64_t d_out, int64_t k, int64_t T, int ncta, size_t smem_budget) {
  BatchPlan p{};
  p.ok = false;
  if (T < kBatchMinT || T > kBatchMaxT || ncta < kBatchCluster || ncta % kBatchCluster) return p;
  if (k % 64 || k > kBatchMaxK || d % 8 || d < 16 || d_out < 1) return p;
  if (ncta > kBatchCluster * kBatchMaxClusters) return p;
  p.T = int(T);
  p.ncta = ncta;
  p.vr = int(rup(cdiv(d, ncta), 16));
  p.rpc = int(rup(cdiv(d_out, ncta), 16));
  if (p.vr > 256 || p.rpc > 16 * kBatchMaxMt) return p;
  p.ks = int(k / kBatchCluster);
  p.kb = int(k / 64);
  p.gbf_pitch = int(k * 2 + 16);
  p.xs_pitch = p.vr * 2 + 16;
  size_t off = 1024;  // mbarriers and CTA words
  auto take = [&](size_t bytes, size_t align) {
    off = (off + align - 1) / align * align;
    const size_t at = off;
    off += bytes;
    return int(at);
  };
  p.off_gbf = take(size_t(2) * kBatchMaxT * p.gbf_pitch, 128);
  p.off_dec = take(size_t(2) * kBatchMaxT * 4, 128);
  p.off_wsh = take(size_t(kBatchWarps) * kBatchMaxT * 2 * 4, 128);
  p.off_fs = take(size_t(T) * p.ks * 4 + kBatchMaxT * 4, 128);  // this rank's final slice of G, then the norms
  p.off_nx = take(kBatchMaxT * 4, 128);                          // the CTA's slab norms
  p.off_scr = take(0, 1024);
  p.off_v = take(size_t(p.kb) * p.vr * 128, 1024);
  p.off_xs = take(size_t(kBatchMaxT) * p.xs_pitch, 128);
  p.off_in = take(size_t(kBatchCluster) * T * p.ks * 4, 128);
  p.off_nin = take(size_t(kBatchCluster) * kBatchMaxT * 4, 128);
  p.off_g32 = take(size_t(T) * k * 4 + kBatchMaxT * 4, 128);  // g, then the 16 norms
  p.off_qin = take(size_t(kBatchCluster) * kBatchMaxT * 8, 128);
  p.off_gram = take(size_t(p.ks) * k * 4, 128);
  p.off_m = take(size_t(p.kb) * p.rpc * 128, 1024);
  const size_t end_m = off;
  p.stage_bytes = int(rup(int64_t(p.rpc) * 256 + kBatchMaxT * 256, 1024));
  const size_t budget = smem_budget > kBatchSmemSlack ? smem_budget - kBatchSmemSlack : 0;
  if (end_m > budget) return p;
  int s = int((budget - size_t(p.off_scr)) / size_t(p.stage_bytes));
  if (s > kBatchMaxStages) s = kBatchMaxStages;
  if (s < 2) return p;
  // the warps' partial sums [8][16][rpc] float32 reuse the ring's stages
  if (size_t(s) * p.stage_bytes < size_t(kBatchWarps) * kBatchMaxT * p.rpc * 4) return p;
  p.stages = s;
  const size_t end_ring = size_t(p.off_scr) + size_t(s) * p.stage_bytes;
  p.smem = (end_ring > end_m ? end_ring : end_m) + kBatchSmemSlack;
  p.ok = p.smem <= smem_budget;
  return p;
}

// Workspace of a small-batch call: the control block, then each cluster's
// projections [clusters][T][k] and norms [clusters][16] as 64-bit
// epoch-tagged words.
struct BatchLayout {
  size_t ctrl, part_g, part_x, total;
};

inline BatchLayout layout_batch(int64_t k, int64_t T) {
  BatchLayout L{};
  size_t off = 0;
  L.ctrl = off;    off += 256;
  L.part_g = off;  off += align256(size_t(kBatchMaxClusters) * T * k * 8);
  L.part_x = off;  off += align256(size_t(kBatchMaxClusters) * kBatchMaxT * 8);
  L.total = off;
  return L;
}

}  // namespace gsi
