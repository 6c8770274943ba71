// Host-side launch plans shared by the C ABI and the kernels' launchers.
// Pure integer arithmetic: the workspace size of a call depends only on the
// map's shape and T, never on the device, so it can be queried without a GPU.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace gsi {

constexpr int kClusterSize = 8;     // CTAs per cluster in the gate kernel
constexpr int kGateThreads = 128;  // small enough to share an SM with a decide-and-apply CTA
constexpr int kApplyThreads = 288;  // 8 consumer warps + 1 copy-producer warp
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
  size_t ctrl, part_g, part_x, g, idx, flags, total;
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
  L.total = off;
  return L;
}

// Workspace layout of one tensor-core-path call.
struct TensorLayout {
  size_t ctrl, vt, g, gbf, gfast, xslow, idx, total;
};

inline TensorLayout layout_tensor(int64_t d, int64_t k, int64_t T) {
  TensorLayout L{};
  size_t off = 0;
  L.ctrl = off;   off += 256;
  L.vt = off;     off += align256(size_t(k) * d * 2);
  L.g = off;      off += align256(size_t(T) * k * 4);
  L.gbf = off;    off += align256(size_t(T) * k * 2);
  L.gfast = off;  off += align256(size_t(T) * k * 2);
  L.xslow = off;  off += align256(size_t(T) * d * 2);
  L.idx = off;    off += align256(size_t(2) * T * 4);
  L.total = off;
  return L;
}

// Token count from which GSI_PATH_AUTO uses the tensor cores for bf16 maps.
constexpr int64_t kTensorMinT = 128;

// Decide-and-apply kernel geometry (see gsi_apply.cu).  The device part
// (how many CTAs are co-resident) comes in as ncta; everything else is
// arithmetic on the shapes.  Each CTA owns rows_per_cta contiguous output
// rows.  Its nine warps stream their own W rows in seg_bytes segments through
// private rings of wstages slots; the rings share one shared-memory region
// with the staged M rows (a call's fast rows are computed before its slow
// rows stream).
struct DecidePlan {
  int tc, grv, ncta, rows_per_cta, seg_bytes, wstages, x_stage_max, stage_m;
  int off_m, off_x, off_g, off_gram;  // off_gram = 0: Gram slice read from global
  size_t smem;
  bool ok;
};

constexpr int kSegBytes = 4096;
constexpr int kWarpStages = 4;
constexpr int kXStage = 16 * 1024;

inline DecidePlan plan_decide(int64_t d, int64_t d_out, int64_t k, int es, int64_t T, int ncta,
                              size_t smem_budget) {
  DecidePlan p{};
  p.ok = true;
  p.tc = T >= 8 ? 8 : T >= 4 ? 4 : T >= 2 ? 2 : 1;
  const int64_t ks = cdiv(k, kClusterSize);
  p.grv = 0;  // Gram slice comes from shared memory (or global when it does not fit)
  const int64_t row_b = d * es;
  p.seg_bytes = int(row_b < kSegBytes ? row_b : kSegBytes);
  p.wstages = kWarpStages;
  const size_t ring = size_t(kApplyThreads / 32) * p.wstages * p.seg_bytes;
  const int64_t xs = kXStage / row_b;
  p.x_stage_max = int(xs < p.tc ? xs : p.tc);
  const size_t g_area = (size_t(p.tc) * k + size_t(p.tc) * ks + 40 * size_t(p.tc) + 40) * 4;
  const size_t bars = size_t(kApplyThreads / 32) * p.wstages * 8 + 16;
  size_t off = (bars + 127) & ~size_t(127);
  // Gram slice of one cluster rank (ks rows of k floats), staged by a bulk copy
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
  p.off_m = int(off);
  p.ncta = ncta;
  p.rows_per_cta = int(cdiv(d_out, ncta));
  const size_t m_bytes = size_t(p.rows_per_cta) * k * es;
  p.stage_m = off + (m_bytes > ring ? m_bytes : ring) <= smem_budget ? 1 : 0;
  p.smem = off + (p.stage_m && m_bytes > ring ? m_bytes : ring);
  p.ok = p.smem <= smem_budget;
  return p;
}

}  // namespace gsi
