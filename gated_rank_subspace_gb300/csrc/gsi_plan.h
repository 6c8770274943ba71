// Host-side launch plans shared by the C ABI and the kernels' launchers.
// Pure integer arithmetic: the workspace size of a call depends only on the
// map's shape and T, never on the device, so it can be queried without a GPU.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace gsi {

constexpr int kClusterSize = 8;     // CTAs per cluster in the gate kernel
constexpr int kGateThreads = 256;
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
                  size_t(p.tc) * k * 4 + size_t(p.tc) * 4;
  size_t fin_b = size_t(p.tc) * p.rs * 4 + size_t(p.tc) * p.ks * 4 + 16 + size_t(p.tc) * k * 4 +
                 size_t(p.tc) * k * 4 + size_t(p.tc) * 4 + 2 * 8 * size_t(p.tc) * 4 + 64;
  p.smem = (main_b > fin_b ? main_b : fin_b) + 64;
  return p;
}

// Workspace layout of one stream-path call (offsets in bytes, 256-aligned).
struct StreamLayout {
  size_t ctrl, part_g, part_x, g, idx, total;
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

// Apply kernel geometry: fast units are `rows_fast` rows of M, slow units
// `rows_slow` rows of W, each handled by one warp.
struct ApplyPlan {
  int vplm;        // 16-byte vectors of an M row per lane (1, 2 or 4)
  int rows_fast;   // M rows per fast unit (16 / vplm)
  int rows_slow;   // W rows per slow unit
  int64_t fast_units, slow_units;
  int x_stage_tokens_max;  // slow tokens whose x fits the staging budget
  int g_stage_tokens_max;  // fast tokens whose g fits the staging budget
  size_t smem;
};

constexpr size_t kApplyXStage = 64 * 1024;
constexpr size_t kApplyGStage = 32 * 1024;

inline ApplyPlan plan_apply(int64_t d, int64_t d_out, int64_t k, int elem_bytes) {
  ApplyPlan p{};
  int64_t nvm = k * elem_bytes / 16;
  p.vplm = nvm <= 32 ? 1 : nvm <= 64 ? 2 : 4;
  p.rows_fast = 16 / p.vplm;
  int64_t row_b = d * elem_bytes;
  p.rows_slow = row_b >= 8192 ? 1 : int(8192 / row_b);
  p.fast_units = cdiv(d_out, p.rows_fast);
  p.slow_units = cdiv(d_out, p.rows_slow);
  p.x_stage_tokens_max = int(kApplyXStage / size_t(row_b));
  p.g_stage_tokens_max = int(kApplyGStage / size_t(k * 4));
  p.smem = kApplyXStage + kApplyGStage;
  return p;
}

}  // namespace gsi
