// C ABI of the gated-subspace linear map: argument validation, workspace
// layout and kernel dispatch.  Declarations and the contract of every entry
// point are in include/gsi.h.

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <mutex>
#include <string>

#include "gsi_common.cuh"
#include "gsi_kernels.h"
#include "gsi_plan.h"

namespace gsi {

static thread_local std::string g_err;
static std::atomic<int> g_fail_after{0};
static std::atomic<int> g_withhold{0};  // test hook: grid-projection launches left to withhold a slice

static gsi_status fail(gsi_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

// Records a message for gsi_last_error() from another translation unit.
gsi_status record_error(gsi_status s, const char* msg) {
  g_err = msg;
  return s;
}

static gsi_status ok() {
  g_err.clear();
  return GSI_OK;
}

// Host-side fault injection: when armed with n, the n-th launch step fails.
static bool injected_failure() {
  int n = g_fail_after.load();
  if (n <= 0) return false;
  if (g_fail_after.fetch_sub(1) == 1) return true;
  return false;
}

static gsi_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return GSI_OK;
  return fail(GSI_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Test hook: the next n launches that need a co-resident grid are refused
// on the host, as the driver refuses a grid that cannot be co-resident.
static std::atomic<int> g_refuse_coresident{0};
static bool refused_coresident() { return g_refuse_coresident.load() > 0 && g_refuse_coresident.fetch_sub(1) > 0; }

// Status of a launch that needs a co-resident grid: a refusal for size is
// GSI_ERR_UNSUPPORTED, on which callers take the two-launch streaming path.
static gsi_status coresident_status(cudaError_t e, const char* what) {
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return fail(GSI_ERR_UNSUPPORTED, "%s: the grid cannot be co-resident on this device now", what);
  }
  return cuda_check(e, what);
}

static int elem_bytes(gsi_dtype dt) { return dt == GSI_BF16 ? 2 : 4; }

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static gsi_status check_dtype(gsi_dtype dt) {
  if (dt != GSI_F32 && dt != GSI_BF16) return fail(GSI_ERR_INVALID_ARG, "unknown dtype %d", int(dt));
  return GSI_OK;
}

static gsi_status check_shape(int64_t d, int64_t d_out, int64_t k, gsi_dtype dt) {
  gsi_status s = check_dtype(dt);
  if (s != GSI_OK) return s;
  if (d <= 0 || d_out <= 0 || k <= 0)
    return fail(GSI_ERR_INVALID_ARG, "sizes must be positive (d=%lld d_out=%lld k=%lld)",
                (long long)d, (long long)d_out, (long long)k);
  if (k > d) return fail(GSI_ERR_INVALID_ARG, "k=%lld exceeds d=%lld", (long long)k, (long long)d);
  if (k > GSI_MAX_K) return fail(GSI_ERR_UNSUPPORTED, "k=%lld exceeds GSI_MAX_K=%d", (long long)k, GSI_MAX_K);
  if (d > (int64_t(1) << 30) || d_out > (int64_t(1) << 30))
    return fail(GSI_ERR_UNSUPPORTED, "dimension above 2^30");
  const int es = elem_bytes(dt);
  if ((d * es) % 16 || (k * es) % 16)
    return fail(GSI_ERR_UNSUPPORTED, "d*%d and k*%d bytes must be multiples of 16 (d=%lld k=%lld)",
                es, es, (long long)d, (long long)k);
  return GSI_OK;
}

static gsi_status check_ptr(const void* p, const char* name) {
  if (!p) return fail(GSI_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned(p, 16)) return fail(GSI_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return GSI_OK;
}

static gsi_status check_map(const gsi_map_desc* m) {
  if (!m) return fail(GSI_ERR_INVALID_ARG, "map descriptor is NULL");
  gsi_status s = check_shape(m->d, m->d_out, m->k, m->dtype);
  if (s != GSI_OK) return s;
  if ((s = check_ptr(m->W, "map.W")) != GSI_OK) return s;
  if ((s = check_ptr(m->V, "map.V")) != GSI_OK) return s;
  if ((s = check_ptr(m->M, "map.M")) != GSI_OK) return s;
  if (m->dtype == GSI_BF16 && !m->gram)
    return fail(GSI_ERR_INVALID_ARG, "bf16 maps need the Gram matrix V^T V (map.gram is NULL)");
  if (m->gram && !aligned(m->gram, 16)) return fail(GSI_ERR_INVALID_ARG, "map.gram is not 16-byte aligned");
  return GSI_OK;
}

static gsi_status check_tokens(int64_t T, float eps) {
  if (T < 0) return fail(GSI_ERR_INVALID_ARG, "T=%lld is negative", (long long)T);
  if (T > (int64_t(1) << 24)) return fail(GSI_ERR_UNSUPPORTED, "T=%lld above 2^24", (long long)T);
  if (std::isnan(eps) || eps < 0.f) return fail(GSI_ERR_INVALID_ARG, "eps must be >= 0 and not NaN");
  return GSI_OK;
}

static gsi_status check_workspace(const void* ws, size_t have, size_t need) {
  if (need == 0) return GSI_OK;
  if (!ws) return fail(GSI_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
  if (!aligned(ws, 256)) return fail(GSI_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if (have < need) return fail(GSI_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", have, need);
  return GSI_OK;
}

// Per-block shared memory a kernel may opt into on sm_100-class GPUs (bytes).
constexpr size_t kSmemOptinSm100 = 232448;

// The fused decode kernel handles T <= 2 when one CTA's slab of V (with a
// grid of at least kFusedMinCtas CTAs) fits in shared memory beside its
// working buffers.  Host-only arithmetic, so workspace sizing needs no device.
constexpr int kFusedMinCtas = 64;
static bool fused_fits(const gsi_map_desc* m, int64_t T) {
  if (T < 1 || T > 2) return false;
  const int es = elem_bytes(m->dtype);
  if (m->k * es / 16 > kApplyThreads) return false;  // one thread per 16-byte vector of a V row
  const DecidePlan p = plan_decide(m->d, m->d_out, m->k, es, T, kFusedMinCtas, kSmemOptinSm100, true, 16);
  return p.ok;
}

// The small-batch decode kernel takes bf16 maps (with their Gram) at
// 2 <= T <= 16 where its plan fits a device of kBatchNominalCtas co-resident
// CTAs (host-only arithmetic; the run-time plan uses the device's own grid
// and falls back where it does not fit).
constexpr int kBatchNominalCtas = 112;
static bool batch_fits(const gsi_map_desc* m, int64_t T) {
  if (m->dtype != GSI_BF16 || m->gram == nullptr) return false;
  return plan_batch(m->d, m->d_out, m->k, T, kBatchNominalCtas, kSmemOptinSm100).ok;
}

// The path a call takes without the small-batch kernel: the single-launch
// decode for T <= 2 where it fits, the tensor cores for bf16 maps from
// kTensorAutoMinT tokens, the two-launch streaming kernels otherwise.
static gsi_path classic_path(const gsi_map_desc* m, int64_t T) {
  if (fused_fits(m, T)) return GSI_PATH_FUSED;  // falls back to STREAM at run time where the device cannot run it
  return (m->dtype == GSI_BF16 && T >= kTensorAutoMinT) ? GSI_PATH_TENSOR : GSI_PATH_STREAM;
}

// Resolve the path for a call: the single-token decode for T = 1, the
// small-batch decode for bf16 maps at 2 <= T <= 16, otherwise classic_path.
static gsi_status resolve_path(const gsi_map_desc* m, int64_t T, gsi_path path, gsi_path* out) {
  if (path == GSI_PATH_AUTO) {
    *out = (T >= 2 && batch_fits(m, T)) ? GSI_PATH_BATCH : classic_path(m, T);
    return GSI_OK;
  }
  if (path == GSI_PATH_BATCH) {
    if (!(T >= kBatchMinT && T <= kBatchMaxT && batch_fits(m, T)))
      return fail(GSI_ERR_UNSUPPORTED,
                  "the small-batch decode takes bf16 maps with their Gram, 2 <= T <= 16, k a multiple of 64 "
                  "(at most 384), d a multiple of 8 and at most 160 output rows a CTA");
    *out = GSI_PATH_BATCH;
    return GSI_OK;
  }
  if (path == GSI_PATH_STREAM) {
    *out = GSI_PATH_STREAM;
    return GSI_OK;
  }
  if (path == GSI_PATH_FUSED) {
    if (!fused_fits(m, T))
      return fail(GSI_ERR_UNSUPPORTED, "the fused decode takes T <= 2 and a slice of V that fits shared memory");
    *out = GSI_PATH_FUSED;
    return GSI_OK;
  }
  if (path == GSI_PATH_TENSOR) {
    if (m->dtype != GSI_BF16)
      return fail(GSI_ERR_UNSUPPORTED, "the tensor-core path takes bf16 maps only");
    *out = GSI_PATH_TENSOR;
    return GSI_OK;
  }
  return fail(GSI_ERR_INVALID_ARG, "unknown path %d", int(path));
}

// Workspace of a path.  The fused decode's is also large enough for the
// streaming path, so a device that cannot run it can fall back to the
// two-launch kernels on the same workspace.
static size_t path_ws(const gsi_map_desc* m, int64_t T, gsi_path p) {
  if (p == GSI_PATH_BATCH) {
    // also large enough for the path a device that cannot run it falls back to
    const size_t b = layout_batch(m->k, T).total, c = path_ws(m, T, classic_path(m, T));
    return b > c ? b : c;
  }
  if (p == GSI_PATH_TENSOR) return layout_tensor(m->d, m->k, T).total;
  const size_t st = layout_stream(m->d, m->k, m->dtype == GSI_BF16 ? 2 : 4, T).total;
  if (p != GSI_PATH_FUSED) return st;
  const size_t fu = layout_fused(m->k, T).total;
  return st > fu ? st : fu;
}

static size_t stream_ws(const gsi_map_desc* m, int64_t T) {
  return layout_stream(m->d, m->k, elem_bytes(m->dtype), T).total;
}

// Device facts the decide-and-apply plans need, queried once per device.
struct DeviceFacts {
  int nsm = 0;
  int smem_optin = 0;
  int clusters[2][2][2] = {};  // co-resident clusters per [dtype][fused][cs == 16]; -1: not possible
  int decode_clusters[2] = {};  // co-resident clusters of the single-token decode kernel per dtype
  int stack_clusters[2][2] = {};  // ... of the persistent stack kernel per [dtype][two vectors a lane]
  int batch_clusters = 0;          // ... of the small-batch decode kernel
};

// Shared memory of the two-launch decide-and-apply kernel: the device limit
// less room for one CTA of the next projection kernel, which starts early.
static size_t decide_smem_budget(int smem_optin) { return size_t(smem_optin) - 16 * 1024; }

static gsi_status device_facts(DeviceFacts** out) {
  static DeviceFacts facts[64];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return cuda_check(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(mu);
  DeviceFacts& f = facts[dev];
  if (f.nsm == 0) {
    if ((e = cudaDeviceGetAttribute(&f.nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_check(e, "SM count");
    if ((e = cudaDeviceGetAttribute(&f.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return cuda_check(e, "shared memory limit");
  }
  *out = &f;
  return GSI_OK;
}

// Co-resident clusters for a decide-and-apply variant (cached); 0 if none.
static int decide_clusters(DeviceFacts* f, gsi_dtype dt, bool fused, int cs) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int& c = f->clusters[dt == GSI_BF16][fused][cs == 16];
  if (c == 0) {
    const size_t smem = fused ? size_t(f->smem_optin) : decide_smem_budget(f->smem_optin);
    const int n = decide_apply_max_clusters(smem, dt, fused, cs);
    c = n > 0 ? n : -1;
  }
  return c > 0 ? c : 0;
}

// Co-resident clusters of the persistent stack kernel (cached); 0 if none.
static int stack_clusters(DeviceFacts* f, gsi_dtype dt, int nv) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int& c = f->stack_clusters[dt == GSI_BF16][nv == 2];
  if (c == 0) {
    const int n = stack_max_clusters(size_t(f->smem_optin), dt, nv);
    c = n > 0 ? n : -1;
  }
  return c > 0 ? c : 0;
}

// Co-resident clusters of the single-token decode kernel (cached); 0 if none.
static int decode_clusters(DeviceFacts* f, gsi_dtype dt) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int& c = f->decode_clusters[dt == GSI_BF16];
  if (c == 0) {
    const int n = decode_max_clusters(size_t(f->smem_optin), dt);
    c = n > 0 ? n : -1;
  }
  return c > 0 ? c : 0;
}

// Co-resident clusters of the small-batch decode kernel (cached); 0 if none.
// Every launch uses this grid, so the workspace's call numbers (tickets / grid
// size) stay consistent across calls.
static int batch_clusters(DeviceFacts* f) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int& c = f->batch_clusters;
  if (c == 0) {
    const int n = batch_max_clusters(size_t(f->smem_optin));
    c = n > 0 ? n : -1;
  }
  return c > 0 ? c : 0;
}

// The single-token decode kernel's plan for a map: the cluster projection
// where the basis fits a cluster, else the grid projection (ok = false when
// neither fits this device).
static DecodePlan decode_plan(const gsi_map_desc* m, DeviceFacts* f) {
  DecodePlan p{};
  const int ncl = decode_clusters(f, m->dtype);
  for (int grid = 0; grid < 2 && ncl > 0 && !p.ok; ++grid)
    p = plan_decode(m->d, m->d_out, m->k, elem_bytes(m->dtype), ncl * kDecodeCluster, size_t(f->smem_optin),
                    grid != 0);
  return p;
}

static void fill_decode_map(DecodeMap& a, const gsi_map_desc* m, const DecodePlan& p, const void* X, float* Y,
                            uint8_t* flags, float* rho) {
  a.X = X;
  a.W = m->W;
  a.V = m->V;
  a.M = m->M;
  a.gram = m->gram;
  a.Y = Y;
  a.flags = flags;
  a.rho = rho;
  a.d = m->d;
  a.d_out = m->d_out;
  a.k = int(m->k);
  a.vr = p.vr;
  a.rw = p.rw;
  a.rpc = p.rpc;
  a.ks = p.ks;
  a.seg_bytes = p.seg_bytes;
  a.sw = p.sw;
  a.red_stride = p.red_stride;
  a.m_late = p.m_late;
  a.off_g = p.off_g;
  a.off_y = p.off_y;
  a.off_in = p.off_in;
  a.off_gram = p.off_gram;
  a.off_red = p.off_red;
  a.off_v = p.off_v;
  a.off_m = p.off_m;
  a.grid = p.grid;
}

// 16-byte vectors of a V / M row per lane in the single-token kernels.
static int decode_nv(const gsi_map_desc* m) { return m->k * elem_bytes(m->dtype) > 512 ? 2 : 1; }

// Enqueue the single-token decode kernel (all arguments validated);
// GSI_ERR_UNSUPPORTED, with nothing launched, when its plan does not fit.
static gsi_status run_decode(const gsi_map_desc* m, const void* X, float eps, float* Y, uint8_t* flags, float* rho,
                             void* ws, cudaStream_t st, DeviceFacts* f, const gsi_map_desc* next) {
  const DecodePlan p = decode_plan(m, f);
  if (!p.ok) return GSI_ERR_UNSUPPORTED;
  Ctrl* ctrl = static_cast<Ctrl*>(ws);
  DecodeArgs a{};
  fill_decode_map(a.m, m, p, X, Y, flags, rho);
  a.eps = eps;
  if (p.grid) {
    const FusedLayout FL = layout_fused(m->k, 1);
    a.part_g = reinterpret_cast<float*>(static_cast<char*>(ws) + FL.part_g);
    a.part_x = reinterpret_cast<float*>(static_cast<char*>(ws) + FL.part_x);
    a.ticket = &ctrl->ticket1[m->dtype == GSI_BF16 ? 1 : 0];
  }
  if (next) {
    const int nes = elem_bytes(next->dtype);
    a.next_v = static_cast<const char*>(next->V);
    a.next_v_bytes = uint64_t(next->d) * next->k * nes;
    a.next_m = static_cast<const char*>(next->M);
    a.next_m_bytes = uint64_t(next->d_out) * next->k * nes;
    a.next_gram = reinterpret_cast<const char*>(next->gram);
    a.next_gram_bytes = next->gram ? uint64_t(next->k) * next->k * 4 : 0;
  }
  a.err = &ctrl->err;
  if (p.grid && g_withhold.load() > 0 && g_withhold.fetch_sub(1) > 0) {
    a.dbg_withhold = 1;
    a.poll_cycles = 20000000;  // ~10 ms
  }
  if (p.grid && refused_coresident())
    return fail(GSI_ERR_UNSUPPORTED, "single-token decode kernel launch: co-resident grid refused (test hook)");
  return coresident_status(launch_decode(a, p, m->dtype, st), "single-token decode kernel launch");
}

// Persistent stack decode over maps[0 .. n) (n >= 2, T = 1, every map with a
// single-token plan, one element type, row width and k): one launch, the
// calls in list order with a grid barrier between them.  GSI_ERR_UNSUPPORTED,
// with nothing launched, when the kernel cannot run here (the caller then
// runs the maps one launch each).
static gsi_status run_stack_decode(const gsi_map_desc* maps, int n, const void* const* X, float eps,
                                   float* const* Y, uint8_t* const* flags, void* ws, cudaStream_t st,
                                   DeviceFacts* f) {
  const gsi_dtype dt = maps[0].dtype;
  const int ncl = decode_clusters(f, dt);
  if (ncl == 0 || stack_clusters(f, dt, decode_nv(&maps[0])) != ncl) return GSI_ERR_UNSUPPORTED;
  static thread_local StackDecodeArgs a;  // 17 KB: kept off the stack
  a = StackDecodeArgs{};
  size_t smem = 0;
  for (int i = 0; i < n; ++i) {
    const DecodePlan p = decode_plan(&maps[i], f);
    if (!p.ok) return GSI_ERR_UNSUPPORTED;
    fill_decode_map(a.maps[i], &maps[i], p, X[i], Y[i], flags[i], nullptr);
    if (p.smem > smem) smem = p.smem;
  }
  Ctrl* ctrl = static_cast<Ctrl*>(ws);
  const FusedLayout FL = layout_fused(maps[0].k, 1);
  a.n_maps = n;
  a.eps = eps;
  a.part_g = reinterpret_cast<float*>(static_cast<char*>(ws) + FL.part_g);
  a.part_x = reinterpret_cast<float*>(static_cast<char*>(ws) + FL.part_x);
  a.ticket = &ctrl->ticket1[dt == GSI_BF16 ? 1 : 0];
  a.arrive = &ctrl->arrive[dt == GSI_BF16 ? 1 : 0];
  a.err = &ctrl->err;
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  if (refused_coresident())
    return fail(GSI_ERR_UNSUPPORTED, "stack decode kernel launch: co-resident grid refused (test hook)");
  return coresident_status(launch_stack_decode(a, smem, ncl * kDecodeCluster, decode_nv(&maps[0]), dt, st),
                           "stack decode kernel launch");
}

// Enqueue the decide-and-apply kernel for one map (all arguments validated).
// mode 0: decide and apply (gsi_linear); 1: decide only (gsi_gate, writes
// G, rho, flags and the compaction); 2: apply the decision stored by a
// preceding gsi_gate on the same workspace (gsi_apply); 3: decide, apply the
// fast tokens and write the compaction (the slow rows are left to the
// tensor-core contraction that follows).
// fused: the single-launch decode (mode 0 only; the cluster projects x on
// its own slices of V).  next: the map that follows in a stack, whose
// weights are staged in L2 while this one runs (nullable).  Returns
// GSI_ERR_UNSUPPORTED before launching anything when the fused decode cannot
// run on this device, so that callers may fall back to the two launches.
static gsi_status run_decide(const gsi_map_desc* m, const void* X, int64_t T, float eps, int mode, float* Y,
                             uint8_t* flags, float* rho, float* G, const float* Gin, void* ws, cudaStream_t st,
                             bool fused = false, const gsi_map_desc* next = nullptr) {
  const int es = elem_bytes(m->dtype);
  const GatePlan gp = plan_gate(m->d, m->k, es, T);
  const StreamLayout L = layout_stream(m->d, m->k, es, T);
  char* base = static_cast<char*>(ws);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(base + L.ctrl);
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  DeviceFacts* f = nullptr;
  gsi_status s = device_facts(&f);
  if (s != GSI_OK) return s;
  DecidePlan dp{};
  if (fused && mode == 0 && T == 1) {
    // one token: the single-token decode kernel where the basis fits a cluster
    s = run_decode(m, X, eps, Y, flags, rho, ws, st, f, next);
    if (s != GSI_ERR_UNSUPPORTED) return s;
  }
  if (fused) {
    // Cluster projection (each cluster projects x on all of V; no grid
    // barrier) where a sixteenth of V fits beside the other buffers, else
    // grid projection.  Both use 16-CTA clusters where the device allows
    // them: consecutive launches with different cluster shapes were measured
    // to cost ~1.4 us each in a sequence of maps (6B layer, batch-1 decode).
    const int nc16 = decide_clusters(f, m->dtype, true, 16);
    if (nc16 > 0) dp = plan_decide(m->d, m->d_out, m->k, es, T, nc16 * 16, size_t(f->smem_optin), true, 16, true);
    if (nc16 == 0 || !dp.ok) {
      const int cs = nc16 > 0 ? 16 : kClusterSize;
      int nc = nc16 > 0 ? nc16 : decide_clusters(f, m->dtype, true, cs);
      if (nc * cs > kFusedMaxCtas) nc = kFusedMaxCtas / cs;
      if (nc > 0) dp = plan_decide(m->d, m->d_out, m->k, es, T, nc * cs, size_t(f->smem_optin), true, cs);
      if (nc == 0 || !dp.ok) return fail(GSI_ERR_UNSUPPORTED, "the fused decode does not fit this device");
    }
  } else {
    const int nc = decide_clusters(f, m->dtype, false, kClusterSize);
    if (nc == 0) return fail(GSI_ERR_CUDA, "cannot size the decide-and-apply grid (cluster occupancy query failed)");
    dp = plan_decide(m->d, m->d_out, m->k, es, T, nc * kClusterSize, decide_smem_budget(f->smem_optin));
    if (!dp.ok) return fail(GSI_ERR_UNSUPPORTED, "the streaming kernels' shared memory does not fit this map");
  }
  DecideArgs a{};
  a.X = X;
  a.W = m->W;
  a.M = m->M;
  a.gram = m->gram;
  a.part_g = reinterpret_cast<const float*>(base + L.part_g);
  a.part_x = reinterpret_cast<const float*>(base + L.part_x);
  a.nclu = gp.n_clusters;
  a.d = m->d;
  a.d_out = m->d_out;
  a.k = int(m->k);
  a.T = int(T);
  a.ks = dp.ks;
  a.eps = eps;
  a.mode = mode;
  a.Y = Y;
  a.G = G;
  a.rho = rho;
  a.flags = mode == 1 ? reinterpret_cast<uint8_t*>(base + L.flags) : flags;
  a.idx = reinterpret_cast<int32_t*>(base + L.idx);
  a.counts = ctrl->counts;
  a.Gin = Gin;
  a.flags_in = reinterpret_cast<const uint8_t*>(base + L.flags);
  a.rows_per_cta = dp.rows_per_cta;
  a.seg_bytes = dp.seg_bytes;
  a.wstages = dp.wstages;
  a.x_stage_max = dp.x_stage_max;
  a.stage_m = dp.stage_m;
  a.off_m = dp.off_m;
  a.off_x = dp.off_x;
  a.off_g = dp.off_g;
  a.off_y = dp.off_y;
  a.off_gram = dp.off_gram;
  if (fused) {
    a.cproj = dp.cproj ? 1 : 0;
    const FusedLayout FL = layout_fused(m->k, T);
    a.fpart_g = reinterpret_cast<float*>(base + FL.part_g);
    a.fpart_x = reinterpret_cast<float*>(base + FL.part_x);
    a.part_g = a.fpart_g;
    a.part_x = a.fpart_x;
    a.nclu = dp.ncta;
    a.ticket = &ctrl->ticket[m->dtype == GSI_BF16 ? 1 : 0];
  }
  a.V = m->V;
  a.v_rows = dp.v_rows;
  a.ngrp = dp.ngrp;
  a.off_v = dp.off_v;
  a.off_xs = dp.off_xs;
  if (next) {
    const int nes = elem_bytes(next->dtype);
    a.next_v = static_cast<const char*>(next->V);
    a.next_v_bytes = uint64_t(next->d) * next->k * nes;
    a.next_m = static_cast<const char*>(next->M);
    a.next_m_bytes = uint64_t(next->d_out) * next->k * nes;
    a.next_gram = reinterpret_cast<const char*>(next->gram);
    a.next_gram_bytes = next->gram ? uint64_t(next->k) * next->k * 4 : 0;
  }
  a.err = &ctrl->err;
  a.flags_user = mode == 1 ? flags : nullptr;  // gsi_gate: also the caller's copy
  if (fused && !dp.cproj && refused_coresident())
    return fail(GSI_ERR_UNSUPPORTED, "decide-and-apply kernel launch: co-resident grid refused (test hook)");
  return coresident_status(launch_decide_apply(a, dp, m->dtype, st), "decide-and-apply kernel launch");
}

// Enqueue the projection kernel, then (mode) the decide-and-apply kernel.
static gsi_status run_stream(const gsi_map_desc* m, const void* X, int64_t T, float eps, float* Y,
                             uint8_t* flags, float* rho, float* G_out, void* ws, cudaStream_t st, bool apply,
                             const gsi_map_desc* next = nullptr) {
  const int es = elem_bytes(m->dtype);
  const GatePlan gp = plan_gate(m->d, m->k, es, T);
  const StreamLayout L = layout_stream(m->d, m->k, es, T);
  char* base = static_cast<char*>(ws);
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  GateArgs ga{};
  ga.X = X;
  ga.V = m->V;
  ga.d = m->d;
  ga.k = int(m->k);
  ga.T = int(T);
  ga.rs = gp.rs;
  ga.nv = gp.nv;
  ga.nrg = gp.nrg;
  ga.ks = gp.ks;
  ga.n_clusters = gp.n_clusters;
  ga.part_g = reinterpret_cast<float*>(base + L.part_g);
  ga.part_x = reinterpret_cast<float*>(base + L.part_x);
  if (apply) {
    ga.pf_m = static_cast<const char*>(m->M);
    ga.pf_m_bytes = uint64_t(m->d_out) * m->k * es;
  }
  if (m->gram) {
    ga.pf_g = reinterpret_cast<const char*>(m->gram);
    ga.pf_g_bytes = uint64_t(m->k) * m->k * 4;
  }
  gsi_status s = cuda_check(launch_gate(ga, gp, m->dtype, st, true), "projection kernel launch");
  if (s != GSI_OK) return s;
  // bf16 maps: the decide-and-apply kernel writes the fast rows and the
  // compaction (mode 3), and the slow rows follow on the tensor cores
  const bool defer = apply && m->dtype == GSI_BF16;
  s = run_decide(m, X, T, eps, apply ? (defer ? 3 : 0) : 1, Y, flags, rho, G_out, nullptr, ws, st, false, next);
  if (s != GSI_OK || !defer) return s;
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(base + L.ctrl);
  s = cuda_check(launch_slow_rows_tc(X, m->W, m->d, m->d_out, T, reinterpret_cast<const int32_t*>(base + L.idx),
                                     ctrl->counts, reinterpret_cast<uint16_t*>(base + L.xslow), Y, &ctrl->err, st),
                 "slow-row contraction launch");
  return s == GSI_OK ? ok() : s;
}


// Enqueue the small-batch decode for one bf16 map (2 <= T <= 16, all
// arguments validated).  GSI_ERR_UNSUPPORTED, with nothing launched, where
// this device cannot run it (the caller then takes classic_path).
static gsi_status run_batch(const gsi_map_desc* m, const void* X, int64_t T, float eps, float* Y, uint8_t* flags,
                            float* rho, void* ws, cudaStream_t st, const gsi_map_desc* next, const void* next_x) {
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  DeviceFacts* f = nullptr;
  gsi_status s = device_facts(&f);
  if (s != GSI_OK) return s;
  const int ncl = batch_clusters(f);
  if (ncl == 0) return fail(GSI_ERR_UNSUPPORTED, "the small-batch decode kernel cannot run on this device");
  const BatchPlan p = plan_batch(m->d, m->d_out, m->k, T, ncl * kBatchCluster, size_t(f->smem_optin));
  if (!p.ok || m->dtype != GSI_BF16 || !m->gram)
    return fail(GSI_ERR_UNSUPPORTED, "the small-batch decode plan does not fit this device");
  const BatchLayout L = layout_batch(m->k, T);
  char* base = static_cast<char*>(ws);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(base + L.ctrl);
  BatchCall c{};
  c.X = X;
  c.W = m->W;
  c.V = m->V;
  c.M = m->M;
  c.gram = m->gram;
  c.Y = Y;
  c.flags = flags;
  c.rho = rho;
  c.d = m->d;
  c.d_out = m->d_out;
  c.k = int(m->k);
  c.T = int(T);
  c.eps = eps;
  c.part_g = reinterpret_cast<unsigned long long*>(base + L.part_g);
  c.part_x = reinterpret_cast<unsigned long long*>(base + L.part_x);
  c.ticket = &ctrl->ticket_b[1];
  c.err = &ctrl->err;
  if (next) {
    const int nes = elem_bytes(next->dtype);
    c.next_v = static_cast<const char*>(next->V);
    c.next_v_bytes = uint64_t(next->d) * next->k * nes;
    c.next_m = static_cast<const char*>(next->M);
    c.next_m_bytes = uint64_t(next->d_out) * next->k * nes;
    c.next_gram = reinterpret_cast<const char*>(next->gram);
    c.next_gram_bytes = next->gram ? uint64_t(next->k) * next->k * 4 : 0;
    if (next_x) {
      c.next_x = static_cast<const char*>(next_x);
      c.next_x_bytes = uint64_t(T) * next->d * nes;
    }
  }
  if (g_withhold.load() > 0 && g_withhold.fetch_sub(1) > 0) {
    c.dbg_withhold = 1;
    c.poll_cycles = 20000000;  // ~10 ms
  }
  if (refused_coresident())
    return fail(GSI_ERR_UNSUPPORTED, "small-batch decode kernel launch: co-resident grid refused (test hook)");
  return coresident_status(launch_batch_decode(c, p, st), "small-batch decode kernel launch");
}

// Enqueue the tensor-core path for one bf16 map.  All arguments validated.
static gsi_status run_tensor(const gsi_map_desc* m, const void* X, int64_t T, float eps, float* Y,
                             uint8_t* flags, float* rho, void* ws, cudaStream_t st) {
  const TensorLayout L = layout_tensor(m->d, m->k, T);
  char* base = static_cast<char*>(ws);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(base + L.ctrl);
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  TensorArgs t{};
  t.X = X;
  t.V = m->V;
  t.W = m->W;
  t.M = m->M;
  t.gram = m->gram;
  t.d = m->d;
  t.d_out = m->d_out;
  t.k = m->k;
  t.T = T;
  t.eps = eps;
  t.Vt = reinterpret_cast<uint16_t*>(base + L.vt);
  t.G = reinterpret_cast<float*>(base + L.g);
  t.Gbf = reinterpret_cast<uint16_t*>(base + L.gbf);
  t.Gfast = reinterpret_cast<uint16_t*>(base + L.gfast);
  t.Xslow = reinterpret_cast<uint16_t*>(base + L.xslow);
  t.idx = reinterpret_cast<int32_t*>(base + L.idx);
  t.counts = ctrl->counts;
  t.rho = rho;
  t.flags = flags;
  t.Y = Y;
  t.err = &ctrl->err;
  t.gT = reinterpret_cast<float*>(base + L.gt);
  t.norms = reinterpret_cast<float2*>(base + L.norms);
  return cuda_check(launch_tensor_path(t, st), "tensor-core path launch");
}

// One gated map along a resolved path (fused falls back to the two-launch
// streaming kernels when the device cannot run it and `strict` is false).
static gsi_status run_path(const gsi_map_desc* m, gsi_path p, bool strict, const void* X, int64_t T, float eps,
                           float* Y, uint8_t* flags, float* rho, void* ws, cudaStream_t st,
                           const gsi_map_desc* next = nullptr, const void* next_x = nullptr) {
  if (p == GSI_PATH_BATCH) {
    const gsi_status s = run_batch(m, X, T, eps, Y, flags, rho, ws, st, next, next_x);
    if (s != GSI_ERR_UNSUPPORTED || strict) return s;
    p = classic_path(m, T);
  }
  if (p == GSI_PATH_TENSOR) return run_tensor(m, X, T, eps, Y, flags, rho, ws, st);
  if (p == GSI_PATH_FUSED) {
    const gsi_status s = run_decide(m, X, T, eps, 0, Y, flags, rho, nullptr, nullptr, ws, st, true, next);
    if (s != GSI_ERR_UNSUPPORTED || strict) return s;
  }
  return run_stream(m, X, T, eps, Y, flags, rho, nullptr, ws, st, true, next);
}

}  // namespace gsi

using namespace gsi;

extern "C" {

const char* gsi_last_error(void) { return g_err.c_str(); }

void gsi_debug_fail_after(int n) { g_fail_after.store(n > 0 ? n : 0); }

void gsi_debug_withhold_slice(int n) { g_withhold.store(n > 0 ? n : 0); }

void gsi_debug_refuse_coresident(int n) { g_refuse_coresident.store(n > 0 ? n : 0); }

gsi_status gsi_build_image(const void* W, const void* V, void* M, float* gram, int64_t d,
                           int64_t d_out, int64_t k, gsi_dtype dtype, void* stream) {
  gsi_status s = check_shape(d, d_out, k, dtype);
  if (s != GSI_OK) return s;
  if ((s = check_ptr(W, "W")) != GSI_OK) return s;
  if ((s = check_ptr(V, "V")) != GSI_OK) return s;
  if ((s = check_ptr(M, "M")) != GSI_OK) return s;
  if (gram && !aligned(gram, 16)) return fail(GSI_ERR_INVALID_ARG, "gram is not 16-byte aligned");
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  s = cuda_check(launch_image(W, V, M, gram, d, d_out, k, dtype, static_cast<cudaStream_t>(stream)),
                 "image kernel launch");
  return s == GSI_OK ? ok() : s;
}

size_t gsi_build_image_work_bytes(int64_t d, int64_t k, gsi_dtype dtype) {
  if (dtype != GSI_BF16 || d < 1 || k < 1) return 0;
  return 256 + align256(size_t(k) * size_t(d) * 2);
}

gsi_status gsi_build_image_ex(const void* W, const void* V, void* M, float* gram, int64_t d, int64_t d_out, int64_t k,
                              gsi_dtype dtype, void* work, size_t work_bytes, void* stream) {
  if (!work || dtype != GSI_BF16) return gsi_build_image(W, V, M, gram, d, d_out, k, dtype, stream);
  gsi_status s = check_shape(d, d_out, k, dtype);
  if (s != GSI_OK) return s;
  if ((s = check_ptr(W, "W")) != GSI_OK) return s;
  if ((s = check_ptr(V, "V")) != GSI_OK) return s;
  if ((s = check_ptr(M, "M")) != GSI_OK) return s;
  if (gram && !aligned(gram, 16)) return fail(GSI_ERR_INVALID_ARG, "gram is not 16-byte aligned");
  if (d > (int64_t(1) << 30) || d_out > (int64_t(1) << 30)) return fail(GSI_ERR_UNSUPPORTED, "dimension above 2^30");
  if ((s = check_workspace(work, work_bytes, gsi_build_image_work_bytes(d, k, dtype))) != GSI_OK) return s;
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  Ctrl* ctrl = static_cast<Ctrl*>(work);
  if ((s = cuda_check(cudaMemsetAsync(ctrl, 0, sizeof(Ctrl), st), "image scratch clear")) != GSI_OK) return s;
  uint16_t* Vt = reinterpret_cast<uint16_t*>(static_cast<char*>(work) + 256);
  if ((s = cuda_check(launch_image_tc(W, V, M, d, d_out, k, Vt, &ctrl->err, st), "image kernel launch")) != GSI_OK)
    return s;
  if (gram) s = cuda_check(launch_gram(V, gram, d, k, dtype, st), "Gram kernel launch");
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_linear_workspace_size(const gsi_map_desc* map, int64_t T, gsi_path path,
                                     size_t* bytes) {
  if (!bytes) return fail(GSI_ERR_INVALID_ARG, "bytes is NULL");
  if (!map) return fail(GSI_ERR_INVALID_ARG, "map descriptor is NULL");
  gsi_status s = check_shape(map->d, map->d_out, map->k, map->dtype);
  if (s != GSI_OK) return s;
  if ((s = check_tokens(T, 0.f)) != GSI_OK) return s;
  gsi_path p;
  if ((s = resolve_path(map, T, path, &p)) != GSI_OK) return s;
  *bytes = path_ws(map, T, p);
  return ok();
}

gsi_status gsi_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace) return fail(GSI_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(GSI_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  gsi_status s = cuda_check(cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream)),
                            "workspace memset");
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_workspace_status(const void* workspace, uint32_t* code, void* stream) {
  if (!workspace || !code) return fail(GSI_ERR_INVALID_ARG, "workspace and code must be non-NULL");
  if (!aligned(workspace, 256)) return fail(GSI_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  const Ctrl* c = static_cast<const Ctrl*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  gsi_status s = cuda_check(cudaMemcpyAsync(code, &c->err, sizeof(uint32_t), cudaMemcpyDeviceToHost, st),
                            "error word copy");
  if (s != GSI_OK) return s;
  s = cuda_check(cudaStreamSynchronize(st), "stream synchronize");
  if (s != GSI_OK) return s;
  if (*code) return fail(GSI_ERR_TIMEOUT, "device error word %u", *code);
  return ok();
}

gsi_status gsi_gate(const gsi_map_desc* map, const void* X, int64_t T, float eps, float* G,
                    float* rho, uint8_t* flags, void* workspace, size_t ws_bytes, void* stream) {
  gsi_status s = check_map(map);
  if (s != GSI_OK) return s;
  if ((s = check_tokens(T, eps)) != GSI_OK) return s;
  if (T == 0) return ok();
  if ((s = check_ptr(X, "X")) != GSI_OK) return s;
  if ((s = check_ptr(G, "G")) != GSI_OK) return s;
  if (!flags) return fail(GSI_ERR_INVALID_ARG, "flags is NULL");
  if (rho && !aligned(rho, 4)) return fail(GSI_ERR_INVALID_ARG, "rho is misaligned");
  if ((s = check_workspace(workspace, ws_bytes, stream_ws(map, T))) != GSI_OK) return s;
  s = run_stream(map, X, T, eps, nullptr, flags, rho, G, workspace,
                 static_cast<cudaStream_t>(stream), false);
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_apply(const gsi_map_desc* map, const void* X, const float* G, int64_t T, float* Y,
                     void* workspace, size_t ws_bytes, void* stream) {
  gsi_status s = check_map(map);
  if (s != GSI_OK) return s;
  if ((s = check_tokens(T, 0.f)) != GSI_OK) return s;
  if (T == 0) return ok();
  if ((s = check_ptr(X, "X")) != GSI_OK) return s;
  if ((s = check_ptr(G, "G")) != GSI_OK) return s;
  if ((s = check_ptr(Y, "Y")) != GSI_OK) return s;
  if ((s = check_workspace(workspace, ws_bytes, stream_ws(map, T))) != GSI_OK) return s;
  s = run_decide(map, X, T, 0.f, 2, Y, nullptr, nullptr, nullptr, G, workspace, static_cast<cudaStream_t>(stream));
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_compact(const uint8_t* flags, int64_t T, int32_t* idx, int32_t* counts, void* stream) {
  if (T < 0 || T > (int64_t(1) << 24)) return fail(GSI_ERR_INVALID_ARG, "bad T=%lld", (long long)T);
  if (!counts) return fail(GSI_ERR_INVALID_ARG, "counts must be non-NULL");
  if (T > 0 && (!flags || !idx)) return fail(GSI_ERR_INVALID_ARG, "flags and idx must be non-NULL");
  if (!aligned(idx, 4) || !aligned(counts, 4)) return fail(GSI_ERR_INVALID_ARG, "idx/counts misaligned");
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  gsi_status s = cuda_check(launch_compact(flags, int(T), idx, counts, static_cast<cudaStream_t>(stream)),
                            "compact kernel launch");
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_linear_ex(const gsi_map_desc* map, const void* X, int64_t T, float eps, float* Y,
                         uint8_t* flags, float* rho, void* workspace, size_t ws_bytes, gsi_path path,
                         void* stream) {
  gsi_status s = check_map(map);
  if (s != GSI_OK) return s;
  if ((s = check_tokens(T, eps)) != GSI_OK) return s;
  gsi_path p;
  if ((s = resolve_path(map, T, path, &p)) != GSI_OK) return s;
  if (T == 0) return ok();
  if ((s = check_ptr(X, "X")) != GSI_OK) return s;
  if ((s = check_ptr(Y, "Y")) != GSI_OK) return s;
  if (!flags) return fail(GSI_ERR_INVALID_ARG, "flags is NULL");
  if (rho && !aligned(rho, 4)) return fail(GSI_ERR_INVALID_ARG, "rho is misaligned");
  if ((s = check_workspace(workspace, ws_bytes, path_ws(map, T, p))) != GSI_OK) return s;
  s = run_path(map, p, path == GSI_PATH_FUSED || path == GSI_PATH_BATCH, X, T, eps, Y, flags, rho, workspace,
               static_cast<cudaStream_t>(stream));
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_linear(const gsi_map_desc* map, const void* X, int64_t T, float eps, float* Y,
                      uint8_t* flags, float* rho, void* workspace, size_t ws_bytes, void* stream) {
  return gsi_linear_ex(map, X, T, eps, Y, flags, rho, workspace, ws_bytes, GSI_PATH_AUTO, stream);
}

gsi_status gsi_path_errors(const gsi_map_desc* map, const void* X, int64_t T, float* Y_fast, float* Y_slow,
                           uint8_t* flags, float* rho, float* err, float* ynorm, void* workspace, size_t ws_bytes,
                           void* stream) {
  gsi_status s = check_map(map);
  if (s != GSI_OK) return s;
  if ((s = check_tokens(T, 0.f)) != GSI_OK) return s;
  gsi_path p;
  if ((s = resolve_path(map, T, GSI_PATH_AUTO, &p)) != GSI_OK) return s;
  if (T == 0) return ok();
  if ((s = check_ptr(X, "X")) != GSI_OK) return s;
  if ((s = check_ptr(Y_fast, "Y_fast")) != GSI_OK) return s;
  if ((s = check_ptr(Y_slow, "Y_slow")) != GSI_OK) return s;
  if (!flags) return fail(GSI_ERR_INVALID_ARG, "flags is NULL");
  if (!rho || !err || !ynorm || !aligned(rho, 4) || !aligned(err, 4) || !aligned(ynorm, 4))
    return fail(GSI_ERR_INVALID_ARG, "rho, err and ynorm must be 4-byte aligned device arrays");
  if ((s = check_workspace(workspace, ws_bytes, path_ws(map, T, p))) != GSI_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float inf = __builtin_huge_valf();
  if ((s = run_path(map, p, false, X, T, inf, Y_fast, flags, rho, workspace, st)) != GSI_OK) return s;
  if ((s = run_path(map, p, false, X, T, 0.f, Y_slow, flags, nullptr, workspace, st)) != GSI_OK) return s;
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  s = cuda_check(launch_path_norms(Y_fast, Y_slow, T, map->d_out, err, ynorm, st), "path-norm kernel launch");
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_eps_sweep(const float* rho, const float* err, const float* ynorm, int64_t T, const float* eps,
                         int64_t n_eps, int64_t tokens_per_call, int32_t* n_slow, int32_t* n_slow_calls,
                         float* rel_err, void* stream) {
  if (T < 0 || n_eps < 0) return fail(GSI_ERR_INVALID_ARG, "T and n_eps must be >= 0");
  if (tokens_per_call < 1) return fail(GSI_ERR_INVALID_ARG, "tokens_per_call must be >= 1");
  if (T > (int64_t(1) << 31) - 1 || n_eps > 65535) return fail(GSI_ERR_UNSUPPORTED, "T or n_eps too large");
  if (n_eps == 0) return ok();
  if (!eps || !n_slow || !n_slow_calls || !rel_err) return fail(GSI_ERR_INVALID_ARG, "a sweep output or eps is NULL");
  if (T > 0 && (!rho || !err || !ynorm)) return fail(GSI_ERR_INVALID_ARG, "rho, err or ynorm is NULL");
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  const gsi_status s = cuda_check(launch_sweep(rho, err, ynorm, T, eps, n_eps, tokens_per_call, n_slow, n_slow_calls,
                                               rel_err, static_cast<cudaStream_t>(stream)),
                                  "sweep kernel launch");
  return s == GSI_OK ? ok() : s;
}

size_t gsi_residual_check_work_bytes(int64_t d, int64_t T) {
  if (d < 1 || T < 1) return 0;
  return residual_check_work_bytes(d, T);
}

gsi_status gsi_residual_check(const gsi_map_desc* map, const void* X, int64_t T, const float* G, const float* rho,
                              float* rho_explicit, float* max_dev, void* work, size_t work_bytes, void* stream) {
  gsi_status s = check_map(map);
  if (s != GSI_OK) return s;
  if ((s = check_tokens(T, 0.f)) != GSI_OK) return s;
  if (T > (int64_t(65535) * 8)) return fail(GSI_ERR_UNSUPPORTED, "the residual check takes T <= 524280");
  if (!max_dev || !aligned(max_dev, 4)) return fail(GSI_ERR_INVALID_ARG, "max_dev is NULL or misaligned");
  if (T == 0) {
    if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
    s = cuda_check(cudaMemsetAsync(max_dev, 0, sizeof(float), static_cast<cudaStream_t>(stream)), "max_dev clear");
    return s == GSI_OK ? ok() : s;
  }
  if ((s = check_ptr(X, "X")) != GSI_OK) return s;
  if ((s = check_ptr(G, "G")) != GSI_OK) return s;
  if (!rho || !rho_explicit || !aligned(rho, 4) || !aligned(rho_explicit, 4))
    return fail(GSI_ERR_INVALID_ARG, "rho and rho_explicit must be 4-byte aligned device arrays");
  const size_t need = residual_check_work_bytes(map->d, T);
  if (!work || !aligned(work, 256) || work_bytes < need)
    return fail(GSI_ERR_WORKSPACE, "work must be 256-byte aligned and hold %zu bytes", need);
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  s = cuda_check(launch_residual_check(X, map->V, G, rho, map->d, int(map->k), T, map->dtype, rho_explicit, max_dev,
                                       work, static_cast<cudaStream_t>(stream)),
                 "residual check launch");
  return s == GSI_OK ? ok() : s;
}

static gsi_status check_basis(int64_t k, int64_t d) {
  if (k < 1 || d < 1) return fail(GSI_ERR_INVALID_ARG, "k and d must be positive");
  if (k > GSI_MAX_K) return fail(GSI_ERR_UNSUPPORTED, "k=%lld above GSI_MAX_K", (long long)k);
  if (k > d) return fail(GSI_ERR_INVALID_ARG, "k=%lld above d=%lld", (long long)k, (long long)d);
  if (d > (int64_t(1) << 31)) return fail(GSI_ERR_UNSUPPORTED, "d above 2^31");
  return GSI_OK;
}

size_t gsi_basis_step_work_bytes(int64_t T, int64_t d, int64_t k) {
  if (T < 1 || d < 1 || k < 1) return 0;
  return align256(size_t(T) * k * 4) + size_t(k) * d * 4;
}

gsi_status gsi_basis_orthonormalize(float* Vt, int64_t k, int64_t d, int32_t* n_reorth, void* stream) {
  gsi_status s = check_basis(k, d);
  if (s != GSI_OK) return s;
  if (!Vt || !aligned(Vt, 4)) return fail(GSI_ERR_INVALID_ARG, "Vt is NULL or misaligned");
  if (n_reorth && !aligned(n_reorth, 4)) return fail(GSI_ERR_INVALID_ARG, "n_reorth is misaligned");
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  s = cuda_check(launch_dgks(Vt, d, int(k), n_reorth, static_cast<cudaStream_t>(stream)), "DGKS kernel launch");
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_basis_step(const void* X, gsi_dtype xdt, int64_t T, int64_t d, int64_t k, float* Vt, void* work,
                          size_t work_bytes, int32_t* n_reorth, void* stream) {
  gsi_status s = check_basis(k, d);
  if (s != GSI_OK) return s;
  if (T < 1) return fail(GSI_ERR_INVALID_ARG, "T must be positive");
  if (xdt != GSI_F32 && xdt != GSI_BF16) return fail(GSI_ERR_INVALID_ARG, "unknown dtype %d", int(xdt));
  if (!X || !aligned(X, xdt == GSI_BF16 ? 2 : 4)) return fail(GSI_ERR_INVALID_ARG, "X is NULL or misaligned");
  if (!Vt || !aligned(Vt, 4)) return fail(GSI_ERR_INVALID_ARG, "Vt is NULL or misaligned");
  const size_t need = gsi_basis_step_work_bytes(T, d, k);
  if (!work || !aligned(work, 256) || work_bytes < need)
    return fail(GSI_ERR_WORKSPACE, "work must be 256-byte aligned and hold %zu bytes", need);
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* P = static_cast<float*>(work);                                              // T x k: X V
  float* Zt = reinterpret_cast<float*>(static_cast<char*>(work) + align256(size_t(T) * k * 4));  // k x d
  // P[t][i] = sum_r X[t][r] Vt[i][r];  Zt[i][r] = sum_t P[t][i] X[t][r]
  if ((s = cuda_check(launch_contract(X, xdt, d, 1, Vt, GSI_F32, 1, d, P, k, T, k, d, st), "X V")) != GSI_OK) return s;
  if ((s = cuda_check(launch_contract(P, GSI_F32, 1, k, X, xdt, d, 1, Zt, d, k, d, T, st), "X^T (X V)")) != GSI_OK)
    return s;
  if ((s = cuda_check(launch_dgks(Zt, d, int(k), n_reorth, st), "DGKS kernel launch")) != GSI_OK) return s;
  s = cuda_check(cudaMemcpyAsync(Vt, Zt, size_t(k) * d * 4, cudaMemcpyDeviceToDevice, st), "basis copy");
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_basis_coherence(const float* Vt_a, const float* Vt_b, int64_t k, int64_t d, float* out, float* work,
                               void* stream) {
  gsi_status s = check_basis(k, d);
  if (s != GSI_OK) return s;
  if (!Vt_a || !Vt_b || !out || !work || !aligned(Vt_a, 4) || !aligned(Vt_b, 4) || !aligned(out, 4) ||
      !aligned(work, 4))
    return fail(GSI_ERR_INVALID_ARG, "Vt_a, Vt_b, out and work must be 4-byte aligned device pointers");
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // S[i][j] = sum_r Vt_a[i][r] Vt_b[j][r]
  if ((s = cuda_check(launch_contract(Vt_a, GSI_F32, d, 1, Vt_b, GSI_F32, 1, d, work, k, k, k, d, st), "Va^T Vb")) !=
      GSI_OK)
    return s;
  s = cuda_check(launch_sumsq(work, k * k, 1.f / float(k), out, st), "coherence reduction");
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_basis_export(const float* Vt, int64_t k, int64_t d, void* V, gsi_dtype dt, void* stream) {
  gsi_status s = check_basis(k, d);
  if (s != GSI_OK) return s;
  if (dt != GSI_F32 && dt != GSI_BF16) return fail(GSI_ERR_INVALID_ARG, "unknown dtype %d", int(dt));
  if (!Vt || !V || !aligned(Vt, 4) || !aligned(V, dt == GSI_BF16 ? 2 : 4))
    return fail(GSI_ERR_INVALID_ARG, "Vt or V is NULL or misaligned");
  if (injected_failure()) return fail(GSI_ERR_CUDA, "injected failure (gsi_debug_fail_after)");
  s = cuda_check(launch_transpose_cast(Vt, k, d, V, dt, static_cast<cudaStream_t>(stream)), "basis export");
  return s == GSI_OK ? ok() : s;
}

gsi_status gsi_stack_workspace_size(const gsi_map_desc* maps, int64_t n_maps, int64_t T, size_t* bytes) {
  if (!bytes) return fail(GSI_ERR_INVALID_ARG, "bytes is NULL");
  if (!maps || n_maps <= 0) return fail(GSI_ERR_INVALID_ARG, "maps is NULL or n_maps <= 0");
  size_t need = 0;
  for (int64_t i = 0; i < n_maps; ++i) {
    size_t b = 0;
    gsi_status s = gsi_linear_workspace_size(&maps[i], T, GSI_PATH_AUTO, &b);
    if (s != GSI_OK) return s;
    if (b > need) need = b;
  }
  *bytes = need;
  return ok();
}

gsi_status gsi_stack(const gsi_map_desc* maps, int64_t n_maps, const void* const* X, int64_t T,
                     float eps, float* const* Y, uint8_t* const* flags, void* workspace,
                     size_t ws_bytes, void* stream) {
  return gsi_stack_ex(maps, n_maps, X, T, eps, Y, flags, workspace, ws_bytes, GSI_STACK_AUTO, stream);
}

gsi_status gsi_stack_ex(const gsi_map_desc* maps, int64_t n_maps, const void* const* X, int64_t T,
                        float eps, float* const* Y, uint8_t* const* flags, void* workspace,
                        size_t ws_bytes, gsi_stack_mode mode, void* stream) {
  if (mode != GSI_STACK_AUTO && mode != GSI_STACK_PER_MAP && mode != GSI_STACK_PERSISTENT)
    return fail(GSI_ERR_INVALID_ARG, "unknown stack mode %d", int(mode));
  if (!maps || n_maps <= 0) return fail(GSI_ERR_INVALID_ARG, "maps is NULL or n_maps <= 0");
  if (!X || !Y || !flags) return fail(GSI_ERR_INVALID_ARG, "X, Y and flags arrays must be non-NULL");
  gsi_status s = check_tokens(T, eps);
  if (s != GSI_OK) return s;
  size_t need = 0;
  for (int64_t i = 0; i < n_maps; ++i) {
    if ((s = check_map(&maps[i])) != GSI_OK)
      return fail(s, "map %lld: %s", (long long)i, g_err.c_str());
    if (T > 0) {
      if ((s = check_ptr(X[i], "X[i]")) != GSI_OK) return fail(s, "map %lld: %s", (long long)i, g_err.c_str());
      if ((s = check_ptr(Y[i], "Y[i]")) != GSI_OK) return fail(s, "map %lld: %s", (long long)i, g_err.c_str());
      if (!flags[i]) return fail(GSI_ERR_INVALID_ARG, "map %lld: flags is NULL", (long long)i);
    }
    gsi_path p;
    if ((s = resolve_path(&maps[i], T, GSI_PATH_AUTO, &p)) != GSI_OK) return s;
    size_t b = path_ws(&maps[i], T, p);
    if (b > need) need = b;
  }
  if (T == 0) return ok();
  if ((s = check_workspace(workspace, ws_bytes, need)) != GSI_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // GSI_STACK_PERSISTENT with one token per map: runs of consecutive maps
  // that the single-token kernel takes (one element type, row width and k)
  // go to the persistent stack kernel, up to kStackMaxMaps per launch; every
  // other map (and a run the device refuses) is one call each.  AUTO and
  // PER_MAP run one call per map: a launch boundary chained by programmatic
  // dependent launch was measured faster than the persistent kernel's grid
  // barrier between maps.
  DeviceFacts* f = nullptr;
  if (T == 1 && mode == GSI_STACK_PERSISTENT && (s = device_facts(&f)) != GSI_OK) return s;
  auto stackable = [&](int64_t j) {
    gsi_path p;
    return resolve_path(&maps[j], 1, GSI_PATH_AUTO, &p) == GSI_OK && p == GSI_PATH_FUSED &&
           decode_plan(&maps[j], f).ok;
  };
  for (int64_t i = 0; i < n_maps;) {
    if (f && stackable(i)) {
      int64_t j = i + 1;
      while (j < n_maps && j - i < kStackMaxMaps && maps[j].dtype == maps[i].dtype && maps[j].k == maps[i].k &&
             stackable(j))
        ++j;
      if (j - i >= 2) {
        s = run_stack_decode(&maps[i], int(j - i), X + i, eps, Y + i, flags + i, workspace, st, f);
        if (s == GSI_OK) {
          i = j;
          continue;
        }
        if (s != GSI_ERR_UNSUPPORTED) return fail(s, "maps %lld-%lld: %s", (long long)i, (long long)(j - 1), g_err.c_str());
      }
    }
    gsi_path p;
    resolve_path(&maps[i], T, GSI_PATH_AUTO, &p);
    s = run_path(&maps[i], p, false, X[i], T, eps, Y[i], flags[i], nullptr, workspace, st,
                 i + 1 < n_maps ? &maps[i + 1] : nullptr, i + 1 < n_maps ? X[i + 1] : nullptr);
    if (s != GSI_OK) return fail(s, "map %lld: %s", (long long)i, g_err.c_str());
    ++i;
  }
  return ok();
}

}  // extern "C"
