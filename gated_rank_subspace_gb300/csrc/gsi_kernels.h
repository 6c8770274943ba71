// Kernel argument blocks and host launchers (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gsi.h"
#include "gsi_plan.h"

namespace gsi {

struct Ctrl;

struct GateArgs {
  const void* X;        // T x d tokens
  const void* V;        // d x k basis
  int64_t d;
  int k, T;
  int rs, nv, nrg, ks, n_clusters;
  float* part_g;        // [n_clusters][T][k]
  float* part_x;        // [n_clusters][T]
  // Speculative L2 prefetch, for the decide-and-apply kernel that follows:
  // the image M (most tokens take the fast path) and the Gram matrix.
  const char* pf_m;
  uint64_t pf_m_bytes;
  const char* pf_g;
  uint64_t pf_g_bytes;
};

// Decide-and-apply kernel arguments (see gsi_apply.cu).
struct DecideArgs {
  const void* X;        // T x d
  const void* W;        // d_out x d
  const void* M;        // d_out x k
  const float* gram;    // k x k, or null (orthonormal)
  const float* part_g;  // [nclu][T][k] projection partials
  const float* part_x;  // [nclu][T]
  int nclu;
  int64_t d, d_out;
  int k, T, ks;
  float eps;
  int mode;             // 0 decide + apply, 1 decide only, 2 apply a stored decision
  float* Y;             // T x d_out (modes 0, 2)
  float* G;             // T x k projections out (mode 1), or null
  float* rho;           // T, or null
  uint8_t* flags;       // T flags out (modes 0, 1)
  uint8_t* flags_user;  // mode 1: the caller's flags (a copy of the stored ones), or null
  int32_t* idx;         // 2T compaction (mode 1)
  int32_t* counts;      // 2 (mode 1)
  const float* Gin;     // T x k stored projections (mode 2)
  const uint8_t* flags_in;  // T stored flags (mode 2)
  int rows_per_cta, seg_bytes, wstages, x_stage_max, stage_m;
  int off_m, off_x, off_g, off_gram;
  int off_y;            // [TC][rows_per_cta] fast outputs computed before the decision (mode 0)
  // fused decode (the grid projects x itself): CTA b projects V rows
  // [b * v_rows, ...), publishes its partials in fpart_g / fpart_x (laid out
  // like the projection kernel's cluster partials, one per CTA) and meets the
  // other CTAs at a grid barrier on the workspace's ticket counter
  const void* V;        // d x k
  int v_rows, ngrp, off_v, off_xs;
  int cproj;            // each cluster projects x on all of V (16-CTA clusters; no grid barrier)
  float* fpart_g;       // [grid][T][k]
  float* fpart_x;       // [grid][T]
  unsigned long long* ticket;
  // weights of the next map of a stack, staged in L2 while this one runs
  const char* next_v;
  uint64_t next_v_bytes;
  const char* next_m;
  uint64_t next_m_bytes;
  const char* next_gram;
  uint64_t next_gram_bytes;
  uint32_t* err;
};


// One map's single-token call (see gsi_decode.cu): the operands and the
// DecodePlan geometry and shared-memory offsets.
struct DecodeMap {
  const void* X;        // 1 x d token
  const void* W;        // d_out x d
  const void* V;        // d x k
  const void* M;        // d_out x k
  const float* gram;    // k x k, or null (orthonormal basis)
  float* Y;             // 1 x d_out
  uint8_t* flags;       // 1
  float* rho;           // 1, or null
  int64_t d, d_out;
  int k;
  int vr, rw, rpc, ks, seg_bytes, sw, red_stride, m_late;
  int off_g, off_y, off_in, off_gram, off_red, off_v, off_m;
  // grid projection: each cluster's slice of g is published as epoch-tagged
  // words in the workspace; 0: the cluster projection
  int grid;
};

// Single-token decode kernel arguments: one call of the gated map for one
// token, decide and apply, in one launch.
struct DecodeArgs {
  DecodeMap m;
  float eps;
  // grid projection: each cluster's partial g [clusters][k] and ||x||^2
  // [clusters] as epoch-tagged words; the call's epoch comes from a ticket
  float* part_g;
  float* part_x;
  unsigned long long* ticket;
  // weights of the next map of a stack, staged in L2 while this one runs
  const char* next_v;
  uint64_t next_v_bytes;
  const char* next_m;
  uint64_t next_m_bytes;
  const char* next_gram;
  uint64_t next_gram_bytes;
  uint32_t* err;        // device error word (bounded waits)
  // test hook (grid projection): cluster 0 withholds its slice words, so the
  // other ranks' polls give up after poll_cycles (0: the default ~2 s)
  int dbg_withhold;
  long long poll_cycles;
};

// Persistent stack decode: one launch runs up to kStackMaxMaps single-token
// calls in list order, the calls separated by a grid barrier (map i + 1
// reads its token only after every CTA has finished map i).  The maps share
// one element type and row width (one kernel instantiation).
constexpr int kStackMaxMaps = 112;

struct StackDecodeArgs {
  DecodeMap maps[kStackMaxMaps];
  int n_maps;
  float eps;
  float* part_g;                // as DecodeArgs
  float* part_x;
  unsigned long long* ticket;   // shared with the single-token kernel: numbers the launch
  unsigned long long* arrive;   // arrivals at the barriers between maps
  uint32_t* err;
};

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& p, gsi_dtype dt, cudaStream_t s);
// The persistent stack kernel with `smem` bytes of shared memory (the
// largest plan of its maps) and `ncta` CTAs (the single-token kernel's grid).
cudaError_t launch_stack_decode(const StackDecodeArgs& a, size_t smem, int ncta, int nv, gsi_dtype dt,
                                cudaStream_t s);
// Co-resident kDecodeCluster-CTA clusters of the single-token decode kernel
// with `smem` bytes of shared memory per CTA; 0 if none.
int decode_max_clusters(size_t smem, gsi_dtype dt);
// The same for the persistent stack kernel (nv vectors of a row per lane).
int stack_max_clusters(size_t smem, gsi_dtype dt, int nv);

// Small-batch decode (see gsi_batch.cu): one call of a bf16 map for
// 2 <= T <= 16 tokens in one launch.  Device pointers; part_g / part_x are
// the workspace's epoch-tagged words (BatchLayout).
struct BatchCall {
  const void* X;        // T x d tokens
  const void* W;        // d_out x d
  const void* V;        // d x k
  const void* M;        // d_out x k
  const float* gram;    // k x k
  float* Y;             // T x d_out
  uint8_t* flags;       // T
  float* rho;           // T, or null
  int64_t d, d_out;
  int k, T;
  float eps;
  unsigned long long* part_g;  // [clusters][T][k]
  unsigned long long* part_x;  // [clusters][16]
  unsigned long long* ticket;  // numbers the calls (the words' epochs)
  uint32_t* err;               // device error word
  // weights of the next map of a stack, staged in L2 while this one runs
  const char* next_v;
  uint64_t next_v_bytes;
  const char* next_m;
  uint64_t next_m_bytes;
  const char* next_gram;
  uint64_t next_gram_bytes;
  const char* next_x;  // the next map's tokens
  uint64_t next_x_bytes;
  // test hook: cluster 0 withholds its words, so the other clusters' polls
  // give up after poll_cycles (0: the default ~2 s)
  int dbg_withhold;
  long long poll_cycles;
};

cudaError_t launch_batch_decode(const BatchCall& c, const BatchPlan& p, cudaStream_t s);
// Co-resident kBatchCluster-CTA clusters of the small-batch kernel at the
// largest shared-memory request; 0 if none.
int batch_max_clusters(size_t smem);

// Tensor-core path (bf16, prefill-sized T).  All pointers are device pointers;
// Vt, G, Gbf, Gfast, Xslow and idx live in the call's workspace.
struct TensorArgs {
  const void* X;        // T x d
  const void* V;        // d x k
  const void* W;        // d_out x d
  const void* M;        // d_out x k
  const float* gram;    // k x k
  int64_t d, d_out, k, T;
  float eps;
  uint16_t* Vt;         // k x d
  float* G;             // T x k fp32
  uint16_t* Gbf;        // T x k bf16
  uint16_t* Gfast;      // T x k bf16 (gathered fast rows)
  uint16_t* Xslow;      // T x d bf16 (gathered slow rows)
  int32_t* idx;         // 2T
  int32_t* counts;      // 2
  float* rho;           // T or null
  uint8_t* flags;       // T
  float* Y;             // T x d_out
  uint32_t* err;        // device error word
  float* gT;            // float32 g by chunks of 8 tokens: [chunk][k][8]
  float2* norms;        // per token (||g||^2, ||x||^2)
};

cudaError_t launch_tensor_path(const TensorArgs& t, cudaStream_t s);
// The slow rows of a call whose decision, compaction (idx: fast tokens, then
// slow tokens from idx + T; counts = {n_fast, n_slow}) and fast rows are done:
// the slow tokens' x gathered into Xslow (T x d bf16 scratch), then
// Y[slow] = X_slow W^T as the few-token tensor-core contraction.
cudaError_t launch_slow_rows_tc(const void* X, const void* W, int64_t d, int64_t d_out, int64_t T,
                                const int32_t* idx, const int32_t* counts, uint16_t* Xslow, float* Y, uint32_t* err,
                                cudaStream_t s);
// M = W V_k (bf16) on the tensor cores; Vt: k x d bf16 scratch.
cudaError_t launch_image_tc(const void* W, const void* V, void* M, int64_t d, int64_t d_out, int64_t k,
                            uint16_t* Vt, uint32_t* err, cudaStream_t s);
// The Gram matrix V_k^T V_k (k x k float32) on the CUDA cores.
cudaError_t launch_gram(const void* V, float* gram, int64_t d, int64_t k, gsi_dtype dt, cudaStream_t s);

// Sets the calling thread's gsi_last_error() message and returns s.
gsi_status record_error(gsi_status s, const char* msg);

cudaError_t launch_gate(const GateArgs& a, const GatePlan& p, gsi_dtype dt, cudaStream_t s,
                        bool pdl);
cudaError_t launch_compact(const uint8_t* flags, int T, int32_t* idx, int32_t* counts,
                           cudaStream_t s);
cudaError_t launch_decide_apply(const DecideArgs& a, const DecidePlan& p, gsi_dtype dt, cudaStream_t s);
int decide_apply_max_clusters(size_t smem, gsi_dtype dt, bool fused, int cs);
cudaError_t launch_path_norms(const float* Yf, const float* Ys, int64_t T, int64_t d_out, float* err, float* ynorm,
                              cudaStream_t s);
cudaError_t launch_sweep(const float* rho, const float* err, const float* ynorm, int64_t T, const float* eps,
                         int64_t n_eps, int64_t tokens_per_call, int32_t* n_slow, int32_t* n_slow_calls,
                         float* rel_err, cudaStream_t s);
cudaError_t launch_contract(const void* A, gsi_dtype adt, int64_t sam, int64_t sak, const void* B, gsi_dtype bdt,
                            int64_t sbk, int64_t sbn, float* C, int64_t ldc, int64_t Md, int64_t Nd, int64_t Kd,
                            cudaStream_t s);
// Basis construction (see gsi_basis.cu).
cudaError_t launch_dgks(float* Qt, int64_t d, int k, int32_t* n_reorth, cudaStream_t s);
cudaError_t launch_sumsq(const float* S, int64_t n, float scale, float* out, cudaStream_t s);
cudaError_t launch_transpose_cast(const float* Qt, int64_t k, int64_t d, void* V, gsi_dtype dt, cudaStream_t s);
// Explicit-residual check of the gate (see gsi_check.cu).
size_t residual_check_work_bytes(int64_t d, int64_t T);
cudaError_t launch_residual_check(const void* X, const void* V, const float* G, const float* rho, int64_t d, int k,
                                  int64_t T, gsi_dtype dt, float* rho_x, float* max_dev, void* work,
                                  cudaStream_t s);
cudaError_t launch_image(const void* W, const void* V, void* M, float* gram, int64_t d,
                         int64_t d_out, int64_t k, gsi_dtype dt, cudaStream_t s);

}  // namespace gsi
