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
  const float* gram;    // k x k V^T V, or null (orthonormal)
  int64_t d;
  int k, T;
  float eps;
  int rs, nv, nrg, ks, n_clusters;
  float* part_g;        // [n_clusters][T][k]
  float* part_x;        // [n_clusters][T]
  float* G;             // [T][k] projections (output)
  float* rho;           // [T] or null
  uint8_t* flags;       // [T]
  int32_t* idx;         // [2T] compaction lists, or null
  Ctrl* ctrl;
  const char* pf_base;  // L2 prefetch of the image M (speculative fast path)
  uint64_t pf_share;    // bytes per CTA (multiple of 16), 0 = off
  uint64_t pf_total;
  uint64_t gram_share;  // L2 prefetch of the Gram: bytes per CTA (multiple of 16), 0 = off
};

struct ApplyArgs {
  const void* W;        // d_out x d
  const void* M;        // d_out x k
  const void* X;        // T x d
  const float* G;       // T x k
  float* Y;             // T x d_out
  const int32_t* idx;   // [2T]
  const Ctrl* ctrl;
  int64_t d, d_out;
  int k, T;
  int rows_slow;
  int64_t fast_units, slow_units;
  int x_stage_max, g_stage_max;
};

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
};

cudaError_t launch_tensor_path(const TensorArgs& t, cudaStream_t s);

// Sets the calling thread's gsi_last_error() message and returns s.
gsi_status record_error(gsi_status s, const char* msg);

cudaError_t launch_gate(const GateArgs& a, const GatePlan& p, gsi_dtype dt, cudaStream_t s,
                        bool pdl);
cudaError_t launch_compact(const uint8_t* flags, int T, int32_t* idx, int32_t* counts,
                           cudaStream_t s);
cudaError_t launch_apply(const ApplyArgs& a, const ApplyPlan& p, gsi_dtype dt, int nsm,
                         cudaStream_t s, bool pdl);
cudaError_t launch_image(const void* W, const void* V, void* M, float* gram, int64_t d,
                         int64_t d_out, int64_t k, gsi_dtype dt, cudaStream_t s);

}  // namespace gsi
