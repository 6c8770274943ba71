// gsi_linear_noalloc: the gated linear map for callers that cannot allocate.
//
// Some callers have no way to hand the library a workspace: code running
// where device allocation is forbidden or unavailable (an allocator hook that
// must not recurse into cudaMalloc, a plug-in loaded into a host program that
// owns all device memory, a real-time loop that may not allocate at all).
// For them this file keeps the scratch the streaming kernels need in one
// file-scope device array, sized once at load time and held by every GPU that
// loads the library until the process exits.  The caller still owns and
// passes the inputs and outputs; nothing here calls cudaMalloc, cudaFree or
// an allocating library routine.

#include <cstdio>
#include <mutex>

#include "gsi_common.cuh"
#include "gsi_kernels.h"
#include "gsi_plan.h"

namespace {

// Largest workspace a call may need: 4 MiB covers decode-sized calls of the
// 6B / 13B shapes (e.g. d = 16384, k = 256 up to 64 tokens).
constexpr size_t kScratchBytes = size_t(4) << 20;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, never a device address: the address comes from
// cudaGetSymbolAddress, looked up once per device below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up on first use).
gsi_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    char msg[256];
    snprintf(msg, sizeof msg, "gsi_linear_noalloc: no usable current device (%s)", cudaGetErrorString(e));
    return gsi::record_error(GSI_ERR_CUDA, msg);
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof msg, "gsi_linear_noalloc: cudaGetSymbolAddress failed (%s)", cudaGetErrorString(e));
      return gsi::record_error(GSI_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GSI_OK;
}

}  // namespace

extern "C" size_t gsi_linear_noalloc_max_bytes(void) { return kScratchBytes; }

extern "C" gsi_status gsi_linear_noalloc_status(uint32_t* code, void* stream) {
  if (!code) return gsi::record_error(GSI_ERR_INVALID_ARG, "gsi_linear_noalloc_status: code is NULL");
  void* ws = nullptr;
  gsi_status s = scratch_address(&ws);
  if (s != GSI_OK) return s;
  // the error word sits in the control block at the head of the scratch
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint32_t* err = &static_cast<const gsi::Ctrl*>(ws)->err;
  cudaError_t e = cudaMemcpyAsync(code, err, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "gsi_linear_noalloc_status: reading the error word failed (%s)", cudaGetErrorString(e));
    return gsi::record_error(GSI_ERR_CUDA, msg);
  }
  if (*code) {
    char msg[128];
    snprintf(msg, sizeof msg, "gsi_linear_noalloc: a bounded device wait gave up (error word %u)", *code);
    return gsi::record_error(GSI_ERR_TIMEOUT, msg);
  }
  return gsi::record_error(GSI_OK, "");
}

extern "C" gsi_status gsi_linear_noalloc(const gsi_map_desc* map, const void* X, int64_t T, float eps,
                                         float* Y, uint8_t* flags, float* rho, void* stream) {
  size_t need = 0;
  gsi_status s = gsi_linear_workspace_size(map, T, GSI_PATH_STREAM, &need);
  if (s != GSI_OK) return s;
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "gsi_linear_noalloc: this call needs %zu bytes of scratch but the built-in area holds %zu; "
             "use gsi_linear with a caller workspace",
             need, kScratchBytes);
    return gsi::record_error(GSI_ERR_WORKSPACE, msg);
  }
  if (T == 0) return gsi_linear_ex(map, X, T, eps, Y, flags, rho, nullptr, 0, GSI_PATH_STREAM, stream);
  void* ws = nullptr;
  if ((s = scratch_address(&ws)) != GSI_OK) return s;
  // The area keeps the previous call's contents; the control block (arrival
  // ticket, error word, counts) must start at zero.
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(gsi::Ctrl), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "gsi_linear_noalloc: clearing the scratch control block failed (%s)",
             cudaGetErrorString(e));
    return gsi::record_error(GSI_ERR_CUDA, msg);
  }
  return gsi_linear_ex(map, X, T, eps, Y, flags, rho, ws, kScratchBytes, GSI_PATH_STREAM, stream);
}
