// Asynchronous-copy, mbarrier and cluster-exchange wrappers shared by the
// decode kernels (sm_103a inline PTX).  Every wait is bounded: after ~2 s of
// clock it sets the caller's error word and returns false.
#pragma once

#include "gsi_common.cuh"

namespace gsi {

__device__ __forceinline__ uint32_t sa(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(n) : "memory");
}
// A barrier's memory is reused for a new barrier only after the old one is
// invalidated (init on a valid mbarrier object is undefined).
__device__ __forceinline__ void bar_inval(uint64_t* b) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(sa(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
constexpr long long kSpinCycles = 4000000000LL;  // ~2 s at 2 GHz
// After an earlier wait of the same launch gave up, the remaining waits use
// this short limit (~1 ms): every wait still runs, so no CTA leaves while a
// peer may write into its shared memory, but the launch ends promptly.
constexpr long long kSpinCyclesAfterError = 2000000LL;
// `site` (a bit above kErrTimeout) records which wait gave up.
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t parity, uint32_t* err, long long lim = kSpinCycles,
                                         uint32_t site = 0) {
  if (bar_try(b, parity)) return true;
  const long long t0 = clock64();
  while (!bar_try(b, parity)) {
    if (clock64() - t0 > lim) {
      atomicOr(err, kErrTimeout | site);
      return false;
    }
  }
  return true;
}
// Grid barrier of the fused decode on a ticket counter in the workspace.
// One thread per CTA, after a __syncthreads that follows the CTA's stores:
// publish them (fence), take a ticket, and wait, bounded, until the n CTAs of
// this barrier episode have all taken theirs.  Episodes never overlap: a
// call's CTAs reach the barrier only after the dependency wait on the previous
// kernel, and every call's grid has the same n for an element type, so the
// episode of ticket t ends at (t / n + 1) * n.  The grid is sized so that all
// its CTAs are co-resident.  (Measured: taking the ticket with a returning
// atomic beats a fire-and-forget add against a count read in advance.)
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool grid_barrier(unsigned long long* ticket, unsigned long long n, uint32_t* err) {
  __threadfence();
  const unsigned long long mine = atomicAdd(ticket, 1ull);
  const unsigned long long target = (mine / n + 1) * n;
  if (ld_acquire_gpu(ticket) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire_gpu(ticket) < target) {
    if (clock64() - t0 > kSpinCycles) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
  return true;
}

// Epoch-tagged words across the grid: a 64-bit word (epoch << 32 | value
// bits) is stored and loaded whole, so a reader that sees the current epoch
// also sees that value, with no fence or flag between them.
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Exchanges inside a cluster: st.async stores into a peer's shared memory
// that complete on the peer's mbarrier, so each CTA waits (acquire at
// cluster scope, bounded) only for the bytes it receives.
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, int r) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(saddr), "r"(r));
  return out;
}
__device__ __forceinline__ void st_async_f32(uint32_t raddr, float v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr),
               "r"(__float_as_uint(v)), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ void st_async_v4(uint32_t raddr, float4 v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(raddr),
               "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
               "r"(__float_as_uint(v.w)), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ bool bar_try_cluster(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(sa(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool bar_wait_cluster(uint64_t* b, uint32_t parity, uint32_t* err,
                                                 long long lim = kSpinCycles, uint32_t site = 0) {
  if (bar_try_cluster(b, parity)) return true;
  const long long t0 = clock64();
  while (!bar_try_cluster(b, parity)) {
    if (clock64() - t0 > lim) {
      atomicOr(err, kErrTimeout | site);
      return false;
    }
  }
  return true;
}

// 1-D bulk copy global -> shared (16-byte aligned, multiple of 16 bytes).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   sa(dst)),
               "l"(src), "r"(bytes), "r"(sa(b))
               : "memory");
}

template <bool B>
struct BoolC {
  static constexpr bool value = B;
};
template <int N>
struct IntC {
  static constexpr int value = N;
};

}  // namespace gsi
