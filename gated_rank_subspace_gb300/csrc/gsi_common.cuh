// Shared device helpers for the gated-subspace kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cooperative_groups.h>
#include <stdint.h>
#include <cstdlib>

#include "../../include/gsi.h"

namespace gsi {

namespace cg = cooperative_groups;

// ---------------------------------------------------------------- packed float pairs
// Two float32 lanes in one 64-bit register, for the paired FMA of sm_100-class
// GPUs (fma.rn.f32x2: two independent float32 FMAs, each rounded once).
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
  return make_float2(a, b);
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// ---------------------------------------------------------------- element types
// Both storage types are read as 16-byte vectors: 4 float32 or 8 bf16.
struct F32 {
  static constexpr int kBytes = 4;
  static constexpr int kPerVec = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static float load1(const void* base, int64_t i) {
    return reinterpret_cast<const float*>(base)[i];
  }
  __device__ __forceinline__ static void store1(void* base, int64_t i, float v) {
    reinterpret_cast<float*>(base)[i] = v;
  }
  __device__ __forceinline__ static float load1_cg(const void* base, int64_t i) {
    return __ldcg(reinterpret_cast<const float*>(base) + i);
  }
  // acc[e] += x * w[e] for the 4 elements of w
  __device__ __forceinline__ static void axpy(const uint4& w, float x, float* acc) {
    acc[0] = fmaf(x, __uint_as_float(w.x), acc[0]);
    acc[1] = fmaf(x, __uint_as_float(w.y), acc[1]);
    acc[2] = fmaf(x, __uint_as_float(w.z), acc[2]);
    acc[3] = fmaf(x, __uint_as_float(w.w), acc[3]);
  }
  // sum over the vector of w[e] g[e], in element order
  __device__ __forceinline__ static float dot_vec(const uint4& w, const float* g) {
    float p = __uint_as_float(w.x) * g[0];
    p = fmaf(__uint_as_float(w.y), g[1], p);
    p = fmaf(__uint_as_float(w.z), g[2], p);
    p = fmaf(__uint_as_float(w.w), g[3], p);
    return p;
  }
  // a0 += w.x*x.x + w.z*x.z, a1 += w.y*x.y + w.w*x.w (in that order)
  __device__ __forceinline__ static void dot_acc(const uint4& w, const uint4& x, float& a0, float& a1) {
    a0 = fmaf(__uint_as_float(w.x), __uint_as_float(x.x), a0);
    a1 = fmaf(__uint_as_float(w.y), __uint_as_float(x.y), a1);
    a0 = fmaf(__uint_as_float(w.z), __uint_as_float(x.z), a0);
    a1 = fmaf(__uint_as_float(w.w), __uint_as_float(x.w), a1);
  }
};

struct BF16 {
  static constexpr int kBytes = 2;
  static constexpr int kPerVec = 8;
  // bf16 -> f32 widening is exact: the bf16 bits are the high half of the f32.
  __device__ __forceinline__ static void unpack2(uint32_t u, float& lo, float& hi) {
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xffff0000u);
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    unpack2(v.x, f[0], f[1]);
    unpack2(v.y, f[2], f[3]);
    unpack2(v.z, f[4], f[5]);
    unpack2(v.w, f[6], f[7]);
  }
  __device__ __forceinline__ static float load1(const void* base, int64_t i) {
    uint16_t b = reinterpret_cast<const uint16_t*>(base)[i];
    return __uint_as_float(uint32_t(b) << 16);
  }
  __device__ __forceinline__ static void store1(void* base, int64_t i, float v) {
    reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  }
  __device__ __forceinline__ static float load1_cg(const void* base, int64_t i) {
    unsigned short b = __ldcg(reinterpret_cast<const unsigned short*>(base) + i);
    return __uint_as_float(uint32_t(b) << 16);
  }
  // lo += lo(w) * lo(x); hi += hi(w) * hi(x) for one word of two bf16 each:
  // the mixed-precision FMA takes the bf16 halves as they are (the product
  // of two bf16 is exact in f32) and rounds once into the f32 sum, which is
  // what widening both and calling fmaf computes.
  __device__ __forceinline__ static void fma2(uint32_t w, uint32_t x, float& lo, float& hi) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\tmov.b32 {wl, wh}, %2;\n\tmov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\tfma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(w), "r"(x));
  }
  // acc[e] += x * w[e] for the 8 elements of w, x a widened bf16 value: the
  // mixed-precision FMA on x's bf16 bits (its f32 image's upper half) and
  // the halves of w, one rounding each -- what fmaf on the widened values gives
  __device__ __forceinline__ static void axpy(const uint4& w, float x, float* acc) {
    const unsigned short xb = static_cast<unsigned short>(__float_as_uint(x) >> 16);
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      asm("{\n\t.reg .b16 wl, wh;\n\tmov.b32 {wl, wh}, %2;\n\t"
          "fma.rn.f32.bf16 %0, wl, %3, %0;\n\tfma.rn.f32.bf16 %1, wh, %3, %1;\n\t}"
          : "+f"(acc[2 * c]), "+f"(acc[2 * c + 1])
          : "r"(wv[c]), "h"(xb));
  }
  // sum over the vector of w[e] g[e] (g float32): the even elements and the
  // odd ones in two lanes of paired FMAs (each in element order), then added
  __device__ __forceinline__ static float dot_vec(const uint4& w, const float* g) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    unsigned long long acc = f2_pack(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      acc = f2_fma(f2_pack(__uint_as_float(wv[c] << 16), __uint_as_float(wv[c] & 0xffff0000u)),
                   f2_pack(g[2 * c], g[2 * c + 1]), acc);
    const float2 r = f2_unpack(acc);
    return r.x + r.y;
  }
  // a0 += the products of the even elements, a1 of the odd ones, in order
  __device__ __forceinline__ static void dot_acc(const uint4& w, const uint4& x, float& a0, float& a1) {
    fma2(w.x, x.x, a0, a1);
    fma2(w.y, x.y, a0, a1);
    fma2(w.z, x.z, a0, a1);
    fma2(w.w, x.w, a0, a1);
  }
};

// ---------------------------------------------------------------- memory access
// Read-only weights (W, V, M, Gram): 16-byte non-coherent loads that do not
// allocate in L1 (each byte is used once per CTA).
__device__ __forceinline__ uint4 ld_weight_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Data written by an earlier kernel of the stream (tokens, projections,
// counts, index lists): read at L2 so no stale L1 line can be hit.
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  return __ldcg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint32_t ld_cg_u8(const uint8_t* p) {
  uint32_t r;
  asm volatile("ld.global.cg.u8 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// Speculative L2 prefetch of a byte range (16-byte aligned, multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- programmatic dependent launch
// launch_dependents lets the next kernel of the stream start its prologue
// (weight prefetch) early; wait blocks until every kernel this one depends on
// has finished and its writes are visible.  Both are no-ops when the kernel
// was launched without the programmatic-serialisation attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- cluster barrier halves
// A relaxed arrive early in the kernel and the matching wait just before the
// first access to a peer's shared memory: the "every CTA of the cluster has
// started" barrier then overlaps the kernel's weight loads.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Reduce R per-lane partial sums (R = 1, 2, 4, 8, 16 or 32) across the warp
// with R - 1 + 5 - log2(R) shuffles instead of 5 R: each butterfly stage halves
// the number of live values while doubling the lanes each one covers.
// On return, lane l holds the full sum of value index
//   idx(l) = bits of l above position 5 - log2(R)  (see row_of_lane).
template <int R>
__device__ __forceinline__ float warp_reduce_multi(float (&v)[R], int lane) {
  static_assert(R == 1 || R == 2 || R == 4 || R == 8 || R == 16 || R == 32, "R power of 2");
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int off = 16 >> st;
    const int n = R >> st;  // live values before this stage (compile-time per stage)
    if (n > 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        // Upper lanes keep the upper half of the live values, the others the
        // lower half; each sends the half it does not keep to its partner.
        const float send = upper ? v[i] : v[i + n / 2];
        const float keep = upper ? v[i + n / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
  return v[0];
}

// Value index whose total lane `lane` holds after warp_reduce_multi<R>:
// the stage with offset 16 >> st sets bit (R >> (st + 1)) of the index.
template <int R>
__device__ __forceinline__ int row_of_lane(int lane) {
  int idx = 0;
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int n = R >> st;
    if (n > 1 && (lane & (16 >> st))) idx += n / 2;
  }
  return idx;
}

// One warp: stable compaction of T flags into fast / slow index lists
// (fast list at idx[0..), slow list at idx[T..)) and their counts.
__device__ __forceinline__ void compact_warp(const uint8_t* flags, int T, int32_t* idx, int32_t* counts,
                                             int lane) {
  int nf = 0, ns = 0;
  for (int base = 0; base < T; base += 32) {
    const int t = base + lane;
    const bool valid = t < T;
    const bool slow = valid && ld_cg_u8(flags + t) != 0;
    const unsigned ms = __ballot_sync(0xffffffffu, slow);
    const unsigned mf = __ballot_sync(0xffffffffu, valid && !slow);
    const unsigned lt = (1u << lane) - 1u;
    if (valid && idx) {
      if (slow)
        idx[T + ns + __popc(ms & lt)] = t;
      else
        idx[nf + __popc(mf & lt)] = t;
    }
    nf += __popc(mf);
    ns += __popc(ms);
  }
  if (lane == 0 && counts) {
    counts[0] = nf;
    counts[1] = ns;
  }
}

// Every kernel of the decode path asks for the largest shared-memory
// carve-out: consecutive kernels then run in one L1 / shared-memory
// configuration, so an SM never has to drain and reconfigure between the
// projection kernel and the decide-and-apply kernel that overlaps it.
template <class K>
inline cudaError_t set_kernel_smem(K kern, size_t dyn_bytes) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       int(cudaSharedmemCarveoutMaxShared));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn_bytes));
}

// ---------------------------------------------------------------- co-resident launches
// Kernels whose CTAs wait on CTAs of other clusters (a grid barrier, polled
// epoch words) are launched with the cooperative attribute: a grid that
// cannot be co-resident (other work holding SMs, or a smaller device share)
// is then refused at launch instead of running into its bounded waits.
// Where the driver refuses the attribute together with a cluster shape, the
// refusal is remembered in *no_coop and the launch is repeated without it
// (the waits stay bounded).  A refusal for size comes back as
// cudaErrorCooperativeLaunchTooLarge, for the caller to take another path.
// GSI_COOPERATIVE=0 in the environment launches these kernels without the
// attribute, sized as before from the occupancy query (for tools that
// relaunch kernels themselves and do not keep the cooperative attribute
// together with the cluster shape; the waits stay bounded).
inline bool cooperative_launch_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("GSI_COOPERATIVE");
    return !(v && v[0] == '0' && v[1] == '\0');
  }();
  return on;
}

template <class K, class A>
inline cudaError_t launch_maybe_coop(cudaLaunchConfig_t cfg, cudaLaunchAttribute* attrs, int n_attrs, bool coop,
                                     int* no_coop, K kern, const A& args) {
  if (coop && !*no_coop && cooperative_launch_enabled()) {
    attrs[n_attrs].id = cudaLaunchAttributeCooperative;
    attrs[n_attrs].val.cooperative = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = unsigned(n_attrs + 1);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e == cudaSuccess || e == cudaErrorCooperativeLaunchTooLarge) return e;
    if (e != cudaErrorInvalidValue && e != cudaErrorNotSupported && e != cudaErrorInvalidConfiguration) return e;
    cudaGetLastError();
    *no_coop = 1;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = unsigned(n_attrs);
  return cudaLaunchKernelEx(&cfg, kern, args);
}

// ---------------------------------------------------------------- workspace layout
// Control words at the head of every workspace (256 bytes).
struct Ctrl {
  uint32_t reserved;
  uint32_t err;        // device error word (0 = ok); set by bounded waits
  int32_t counts[2];   // {n_fast, n_slow} of the last gate
  // fused decode's grid barrier, one ticket counter per element type: the
  // arrivals of all calls so far (zeroed by gsi_workspace_init, never reset)
  unsigned long long ticket[2];
  // the single-token decode's call numbers (the grid projection's epochs),
  // per element type; also numbers the persistent stack kernel's launches
  unsigned long long ticket1[2];
  // the persistent stack kernel's arrivals at its barriers between maps
  unsigned long long arrive[2];
  uint32_t unused0;
  // the small-batch decode's call numbers (its grid projection's epochs), per
  // element type
  unsigned long long ticket_b[2];
  uint32_t pad[42];
};
static_assert(sizeof(Ctrl) == 256, "Ctrl is 256 bytes");

constexpr uint32_t kErrTimeout = 1;
// Which bounded wait gave up (bits above kErrTimeout, or-ed into the error
// word of the single-token and stack decode kernels).
constexpr uint32_t kWaitV = 1u << 4, kWaitGram = 1u << 5, kWaitM = 1u << 6, kWaitPartials = 1u << 7,
                   kWaitGathered = 1u << 8, kWaitShares = 1u << 9, kWaitRing = 1u << 10, kWaitSlices = 1u << 11,
                   kWaitGrid = 1u << 12;
// The kernel found itself running without the cluster shape it was built
// for (or with a grid its exchanges cannot address) and returned before its
// first access to another CTA's shared memory.
constexpr uint32_t kErrLaunchShape = 1u << 13;

// True when this CTA's cluster has `ctas` CTAs: every rank a kernel maps a
// shared-memory address to (mapa, st.async) then exists.
__device__ __forceinline__ bool cluster_shape_ok(unsigned ctas) {
  unsigned n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n == ctas;
}

}  // namespace gsi
