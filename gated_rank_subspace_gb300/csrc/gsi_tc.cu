// Tensor-core path for prefill-sized token counts (sm_103a tcgen05 + TMEM + TMA).
//
// "Gated Subspace Inference for Transformer Acceleration", §2.1-§2.2 at large
// T: the projections G = X V_k, the fast outputs Y_fast = G_fast M^T and the
// slow outputs Y_slow = X_slow W^T are dense contractions, so they run on the
// 5th-generation tensor cores:
//
//   1. transpose V_k (d x k) into V_k^T (k x d) so both operands of the
//      projection are K-major;
//   2. G = X V_k                       (tcgen05, fp32 accumulate in TMEM);
//   3. per token ||x||^2, g^T Gram g, rho, flag, and g rounded to bf16
//      (CUDA cores, float32 -- the gate needs more precision than bf16);
//   4. compaction and gathers: X_slow (slow tokens' rows of X) and G_fast;
//   5. Y[idx_fast] = G_fast M^T and Y[idx_slow] = X_slow W^T
//      (tcgen05; the epilogue scatters rows to their token positions).
//
// The GEMM kernel: one 128 x BN output tile per CTA, 128 threads.  Thread 0
// issues TMA tile loads (128-byte swizzle) into a STAGES-deep shared-memory
// ring guarded by mbarriers; thread 32 issues tcgen05.mma (M = 128, N = BN,
// K = 16 per instruction) into a TMEM accumulator and commits each stage back
// to the producer; after the last k-block all four warps read their 32 TMEM
// lanes with tcgen05.ld and write fp32 rows.  Every wait is bounded (about
// two seconds of clock): on expiry the CTA records an error in the workspace
// word, waits (bounded) for its own in-flight copies, frees its TMEM and
// returns.  The valid row count can come from device memory (the fast / slow
// counts), so the grid is sized for T and surplus tiles exit at once.

#include <cuda.h>

#include "gsi_common.cuh"
#include "gsi_kernels.h"
#include "gsi_plan.h"

namespace gsi {

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz

// Bounded wait on an mbarrier phase; false (and the error word set) on expiry.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
  return true;
}

// The same wait with a suspend-time hint: a waiting thread sleeps until the
// phase completes (or ~0.1 ms pass) instead of spinning on the barrier, so it
// takes no issue slots from the warps that compute.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(100000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// 1-D bulk copy shared -> global in the thread's bulk group (both addresses
// 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_store_1d(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_store_commit_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// 1-D bulk copy global -> shared completing on an mbarrier (both addresses
// 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// tcgen05.ld of 16 columns without the wait: several loads in flight, then
// one tmem_ld_wait() before any of their registers is read.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand tile written by TMA with
// 128-byte swizzle (rows of 64 bf16, 8-row / 1024-byte swizzle atoms).
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* tile) {
  uint64_t d = 0;
  d |= uint64_t((smem_u32(tile) & 0x3FFFFu) >> 4);  // start address
  d |= uint64_t(1) << 16;                           // leading byte offset (unused for SW128 K-major)
  d |= uint64_t(1024 >> 4) << 32;                   // stride byte offset: next 8-row atom
  d |= uint64_t(1) << 46;                           // descriptor version
  d |= uint64_t(2) << 61;                           // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, A = B = bf16, D = f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// ------------------------------------------------------------------ GEMM kernel
struct TcArgs {
  int rows;               // valid rows of A (used when rows_dev is null)
  const int32_t* rows_dev;  // device count of valid rows, or null
  int N, K;
  float* C;
  int64_t ldc;
  const int32_t* row_map;  // output row of A-row m is row_map[m] (null: m)
  uint32_t* err;
  int ksplit;              // K is cut into ksplit slices (grid z); 0 or 1: none
  int64_t c_split;         // elements between the slices' outputs
  int c_bf16;              // C is bf16 (rounded to nearest even), not float32
};

constexpr int kBM = 128, kBK = 64;

// SG: pipeline stages (0: the default -- 4 for BN = 256, else 6; 3 when the
// CTA takes two row tiles).  Short contractions (K <= 256, BN = 128) take 2
// stages, so three CTAs share an SM and their epilogues (staged 64 columns at
// a time) overlap the others' loads and MMAs.
// MT: 128-row tiles of A per CTA; with MT = 2 every B tile feeds two MMAs
// into two TMEM accumulators (B is read from L2 half as often).
template <int BN, int SG = 0, int MT = 1>
struct TcCfg {
  static constexpr int STAGES = SG > 0 ? SG : (MT > 1 ? 3 : (BN >= 256 ? 4 : 6));
  static constexpr uint32_t A_TILE = kBM * kBK * 2;  // one 128-row tile of a stage
  static constexpr uint32_t A_BYTES = MT * A_TILE;
  static constexpr int TMEM_COLS = BN * MT;
  static_assert(TMEM_COLS <= 512, "TMEM holds 512 columns");
  static constexpr uint32_t B_BYTES = BN * kBK * 2;
  static constexpr size_t SMEM = 1024 + size_t(STAGES) * (A_BYTES + B_BYTES) + 256;
  // epilogue column chunk: all BN columns where 128 staged rows of them fit
  // the idle ring, else the widest multiple of 64 that does
  static constexpr int CW = size_t(kBM) * (BN + 4) * 4 <= size_t(STAGES) * (A_BYTES + B_BYTES) ? BN
                          : size_t(kBM) * (BN / 2 + 4) * 4 <= size_t(STAGES) * (A_BYTES + B_BYTES) ? BN / 2
                                                                                                    : 64;
};

template <int BN, int SG, int MT>
__global__ void __launch_bounds__(128, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, TcArgs a) {
  using C = TcCfg<BN, SG, MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::STAGES * C::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* done = empty + C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x, n_tile = blockIdx.y;
  pdl_wait();
  const int rows = a.rows_dev ? __ldcg(a.rows_dev) : a.rows;
  if (m_tile * kBM * MT >= rows) return;  // whole CTA, before any barrier or TMEM

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // this CTA's slice of K (grid z): k-blocks [kb0, kb0 + nk)
  const int nk_all = (a.K + kBK - 1) / kBK;
  const int ns = a.ksplit > 1 ? a.ksplit : 1;
  const int kb0 = int(int64_t(nk_all) * blockIdx.z / ns);
  const int nk = int(int64_t(nk_all) * (blockIdx.z + 1) / ns) - kb0;
  __shared__ int s_issued;  // k-blocks whose TMA loads were issued

  if (threadIdx.x == 0) {
    int kb = 0;
    for (; kb < nk; ++kb) {
      const int s = kb % C::STAGES;
      const uint32_t ph = (kb / C::STAGES) & 1;
      if (kb >= C::STAGES && !mbar_wait(&empty[s], ph ^ 1, a.err)) break;
      mbar_expect_tx(&full[s], C::A_BYTES + C::B_BYTES);
      tma_load_2d(sA + s * C::A_BYTES, &ta, &full[s], (kb0 + kb) * kBK, m_tile * kBM * MT);
      tma_load_2d(sB + s * C::B_BYTES, &tb, &full[s], (kb0 + kb) * kBK, n_tile * BN);
    }
    s_issued = kb;
  } else if (threadIdx.x == 32) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % C::STAGES;
      const uint32_t ph = (kb / C::STAGES) & 1;
      if (!mbar_wait(&full[s], ph, a.err)) break;
      tc_fence_after();
      const uint64_t bd = smem_desc_sw128(sB + s * C::B_BYTES);
#pragma unroll
      for (int u = 0; u < MT; ++u) {  // row tile u accumulates in TMEM columns [u * BN, (u + 1) * BN)
        const uint64_t ad = smem_desc_sw128(sA + s * C::A_BYTES + u * C::A_TILE);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)  // advance 16 bf16 = 32 bytes inside the swizzle row
          umma_bf16(tmem + uint32_t(u * BN), ad + uint64_t(kk * 2), bd + uint64_t(kk * 2), idesc, (kb | kk) != 0);
      }
      umma_commit(&empty[s]);
    }
    umma_commit(done);  // fires once every MMA issued above has completed
  }
  __syncwarp();
  const bool ok = mbar_wait(done, 0, a.err);
  tc_fence_after();
  // tcgen05.ld is warp-collective: decide per warp, never per thread.
  const bool go = __all_sync(0xffffffffu, ok && *reinterpret_cast<volatile uint32_t*>(a.err) == 0);
  if (go) {
    // The pipeline buffers are idle (every MMA, and so every operand load,
    // has completed): each warp stages its 32 rows x CW columns there at a
    // time (CW = BN where the buffers hold all of it), then writes whole row
    // segments -- consecutive lanes on consecutive columns, 16-byte stores --
    // instead of one 16-byte piece of 32 rows per store.
    constexpr int CW = C::CW;
    constexpr int LD = CW + 4;  // staged row stride in floats (conflict-free 16-byte accesses)
    static_assert(size_t(kBM) * LD * 4 <= size_t(C::STAGES) * (C::A_BYTES + C::B_BYTES), "staging fits");
    static_assert(BN % CW == 0 && CW % 64 == 0, "column chunks");
    float* st = reinterpret_cast<float*>(sA) + size_t(warp) * 32 * LD;
    const bool vec = (a.ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.C) & 15) == 0);
    // float32 rows with 16-byte aligned starts and lengths leave by bulk
    // copies: lane i sends the staged row i, and the warp waits only until
    // the copies have read the staging buffer, so the writes drain to memory
    // while the CTA finishes and the next CTA of the SM loads its operands
    const bool bulk = !a.c_bf16 && vec && (a.N % 4 == 0) && (a.c_split % 4 == 0);
#pragma unroll 1
    for (int u = 0; u < MT; ++u) {
    const int r_base = (m_tile * MT + u) * kBM + warp * 32;
    const int my_r = r_base + lane;
    const int64_t my_orow = my_r < rows ? (a.row_map ? int64_t(__ldcg(&a.row_map[my_r])) : int64_t(my_r)) : 0;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += CW) {
#pragma unroll 1
    for (int c = 0; c < CW; c += 64) {  // four 16-column loads in flight, one wait
      uint32_t r[4][16];
#pragma unroll
      for (int h = 0; h < 4; ++h)
        tmem_ld16_nowait(tmem + (uint32_t(warp * 32) << 16) + uint32_t(u * BN + c0 + c + 16 * h), r[h]);
      tmem_ld_wait();
#pragma unroll
      for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4*>(st + lane * LD + c + 16 * h + 4 * q) =
              make_float4(__uint_as_float(r[h][4 * q]), __uint_as_float(r[h][4 * q + 1]),
                          __uint_as_float(r[h][4 * q + 2]), __uint_as_float(r[h][4 * q + 3]));
    }
    __syncwarp();
    const int col0 = n_tile * BN + c0;  // first output column of this chunk
    if (bulk) {
      const int ncols = a.N - col0 < CW ? a.N - col0 : CW;
      if (my_r < rows && ncols > 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // this lane's staged row -> async proxy
        bulk_store_1d(a.C + int64_t(blockIdx.z) * a.c_split + my_orow * a.ldc + int64_t(col0), st + lane * LD,
                      uint32_t(ncols) * 4);
      }
      bulk_store_commit_wait_read();
      __syncwarp();
      continue;
    }
    for (int i = 0; i < 32 && r_base + i < rows; ++i) {
      const int64_t orow = __shfl_sync(0xffffffffu, my_orow, i);
      const int64_t cofs = int64_t(blockIdx.z) * a.c_split + orow * a.ldc + int64_t(col0);
      const float* srow = st + i * LD;
      if (a.c_bf16) {
        // four columns a lane: 8-byte stores of bf16 pairs (ldc and the
        // column offsets are multiples of 4 elements)
        __nv_bfloat16* crow = reinterpret_cast<__nv_bfloat16*>(a.C) + cofs;
        for (int q = lane; q < CW / 4; q += 32) {
          const int col = col0 + 4 * q;
          const float4 v = *reinterpret_cast<const float4*>(srow + 4 * q);
          if (col + 4 <= a.N) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
            uint2 u;
            u.x = *reinterpret_cast<const uint32_t*>(&lo);
            u.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(crow + 4 * q) = u;
          } else {
            const float f[4] = {v.x, v.y, v.z, v.w};
            for (int e2 = 0; e2 < 4; ++e2)
              if (col + e2 < a.N) crow[4 * q + e2] = __float2bfloat16_rn(f[e2]);
          }
        }
        continue;
      }
      float* crow = a.C + cofs;
      for (int q = lane; q < CW / 4; q += 32) {
        const int col = col0 + 4 * q;
        if (vec && col + 4 <= a.N) {
          *reinterpret_cast<float4*>(crow + 4 * q) = *reinterpret_cast<const float4*>(srow + 4 * q);
        } else {
          for (int e2 = 0; e2 < 4; ++e2)
            if (col + e2 < a.N) crow[4 * q + e2] = srow[4 * q + e2];
        }
      }
    }
    __syncwarp();  // the staging rows are read before the next chunk overwrites them
    }
    }
  }
  // Bounded drain of this CTA's own copies before its shared memory goes away
  // (only reached with copies in flight after a timeout).
  if (threadIdx.x == 0 && !ok) {
    for (int kb = 0; kb < s_issued; ++kb)
      mbar_wait(&full[kb % C::STAGES], (kb / C::STAGES) & 1, a.err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ------------------------------------------------------------------ persistent contraction (Y_fast)
// C[row_map(m)][n] = sum_k A[m][k] B[n][k] over 128 x 128 tiles, float32 C,
// one CTA an SM looping over the tiles t = blockIdx.x, + gridDim.x, ...
// (tile t: row tile t % n_m, column tile t / n_m).  Warp 0 (one thread)
// streams the operand k-blocks of its tiles through a kPS-stage ring, running
// ahead across tile boundaries; warp 1 allocates two TMEM accumulators and
// one thread of it issues the MMAs of tile j into accumulator j % 2; warps
// 2-5 drain accumulator j % 2 (warp w reads TMEM lanes 32 (w % 4) ..) into
// staging rows, hand it back, and send each row by one bulk copy while the
// MMAs of tile j + 1 run.  Each output is summed in the same k-block and MMA
// order as in tc_gemm_kernel<128>.
constexpr int kPS = 4;
constexpr int kPBN = 128;
constexpr uint32_t kPTile = uint32_t(kBM) * kBK * 2;  // one 128-row tile of a stage (A or B)
constexpr int kPLD = kPBN + 4;                          // staged row stride (floats)
constexpr size_t kPSmem = 1024 + size_t(kPS) * 2 * kPTile + size_t(kBM) * kPLD * 4 + 256;
constexpr int kPThreads = 192;

__global__ void __launch_bounds__(kPThreads, 1)
    tc_gemm_persist_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* staging = reinterpret_cast<float*>(base + size_t(kPS) * 2 * kPTile);
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + size_t(kBM) * kPLD);
  uint64_t* empty = full + kPS;
  uint64_t* tfull = empty + kPS;  // accumulator j % 2 holds tile j (tcgen05.commit)
  uint64_t* tempty = tfull + 2;   // accumulator drained (the four epilogue warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  const int rows = a.rows_dev ? __ldcg(a.rows_dev) : a.rows;
  const int n_m = (rows + kBM - 1) / kBM, n_n = (a.N + kPBN - 1) / kPBN;
  const int n_tiles = n_m * n_n;
  if (int(blockIdx.x) >= n_tiles) return;  // whole CTA, before any barrier or TMEM
  const int nk = (a.K + kBK - 1) / kBK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(&tfull[u], 1);
      mbar_init(&tempty[u], 4);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * kPBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0) {
    if (lane == 0) {
      // ---- operand loads
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        const int m_tile = t % n_m, n_tile = t / n_m;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = int(it % kPS);
          if (it >= uint32_t(kPS) && !mbar_wait(&empty[s], ((it / kPS) & 1u) ^ 1u, a.err)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[s], 2 * kPTile);
          tma_load_2d(base + size_t(s) * 2 * kPTile, &ta, &full[s], kb * kBK, m_tile * kBM);
          tma_load_2d(base + size_t(s) * 2 * kPTile + kPTile, &tb, &full[s], kb * kBK, n_tile * kPBN);
        }
      }
      // bounded drain: the last issue of every stage has landed before the
      // CTA's shared memory can go away (already so on the normal path)
      for (uint32_t i = it > uint32_t(kPS) ? it - kPS : 0u; i < it; ++i)
        mbar_wait(&full[i % kPS], (i / kPS) & 1u, a.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMAs
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kPBN);
      uint32_t it = 0;
      int j = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++j) {
        const int acc = j & 1;
        if (j >= 2 && !mbar_wait(&tempty[acc], uint32_t((j >> 1) - 1) & 1u, a.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + uint32_t(acc * kPBN);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = int(it % kPS);
          if (!mbar_wait(&full[s], (it / kPS) & 1u, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = smem_desc_sw128(base + size_t(s) * 2 * kPTile);
          const uint64_t bd = smem_desc_sw128(base + size_t(s) * 2 * kPTile + kPTile);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(d_tmem, ad + uint64_t(kk * 2), bd + uint64_t(kk * 2), idesc, (kb | kk) != 0);
          umma_commit(&empty[s]);
        }
        if (ok) umma_commit(&tfull[acc]);
      }
    }
  } else {
    // ---- epilogue: TMEM lane quarter q, staged rows, one bulk copy a row
    const int q = warp & 3;
    float* st = staging + size_t(q) * 32 * kPLD;
    int j = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++j) {
      const int acc = j & 1;
      const int m_tile = t % n_m, n_tile = t / n_m;
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], uint32_t(j >> 1) & 1u, a.err))) break;
      tc_fence_after();
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // the previous tile's rows have left
      __syncwarp();
#pragma unroll 1
      for (int c = 0; c < kPBN; c += 64) {  // four 16-column loads in flight, one wait
        uint32_t r[4][16];
#pragma unroll
        for (int h = 0; h < 4; ++h)
          tmem_ld16_nowait(tmem + (uint32_t(q * 32) << 16) + uint32_t(acc * kPBN + c + 16 * h), r[h]);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
          for (int v = 0; v < 4; ++v)
            *reinterpret_cast<float4*>(st + lane * kPLD + c + 16 * h + 4 * v) =
                make_float4(__uint_as_float(r[h][4 * v]), __uint_as_float(r[h][4 * v + 1]),
                            __uint_as_float(r[h][4 * v + 2]), __uint_as_float(r[h][4 * v + 3]));
      }
      // the accumulator is read: the MMAs of tile j + 2 may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      const int my_r = m_tile * kBM + q * 32 + lane;
      const int col0 = n_tile * kPBN;
      const int ncols = a.N - col0 < kPBN ? a.N - col0 : kPBN;
      if (my_r < rows) {
        const int64_t orow = a.row_map ? int64_t(__ldcg(&a.row_map[my_r])) : int64_t(my_r);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // this lane's staged row -> async proxy
        bulk_store_1d(a.C + orow * a.ldc + int64_t(col0), st + lane * kPLD, uint32_t(ncols) * 4);
      }
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 2 * kPBN);
}

// ------------------------------------------------------------------ few-token contraction
// Y[tok(j)][r] = sum_kk A[r][kk] B[j][kk] for the rows r of a weight matrix A
// (W or M: n_rows x K, bf16, K-major) and the first n_tok rows of a token
// matrix B (X_slow or G_fast: K-major), NT token rows per CTA (grid z).  The
// weight rows are the MMA's M side (128-row tiles) and the tokens its N side
// (NT columns of TMEM), so a call with few tokens spends no tensor-core work on padding
// token rows, and the weight stream is spread over the n_rows / 128 tiles
// times `splits` slices of K.  The slices of one tile are one thread-block
// cluster (grid x): after its MMAs each CTA stages its partial 128 x NT tile
// in shared memory, and after a cluster barrier CTA q adds rows
// [q R, (q + 1) R) over the cluster's CTAs in rank order (distributed shared
// memory) and writes them, so every output has one fixed summation order.
// Threads: 0 issues the TMA loads, 32 the MMAs, all four warps the epilogue
// (warp w reads TMEM lanes 32 w .. 32 w + 31 = weight rows).
struct SkinnyArgs {
  int n_rows, K;
  int n_tok;                 // token rows (used when n_tok_dev is null)
  const int32_t* n_tok_dev;  // device count of token rows, or null
  float* Y;
  int64_t ldy;
  const int32_t* tok_map;    // output row of token row j is tok_map[j] (null: j)
  uint32_t* err;
};

template <int NT>
struct SkinnyCfg {
  static constexpr uint32_t A_BYTES = kBM * kBK * 2;
  static constexpr uint32_t B_BYTES = NT * kBK * 2;
  static constexpr int STAGES = (100 * 1024) / (A_BYTES + B_BYTES) > 3 ? (100 * 1024) / (A_BYTES + B_BYTES) : 3;
  static constexpr int TMEM_COLS = NT < 32 ? 32 : NT;
  static constexpr int LDS = NT + 4;  // staged partial tile row stride (floats)
  static_assert(size_t(kBM) * LDS * 4 <= size_t(STAGES) * (A_BYTES + B_BYTES), "staging fits");
  static constexpr size_t SMEM = 1024 + size_t(STAGES) * (A_BYTES + B_BYTES) + 256;
};

template <int NT>
__global__ void __launch_bounds__(128, 1)
    tc_skinny_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, SkinnyArgs a) {
  using C = SkinnyCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::STAGES * C::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* done = empty + C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  __shared__ int s_issued;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int splits = int(gridDim.x), sl = int(blockIdx.x);  // K slice = rank in the cluster
  const int row0 = int(blockIdx.y) * kBM;
  const int tok0 = int(blockIdx.z) * NT;  // this CTA's token rows [tok0, tok0 + NT)
  pdl_wait();
  int n_tok = (a.n_tok_dev ? __ldcg(a.n_tok_dev) : a.n_tok) - tok0;
  if (n_tok <= 0) return;  // the whole cluster leaves together (same count everywhere)
  if (n_tok > NT) n_tok = NT;
  const int32_t* tok_map = a.tok_map ? a.tok_map + tok0 : nullptr;
  if (splits > 1 && !cluster_shape_ok(unsigned(splits))) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrTimeout | kErrLaunchShape);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nk_all = (a.K + kBK - 1) / kBK;
  const int kb0 = int(int64_t(nk_all) * sl / splits);
  const int nk = int(int64_t(nk_all) * (sl + 1) / splits) - kb0;

  if (threadIdx.x == 0) {
    int kb = 0;
    for (; kb < nk; ++kb) {
      const int s = kb % C::STAGES;
      const uint32_t ph = (kb / C::STAGES) & 1;
      if (kb >= C::STAGES && !mbar_wait(&empty[s], ph ^ 1, a.err)) break;
      mbar_expect_tx(&full[s], C::A_BYTES + C::B_BYTES);
      tma_load_2d(sA + s * C::A_BYTES, &ta, &full[s], (kb0 + kb) * kBK, row0);
      tma_load_2d(sB + s * C::B_BYTES, &tb, &full[s], (kb0 + kb) * kBK, tok0);
    }
    s_issued = kb;
  } else if (threadIdx.x == 32) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, NT);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % C::STAGES;
      const uint32_t ph = (kb / C::STAGES) & 1;
      if (!mbar_wait(&full[s], ph, a.err)) break;
      tc_fence_after();
      const uint64_t ad = smem_desc_sw128(sA + s * C::A_BYTES);
      const uint64_t bd = smem_desc_sw128(sB + s * C::B_BYTES);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)  // advance 16 bf16 = 32 bytes inside the swizzle row
        umma_bf16(tmem, ad + uint64_t(kk * 2), bd + uint64_t(kk * 2), idesc, (kb | kk) != 0);
      umma_commit(&empty[s]);
    }
    umma_commit(done);  // fires once every MMA issued above has completed
  }
  __syncwarp();
  const bool ok = mbar_wait(done, 0, a.err);
  tc_fence_after();
  // tcgen05.ld is warp-collective: decide per warp, never per thread
  const bool go = __all_sync(0xffffffffu, ok && nk > 0 && *reinterpret_cast<volatile uint32_t*>(a.err) == 0);
  const int row = warp * 32 + lane;  // this lane's weight row in the tile
  if (splits == 1) {
    if (go) {
#pragma unroll 1
      for (int c = 0; c < NT; c += 16) {
        if (c >= n_tok) break;  // warp-uniform
        float v[16];
        tmem_ld16(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c), v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = c + i;
          if (j < n_tok && row0 + row < a.n_rows) {
            const int64_t orow = tok_map ? int64_t(__ldcg(&tok_map[j])) : int64_t(tok0 + j);
            a.Y[orow * a.ldy + row0 + row] = v[i];
          }
        }
      }
    }
  } else {
    // stage this slice's partial tile in the (idle) pipeline buffers: every
    // MMA, and so every operand copy into them, has completed
    float* st = reinterpret_cast<float*>(base);
    if (go) {
#pragma unroll 1
      for (int c = 0; c < NT; c += 16) {
        float v[16];
        tmem_ld16(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c), v);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4*>(st + row * C::LDS + c + 4 * q) =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
    // every CTA of the cluster passes both barriers, with or without an error
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // the partial tiles are staged
    const bool all_ok = __syncthreads_and(go) != 0;
    const bool any_err = *reinterpret_cast<volatile uint32_t*>(a.err) != 0;
    if (all_ok && !any_err) {
      const int R = (kBM + splits - 1) / splits;
      const int rb = sl * R, rn = kBM - rb < R ? (kBM - rb > 0 ? kBM - rb : 0) : R;
      for (int e = threadIdx.x; e < rn * n_tok; e += 128) {
        const int j = e / rn, r = rb + (e - (e / rn) * rn);
        float sum = 0.f;
        for (int q = 0; q < splits; ++q) sum += cluster.map_shared_rank(st, q)[r * C::LDS + j];
        if (row0 + r < a.n_rows) {
          const int64_t orow = tok_map ? int64_t(__ldcg(&tok_map[j])) : int64_t(tok0 + j);
          a.Y[orow * a.ldy + row0 + r] = sum;
        }
      }
    }
    cluster.sync();  // the peers' reads of this CTA's tile are done
  }
  // bounded drain of this CTA's own copies before its shared memory goes away
  // (only reached with copies in flight after a timeout)
  if (threadIdx.x == 0 && !ok) {
    for (int kb = 0; kb < s_issued; ++kb) mbar_wait(&full[kb % C::STAGES], (kb / C::STAGES) & 1, a.err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ------------------------------------------------------------------ helpers on CUDA cores
// V_k (d x k) -> V_k^T (k x d), bf16, 32 x 32 tiles through shared memory.
__global__ void transpose_bf16_kernel(const uint16_t* __restrict__ V, uint16_t* __restrict__ Vt, int d, int k) {
  __shared__ uint16_t tile[32][33];
  const int i0 = blockIdx.y * 32, j0 = blockIdx.x * 32;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int i = i0 + r, j = j0 + threadIdx.x;
    tile[r][threadIdx.x] = (i < d && j < k) ? V[int64_t(i) * k + j] : uint16_t(0);
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int j = j0 + r, i = i0 + threadIdx.x;
    if (j < k && i < d) Vt[int64_t(j) * d + i] = tile[threadIdx.x][r];
  }
}

// The finalize: per token ||x||^2, ||g||^2, g^T Gram g, rho, flag and g
// rounded to bf16, in two kernels.
//
// tc_norms_kernel, one CTA of 64 threads a token: adds the split-K slices of
// g in slice order (four columns a thread, every slice's 16-byte load in
// flight together with the first batch of x's vectors), writes the bf16 g and
// the float32 g into gT, laid out by chunks of kFinTok tokens as
// [chunk][column j][token slot] so that a chunk is one contiguous block with
// the chunk's g_j side by side, and stores (||g||^2, ||x||^2).
//
// tc_gramq_kernel, CTA (c, b) of a (1, nb, 1) cluster: the chunk's g lands by
// one bulk copy; Gram rows [k b / nb, k (b + 1) / nb) stream through a ring
// of kFinStages shared-memory stages, one bulk copy a row into a fixed row
// stride.  Register-tiled Gram form: thread (to, cq) keeps h[t][v] = sum over
// the block's rows i of g_t[i] Gram[i][c + v] for the eight tokens t of octet
// to and the four columns c + v of quad cq in each 256-column pass (three
// 16-byte shared loads per 32 FMAs), then adds g_t[c + v] h[t][v].  The
// blocks' partial sums meet in the cluster's rank 0, which adds them in block
// order and takes rho and the flag.  Every sum has one fixed order.
__device__ __forceinline__ void fin_token(float qq, float nn, float x2, float eps, float* rho_out, uint8_t* flags,
                                          int t) {
  float rr = x2 - 2.f * nn + qq;
  rr = rr < 0.f ? 0.f : rr;
  const float rho = x2 == 0.f ? 0.f : sqrtf(rr / x2);
  if (rho_out) rho_out[t] = rho;
  flags[t] = (rho < eps) ? uint8_t(0) : uint8_t(1);
}

template <int GS>
__global__ void __launch_bounds__(kNormThreads) tc_norms_kernel(const uint16_t* __restrict__ X,
                                                                const float* __restrict__ G, int64_t d, int k,
                                                                int T, int gsplit, float* __restrict__ gT,
                                                                uint16_t* __restrict__ Gbf,
                                                                float2* __restrict__ norms) {
  __shared__ float red[2][2];
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  const uint4* xr = reinterpret_cast<const uint4*>(X + int64_t(t) * d);
  const int64_t nv = d / 8;
  // the first batch of x's 16-byte vectors, in flight while g is summed
  uint4 xq[8];
#pragma unroll
  for (int u = 0; u < 8; ++u)
    xq[u] = tid + kNormThreads * u < nv ? ld_cg_v4(xr + tid + kNormThreads * u) : make_uint4(0u, 0u, 0u, 0u);
  const int kq = k / 4;
  const int64_t ss4 = int64_t(T) * kq;  // slice stride in 16-byte units
  const float4* g0 = reinterpret_cast<const float4*>(G) + int64_t(t) * kq;
  float* gc = gT + int64_t(t / kFinTok) * k * kFinTok + (t % kFinTok);
  float nn = 0.f;
  for (int j4 = tid; j4 < kq; j4 += kNormThreads) {
    float4 v[GS];
#pragma unroll
    for (int sl = 0; sl < GS; ++sl) v[sl] = sl < gsplit ? __ldcg(g0 + sl * ss4 + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int sl = 0; sl < GS; ++sl) {
      g.x += v[sl].x;
      g.y += v[sl].y;
      g.z += v[sl].z;
      g.w += v[sl].w;
    }
    const int j = 4 * j4;
    gc[(j + 0) * kFinTok] = g.x;
    gc[(j + 1) * kFinTok] = g.y;
    gc[(j + 2) * kFinTok] = g.z;
    gc[(j + 3) * kFinTok] = g.w;
    __nv_bfloat162 lo = __floats2bfloat162_rn(g.x, g.y), hi = __floats2bfloat162_rn(g.z, g.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(Gbf + int64_t(t) * k + j) = pk;
    nn = fmaf(g.x, g.x, nn);
    nn = fmaf(g.y, g.y, nn);
    nn = fmaf(g.z, g.z, nn);
    nn = fmaf(g.w, g.w, nn);
  }
  // ||x||^2: squares in vector order a thread
  float xx = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    float f[8];
    BF16::unpack(xq[u], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) xx = fmaf(f[e], f[e], xx);
  }
  for (int64_t vb = tid + kNormThreads * 8; vb < nv; vb += kNormThreads * 8) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      xq[u] = vb + kNormThreads * u < nv ? ld_cg_v4(xr + vb + kNormThreads * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float f[8];
      BF16::unpack(xq[u], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) xx = fmaf(f[e], f[e], xx);
    }
  }
  nn = warp_sum(nn);
  xx = warp_sum(xx);
  if (lane == 0) {
    red[warp][0] = nn;
    red[warp][1] = xx;
  }
  __syncthreads();
  if (tid == 0) norms[t] = make_float2(red[0][0] + red[1][0], red[0][1] + red[1][1]);
}

// h[t][v] += g_t m_v for the eight tokens of an octet (ga: tokens 0-3, gb: 4-7).
__device__ __forceinline__ void octet_fma(float (&h)[8][4], const float4 ga, const float4 gb, const float4 m) {
  const float gt[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    h[t][0] = fmaf(gt[t], m.x, h[t][0]);
    h[t][1] = fmaf(gt[t], m.y, h[t][1]);
    h[t][2] = fmaf(gt[t], m.z, h[t][2]);
    h[t][3] = fmaf(gt[t], m.w, h[t][3]);
  }
}

// nr Gram rows of one ring stage (row stride KS) into the first NL passes'
// accumulators, in row order.
template <int NP, int NL, int R, int KS>
__device__ __forceinline__ void gram_rows(float (&h)[NP][8][4], const float* sg, const float* gr, int nr) {
  if (nr == R) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float4 ga = *reinterpret_cast<const float4*>(gr + r * kFinTok);
      const float4 gb = *reinterpret_cast<const float4*>(gr + r * kFinTok + 4);
#pragma unroll
      for (int p = 0; p < NL; ++p)
        octet_fma(h[p], ga, gb, *reinterpret_cast<const float4*>(sg + r * KS + p * kFinCols));
    }
  } else {
    for (int r = 0; r < nr; ++r) {
      const float4 ga = *reinterpret_cast<const float4*>(gr + r * kFinTok);
      const float4 gb = *reinterpret_cast<const float4*>(gr + r * kFinTok + 4);
#pragma unroll
      for (int p = 0; p < NL; ++p)
        octet_fma(h[p], ga, gb, *reinterpret_cast<const float4*>(sg + r * KS + p * kFinCols));
    }
  }
}

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_cluster_f32(const float* local, uint32_t rank, float v) {
  uint32_t raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(raddr), "f"(v) : "memory");
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// NP: 256-column passes over the Gram (k <= 256 NP).  Warps 0-3 compute;
// warp 4 fills the ring: a stage is refilled once the four compute warps
// have arrived on its "empty" barrier.
template <int NP>
__global__ void __launch_bounds__(kFinThreads + 32) tc_gramq_kernel(const float* __restrict__ gT,
                                                                    const float* __restrict__ gram,
                                                                    const float2* __restrict__ norms, int k, int T,
                                                                    float eps, float* __restrict__ rho_out,
                                                                    uint8_t* __restrict__ flags, int nb,
                                                                    uint32_t* err) {
  constexpr int KS = NP * kFinCols;                    // ring row stride (floats)
  constexpr int R = int(kFinStageBytes / (KS * 4));    // Gram rows a stage
  extern __shared__ float4 fsm4[];
  __shared__ uint64_t full[kFinStages], empty[kFinStages], gbar;
  __shared__ float qred[kFinMaxBlocks][kFinTok];       // rank 0: the blocks' q partials
  float* ring = reinterpret_cast<float*>(fsm4);        // [kFinStages][R][KS]
  float* gs = ring + kFinStages * R * KS;              // [k][kFinTok]
  float* red = gs + kFinTok * k;                       // [4 warps][kFinTok]: q partials
  const int cb = blockIdx.x, blk = blockIdx.y;         // blk: rank in the (1, nb, 1) cluster
  const int t0 = cb * kFinTok;
  const int tn = T - t0 < kFinTok ? T - t0 : kFinTok;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = int(int64_t(k) * blk / nb), i1 = int(int64_t(k) * (blk + 1) / nb);
  const int nchunk = gram ? (i1 - i0 + R - 1) / R : 0;
  if (nb > 1) cluster_arrive_relaxed();
  if (tid == kFinThreads) {
    for (int s = 0; s < kFinStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    mbar_init(&gbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  float qq = 0.f;
  if (warp == 4) {
    // ---- producer: the chunk's g, then the block's Gram rows, lane r a row
    if (lane == 0) {
      mbar_expect_tx(&gbar, uint32_t(kFinTok) * k * 4);
      bulk_load_1d(gs, gT + int64_t(cb) * kFinTok * k, uint32_t(kFinTok) * k * 4, &gbar);
    }
    for (int ch = 0; ch < nchunk; ++ch) {
      const int st = ch % kFinStages;
      const int r0 = i0 + ch * R, nr = i1 - r0 < R ? i1 - r0 : R;
      if (ch >= kFinStages &&
          !__all_sync(0xffffffffu, mbar_wait_sleep(&empty[st], uint32_t(ch / kFinStages - 1) & 1u, err)))
        break;  // a compute warp never released the stage (error word set)
      if (lane == 0) mbar_expect_tx(&full[st], uint32_t(nr) * k * 4);
      __syncwarp();
      if (lane < nr)
        bulk_load_1d(ring + (size_t(st) * R + lane) * KS, gram + int64_t(r0 + lane) * k, uint32_t(k) * 4,
                     &full[st]);
    }
  } else {
    // ---- compute warps
    bool failed = !mbar_wait_sleep(&gbar, 0, err);
    // token slots past T hold whatever the workspace held: zero them
    if (tn < kFinTok) {
      for (int e = tid; e < kFinTok * k; e += kFinThreads)
        if (e % kFinTok >= tn) gs[e] = 0.f;
      consumer_sync();
    }
    // this block's share of g^T Gram g, the Gram rows in row order
    const int to = tid >> 6, cq = tid & 63;
    const bool live0 = 4 * cq < k;                       // k % 8 == 0: a quad is whole or absent
    const bool live1 = NP == 2 && kFinCols + 4 * cq < k;
    float h[NP][8][4];
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
      for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int v = 0; v < 4; ++v) h[p][t][v] = 0.f;
    for (int ch = 0; ch < nchunk; ++ch) {
      const int st = ch % kFinStages;
      const int r0 = i0 + ch * R, nr = i1 - r0 < R ? i1 - r0 : R;
      if (!failed && !mbar_wait_sleep(&full[st], uint32_t(ch / kFinStages) & 1u, err)) failed = true;
      const float* sg = ring + size_t(st) * R * KS + 4 * cq;
      const float* gr = gs + r0 * kFinTok + 8 * to;
      if (live1)
        gram_rows<NP, (NP > 1 ? 2 : 1), R, KS>(h, sg, gr, nr);
      else if (live0)
        gram_rows<NP, 1, R, KS>(h, sg, gr, nr);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage
    }
    // q_t over the thread's columns: sum of g_t[c + v] h[t][v]
    float q[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) q[t] = 0.f;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      if (!(p == 0 ? live0 : live1)) continue;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float* gc = gs + (p * kFinCols + 4 * cq + v) * kFinTok + 8 * to;
        const float4 ga = *reinterpret_cast<const float4*>(gc), gb = *reinterpret_cast<const float4*>(gc + 4);
        const float gt[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) q[t] = fmaf(gt[t], h[p][t][v], q[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const float a = warp_sum(q[t]);
      if (lane == 0) red[warp * kFinTok + 8 * to + t] = a;
    }
    consumer_sync();
    if (tid < kFinTok) {
      const int w0 = (tid >> 3) * 2;  // the two warps of this token's octet
      qq = red[w0 * kFinTok + tid] + red[(w0 + 1) * kFinTok + tid];
    }
  }
  if (nb > 1) {
    cluster_wait();  // every CTA of the cluster runs: rank 0's shared memory is live
    if (tid < kFinTok) st_cluster_f32(&qred[blk][tid], 0u, qq);
    cluster_arrive_release();
    cluster_wait();
    if (blk != 0) return;
    if (tid < kFinTok) {
      qq = 0.f;
      for (int b = 0; b < nb; ++b) qq += qred[b][tid];
    }
  }
  if (tid < tn) {
    const float2 nx = __ldcg(&norms[t0 + tid]);
    // (without a Gram matrix the basis is taken as orthonormal: g^T g)
    fin_token(gram ? qq : nx.x, nx.x, nx.y, eps, rho_out, flags, t0 + tid);
  }
}

// Two row gathers in one launch (the prefill path's X_slow and G_fast): CTAs
// [0, nb0) copy dst0[j] = src0[idx0[j]] for j < count0, the others
// dst1[j] = src1[idx1[j]] for j < count1 (16-byte vectors).
struct GatherJob {
  const uint4* src;
  uint4* dst;
  const int32_t* idx;
  const int32_t* count;
  int64_t row_vecs;
};
__global__ void gather_rows2_kernel(GatherJob j0, GatherJob j1, int nb0) {
  pdl_wait();
  const bool second = int(blockIdx.x) >= nb0;
  const uint4* src = second ? j1.src : j0.src;
  uint4* dst = second ? j1.dst : j0.dst;
  const int32_t* idx = second ? j1.idx : j0.idx;
  const int64_t rv = second ? j1.row_vecs : j0.row_vecs;
  const int b = second ? int(blockIdx.x) - nb0 : int(blockIdx.x);
  const int nbk = second ? int(gridDim.x) - nb0 : nb0;
  const int n = __ldcg(second ? j1.count : j0.count);
  const int64_t total = int64_t(n) * rv;
  for (int64_t e = int64_t(b) * blockDim.x + threadIdx.x; e < total; e += int64_t(nbk) * blockDim.x) {
    const int64_t j = e / rv, v = e - j * rv;
    const int32_t t = __ldcg(&idx[j]);
    dst[e] = ld_cg_v4(src + int64_t(t) * rv + v);
  }
}

// Gather rows: dst[j] = src[idx[j]] for j < count (16-byte vectors).
__global__ void gather_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, const int32_t* idx,
                                   const int32_t* count, int64_t row_vecs, int T) {
  pdl_wait();
  const int n = __ldcg(count);
  const int64_t total = int64_t(n) * row_vecs;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total; e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t j = e / row_vecs, v = e - j * row_vecs;
    const int32_t t = __ldcg(&idx[j]);
    dst[e] = ld_cg_v4(src + int64_t(t) * row_vecs + v);
  }
  (void)T;
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 tensor map over a row-major (rows x cols) matrix, box of
// box_rows x 64 columns, 128-byte swizzle, zero fill outside.
static cudaError_t make_map_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  cuuint32_t box[2] = {cuuint32_t(kBK), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int BN, int SG = 0, int MT = 1>
static cudaError_t launch_tc_gemm_t(const void* A, int64_t a_rows, const void* B, int64_t b_rows, int K,
                                    const TcArgs& args, cudaStream_t s) {
  CUtensorMap ta, tb;
  cudaError_t e = make_map_2d(&ta, A, a_rows, K, kBM * MT);
  if (e != cudaSuccess) return e;
  if ((e = make_map_2d(&tb, B, b_rows, K, BN)) != cudaSuccess) return e;
  auto kern = tc_gemm_kernel<BN, SG, MT>;
  static bool attr = false;
  if (!attr) {
    if ((e = set_kernel_smem(kern, TcCfg<BN, SG, MT>::SMEM)) != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(cdiv(a_rows, kBM * MT)), unsigned(cdiv(b_rows, BN)), unsigned(args.ksplit > 1 ? args.ksplit : 1));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = TcCfg<BN, SG, MT>::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, args);
}

// C[row_map(m)][n] = sum_k A[m][k] B[n][k]; A: a_rows x K, B: b_rows x K, bf16.
// mt = 2 (bn = 256 only): each CTA takes 256 rows of A as two 128-row tiles.
cudaError_t launch_tc_gemm(const void* A, int64_t a_rows, const void* B, int64_t b_rows, int K, int bn,
                           const TcArgs& args, cudaStream_t s, int mt = 1) {
  if (mt == 2 && bn == 256) return launch_tc_gemm_t<256, 0, 2>(A, a_rows, B, b_rows, K, args, s);
  switch (bn) {
    case 64: return launch_tc_gemm_t<64>(A, a_rows, B, b_rows, K, args, s);
    case 128:
      return K <= 256 ? launch_tc_gemm_t<128, 2>(A, a_rows, B, b_rows, K, args, s)
                      : launch_tc_gemm_t<128, 3>(A, a_rows, B, b_rows, K, args, s);
    default: return launch_tc_gemm_t<256>(A, a_rows, B, b_rows, K, args, s);
  }
}

// The persistent 128 x 128 contraction (float32 C with 16-byte aligned rows):
// one CTA an SM, at most as many as the tiles of a_rows rows.
static cudaError_t launch_tc_gemm_persist(const void* A, int64_t a_rows, const void* B, int64_t b_rows, int K,
                                          const TcArgs& args, cudaStream_t s) {
  CUtensorMap ta, tb;
  cudaError_t e = make_map_2d(&ta, A, a_rows, K, kBM);
  if (e != cudaSuccess) return e;
  if ((e = make_map_2d(&tb, B, b_rows, K, kPBN)) != cudaSuccess) return e;
  static bool attr = false;
  if (!attr) {
    if ((e = set_kernel_smem(tc_gemm_persist_kernel, kPSmem)) != cudaSuccess) return e;
    attr = true;
  }
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t tiles = cdiv(a_rows, kBM) * cdiv(b_rows, kPBN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(tiles < sms ? tiles : sms));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_persist_kernel, ta, tb, args);
}

// Few-token contraction (see tc_skinny_kernel): A = weights (a_rows x K),
// B = token rows (b_rows x K) in tiles of NT (grid z), K cut into `splits`
// slices (one cluster per 128-row tile of A; splits <= 8 and <= the k-blocks).
template <int NT>
static cudaError_t launch_skinny_t(const void* A, int64_t a_rows, const void* B, int64_t b_rows, int K, int splits,
                                   const SkinnyArgs& args, cudaStream_t s) {
  CUtensorMap ta, tb;
  cudaError_t e = make_map_2d(&ta, A, a_rows, K, kBM);
  if (e != cudaSuccess) return e;
  if ((e = make_map_2d(&tb, B, b_rows, K, NT)) != cudaSuccess) return e;
  auto kern = tc_skinny_kernel<NT>;
  static bool attr = false;
  if (!attr) {
    if ((e = set_kernel_smem(kern, SkinnyCfg<NT>::SMEM)) != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(splits), unsigned(cdiv(a_rows, kBM)), unsigned(cdiv(b_rows, NT)));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = SkinnyCfg<NT>::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = unsigned(splits);
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, args);
}

static cudaError_t launch_skinny(const void* A, int64_t a_rows, const void* B, int64_t b_rows, int K, int max_tok,
                                 const SkinnyArgs& args, cudaStream_t s) {
  // K slices: enough CTAs for two a SM over the 128-row tiles, at most 8 (one
  // portable cluster) and at least 4 k-blocks a slice
  const int64_t tiles = cdiv(a_rows, kBM), nk = cdiv(K, kBK);
  int64_t splits = cdiv(2 * 152, tiles);
  if (splits > 8) splits = 8;
  if (splits > nk / 4) splits = nk / 4;
  if (splits < 1) splits = 1;
  const int sp = int(splits);
  if (max_tok <= 16) return launch_skinny_t<16>(A, a_rows, B, b_rows, K, sp, args, s);
  if (max_tok <= 32) return launch_skinny_t<32>(A, a_rows, B, b_rows, K, sp, args, s);
  if (max_tok <= 64) return launch_skinny_t<64>(A, a_rows, B, b_rows, K, sp, args, s);
  return launch_skinny_t<128>(A, a_rows, B, b_rows, K, sp, args, s);
}

// cluster_y > 1: thread-block clusters of (1, cluster_y, 1).
static cudaError_t launch_pdl(const void* kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args,
                              unsigned cluster_y = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cluster_y > 1) {
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = 1;
    at[1].val.clusterDim.y = cluster_y;
    at[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelExC(&cfg, kern, args);
}

// Image build on the tensor cores (bf16 maps): V_k^T into the scratch, then
// M = W V_k as the contraction of W (d_out x d) with V_k^T (k x d), stored in
// bf16 by the epilogue (accumulation in TMEM; each output summed in one fixed
// order).  The Gram matrix is not formed here: the gate's residual needs it
// to float32 accuracy over sums of up to d terms, which the tensor cores'
// accumulation does not give (measured: rho^2 off by 2.4e-5 at d = 8200).
cudaError_t launch_image_tc(const void* W, const void* V, void* M, int64_t d, int64_t d_out, int64_t k,
                            uint16_t* Vt, uint32_t* err, cudaStream_t s) {
  cudaError_t e;
  {
    dim3 grid(unsigned(cdiv(k, 32)), unsigned(cdiv(d, 32)));
    transpose_bf16_kernel<<<grid, dim3(32, 8), 0, s>>>(static_cast<const uint16_t*>(V), Vt, int(d), int(k));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int bn = k >= 256 ? 256 : (k >= 128 ? 128 : 64);
  TcArgs a{};
  a.rows = int(d_out);
  a.N = int(k);
  a.K = int(d);
  a.C = static_cast<float*>(M);
  a.ldc = k;
  a.err = err;
  a.c_bf16 = 1;
  return launch_tc_gemm(W, d_out, Vt, k, int(d), bn, a, s);
}

cudaError_t launch_slow_rows_tc(const void* X, const void* W, int64_t d, int64_t d_out, int64_t T,
                                const int32_t* idx, const int32_t* counts, uint16_t* Xslow, float* Y, uint32_t* err,
                                cudaStream_t s) {
  cudaError_t e;
  {
    const uint4* src = static_cast<const uint4*>(X);
    uint4* dst = reinterpret_cast<uint4*>(Xslow);
    const int32_t* sidx = idx + T;
    const int32_t* cnt = counts + 1;
    int64_t rv = d * 2 / 16;
    int TT = int(T);
    void* args[] = {&src, &dst, &sidx, &cnt, &rv, &TT};
    if ((e = launch_pdl(reinterpret_cast<const void*>(gather_rows_kernel), dim3(296), dim3(256), 0, s, args)) !=
        cudaSuccess)
      return e;
  }
  SkinnyArgs sl{};
  sl.n_rows = int(d_out);
  sl.K = int(d);
  sl.n_tok_dev = counts + 1;
  sl.Y = Y;
  sl.ldy = d_out;
  sl.tok_map = idx + T;
  sl.err = err;
  return launch_skinny(W, d_out, Xslow, T, int(d), int(T), sl, s);
}

cudaError_t launch_tensor_path(const TensorArgs& t, cudaStream_t s) {
  cudaError_t e;
  const int64_t d = t.d, k = t.k, T = t.T, d_out = t.d_out;
  // 1. V^T
  {
    dim3 grid(unsigned(cdiv(k, 32)), unsigned(cdiv(d, 32)));
    transpose_bf16_kernel<<<grid, dim3(32, 8), 0, s>>>(static_cast<const uint16_t*>(t.V), t.Vt, int(d), int(k));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // 2. G = X V
  TcArgs g{};
  g.rows = int(T);
  g.N = int(k);
  g.K = int(d);
  g.C = t.G;
  g.ldc = k;
  g.err = t.err;
  // Prefill-sized T: 128 x 128 tiles where k >= 256 (X read from L2 once
  // per 128 columns of G; 3 stages, two CTAs an SM, so the grid of 16 x 2 x 8
  // CTAs at T = 2048, k = 256 is one wave); small T: 128 x 64 tiles (one
  // 128-row tile holds every token, so narrower tiles give more CTAs).  K is
  // cut into g_split(T) slices for parallelism; the finalize adds the slices.
  const int gsplit = int(cdiv(d, kBK)) < g_split(T) ? int(cdiv(d, kBK)) : g_split(T);  // each slice >= 1 k-block
  g.ksplit = gsplit;
  g.c_split = T * k;
  const int g_bn = (T >= kTensorMinT && k >= 256) ? 128 : 64;
  if ((e = launch_tc_gemm(t.X, T, t.Vt, k, int(d), g_bn, g, s)) != cudaSuccess) return e;
  // 3. rho, flags, bf16 g: the per-token pass, then the Gram form
  {
    const uint16_t* X = static_cast<const uint16_t*>(t.X);
    const float* G = t.G;
    int64_t dd = d;
    int kk = int(k), TT = int(T), gs = gsplit;
    float* gT = t.gT;
    uint16_t* Gbf = t.Gbf;
    float2* norms = t.norms;
    void* args[] = {&X, &G, &dd, &kk, &TT, &gs, &gT, &Gbf, &norms};
    const void* kern = gsplit > 8 ? reinterpret_cast<const void*>(tc_norms_kernel<kGSplitMax>)
                                  : reinterpret_cast<const void*>(tc_norms_kernel<8>);
    if ((e = launch_pdl(kern, dim3(unsigned(T)), dim3(kNormThreads), 0, s, args)) != cudaSuccess) return e;
  }
  {
    const float* gT = t.gT;
    const float* gram = t.gram;
    const float2* norms = t.norms;
    int kk = int(k), TT = int(T);
    float eps = t.eps;
    float* rho = t.rho;
    uint8_t* flags = t.flags;
    int nb = fin_blocks(T, k);
    uint32_t* err = t.err;
    void* args[] = {&gT, &gram, &norms, &kk, &TT, &eps, &rho, &flags, &nb, &err};
    const size_t smem = fin_smem(k);
    const void* kern = k > kFinCols ? reinterpret_cast<const void*>(tc_gramq_kernel<2>)
                                    : reinterpret_cast<const void*>(tc_gramq_kernel<1>);
    if (smem > 48 * 1024) {
      if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess)
        return e;
    }
    if ((e = launch_pdl(kern, dim3(unsigned(cdiv(T, kFinTok)), unsigned(nb)), dim3(kFinThreads + 32), smem, s,
                        args, unsigned(nb))) != cudaSuccess)
      return e;
  }
  // 4. compaction and gathers
  if ((e = launch_compact(t.flags, int(T), t.idx, t.counts, s)) != cudaSuccess) return e;
  {
    GatherJob xs{static_cast<const uint4*>(t.X), reinterpret_cast<uint4*>(t.Xslow), t.idx + T, t.counts + 1,
                 d * 2 / 16};
    GatherJob gf{reinterpret_cast<const uint4*>(t.Gbf), reinterpret_cast<uint4*>(t.Gfast), t.idx, t.counts,
                 k * 2 / 16};
    int nb0 = 296;
    void* args[] = {&xs, &gf, &nb0};
    if ((e = launch_pdl(reinterpret_cast<const void*>(gather_rows2_kernel), dim3(296 + 148), dim3(256), 0, s,
                        args)) != cudaSuccess)
      return e;
  }
  // 5. Y_fast = G_fast M^T, Y_slow = X_slow W^T (rows scattered to token
  // positions).  Below prefill size the weights are the MMA's 128-row side
  // and the tokens its narrow side (the few-token contraction).
  if (T < kTensorMinT) {
    SkinnyArgs f{};
    f.n_rows = int(d_out);
    f.K = int(k);
    f.n_tok_dev = t.counts;
    f.Y = t.Y;
    f.ldy = d_out;
    f.tok_map = t.idx;
    f.err = t.err;
    if ((e = launch_skinny(t.M, d_out, t.Gfast, T, int(k), int(T), f, s)) != cudaSuccess) return e;
    SkinnyArgs sl{};
    sl.n_rows = int(d_out);
    sl.K = int(d);
    sl.n_tok_dev = t.counts + 1;
    sl.Y = t.Y;
    sl.ldy = d_out;
    sl.tok_map = t.idx + T;
    sl.err = t.err;
    return launch_skinny(t.W, d_out, t.Xslow, T, int(d), int(T), sl, s);
  }
  TcArgs f{};
  f.rows_dev = t.counts;
  f.N = int(d_out);
  f.K = int(k);
  f.C = t.Y;
  f.ldc = d_out;
  f.row_map = t.idx;
  f.err = t.err;
  // float32 rows that bulk copies can send: the persistent contraction
  const bool persist = d_out % 4 == 0 && (reinterpret_cast<uintptr_t>(t.Y) & 15) == 0;
  if ((e = persist ? launch_tc_gemm_persist(t.Gfast, T, t.M, d_out, int(k), f, s)
                   : launch_tc_gemm(t.Gfast, T, t.M, d_out, int(k), 128, f, s)) != cudaSuccess)
    return e;
  TcArgs sl{};
  sl.rows_dev = t.counts + 1;
  sl.N = int(d_out);
  sl.K = int(d);
  sl.C = t.Y;
  sl.ldc = d_out;
  sl.row_map = t.idx + T;
  sl.err = t.err;
  // 256 token rows per CTA (two 128-row tiles), so W is read from L2 once
  // per 256 slow tokens
  return launch_tc_gemm(t.Xslow, T, t.W, d_out, int(d), 256, sl, s, 2);
}

}  // namespace gsi
