// Device helpers shared by the dispatch / combine kernels (sm_103a).
//
// Inline PTX for: mbarriers, TMA bulk copies (cp.async.bulk, no tensor map, no
// multicast), bulk-group completion, cross-proxy fences, programmatic dependent
// launch (griddepcontrol), acquire/release flags and %globaltimer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace crs {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- errors

// Record the first device-side error of the workspace (later ones are dropped).
__device__ __forceinline__ void set_error(int* status, int code) {
  atomicCAS(status, 0, code);
}

// Bounds checks of checked builds (-DMOE_BOUNDS_CHECK): an index outside its
// buffer records MOE_ERR_OUT_OF_BOUNDS and the guarded access is skipped.
// Ordinary builds compile every check to `true`.
__device__ __forceinline__ bool in_bounds_checked(int* status, long long idx, long long n) {
  if (idx >= 0 && idx < n) return true;
  set_error(status, MOE_ERR_OUT_OF_BOUNDS);
  return false;
}
#ifdef MOE_BOUNDS_CHECK
#define MOE_IN_BOUNDS(status, idx, n) ::crs::in_bounds_checked((status), (long long)(idx), (long long)(n))
#else
#define MOE_IN_BOUNDS(status, idx, n) true
#endif

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- phase times
// Test builds only (-DMOE_PHASE_TIMES): thread 0 of every CTA of a kernel
// records, in the 4 words of the kernel's slot, the earliest CTA start and the
// earliest CTA past griddepcontrol.wait (both kept inverted, so that
// atomicMax keeps the minimum), the latest CTA past it, and the latest CTA end
// (%globaltimer ns). Other builds compile the marks to nothing.
#ifdef MOE_PHASE_TIMES
struct PhaseScope {
  unsigned long long* t;
  __device__ PhaseScope(unsigned long long* base, int slot) : t(base ? base + slot * 4 : nullptr) {
    if (t && threadIdx.x == 0) atomicMax(t + 0, ~globaltimer_ns());
  }
  __device__ void past_wait() {
    if (t && threadIdx.x == 0) {
      const unsigned long long g = globaltimer_ns();
      atomicMax(t + 1, ~g);
      atomicMax(t + 2, g);
    }
  }
  __device__ ~PhaseScope() {
    if (t && threadIdx.x == 0) atomicMax(t + 3, globaltimer_ns());
  }
};
#define MOE_PHASE_BEGIN(params, slot) ::crs::PhaseScope moe_phase_scope((params).phase, (slot))
#define MOE_PHASE_PAST_WAIT() moe_phase_scope.past_wait()
#else
#define MOE_PHASE_BEGIN(params, slot) ((void)0)
#define MOE_PHASE_PAST_WAIT() ((void)0)
#endif
enum { kPhaseRoute = 0, kPhaseScatter = 1, kPhaseInverse = 2, kPhaseReduce = 3 };

// ---------------------------------------------------------------- PDL

// Wait until the previous kernel in the stream has completed and its memory
// is visible (no-op when the launch had no programmatic dependency).
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Let the next kernel in the stream start its prologue.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA) and other threads.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Plain arrival (no transaction bytes): completes the phase of a count-1
// barrier at once, with release semantics for this thread's earlier writes.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on a phase of an mbarrier. Returns false (and records
// MOE_ERR_TIMEOUT) if the phase did not complete within `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) {
      set_error(status, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA bulk

// global -> shared, completion counted on `bar` (bytes multiple of 16, both
// addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// shared -> global, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_s2g(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N of this thread's bulk groups are incomplete (writes done).
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Order completed async-proxy global writes before later generic accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------- flags

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------- vectors

__device__ __forceinline__ int4 ld_nc_v4(const void* p) {
  int4 v;
  asm("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_v4(void* p, int4 v) {
  asm volatile("st.global.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Lane mask of lanes below this one.
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace crs

namespace crs {

// Class of pick (s, t, k): the routed expert id in [0, E), or a negative code.
enum : int { kPickInactive = -1, kPickZero = -2, kPickCopy = -3, kPickBad = -4 };

__device__ __forceinline__ int classify_pick(const int32_t* ids, const uint8_t* mask, const Shape& sh,
                                             size_t tok, int k) {
  if (sh.mask_kind == 1 && mask[tok] == 0) return kPickInactive;
  if (sh.mask_kind == 2 && mask[tok * sh.K + k] == 0) return kPickInactive;
  const int e = ids[tok * sh.K + k];
  if (e < 0) return kPickBad;
  if (e < sh.E) return e;
  const long long r = (long long)e - sh.E;
  if (r < sh.Z) return kPickZero;
  if (r < (long long)sh.Z + sh.C) return kPickCopy;
  return kPickBad;
}

// Exclusive prefix sum over the block (blockDim.x a multiple of 32, <= 1024).
// `scratch` holds 32 ints of shared memory.
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nwarps ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  return (warp > 0 ? scratch[warp - 1] : 0) + x - v;
}

}  // namespace crs
