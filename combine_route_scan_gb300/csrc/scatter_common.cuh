// Pieces shared by the dispatch payload kernels (scatter.cu, and the
// quantising variants in scatter_quant.cu): the per-token destination list
// built by warp 0, ready-flag publication and the per-rank communication
// timer (aclnnMoeDistributeDispatchV4, 参数说明 performanceInfoOptional).
#pragma once

#include "common.cuh"

namespace crs {

constexpr int kScatterThreads = 256;
constexpr int kScatterWarps = kScatterThreads / 32;
constexpr int kMaxK = 32;

__host__ __device__ __forceinline__ size_t align128(size_t v) { return (v + 127) & ~size_t(127); }

// Per-token destination list, built by warp 0. Three of them rotate by token,
// so the ready-flag publisher can still read the last two tokens' lists.
struct PickTable {
  long long sm_dst[kMaxK];    // flat expand_x rows (d*A + row) on the store plane
  long long bulk_dst[kMaxK];  // ... on the bulk plane
  int sm_seg[kMaxK];          // their segments g = e*W + s
  int bulk_seg[kMaxK];
  int n_sm, n_bulk;
};

// One more row of segment g is in place; the last one releases the flag.
// The caller has fenced after the row's stores became visible.
__device__ __forceinline__ void publish_row(const ScatterParams& p, int g) {
  if (atomicAdd(p.landed + g, 1u) + 1u == (uint32_t)p.cnt[g]) {
    __threadfence();
    st_release_gpu(p.seg_ready + g, p.ticket);
  }
}

// Ready flags by the lanes of one warp: lane j counts row j in (a token's rows
// lie in distinct segments, so the atomics hit distinct counters and run in
// parallel). Every lane fences first; the caller has made the rows' stores
// visible to this warp (a CTA barrier; for bulk copies, lane 0 waited for
// their completion and fenced the async proxy before a __syncwarp).
__device__ __forceinline__ void publish_rows_warp(const ScatterParams& p, const int* segs, int n) {
  __threadfence();
  if ((int)(threadIdx.x & 31) < n) publish_row(p, segs[threadIdx.x & 31]);
}

// Builds the destination list of token `tau` (warp 0 only) and writes the
// per-row metadata. Returns nothing; results land in `tab`.
__device__ __forceinline__ void build_picks(const ScatterParams& p, size_t tau, int s, int t, PickTable& tab) {
  const Shape& sh = p.sh;
  const int lane = threadIdx.x & 31;
  long long dst = -1;
  int bulk = 0;
  if (lane < sh.K) {
    // position and id are independent loads: issue both before using either
    const int r = p.rank[tau * sh.K + lane];
    const int e = p.ids[tau * sh.K + lane];
    if (r >= 0 && MOE_IN_BOUNDS(p.status, e, sh.E)) {
      const int d = e / sh.L;
      const size_t g = (size_t)e * sh.W + s;
      const long long row = (long long)p.base[g] + r;
      if (row < sh.A && MOE_IN_BOUNDS(p.status, (long long)d * sh.A + row, (long long)sh.W * sh.A)) {
        dst = (long long)d * sh.A + row;
        bulk = p.plane[g];
        if (p.inv) p.inv[tau * sh.K + lane] = (int32_t)dst;
        int32_t* a = p.assist + dst * 3;
        a[0] = s;
        a[1] = t;
        a[2] = lane;
        if (p.expand_scales)
          reinterpret_cast<uint32_t*>(p.expand_scales)[dst] =
              reinterpret_cast<const uint32_t*>(p.scales)[tau * sh.K + lane];
      } else {
        set_error(p.status, MOE_ERR_CAPACITY);
      }
    }
  }
  const uint32_t m_sm = __ballot_sync(0xffffffffu, dst >= 0 && !bulk);
  const uint32_t m_bk = __ballot_sync(0xffffffffu, dst >= 0 && bulk);
  const int seg = dst >= 0 ? p.ids[tau * sh.K + lane] * sh.W + s : -1;
  if (dst >= 0 && !bulk) {
    const int j = __popc(m_sm & lanemask_lt());
    tab.sm_dst[j] = dst;
    tab.sm_seg[j] = seg;
  }
  if (dst >= 0 && bulk) {
    const int j = __popc(m_bk & lanemask_lt());
    tab.bulk_dst[j] = dst;
    tab.bulk_seg[j] = seg;
  }
  if (lane == 0) {
    tab.n_sm = __popc(m_sm);
    tab.n_bulk = __popc(m_bk);
  }
}

// The loads of build_picks issued ahead of their use (warp 0, lanes < K):
// a pick's position, expert id and weight one token ahead, its segment's
// first row and plane, which need the id, on the next token; the list is then
// built without waiting on memory (build_picks_from).
struct PickAhead {
  int r, e;    // position in the segment (-1: not routed), expert id
  uint32_t w;  // expert_scales bits (when expand_scales is written)
  int base;    // first row of segment e*W + s
  int plane;   // its plane
};

__device__ __forceinline__ void pick_load_first(const ScatterParams& p, size_t tau, PickAhead& a) {
  const int lane = threadIdx.x & 31;
  a.r = -1;
  a.e = -1;
  a.w = 0u;
  if (lane < p.sh.K) {
    a.r = p.rank[tau * p.sh.K + lane];
    a.e = p.ids[tau * p.sh.K + lane];
    if (p.expand_scales) a.w = reinterpret_cast<const uint32_t*>(p.scales)[tau * p.sh.K + lane];
  }
}

__device__ __forceinline__ void pick_load_second(const ScatterParams& p, int s, PickAhead& a) {
  a.base = 0;
  a.plane = 0;
  if (a.r >= 0 && a.e >= 0 && a.e < p.sh.E) {
    const size_t g = (size_t)a.e * p.sh.W + s;
    a.base = p.base[g];
    a.plane = p.plane[g];
  }
}

// build_picks on values loaded ahead (same results, same metadata writes).
__device__ __forceinline__ void build_picks_from(const ScatterParams& p, size_t tau, int s, int t, PickTable& tab,
                                                 const PickAhead& a) {
  const Shape& sh = p.sh;
  const int lane = threadIdx.x & 31;
  long long dst = -1;
  int bulk = 0;
  if (lane < sh.K && a.r >= 0 && MOE_IN_BOUNDS(p.status, a.e, sh.E)) {
    const int d = a.e / sh.L;
    const long long row = (long long)a.base + a.r;
    if (row < sh.A && MOE_IN_BOUNDS(p.status, (long long)d * sh.A + row, (long long)sh.W * sh.A)) {
      dst = (long long)d * sh.A + row;
      bulk = a.plane;
      if (p.inv) p.inv[tau * sh.K + lane] = (int32_t)dst;
      int32_t* as = p.assist + dst * 3;
      as[0] = s;
      as[1] = t;
      as[2] = lane;
      if (p.expand_scales) reinterpret_cast<uint32_t*>(p.expand_scales)[dst] = a.w;
    } else {
      set_error(p.status, MOE_ERR_CAPACITY);
    }
  }
  const uint32_t m_sm = __ballot_sync(0xffffffffu, dst >= 0 && !bulk);
  const uint32_t m_bk = __ballot_sync(0xffffffffu, dst >= 0 && bulk);
  const int seg = dst >= 0 ? a.e * sh.W + s : -1;
  if (dst >= 0 && !bulk) {
    const int j = __popc(m_sm & lanemask_lt());
    tab.sm_dst[j] = dst;
    tab.sm_seg[j] = seg;
  }
  if (dst >= 0 && bulk) {
    const int j = __popc(m_bk & lanemask_lt());
    tab.bulk_dst[j] = dst;
    tab.bulk_seg[j] = seg;
  }
  if (lane == 0) {
    tab.n_sm = __popc(m_sm);
    tab.n_bulk = __popc(m_bk);
  }
}

// Per-rank communication time (performance info): the earliest CTA start,
// the latest row-store time per source rank, and the last CTA to finish adds
// each rank's span to the caller's array and resets the workspace fields.
__device__ __forceinline__ void perf_begin(const ScatterParams& p) {
  atomicMax(&p.hdr->perf_start_inv, ~(unsigned long long)globaltimer_ns());
}
__device__ __forceinline__ void perf_mark(const ScatterParams& p, size_t tau) {
  atomicMax(p.perf_end + tau / p.sh.bs, (unsigned long long)globaltimer_ns());
}
__device__ __forceinline__ void perf_finish(const ScatterParams& p, int* s_last) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    *s_last = atomicAdd(&p.hdr->scatter_done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (*s_last) {
    __threadfence();
    const unsigned long long start = ~atomicAdd(&p.hdr->perf_start_inv, 0ull);
    for (int s = threadIdx.x; s < p.sh.W; s += blockDim.x) {
      const unsigned long long end = atomicExch(p.perf_end + s, 0ull);
      if (end > start) p.perf[s] += (long long)(end - start);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      p.hdr->perf_start_inv = 0ull;
      p.hdr->scatter_done = 0u;
    }
  }
}

#ifdef MOE_FLAG_OBSERVER
// Test builds only. The last CTA of a dispatch payload grid (launched
// cooperatively, so it runs alongside the storing CTAs) watches every
// segment's ready flag with acquire loads and, the moment a flag holds the
// call's ticket, copies the segment's rows, assist_info entries and dynamic
// scales into the observer's buffers. A flag published before its rows were
// visible would leave rows in the copies that differ from the final output.
// Warp w takes segments w, w + nwarps, ...; every wait is bounded by the
// call's timeout (a segment never seen records MOE_ERR_TIMEOUT).
__device__ __forceinline__ void observe_flags(const ScatterParams& p) {
  const Shape& sh = p.sh;
  const int lane = threadIdx.x & 31, nthr = blockDim.x;
  const int nseg = sh.E * sh.W;  // at most 64 * nthr (host check)
  const uint32_t row_out = (uint32_t)sh.row_out;
  const int dyn_row = sh.quant == 4 ? sh.ngroups : sh.ngroups * 4;  // dynamic-scale bytes of a row
  pdl_wait();
  const uint64_t t0 = globaltimer_ns();
  // thread i watches segments i, i + nthr, ... (bit k of pend: segment i + k * nthr)
  uint64_t pend = 0;
  for (int k = 0; k < 64; ++k)
    if ((int)threadIdx.x + k * nthr < nseg) pend |= 1ull << k;
  while (__any_sync(0xffffffffu, pend != 0)) {
    // poll every pending flag with relaxed loads (all in flight together);
    // a segment is read only after its flag is acquired below
    int found = -1;
    for (uint64_t m = pend; m; m &= m - 1) {
      const int k = __ffsll((long long)m) - 1;
      uint32_t f;
      asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(f) : "l"(p.seg_ready + threadIdx.x + k * nthr) : "memory");
      if (f == p.ticket && found < 0) {
        found = (int)threadIdx.x + k * nthr;
        pend &= ~(1ull << k);
      }
    }
    // the warp copies every segment a lane just saw, one after another
    for (uint32_t b = __ballot_sync(0xffffffffu, found >= 0); b; b &= b - 1) {
      const int gs = __shfl_sync(0xffffffffu, found, __ffs(b) - 1);
      // every lane acquires the flag itself before reading the segment
      if (ld_acquire_gpu(p.seg_ready + gs) != p.ticket) set_error(p.status, MOE_ERR_BAD_ASSIST);
      const int e = gs / sh.W, d = e / sh.L;
      const long long b0 = min((long long)max(p.base[gs], 0), (long long)sh.A);
      const long long r0 = (long long)d * sh.A + b0, n = min((long long)max(p.cnt[gs], 0), (long long)sh.A - b0);
      const uint8_t* from = static_cast<const uint8_t*>(p.expand_x) + r0 * row_out;
      uint8_t* to = p.obs.rows + r0 * row_out;
      const long long bytes = n * (long long)row_out;
      // four 16-byte loads a lane in flight, then their stores
      for (long long o = (long long)lane * 16; o < bytes; o += 4 * 32 * 16) {
        int4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (o + j * 512 < bytes) v[j] = *reinterpret_cast<const int4*>(from + o + j * 512);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (o + j * 512 < bytes) *reinterpret_cast<int4*>(to + o + j * 512) = v[j];
      }
      for (long long o = lane; o < n * 3; o += 32) p.obs.assist[r0 * 3 + o] = p.assist[r0 * 3 + o];
      if (p.obs.dyn)
        for (long long o = lane; o < n * dyn_row; o += 32)
          p.obs.dyn[r0 * dyn_row + o] = static_cast<const uint8_t*>(p.dyn_scales)[r0 * dyn_row + o];
      __syncwarp();
      if (lane == 0) {
        p.obs.seen_ns[gs] = globaltimer_ns();  // every read of the segment has returned
        atomicAdd(p.obs.n_seen, 1u);
      }
    }
    if (pend && globaltimer_ns() - t0 > p.timeout_ns) {
      set_error(p.status, MOE_ERR_TIMEOUT);
      pend = 0;
    }
  }
}

// An observed payload grid: `grid` CTAs (the storing ones and the observer)
// as one cooperative launch, so that all of them are resident together.
template <typename KernelT>
static cudaError_t launch_observed(KernelT kernel, const ScatterParams& p, cudaStream_t st, int grid, size_t smem,
                                   int threads = kScatterThreads) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeCooperative;
  a[0].val.cooperative = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// A storing CTA of an observed grid ends: its time for the observer.
__device__ __forceinline__ void observer_producer_end(const ScatterParams& p) {
  if (p.observe && threadIdx.x == 0) atomicMax(p.obs.producer_end_ns, (unsigned long long)globaltimer_ns());
}
#endif

}  // namespace crs
