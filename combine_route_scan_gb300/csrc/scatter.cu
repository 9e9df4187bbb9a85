// Dispatch payload without quantisation: expandXOut = AllToAllV(X)
// (aclnnMoeDistributeDispatchV4, 接口功能), with the two data planes of the
// combine_doubleplane README (方案设计) applied to the dispatch direction:
// plain SM stores for local, small or average segments, TMA bulk copies for
// large remote ones. (The quantised modes run in scatter_quant.cu.)
//
// Token-major and persistent: each CTA starts with tokens blockIdx.x, +grid,
// ... and then takes tokens from a shared ticket counter until none is left.
// A ring of STAGES shared-memory slots is filled by TMA bulk loads
// (cp.async.bulk global->shared, completion on an mbarrier), so every source
// row is read from HBM exactly once however many ranks it goes to. For each
// token, warp 0 builds the list of destination rows (rank d, row base + rank)
// and writes assist_info / expand_scales; then
//   * bulk-plane picks: one thread issues cp.async.bulk shared->global of the
//     whole row (no multicast), one bulk group per token, at most STAGES groups
//     in flight (the page's bounded backlog: quiet every 256 issues);
//   * store-plane picks: all threads copy the row from shared memory with
//     16-byte st.global.v4, coalesced.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "scatter_common.cuh"

namespace crs {

// Ready flags, called by warp 0 right after the first barrier of token i:
//   * token i-1's store-plane rows: every thread passed the barrier after
//     storing them, so a fence makes them visible before the count;
//   * token i-2's bulk-plane rows: its bulk group is complete once at most one
//     newer group (token i-1's) is pending (lane 0 issued them and waits);
//     then an async-proxy fence.
__device__ __forceinline__ void publish_earlier(const ScatterParams& p, const PickTable* tabs, int i) {
  if (i >= 1) {
    const PickTable& a = tabs[(i - 1) % 3];
    publish_rows_warp(p, a.sm_seg, a.n_sm);
  }
  if (i >= 2) {
    const PickTable& b = tabs[(i - 2) % 3];
    if (b.n_bulk > 0) {
      if ((threadIdx.x & 31) == 0) {
        bulk_wait_all<1>();
        fence_proxy_async_global();
      }
      __syncwarp();
      publish_rows_warp(p, b.bulk_seg, b.n_bulk);
    }
  }
}

// Thread 0 fills a ring slot with token `tau`: records the token, then either
// starts the TMA load of its row or, with tau < 0 (no token left), completes
// the slot's barrier phase by a plain arrival. Either way the barrier phase
// publishes s_tok[slot] to the threads that wait on it.
__device__ __forceinline__ void fill_slot(uint64_t* bar, int* s_tok, uint8_t* dst, const uint8_t* x, int tau,
                                          uint32_t row_in) {
  *s_tok = tau;
  if (tau >= 0) {
    mbar_arrive_expect_tx(bar, row_in);
    bulk_g2s(dst, x + (size_t)tau * row_in, row_in, bar);
  } else {
    mbar_arrive(bar);
  }
}

// Streaming store (st.global.cs: evict first from L2).
__device__ __forceinline__ void st_v4_cs(void* p, int4 v) {
  asm volatile("st.global.cs.v4.s32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// STREAM: the call writes far more than the L2 holds, so store-plane rows of
// tokens below p.stream_below use streaming stores and leave L2 early instead
// of as dirty lines that the next kernel's loads must first write back
// (measured at W16 bs256 h7168: dispatch + combine 156.9 -> 152.8 us); the
// last tokens, and a batch whose rows fit in L2, keep plain stores, so that
// the consumer can still find them there.
// 16 warps a CTA: more stores in flight per SM than 8 (three CTAs per SM
// either way, bounded by the ring's shared memory; measured at 16 x 256
// tokens, h 7168: scatter 75.2 -> 74.5 us)
constexpr int kTmaThreads = 512;
template <int STAGES, bool STREAM>
__global__ void __launch_bounds__(kTmaThreads) scatter_tma_kernel(ScatterParams p) {
  MOE_PHASE_BEGIN(p, kPhaseScatter);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ int s_tok[STAGES];  // token held by each slot, -1 once the tokens ran out
  __shared__ PickTable tabs[3];
  __shared__ int s_abort;

  const Shape sh = p.sh;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int n_tok = sh.W * sh.bs;
#ifdef MOE_FLAG_OBSERVER
  if (p.observe && blockIdx.x == gridDim.x - 1) {
    observe_flags(p);
    return;
  }
  const int G = gridDim.x - (p.observe ? 1 : 0);
#else
  const int G = gridDim.x;
#endif
  const uint32_t row_in = (uint32_t)sh.row_in, row_out = (uint32_t)sh.row_out;
  const size_t slot_in = align128(row_in);
  uint8_t* xin = smem;                         // [STAGES][slot_in]
  const uint8_t* x = static_cast<const uint8_t*>(p.x);
  uint8_t* out = static_cast<uint8_t*>(p.expand_x);

  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      s_tok[i] = -1;  // slots past the end of the tokens are never filled
    }
    mbar_fence_init();
    s_abort = 0;
  }
  __syncthreads();
  // Token hand-out (thread 0): the CTA's first STAGES tokens are blockIdx.x +
  // i*G, prefetched before the routing ends (x is never written by the routing
  // kernel, which lets this grid start only after its own predecessor ended);
  // every later one is STAGES*G + a ticket from a counter shared by all CTAs,
  // so CTAs that finish early take more tokens and the grid ends together.
  bool exhausted = false;  // thread 0: a slot got -1, no further fills
  if (tid == 0) {
    for (int i = 0; i < STAGES && !exhausted; ++i) {
      const long long tau = blockIdx.x + (long long)i * G;
      exhausted = tau >= n_tok;
      fill_slot(&full_bar[i], &s_tok[i], xin + i * slot_in, x, exhausted ? -1 : (int)tau, row_in);
    }
  }
  pdl_wait();  // routing results (and the zeroed ticket counter) are visible from here on
  MOE_PHASE_PAST_WAIT();
  pdl_launch_dependents();
  if (p.perf && tid == 0) perf_begin(p);
  // thread 0 claims each ticket one token ahead of its use, so the atomic's
  // latency overlaps a token's stores
  unsigned ticket = 0;
  if (tid == 0 && !exhausted) ticket = atomicAdd(&p.hdr->scatter_next, 1u);
  int prev_tau = -1;  // thread 0: last token handled (performance info)
  int n_done = 0;
  for (int i = 0;; ++i) {
    const int stage = i % STAGES;
    const uint32_t parity = (uint32_t)(i / STAGES) & 1u;
    PickTable& tab = tabs[i % 3];
    const uint8_t* row = xin + stage * slot_in;

    const bool ok = mbar_wait_bounded(&full_bar[stage], parity, p.status, p.timeout_ns);
    if (!ok) s_abort = 1;
    if (warp == 0) {
      const int tw = s_tok[stage];
      if (tw >= 0) build_picks(p, (size_t)tw, tw / sh.bs, tw % sh.bs, tab);
    }
    __syncthreads();
    const int tau = s_tok[stage];
    if (tau < 0 || s_abort) break;
    if (p.seg_ready && warp == 0) publish_earlier(p, tabs, i);
    if (p.perf && tid == 0 && i >= 1) perf_mark(p, (size_t)prev_tau);
    const int nb = tab.n_bulk, ns = tab.n_sm;
    if (tid == 0) {
      // refill the slot of the previous token once its bulk group has read it
      if (i >= 1 && !exhausted) {
        bulk_wait_read<0>();
        const int ps = (i - 1) % STAGES;
        const long long tn = (long long)STAGES * G + ticket;
        exhausted = tn >= n_tok;
        fill_slot(&full_bar[ps], &s_tok[ps], xin + ps * slot_in, x, exhausted ? -1 : (int)tn, row_in);
        if (!exhausted) ticket = atomicAdd(&p.hdr->scatter_next, 1u);
      }
      for (int j = 0; j < nb; ++j) bulk_s2g(out + tab.bulk_dst[j] * row_out, row, row_out);
      bulk_commit();
      prev_tau = tau;
    }
    if (ns > 0) {
      const bool cs = STREAM && tau < p.stream_below;
      for (uint32_t v = tid; v < row_in / 16; v += kTmaThreads) {
        const int4 val = *reinterpret_cast<const int4*>(row + v * 16);
        for (int j = 0; j < ns; ++j) {
          if (cs) st_v4_cs(out + tab.sm_dst[j] * row_out + v * 16, val);
          else st_v4(out + tab.sm_dst[j] * row_out + v * 16, val);
        }
      }
    }
    ++n_done;
  }
  // all bulk stores of this CTA complete before it exits
  if (p.seg_ready) {
    __syncthreads();  // every thread's stores of the last token are issued
    if (warp == 0 && !s_abort) {
      if (tid == 0) {
        bulk_wait_all<0>();
        fence_proxy_async_global();
      }
      __syncwarp();
      const int last = n_done - 1;
      if (last >= 0) {
        const PickTable& a = tabs[last % 3];
        publish_rows_warp(p, a.sm_seg, a.n_sm);
        publish_rows_warp(p, a.bulk_seg, a.n_bulk);
      }
      if (last >= 1) {
        const PickTable& b = tabs[(last - 1) % 3];
        publish_rows_warp(p, b.bulk_seg, b.n_bulk);
      }
    }
  }
  if (tid == 0) bulk_wait_all<0>();
#ifdef MOE_FLAG_OBSERVER
  observer_producer_end(p);
#endif
  if (p.perf) {
    if (tid == 0 && n_done > 0 && !s_abort) perf_mark(p, (size_t)prev_tau);
    __shared__ int s_last;
    perf_finish(p, &s_last);
  }
}

// Fallback for rows that are not 16-byte multiples: element-wise copies, all
// segments on the store plane.
__global__ void __launch_bounds__(kScatterThreads) scatter_plain_kernel(ScatterParams p) {
  __shared__ PickTable tab;
  const Shape sh = p.sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_tok = sh.W * sh.bs;
  pdl_wait();
  pdl_launch_dependents();
  if (p.perf && tid == 0) perf_begin(p);
  for (size_t tau = blockIdx.x; tau < (size_t)n_tok; tau += gridDim.x) {
    const int s = (int)(tau / sh.bs), t = (int)(tau % sh.bs);
    if (warp == 0) {
      build_picks(p, tau, s, t, tab);
      __syncwarp();
      // both planes are carried by plain stores here
      if (lane == 0) {
        for (int j = 0; j < tab.n_bulk; ++j) {
          tab.sm_dst[tab.n_sm + j] = tab.bulk_dst[j];
          tab.sm_seg[tab.n_sm + j] = tab.bulk_seg[j];
        }
        tab.n_sm += tab.n_bulk;
        tab.n_bulk = 0;
      }
    }
    __syncthreads();
    const int ns = tab.n_sm;
    if (sh.es == 4) {
      const uint32_t* xr = static_cast<const uint32_t*>(p.x) + tau * sh.h;
      uint32_t* out = static_cast<uint32_t*>(p.expand_x);
      for (int j = tid; j < sh.h; j += kScatterThreads) {
        const uint32_t v = xr[j];
        for (int k = 0; k < ns; ++k) out[tab.sm_dst[k] * sh.h + j] = v;
      }
    } else {
      const uint16_t* xr = static_cast<const uint16_t*>(p.x) + tau * sh.h;
      uint16_t* out = static_cast<uint16_t*>(p.expand_x);
      for (int j = tid; j < sh.h; j += kScatterThreads) {
        const uint16_t v = xr[j];
        for (int k = 0; k < ns; ++k) out[tab.sm_dst[k] * sh.h + j] = v;
      }
    }
    __syncthreads();
    // every thread's rows of this token are stored
    if (p.seg_ready && warp == 0) publish_rows_warp(p, tab.sm_seg, ns);
    if (p.perf && tid == 0) perf_mark(p, tau);
    __syncthreads();
  }
  if (p.perf) {
    __shared__ int s_last;
    perf_finish(p, &s_last);
  }
}

template <typename KernelT>
static cudaError_t launch_persistent(KernelT kernel, const ScatterParams& p, cudaStream_t st, int num_sms,
                                     size_t smem) {
  int per_sm = 0;
  const cudaError_t e = resident_blocks((const void*)kernel, kTmaThreads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int n_tok = p.sh.W * p.sh.bs;
#ifdef MOE_FLAG_OBSERVER
  if (p.observe) return launch_observed(kernel, p, st, min(n_tok, num_sms * per_sm - 1) + 1, smem, kTmaThreads);
#endif
  const int grid = max(1, min(n_tok, num_sms * per_sm));
  PdlLaunch L(dim3(grid), dim3(kTmaThreads), smem, st);
  return cudaLaunchKernelEx(&L.cfg, kernel, p);
}

// L2 size of the current device in bytes (cached per device; 0 if unknown).
static long long l2_bytes_of_current_device() {
  static std::atomic<long long> l2[64] = {};  // callers may be on several host threads
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  long long b = l2[dev].load(std::memory_order_relaxed);
  if (b == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    b = v;
    l2[dev].store(b, std::memory_order_relaxed);
  }
  return b;
}

// Shared-memory budget of the TMA scatter for `stages` slots.
static size_t scatter_smem(const Shape& sh, int stages) {
  return (size_t)stages * align128((size_t)sh.row_in);
}

bool scatter_tma_fits(const Shape& sh) { return scatter_smem(sh, 2) <= 200 * 1024; }

cudaError_t launch_scatter(const ScatterParams& p, cudaStream_t st, int num_sms, bool tma) {
  const Shape& sh = p.sh;
  if (sh.W * sh.bs == 0) return cudaSuccess;
  if (p.hdr == nullptr) return cudaErrorInvalidValue;  // the token tickets live in the workspace header
  if (!tma) {
    const int grid = max(1, min(sh.W * sh.bs, num_sms * 4));
    PdlLaunch L(dim3(grid), dim3(kScatterThreads), 0, st);
    return cudaLaunchKernelEx(&L.cfg, scatter_plain_kernel, p);
  }
  const bool four = scatter_smem(sh, 4) <= 110 * 1024;
  const size_t smem = scatter_smem(sh, four ? 4 : 2);
  const bool stream = (long long)sh.W * sh.bs * sh.K * sh.row_out > 2 * l2_bytes_of_current_device();
  // the last tokens' rows, about 3/8 of the L2, keep plain stores: the
  // combine reduce reads the highest tokens first and finds them in L2
  // (measured on GB300 at 16 x 256 tokens, h 7168: reduce 74.4 -> 73.1 us,
  // step 150.7 -> 149.6 us; keeping all of the L2 or none was slower)
  ScatterParams q = p;
  {
    const long long per_tok = (long long)sh.K * sh.row_out;
    const long long keep = per_tok > 0 ? l2_bytes_of_current_device() * 3 / 8 / per_tok : 0;
    q.stream_below = (int)std::max(0LL, (long long)sh.W * sh.bs - keep);
  }
  if (stream)
    return four ? launch_persistent(scatter_tma_kernel<4, true>, q, st, num_sms, smem)
                : launch_persistent(scatter_tma_kernel<2, true>, q, st, num_sms, smem);
  return four ? launch_persistent(scatter_tma_kernel<4, false>, q, st, num_sms, smem)
              : launch_persistent(scatter_tma_kernel<2, false>, q, st, num_sms, smem);
}

}  // namespace crs
