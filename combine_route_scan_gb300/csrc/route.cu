// Routing for MoE dispatch: classify every pick, count the rows of every
// (expert, source) segment, give each routed pick its position inside its
// segment, and turn the counts into the running receive counts and segment
// offsets of every rank.
//
// aclnnMoeDistributeDispatchV4 (参数说明, 约束说明): active masks, zero / copy
// expert id ranges, epRecvCountsOut of shape epWorldSize * localExpertNum,
// deterministic results. combine_doubleplane README (功能说明, 方案设计):
// expand_x grouped by expert, ep_recv_count = running counts over the
// (local_expert, src_rank) segments, the SDMA / MTE plane rule.
//
// One CTA per source rank s. A warp iteration covers floor(32/K) whole tokens
// (lane = token-in-group * K + k), so the picks of a token sit in adjacent
// lanes and a repeated routed id is found with K-1 register shuffles. Tokens
// are split into contiguous runs, one per warp, in token order. A warp groups
// equal expert ids with __match_any_sync: the leader of each group adds the
// group size to the warp's counter for that expert. A scan of the warp counters
// over warps gives each warp its starting position per expert; a second walk
// hands every pick base + (equal ids in earlier lanes). Positions therefore
// follow (t, k) order exactly and no atomic decides any order. The first walk
// leaves each pick's expert id (or -1) in the rank array; the second walk
// reads it back and overwrites it with the position.
//
// The per-rank scan of the W*L*W segment counts into ep_recv_count (inclusive)
// and segment offsets (exclusive) then takes one of two forms:
//   * W <= 16: the W CTAs run as one thread-block cluster. Each CTA sets up a
//     receive barrier (an mbarrier expecting L*W counts) and arrives at a
//     cluster barrier before anything else; once its totals are known, CTA s
//     pushes the count of segment (le, s) into CTA d's shared memory with
//     st.async, whose completion is counted in bytes on CTA d's receive
//     barrier. CTA d waits for its L*W counts and scans rank d's segments: all
//     ranks in parallel, no fence, no global atomic. A last cluster barrier at
//     the very end keeps every CTA alive until all pushes have landed.
//   * otherwise: the last CTA to finish (completion counter in the workspace)
//     scans all counts, tile by tile through shared memory.
#include "common.cuh"

namespace crs {

constexpr int kRouteThreadsMax = 1024;
constexpr int kScanTile = 4096;
constexpr int kRegIters = 4;  // warp iterations whose keys walk 1 keeps in registers

// Split cluster barrier: arrive (release: this thread's earlier writes become
// visible to the cluster; relaxed: no ordering) and wait (acquire).
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
// 4-byte store into another CTA's shared memory; its completion is counted
// (4 bytes) on that CTA's mbarrier `bar` (both cluster addresses).
__device__ __forceinline__ void st_async_u32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(addr), "r"(v),
               "r"(bar)
               : "memory");
}
// Bounded wait on a phase of this CTA's mbarrier whose bytes other CTAs of the
// cluster deliver (acquire at cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int* status, uint64_t limit_ns) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (it == 0) t0 = globaltimer_ns();
    else if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) {
      set_error(status, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}

constexpr uint64_t kExchangeTimeoutNs = 2000000000ull;  // bound on the count exchange (never reached when healthy)

// THREADS: 256 for sources with at most 1024 picks (every warp then has at most
// kRegIters iterations and barriers are short), else 1024.
template <bool CLUSTER, int THREADS>
__global__ void __launch_bounds__(THREADS) route_kernel(RouteParams p) {
  MOE_PHASE_BEGIN(p, kPhaseRoute);
  constexpr int kRouteThreads = THREADS;
  constexpr int kRouteWarps = THREADS / 32;
  // wcnt [kRouteWarps][E], tot [E], recv [E] (cluster form: the L*W counts
  // this rank receives, index le*W + s); later the scan tiles
  extern __shared__ __align__(16) int32_t rsm[];
  __shared__ __align__(8) uint64_t recv_bar;
  __shared__ long long s_scan[32];
  __shared__ long long s_total;
  __shared__ int s_last;
  const Shape sh = p.sh;
  const int s = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = sh.E, K = sh.K;
  const int G = 32 / K;  // whole tokens per warp iteration
  int32_t* wcnt = rsm;
  int32_t* tot = rsm + kRouteWarps * E;
  int32_t* recv = tot + E;

  if constexpr (CLUSTER) {
    // the receive barrier expects one 4-byte count per (le, s) segment; every
    // CTA's barrier is set up before any CTA passes the first cluster wait
    if (tid == 0) {
      mbar_init(&recv_bar, 1);
      mbar_fence_init();
      mbar_arrive_expect_tx(&recv_bar, (uint32_t)E * 4u);
    }
    cluster_arrive_relaxed();
  }
  pdl_wait();
  MOE_PHASE_PAST_WAIT();
  pdl_launch_dependents();

  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) wcnt[i] = 0;
  if (sh.mask_kind == 1) {
    const uint8_t* m = p.mask + (size_t)s * sh.bs;
    for (int t = tid + 1; t < sh.bs; t += kRouteThreads)
      if (m[t] != 0 && m[t - 1] == 0) set_error(p.status, MOE_ERR_MASK_ORDER);
  }
  __syncthreads();

  const int n_iter = (sh.bs + G - 1) / G;
  const int per_warp = (n_iter + kRouteWarps - 1) / kRouteWarps;
  const int it0 = min(n_iter, warp * per_warp), it1 = min(n_iter, it0 + per_warp);
  const size_t tok0 = (size_t)s * sh.bs;
  const int tl = lane / K, k = lane - tl * K;
  int32_t* keys = p.rank + tok0 * K;

  // walk 1: classify, reject repeated routed ids, count per warp and expert.
  // When a warp has at most kRegIters iterations (the common case), all its
  // ids and mask bytes are loaded up front so the loads are in flight
  // together, and the keys stay in registers for walk 2.
  const bool in_regs = per_warp <= kRegIters;
  int keyr[kRegIters];
  int locr[kRegIters];  // position among the warp's earlier picks of the same expert
  if (in_regs) {
    int raw[kRegIters];
    bool act[kRegIters];
#pragma unroll
    for (int j = 0; j < kRegIters; ++j) {
      const int t = (it0 + j) * G + tl;
      const bool valid = it0 + j < it1 && tl < G && t < sh.bs;
      const size_t tok = tok0 + t;
      raw[j] = valid ? p.ids[tok * K + k] : -1;
      act[j] = valid && (sh.mask_kind == 0 || (sh.mask_kind == 1 ? p.mask[tok] != 0 : p.mask[tok * K + k] != 0));
    }
#pragma unroll
    for (int j = 0; j < kRegIters; ++j) {
      if (it0 + j >= it1) {
        keyr[j] = -1;
        locr[j] = -1;
        continue;
      }
      int key = -1;
      if (act[j]) {
        const int e = raw[j];
        const long long z = (long long)e - sh.E;
        if (e < 0 || z >= (long long)sh.Z + sh.C) set_error(p.status, MOE_ERR_BAD_EXPERT_ID);
        else if (e < sh.E) key = e;
      }
      bool dup = false;
      for (int dd = 1; dd < K; ++dd) {
        const int other = __shfl_up_sync(0xffffffffu, key, dd);
        if (dd <= k && key >= 0 && other == key) dup = true;
      }
      if (dup) {
        set_error(p.status, MOE_ERR_BAD_EXPERT_ID);
        key = -1;
      }
      keyr[j] = key;
      // the group leader bumps the warp's counter for this expert and hands
      // the old value to its group, so walk 2 needs no second match
      const uint32_t peers = __match_any_sync(0xffffffffu, key);
      const int leader = __ffs(peers) - 1;
      int before = 0;
      if (key >= 0 && lane == leader) {
        before = wcnt[warp * E + key];
        wcnt[warp * E + key] = before + __popc(peers);
      }
      __syncwarp();  // the next iteration's leaders read what this one wrote
      before = __shfl_sync(0xffffffffu, before, leader);
      locr[j] = key >= 0 ? before + __popc(peers & lanemask_lt()) : -1;
    }
  } else {
    for (int it = it0; it < it1; ++it) {
      const int t = it * G + tl;
      const bool valid = tl < G && t < sh.bs;
      int key = -1;
      if (valid) {
        const int c = classify_pick(p.ids, p.mask, sh, tok0 + t, k);
        if (c == kPickBad) set_error(p.status, MOE_ERR_BAD_EXPERT_ID);
        key = c >= 0 ? c : -1;
      }
      bool dup = false;
      for (int dd = 1; dd < K; ++dd) {
        const int other = __shfl_up_sync(0xffffffffu, key, dd);
        if (dd <= k && key >= 0 && other == key) dup = true;
      }
      if (dup) {
        set_error(p.status, MOE_ERR_BAD_EXPERT_ID);
        key = -1;
      }
      if (valid) keys[(size_t)t * K + k] = key;
      const uint32_t peers = __match_any_sync(0xffffffffu, key);
      if (key >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + key] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();

  // scan over warps per expert; totals; rows sent to other ranks
  long long remote = 0;
  for (int e = tid; e < E; e += kRouteThreads) {
    int run = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
    tot[e] = run;
    if (e / sh.L != s) remote += run;
  }
  // cluster form: push each total to the rank that receives the segment
  // (e = d*L + le goes to CTA d, slot le*W + s); this thread wrote tot[e]
  if constexpr (CLUSTER) {
    cluster_wait_acquire();  // every receive barrier is set up
    for (int e = tid; e < E; e += kRouteThreads) {
      const int d = e / sh.L, le = e - d * sh.L;
      st_async_u32(cluster_map(recv + le * sh.W + s, (uint32_t)d), (uint32_t)tot[e],
                   cluster_map(&recv_bar, (uint32_t)d));
    }
  }
  {
    const long long ex = block_exclusive_scan(remote, s_scan);
    if (tid == kRouteThreads - 1) s_total = ex + remote;
    __syncthreads();
    remote = s_total;
  }

  // counts and plane of each segment sent by s (the page's rule with s as the
  // writer): bulk iff remote, non-empty, >= bulk_min_bytes and above the mean
  // remote segment; rows*den > remote is the page's cross multiply with the
  // row size divided out of both sides.
  const long long den = (long long)(sh.W - 1 > 1 ? sh.W - 1 : 1) * sh.L;
  for (int e = tid; e < E; e += kRouteThreads) {
    const int d = e / sh.L;
    const long long rows = tot[e];
    const size_t g = (size_t)e * sh.W + s;
    p.cnt[g] = (int32_t)rows;
    if (p.seg_ready) {  // ready flags: count this call's rows from zero; empty segments are ready now
      p.landed[g] = 0u;
      if (rows == 0) st_release_gpu(p.seg_ready + g, p.ticket);
    }
    int use = 0;
    if (p.bulk_ok && d != s && rows > 0) {
      if (p.plane_policy == MOE_PLANE_BULK_ALL) {
        use = 1;
      } else if (p.plane_policy == MOE_PLANE_RULE) {
        use = rows * sh.row_out >= p.bulk_min_bytes && rows * den > remote;
      }
    }
    p.plane[g] = (uint8_t)use;
    if (p.seg_plane_out) p.seg_plane_out[g] = (uint8_t)use;
  }

  if constexpr (CLUSTER) {
    // CTA s scans the L*W segments (le, s') of receiving rank d = s
    // (L*W = E <= 1024) once all of their counts have landed
    mbar_wait_cluster(&recv_bar, 0, p.status, kExchangeTimeoutNs);
    // all pushes into this CTA are done; the matching wait is at the very end
    cluster_arrive_relaxed();
    const int d = s, LW = sh.L * sh.W;
    constexpr int kPer = (kRouteThreadsMax + kRouteThreads - 1) / kRouteThreads;
    // thread tid owns the contiguous segments [j0, j1) of rank d (at most kPer)
    const int per = (LW + kRouteThreads - 1) / kRouteThreads;
    const int j0 = min(LW, tid * per), j1 = min(LW, j0 + per);
    long long cv[kPer];
    long long local = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int j = j0 + q;
      cv[q] = 0;
      if (j < j1) cv[q] = recv[j];
      local += cv[q];
    }
    long long run = block_exclusive_scan(local, s_scan);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int j = j0 + q;
      if (j < j1) {
        const size_t g = (size_t)d * LW + j;
        p.base[g] = (int32_t)run;
        p.ep_recv_count[g] = (int32_t)(run + cv[q]);
        run += cv[q];
        if (j == LW - 1 && run > sh.A) set_error(p.status, MOE_ERR_CAPACITY);
      }
    }
  } else {
    __syncthreads();
  }

  // walk 2: position of every routed pick inside its segment
  for (int j = 0; j < per_warp; ++j) {
    const int it = it0 + j;
    if (it >= it1) break;
    const int t = it * G + tl;
    const bool valid = tl < G && t < sh.bs;
    int r = -1;
    if (in_regs) {
      // wcnt now holds each expert's count over earlier warps
      int key = -1, loc = -1;
#pragma unroll
      for (int q = 0; q < kRegIters; ++q)
        if (q == j) {
          key = keyr[q];
          loc = locr[q];
        }
      if (key >= 0) r = wcnt[warp * E + key] + loc;
    } else {
      const int key = valid ? keys[(size_t)t * K + k] : -1;
      const uint32_t peers = __match_any_sync(0xffffffffu, key);
      if (key >= 0) r = wcnt[warp * E + key] + __popc(peers & lanemask_lt());
      __syncwarp();
      if (key >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + key] += __popc(peers);
      __syncwarp();
    }
    if (valid) keys[(size_t)t * K + k] = r;
  }

  // counters of the kernels that follow in the same call start from zero
  if (s == 0)
    for (int i = tid; i < p.n_zero_words; i += kRouteThreads) p.zero_words[i] = 0u;
  // the scatter that follows writes the pick -> row map and hands out tokens
  // by ticket; these stores come after every release of this CTA, so no
  // barrier waits for them
  if (s == 0 && tid == 0 && p.hdr) {
    p.hdr->inv_assist = (unsigned long long)(uintptr_t)p.assist_out;
    p.hdr->inv_ep = (unsigned long long)(uintptr_t)p.ep_recv_count;
    p.hdr->inv_valid = 1u;
    p.hdr->scatter_next = 0u;
  }

  if constexpr (CLUSTER) {
    cluster_wait_acquire();  // no CTA leaves while pushes into another may be in flight
    return;
  }

  // the last CTA turns the counts of all sources into offsets
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atomicAdd(p.done, 1u);
    s_last = (prev == (uint32_t)sh.W - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int LW = sh.L * sh.W;
  const int N = sh.W * LW;  // == E * W, indexed g = e*W + s = d*LW + le*W + s
  long long* pstart = reinterpret_cast<long long*>(rsm);  // [W] prefix at each rank's start
  int32_t* tile = reinterpret_cast<int32_t*>(pstart + sh.W);
  long long carry = 0;
  for (int t0 = 0; t0 < N; t0 += kScanTile) {
    const int n = min(kScanTile, N - t0);
    for (int j = tid; j < n; j += kRouteThreads) tile[j] = __ldcg(p.cnt + t0 + j);
    __syncthreads();
    const int chunk = (n + kRouteThreads - 1) / kRouteThreads;
    const int j0 = min(n, tid * chunk), j1 = min(n, j0 + chunk);
    long long local = 0;
    for (int j = j0; j < j1; ++j) local += tile[j];
    const long long ex = block_exclusive_scan(local, s_scan);
    const long long off = carry + ex;
    long long run = off;
    for (int j = j0; j < j1; ++j) {
      if ((t0 + j) % LW == 0) pstart[(t0 + j) / LW] = run;
      run += tile[j];
    }
    if (tid == kRouteThreads - 1) s_total = ex + local;
    __syncthreads();
    run = off;
    for (int j = j0; j < j1; ++j) {
      const int g = t0 + j;
      const int c = tile[j];
      const long long before = run - pstart[g / LW];
      run += c;
      p.base[g] = (int32_t)before;
      p.ep_recv_count[g] = (int32_t)(before + c);
      if ((g + 1) % LW == 0 && before + c > sh.A) set_error(p.status, MOE_ERR_CAPACITY);
    }
    carry += s_total;
    __syncthreads();
  }
  if (tid == 0) *p.done = 0;  // ready for the next call (stream order)
}

// Dynamic shared memory of the walks: wcnt [threads/32][E], tot [E], recv [E].
static size_t route_walk_smem(int E, int threads) { return (size_t)(threads / 32 + 2) * E * sizeof(int32_t); }

static size_t route_smem(const Shape& sh, int threads) {
  const size_t walk = route_walk_smem(sh.E, threads);
  const size_t scan = (size_t)sh.W * sizeof(long long) + kScanTile * sizeof(int32_t);
  return walk > scan ? walk : scan;
}

// Is a cluster of W route CTAs schedulable on this device? Cached per (device, W, size).
template <int THREADS>
static bool cluster_route_ok(int dev, int W, size_t smem) {
  static signed char ok[64][17] = {};
  if (W > 16) return false;
  if (ok[dev][W] != 0) return ok[dev][W] > 0;
  bool good = cudaFuncSetAttribute(route_kernel<true, THREADS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                  cudaSuccess &&
              cudaFuncSetAttribute(route_kernel<true, THREADS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)route_walk_smem(1024, THREADS)) == cudaSuccess;
  if (good) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(W);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = W;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int n = 0;
    good = cudaOccupancyMaxActiveClusters(&n, route_kernel<true, THREADS>, &cfg) == cudaSuccess && n >= 1;
  }
  cudaGetLastError();  // a refused query leaves no sticky error behind
  ok[dev][W] = good ? 1 : -1;
  return good;
}

template <int THREADS>
static cudaError_t launch_route_t(const RouteParams& p, cudaStream_t st, int dev) {
  const size_t walk = route_walk_smem(p.sh.E, THREADS);
  if (cluster_route_ok<THREADS>(dev, p.sh.W, walk)) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.sh.W);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = walk;
    cfg.stream = st;
    cudaLaunchAttribute a[2];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = p.sh.W;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    a[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = a;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, route_kernel<true, THREADS>, p);
  }
  const size_t smem = route_smem(p.sh, THREADS);
  static size_t attr_bytes[64] = {};
  if (attr_bytes[dev] < smem) {
    cudaError_t e =
        cudaFuncSetAttribute(route_kernel<false, THREADS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_bytes[dev] = smem;
  }
  PdlLaunch L(dim3(p.sh.W), dim3(THREADS), smem, st);
  return cudaLaunchKernelEx(&L.cfg, route_kernel<false, THREADS>, p);
}

cudaError_t launch_route(const RouteParams& p, cudaStream_t st) {
  if (p.sh.K > 32) return cudaErrorInvalidValue;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if ((long long)p.sh.bs * p.sh.K <= 1024) return launch_route_t<256>(p, st, dev);
  return launch_route_t<kRouteThreadsMax>(p, st, dev);
}

}  // namespace crs
