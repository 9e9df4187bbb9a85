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
// One CTA per source rank s. Its picks (t, k) are split into contiguous slices,
// one per warp, in (t, k) order. A warp walks its slice 32 picks at a time and
// groups equal expert ids with __match_any_sync: the leader of each group adds
// the group size to the warp's counter for that expert. A scan of the warp
// counters over warps gives each warp its starting position per expert; a
// second walk hands every pick base + (equal ids in earlier lanes). Positions
// therefore follow (t, k) order exactly and no atomic decides any order.
//
// The last CTA to finish (completion counter in the workspace) scans the
// W*L*W segment counts into ep_recv_count (inclusive) and segment offsets
// (exclusive), per receiving rank.
#include "common.cuh"

namespace crs {

constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;

// Routed expert of pick (tok, k), or -1 if it is not routed or repeats a routed
// id of an earlier pick of the same token (an error that is recorded once, in
// the first walk).
__device__ __forceinline__ int routed_key(const RouteParams& p, size_t tok, int k, bool record) {
  const int c = classify_pick(p.ids, p.mask, p.sh, tok, k);
  if (c == kPickBad) {
    if (record) set_error(p.status, MOE_ERR_BAD_EXPERT_ID);
    return -1;
  }
  if (c < 0) return -1;
  for (int k2 = 0; k2 < k; ++k2) {
    if (classify_pick(p.ids, p.mask, p.sh, tok, k2) == c) {
      if (record) set_error(p.status, MOE_ERR_BAD_EXPERT_ID);
      return -1;
    }
  }
  return c;
}

__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteParams p) {
  extern __shared__ int32_t wcnt[];  // [kRouteWarps][E], then tot[E]
  __shared__ long long s_scan[32];
  __shared__ int s_last;
  const Shape sh = p.sh;
  const int s = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = sh.E, K = sh.K;
  const int n = sh.bs * K;  // picks of source s
  int32_t* tot = wcnt + kRouteWarps * E;

  pdl_wait();
  pdl_launch_dependents();

  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) wcnt[i] = 0;
  if (sh.mask_kind == 1) {
    const uint8_t* m = p.mask + (size_t)s * sh.bs;
    for (int t = tid + 1; t < sh.bs; t += kRouteThreads)
      if (m[t] != 0 && m[t - 1] == 0) set_error(p.status, MOE_ERR_MASK_ORDER);
  }
  __syncthreads();

  const int per_warp = (n + kRouteWarps - 1) / kRouteWarps;
  const int lo = min(n, warp * per_warp), hi = min(n, lo + per_warp);
  const size_t tok0 = (size_t)s * sh.bs;

  // walk 1: per-warp counts per expert
  for (int b = lo; b < hi; b += 32) {
    const int pi = b + lane;
    int key = -1;
    if (pi < hi) key = routed_key(p, tok0 + pi / K, pi % K, true);
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + key] += __popc(peers);
    __syncwarp();
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
    p.cnt[(size_t)e * sh.W + s] = run;
    if (e / sh.L != s) remote += run;
  }
  // block sum of `remote` (exclusive scan of the last thread + its own value)
  {
    const long long ex = block_exclusive_scan(remote, s_scan);
    __shared__ long long s_remote;
    if (tid == kRouteThreads - 1) s_remote = ex + remote;
    __syncthreads();
    remote = s_remote;
  }

  // plane of each segment sent by s (the page's rule with s as the writer):
  // bulk iff remote, non-empty, >= bulk_min_bytes and above the mean remote
  // segment; rows*den > remote is the page's cross multiply with the row size
  // divided out of both sides.
  const long long den = (long long)(sh.W - 1 > 1 ? sh.W - 1 : 1) * sh.L;
  for (int e = tid; e < E; e += kRouteThreads) {
    const int d = e / sh.L;
    const long long rows = tot[e];
    int use = 0;
    if (p.bulk_ok && d != s && rows > 0) {
      if (p.plane_policy == MOE_PLANE_BULK_ALL) {
        use = 1;
      } else if (p.plane_policy == MOE_PLANE_RULE) {
        use = rows * sh.row_out >= p.bulk_min_bytes && rows * den > remote;
      }
    }
    const size_t g = (size_t)e * sh.W + s;
    p.plane[g] = (uint8_t)use;
    if (p.seg_plane_out) p.seg_plane_out[g] = (uint8_t)use;
  }
  __syncthreads();

  // walk 2: position of every routed pick inside its segment
  for (int b = lo; b < hi; b += 32) {
    const int pi = b + lane;
    int key = -1;
    if (pi < hi) key = routed_key(p, tok0 + pi / K, pi % K, false);
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    int r = -1;
    if (key >= 0) r = wcnt[warp * E + key] + __popc(peers & lanemask_lt());
    __syncwarp();
    if (key >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + key] += __popc(peers);
    __syncwarp();
    if (pi < hi) p.rank[tok0 * K + pi] = r;
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
  const int chunk = (N + kRouteThreads - 1) / kRouteThreads;
  const int j0 = min(N, tid * chunk), j1 = min(N, j0 + chunk);
  long long local = 0;
  for (int j = j0; j < j1; ++j) local += __ldcg(p.cnt + j);
  const long long off = block_exclusive_scan(local, s_scan);
  long long* pstart = reinterpret_cast<long long*>(wcnt);  // [W] prefix at each rank's start
  long long run = off;
  for (int j = j0; j < j1; ++j) {
    if (j % LW == 0) pstart[j / LW] = run;
    run += __ldcg(p.cnt + j);
  }
  __syncthreads();
  run = off;
  for (int j = j0; j < j1; ++j) {
    const int c = __ldcg(p.cnt + j);
    const long long before = run - pstart[j / LW];
    run += c;
    p.base[j] = (int32_t)before;
    p.ep_recv_count[j] = (int32_t)(before + c);
    if ((j + 1) % LW == 0 && before + c > sh.A) set_error(p.status, MOE_ERR_CAPACITY);
  }
  if (tid == 0) *p.done = 0;  // ready for the next call (stream order)
}

cudaError_t launch_route(const RouteParams& p, cudaStream_t st) {
  const size_t smem = (size_t)(kRouteWarps + 1) * p.sh.E * sizeof(int32_t);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (kRouteWarps + 1) * 1024 * (int)sizeof(int32_t));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  PdlLaunch L(dim3(p.sh.W), dim3(kRouteThreads), smem, st);
  return cudaLaunchKernelEx(&L.cfg, route_kernel, p);
}

}  // namespace crs
