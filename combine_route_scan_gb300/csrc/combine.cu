// MoE combine (combine_doubleplane README, 功能说明, check formula):
//   x_out[token] = sum_k topk_output[token, k] * expert_scales[token, k]
// where topk_output of a routed pick is the expert-output row that
// assist_info_for_combine names for it (rows [0, ep_recv_count[d][L*W-1]) of
// every rank d), a copy expert gives x[token] and a zero expert or an inactive
// pick gives nothing (aclnnMoeDistributeDispatchV4, 参数说明).
//
// GB300 form (one HBM, so no write-back pass is needed): an inverse-map kernel
// turns assist_info (row -> pick) into pick -> row (unless the dispatch that
// produced these very assist_info / ep_recv_count buffers already left that
// map in the workspace), then a gather kernel reads
// each token's K rows with 16-byte loads and reduces them in fp32, k
// ascending, one fused multiply-add per pick, and rounds once to the output
// type. The reduce checks every pick it reads against assist_info, so a row
// map that does not match the routing is reported, not silently used.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace crs {

constexpr int kInvThreads = 256;
constexpr int kReduceThreads = 256;
constexpr int kReduceBatch = 8;  // picks whose loads are in flight together
constexpr int kReduceVpl = 4;    // 16-byte vectors per lane per work item

__global__ void __launch_bounds__(kInvThreads) combine_inverse_kernel(CombineParams p) {
  MOE_PHASE_BEGIN(p, kPhaseInverse);
  const Shape sh = p.sh;
  const int d = blockIdx.y;
  const int LW = sh.L * sh.W;
  pdl_wait();
  MOE_PHASE_PAST_WAIT();
  pdl_launch_dependents();
  // the dispatch that wrote these assist_info / ep_recv_count buffers also
  // wrote the map (the reduce still checks every pick against assist_info);
  // callers without a workspace (moe_combine_noalloc) have no header
  const WsHeader* h = p.hdr;
  if (h && h->inv_valid && h->inv_assist == (unsigned long long)(uintptr_t)p.assist &&
      h->inv_ep == (unsigned long long)(uintptr_t)p.ep_recv_count)
    return;
  long long count = p.ep_recv_count[(size_t)d * LW + LW - 1];
  if (count < 0 || count > sh.A) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_error(p.status, MOE_ERR_BAD_ASSIST);
    count = count < 0 ? 0 : sh.A;
  }
  for (long long row = (long long)blockIdx.x * kInvThreads + threadIdx.x; row < count;
       row += (long long)gridDim.x * kInvThreads) {
    const long long fr = (long long)d * sh.A + row;
    const int s = p.assist[fr * 3 + 0], t = p.assist[fr * 3 + 1], k = p.assist[fr * 3 + 2];
    if (s < 0 || s >= sh.W || t < 0 || t >= sh.bs || k < 0 || k >= sh.K) {
      set_error(p.status, MOE_ERR_BAD_ASSIST);
      continue;
    }
    const long long pk = ((long long)s * sh.bs + t) * sh.K + k;
    if (MOE_IN_BOUNDS(p.status, pk, (long long)sh.W * sh.bs * sh.K) &&
        MOE_IN_BOUNDS(p.status, fr, (long long)sh.W * sh.A))
      p.inv[pk] = (int32_t)fr;
  }
}

// Element traits: 16-byte vectors of T, fp32 (or wrapping int32) accumulators.
template <int DT>
struct Vec;
template <>
struct Vec<MOE_F16> {
  static constexpr int N = 8;
  __device__ static void fma(float* acc, float w, int4 v) {
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h[i]);
      acc[2 * i] = __fmaf_rn(w, f.x, acc[2 * i]);
      acc[2 * i + 1] = __fmaf_rn(w, f.y, acc[2 * i + 1]);
    }
  }
  __device__ static int4 pack(const float* acc) {
    int4 o;
    __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
    return o;
  }
};
template <>
struct Vec<MOE_BF16> {
  static constexpr int N = 8;
  __device__ static void fma(float* acc, float w, int4 v) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      acc[2 * i] = __fmaf_rn(w, f.x, acc[2 * i]);
      acc[2 * i + 1] = __fmaf_rn(w, f.y, acc[2 * i + 1]);
    }
  }
  __device__ static int4 pack(const float* acc) {
    int4 o;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    return o;
  }
};

// Builds the contributing-pick list of token `tau` (warp 0): source row
// pointers and weights in ascending k. Records errors for ids out of range and
// for a row map that does not name this pick.
struct ReduceTable {
  const uint8_t* src[32];
  uint32_t w[32];  // fp32 or int32 bits
  int n;
};

__device__ __forceinline__ void build_reduce_table(const CombineParams& p, size_t tau, ReduceTable& tab) {
  const Shape& sh = p.sh;
  const int lane = threadIdx.x & 31;
  const uint8_t* src = nullptr;
  uint32_t w = 0;
  if (lane < sh.K) {
    const int c = classify_pick(p.ids, p.mask, sh, tau, lane);
    if (c == kPickBad) {
      set_error(p.status, MOE_ERR_BAD_EXPERT_ID);
    } else if (c >= 0) {
      const int s = (int)(tau / sh.bs), t = (int)(tau % sh.bs);
      const long long r = p.inv[tau * sh.K + lane];
      const int LW = sh.L * sh.W;
      const int d = c / sh.L;
      const long long row = r - (long long)d * sh.A;
      bool good = row >= 0 && row < sh.A && row < p.ep_recv_count[(size_t)d * LW + LW - 1];
      if (good) {
        const int32_t* a = p.assist + r * 3;
        good = a[0] == s && a[1] == t && a[2] == lane;
      }
      if (good) {
        src = static_cast<const uint8_t*>(p.expert_out) + r * (long long)sh.row_in;
      } else {
        set_error(p.status, MOE_ERR_BAD_ASSIST);
      }
    } else if (c == kPickCopy) {
      src = static_cast<const uint8_t*>(p.x) + tau * (size_t)sh.row_in;
    }
    if (src) w = reinterpret_cast<const uint32_t*>(p.scales)[tau * sh.K + lane];
  }
  const uint32_t m = __ballot_sync(0xffffffffu, src != nullptr);
  if (src) {
    const int j = __popc(m & lanemask_lt());
    tab.src[j] = src;
    tab.w[j] = w;
  }
  if (lane == 0) tab.n = __popc(m);
}

// One warp per (token, chunk of 32*vpl vectors): lanes < K load the pick's id,
// mask, weight and row in parallel, the warp compacts the contributing picks
// (ascending k) into shared memory, then every lane reduces its 16-byte
// vectors with up to kReduceBatch picks' loads in flight. No CTA-wide barrier.
// The row map is checked against assist_info and ep_recv_count after the data
// loads are issued (rows are bounds-checked against the capacity before any
// read), so the check costs no round trip on the critical path.
template <int DT>
__device__ __forceinline__ void reduce_vector(const uint8_t* const* src, const uint32_t* w, int n, size_t off,
                                              uint8_t* out) {
  if constexpr (DT == MOE_I32) {
    uint32_t acc[4] = {0u, 0u, 0u, 0u};
    for (int j = 0; j < n; j += kReduceBatch) {
      int4 y[kReduceBatch];
#pragma unroll
      for (int g = 0; g < kReduceBatch; ++g)
        if (j + g < n) y[g] = ld_nc_v4(src[j + g] + off);
#pragma unroll
      for (int g = 0; g < kReduceBatch; ++g) {
        if (j + g < n) {
          const uint32_t ww = w[j + g];
          acc[0] += ww * (uint32_t)y[g].x;
          acc[1] += ww * (uint32_t)y[g].y;
          acc[2] += ww * (uint32_t)y[g].z;
          acc[3] += ww * (uint32_t)y[g].w;
        }
      }
    }
    st_v4(out + off, make_int4((int)acc[0], (int)acc[1], (int)acc[2], (int)acc[3]));
  } else {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < n; j += kReduceBatch) {
      int4 y[kReduceBatch];
#pragma unroll
      for (int g = 0; g < kReduceBatch; ++g)
        if (j + g < n) y[g] = ld_nc_v4(src[j + g] + off);
#pragma unroll
      for (int g = 0; g < kReduceBatch; ++g)
        if (j + g < n) Vec<DT>::fma(acc, __uint_as_float(w[j + g]), y[g]);
    }
    st_v4(out + off, Vec<DT>::pack(acc));
  }
}

// At most 64 registers a thread: four CTAs (32 warps) per SM keep enough
// loads in flight to cover HBM latency.
template <int DT>
__global__ void __launch_bounds__(kReduceThreads, 4) combine_reduce_kernel(CombineParams p, int chunks, int vpl) {
  MOE_PHASE_BEGIN(p, kPhaseReduce);
  __shared__ const uint8_t* s_src[kReduceThreads / 32][32];
  __shared__ uint32_t s_w[kReduceThreads / 32][32];
  const Shape sh = p.sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * (kReduceThreads / 32) + warp;
  pdl_wait();
  MOE_PHASE_PAST_WAIT();
  pdl_launch_dependents();
  const long long n_tok = (long long)sh.W * sh.bs;
  if (item >= n_tok * chunks) return;
  // last token first: the dispatch scatter hands out tokens in ascending
  // order, so the rows of the highest tokens are the newest in L2 when this
  // kernel starts, and are read before the reduce's own traffic evicts them
  // (measured on GB300 at 16 ranks x 256 tokens, h 7168: reduce 78.3 -> 74.2
  // us, dispatch + combine step 155.5 -> 150.1 us)
  const size_t tau = (size_t)(n_tok - 1 - item / chunks);
  const int c = (int)(item % chunks);

  const uint8_t* src = nullptr;
  uint32_t w = 0;
  long long r = -1;
  int d = -1;
  if (lane < sh.K) {
    const size_t pk = tau * sh.K + lane;
    r = p.inv[pk];
    w = reinterpret_cast<const uint32_t*>(p.scales)[pk];
    const int cls = classify_pick(p.ids, p.mask, sh, tau, lane);
    if (cls >= 0) {
      d = cls / sh.L;
      const long long row = r - (long long)d * sh.A;
      if (row >= 0 && row < sh.A && MOE_IN_BOUNDS(p.status, r, (long long)sh.W * sh.A)) {
        src = static_cast<const uint8_t*>(p.expert_out) + r * (long long)sh.row_in;
      } else {
        set_error(p.status, MOE_ERR_BAD_ASSIST);
      }
    } else if (cls == kPickCopy) {
      src = static_cast<const uint8_t*>(p.x) + tau * (size_t)sh.row_in;
    } else if (cls == kPickBad) {
      set_error(p.status, MOE_ERR_BAD_EXPERT_ID);
    }
  }
  const uint32_t m = __ballot_sync(0xffffffffu, src != nullptr);
  if (src) {
    const int j = __popc(m & lanemask_lt());
    s_src[warp][j] = src;
    s_w[warp][j] = w;
  }
  __syncwarp();
  const int n = __popc(m);

  // deferred consistency check of the row map (loads issued now, compared last)
  int a0 = 0, a1 = 0, a2 = 0, cnt = 0;
  const bool check = d >= 0 && src != nullptr && c == 0;
  if (check) {
    const int32_t* a = p.assist + r * 3;
    a0 = a[0];
    a1 = a[1];
    a2 = a[2];
    const int LW = sh.L * sh.W;
    cnt = p.ep_recv_count[(size_t)d * LW + LW - 1];
  }

  const int nvec = sh.row_in / 16;
  uint8_t* out = static_cast<uint8_t*>(p.x_out) + tau * (size_t)sh.row_in;
  const int v0 = c * 32 * vpl;
  for (int i = 0; i < vpl; ++i) {
    const int v = v0 + i * 32 + lane;
    if (v >= nvec) break;
    reduce_vector<DT>(s_src[warp], s_w[warp], n, (size_t)v * 16, out);
  }

  if (check) {
    const int s = (int)(tau / sh.bs), t = (int)(tau % sh.bs);
    if (a0 != s || a1 != t || a2 != lane || r - (long long)d * sh.A >= cnt)
      set_error(p.status, MOE_ERR_BAD_ASSIST);
  }
}

// Element-wise fallback for rows that are not 16-byte multiples.
template <int DT>
__global__ void __launch_bounds__(kReduceThreads) combine_reduce_plain_kernel(CombineParams p) {
  __shared__ ReduceTable tab;
  const Shape sh = p.sh;
  pdl_wait();
  pdl_launch_dependents();
  for (size_t tau = blockIdx.x; tau < (size_t)sh.W * sh.bs; tau += gridDim.x) {
    if (threadIdx.x < 32) build_reduce_table(p, tau, tab);
    __syncthreads();
    const int n = tab.n;
    for (int j = threadIdx.x; j < sh.h; j += kReduceThreads) {
      if constexpr (DT == MOE_I32) {
        uint32_t acc = 0;
        for (int q = 0; q < n; ++q) acc += tab.w[q] * reinterpret_cast<const uint32_t*>(tab.src[q])[j];
        reinterpret_cast<uint32_t*>(p.x_out)[tau * sh.h + j] = acc;
      } else {
        float acc = 0.f;
        for (int q = 0; q < n; ++q) {
          const uint16_t b = reinterpret_cast<const uint16_t*>(tab.src[q])[j];
          const float y = DT == MOE_F16 ? __half2float(__ushort_as_half(b))
                                        : __bfloat162float(__ushort_as_bfloat16(b));
          acc = __fmaf_rn(__uint_as_float(tab.w[q]), y, acc);
        }
        uint16_t o = DT == MOE_F16 ? __half_as_ushort(__float2half_rn(acc))
                                   : __bfloat16_as_ushort(__float2bfloat16_rn(acc));
        reinterpret_cast<uint16_t*>(p.x_out)[tau * sh.h + j] = o;
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_combine_inverse(const CombineParams& p, cudaStream_t st) {
  const Shape& sh = p.sh;
  const long long per_rank_blocks = (sh.A + kInvThreads - 1) / kInvThreads;
  const int gx = (int)(per_rank_blocks < 32 ? (per_rank_blocks > 0 ? per_rank_blocks : 1) : 32);
  PdlLaunch L(dim3(gx, sh.W), dim3(kInvThreads), 0, st);
  return cudaLaunchKernelEx(&L.cfg, combine_inverse_kernel, p);
}

cudaError_t launch_combine_reduce(const CombineParams& p, cudaStream_t st, int num_sms) {
  const Shape& sh = p.sh;
  const long long n_tok = (long long)sh.W * sh.bs;
  if (n_tok == 0) return cudaSuccess;
  if (sh.row_in % 16 != 0) {
    const int grid = (int)(n_tok < num_sms * 8LL ? n_tok : num_sms * 8LL);
    PdlLaunch L(dim3(grid), dim3(kReduceThreads), 0, st);
    if (sh.x_dtype == MOE_I32) return cudaLaunchKernelEx(&L.cfg, combine_reduce_plain_kernel<MOE_I32>, p);
    if (sh.x_dtype == MOE_F16) return cudaLaunchKernelEx(&L.cfg, combine_reduce_plain_kernel<MOE_F16>, p);
    return cudaLaunchKernelEx(&L.cfg, combine_reduce_plain_kernel<MOE_BF16>, p);
  }
  const int nvec = sh.row_in / 16;
  // smaller work items when the batch is too small to give every SM ~16 warps
  int vpl = kReduceVpl;
  while (vpl > 1 && n_tok * ((nvec + 32 * vpl - 1) / (32 * vpl)) < (long long)num_sms * 16) vpl >>= 1;
  const int chunks = (nvec + 32 * vpl - 1) / (32 * vpl);
  const long long items = n_tok * chunks;
  const long long grid = (items + kReduceThreads / 32 - 1) / (kReduceThreads / 32);
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  PdlLaunch L(dim3((unsigned)grid), dim3(kReduceThreads), 0, st);
  if (sh.x_dtype == MOE_I32) return cudaLaunchKernelEx(&L.cfg, combine_reduce_kernel<MOE_I32>, p, chunks, vpl);
  if (sh.x_dtype == MOE_F16) return cudaLaunchKernelEx(&L.cfg, combine_reduce_kernel<MOE_F16>, p, chunks, vpl);
  return cudaLaunchKernelEx(&L.cfg, combine_reduce_kernel<MOE_BF16>, p, chunks, vpl);
}

}  // namespace crs
