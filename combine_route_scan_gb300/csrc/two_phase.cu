// Two-phase combine: the write-back protocol of the combine_doubleplane README
// (方案设计, 实现逻辑), with the W EP ranks as partitions of one GPU.
//
// Phase 1 (put, the page's comm_only): every expert-output row of rank d goes
// back to its source's combine window, slot (s, t, k) = what assist_info
// names, and the slot's ready flag is set to the call's epoch. Warps take
// batches of R consecutive rows of one rank (R = 32, one per lane, or fewer
// for small calls, so that all warps have rows to move):
//   * store plane: the warp copies the row with 16-byte loads / stores, then
//     fences and release-stores the flags of its rows;
//   * bulk plane (segments the page's rule picks, writer = rank d): lane 0
//     moves the row through a per-warp two-slot shared ring with TMA bulk
//     copies (global -> shared -> global, no multicast; at most two copies of
//     the warp read shared memory at a time, the page's bounded backlog), waits
//     for the bulk group to complete, issues an async-proxy fence, and only then
//     release-stores the flags (status never visible before its payload).
// Phase 2 (reduce): for each token, lanes acquire-wait (bounded by
// wait_timeout_us) until the flags of its routed picks carry the epoch, then
// x_out = sum_k w_k * window[s][t][k] (copy experts: x), fp32, k ascending,
// fused multiply-add, as the gather combine does.
//
// One cooperative launch: all CTAs are resident, each finishes its puts before
// it waits on anything, so every wait ends. Flags carry an epoch that grows by
// one per call (kept in the workspace header), so no clearing pass is needed
// and a flag left by an earlier call is never taken for a new one.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace crs {

constexpr int kTpThreads = 256;
constexpr int kTpWarps = kTpThreads / 32;
constexpr int kTpSlot = 2048;  // small slots: 32 KB of ring a CTA, four CTAs (32 warps) an SM  // bytes per staging slot of the bulk plane
constexpr int kTpVpl = 4;      // 16-byte vectors per lane per reduce item

__device__ __forceinline__ int4 ld_v4(const void* p) {
  int4 v;
  asm volatile("ld.global.v4.s32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

template <int DT>
__device__ __forceinline__ void fma16(float* acc, float w, int4 v) {
  if constexpr (DT == MOE_F16) {
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h[i]);
      acc[2 * i] = __fmaf_rn(w, f.x, acc[2 * i]);
      acc[2 * i + 1] = __fmaf_rn(w, f.y, acc[2 * i + 1]);
    }
  } else {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      acc[2 * i] = __fmaf_rn(w, f.x, acc[2 * i]);
      acc[2 * i + 1] = __fmaf_rn(w, f.y, acc[2 * i + 1]);
    }
  }
}

template <int DT>
__device__ __forceinline__ int4 pack16(const float* acc) {
  int4 o;
  if constexpr (DT == MOE_F16) {
    __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
  } else {
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
  }
  return o;
}

// Rows of segment j (= le*W + s) of rank d, from the running counts.
__device__ __forceinline__ long long seg_rows(const int32_t* ep, int d, int LW, int j) {
  const int32_t* e = ep + (size_t)d * LW;
  return (long long)e[j] - (j > 0 ? e[j - 1] : 0);
}

template <int DT>
__global__ void __launch_bounds__(kTpThreads, 4) two_phase_kernel(CombineParams p) {
  extern __shared__ __align__(128) uint8_t tsm[];
  __shared__ __align__(8) uint64_t bars[kTpWarps][2];
  __shared__ const uint8_t* s_src[kTpWarps][32];
  __shared__ uint32_t s_w[kTpWarps][32];
  __shared__ int s_last;

  const Shape sh = p.sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = sh.W, LW = sh.L * sh.W;
  const uint32_t row_in = (uint32_t)sh.row_in;
  uint8_t* slots = tsm + (size_t)warp * 2 * kTpSlot;                         // [2][kTpSlot] per warp
  int* bprefix = reinterpret_cast<int*>(tsm + (size_t)kTpWarps * 2 * kTpSlot);  // [W+1] batch prefix
  long long* remote = reinterpret_cast<long long*>(bprefix + ((W + 2) & ~1));    // [W]
  const uint32_t epoch = p.hdr->epoch + 1u;
  const uint8_t* eo = static_cast<const uint8_t*>(p.expert_out);
  uint8_t* win = static_cast<uint8_t*>(p.window);
  const long long den = (long long)(W - 1 > 1 ? W - 1 : 1) * sh.L;

  if (lane == 0) {
    mbar_init(&bars[warp][0], 1);
    mbar_init(&bars[warp][1], 1);
    mbar_fence_init();
  }
  // per rank: rows received from other ranks, and the number of R-row batches
  const int R = p.tp_rows;
  for (int d = tid; d < W; d += kTpThreads) {
    long long own = 0;
    for (int le = 0; le < sh.L; ++le) own += seg_rows(p.ep_recv_count, d, LW, le * W + d);
    long long cnt = p.ep_recv_count[(size_t)d * LW + LW - 1];
    if (cnt < 0 || cnt > sh.A) {  // a count the routing cannot produce: report it, stay inside rank d's rows
      set_error(p.status, MOE_ERR_BAD_ASSIST);
      cnt = cnt < 0 ? 0 : sh.A;
    }
    remote[d] = cnt - own;
    bprefix[d + 1] = (int)((cnt + R - 1) / R);
  }
  __syncthreads();
  if (tid == 0) {
    bprefix[0] = 0;
    for (int d = 0; d < W; ++d) bprefix[d + 1] += bprefix[d];
  }
  __syncthreads();
  // optional copy of the plane decisions (writer = rank d)
  if (p.seg_plane_out) {
    for (long long g = (long long)blockIdx.x * kTpThreads + tid; g < (long long)W * LW;
         g += (long long)gridDim.x * kTpThreads) {
      const int d = (int)(g / LW), j = (int)(g % LW), s = j % W;
      const long long rows = seg_rows(p.ep_recv_count, d, LW, j);
      int use = 0;
      if (p.bulk_ok && s != d && rows > 0) {
        if (p.plane_policy == MOE_PLANE_BULK_ALL) use = 1;
        else if (p.plane_policy == MOE_PLANE_RULE)
          use = rows * sh.row_in >= p.bulk_min_bytes && rows * den > remote[d];
      }
      p.seg_plane_out[g] = (uint8_t)use;
    }
  }

  // ------------------------------------------------------------ phase 1: put
  const int n_batches = bprefix[W];
  const int gwarp = blockIdx.x * kTpWarps + warp, nwarps = gridDim.x * kTpWarps;
  uint32_t uses[2] = {0u, 0u};  // completed phases per staging slot (lane 0)
  const int nvec = (int)(row_in / 16);
  for (int b = gwarp; b < n_batches; b += nwarps) {
    int lo = 0, hi = W;  // rank d with bprefix[d] <= b < bprefix[d+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (bprefix[mid] <= b) lo = mid; else hi = mid;
    }
    const int d = lo;
    const long long cnt = min((long long)sh.A, (long long)p.ep_recv_count[(size_t)d * LW + LW - 1]);
    const long long r = (long long)(b - bprefix[d]) * R + lane;
    long long q = -1;  // window slot of this lane's row
    int bulk = 0;
    if (lane < R && r < cnt && MOE_IN_BOUNDS(p.status, (long long)d * sh.A + r, (long long)W * sh.A)) {
      const long long fr = (long long)d * sh.A + r;
      const int s = p.assist[fr * 3 + 0], t = p.assist[fr * 3 + 1], k = p.assist[fr * 3 + 2];
      if (s >= 0 && s < W && t >= 0 && t < sh.bs && k >= 0 && k < sh.K) {
        const int e = p.ids[((size_t)s * sh.bs + t) * sh.K + k];
        if (e >= 0 && e < sh.E && e / sh.L == d &&
            MOE_IN_BOUNDS(p.status, ((long long)s * sh.bs + t) * sh.K + k, (long long)W * sh.bs * sh.K)) {
          q = ((long long)s * sh.bs + t) * sh.K + k;
          const long long rows = seg_rows(p.ep_recv_count, d, LW, (e % sh.L) * W + s);
          if (p.bulk_ok && s != d && rows > 0) {
            if (p.plane_policy == MOE_PLANE_BULK_ALL) bulk = 1;
            else if (p.plane_policy == MOE_PLANE_RULE)
              bulk = rows * sh.row_in >= p.bulk_min_bytes && rows * den > remote[d];
          }
        }
      }
      if (q < 0) set_error(p.status, MOE_ERR_BAD_ASSIST);
    }
    const uint32_t m_sm = __ballot_sync(0xffffffffu, q >= 0 && !bulk);
    const uint32_t m_bk = __ballot_sync(0xffffffffu, q >= 0 && bulk);
    const long long row0 = (long long)d * sh.A + (long long)(b - bprefix[d]) * R;

    // store plane: the whole warp copies each row
    for (uint32_t m = m_sm; m; m &= m - 1) {
      const int i = __ffs(m) - 1;
      const long long qi = __shfl_sync(0xffffffffu, q, i);
      const uint8_t* src = eo + (row0 + i) * (long long)row_in;
      uint8_t* dst = win + qi * (long long)row_in;
      int v = lane;
      for (; v + 96 < nvec; v += 128) {
        const int4 a0 = ld_nc_v4(src + (size_t)v * 16), a1 = ld_nc_v4(src + (size_t)(v + 32) * 16);
        const int4 a2 = ld_nc_v4(src + (size_t)(v + 64) * 16), a3 = ld_nc_v4(src + (size_t)(v + 96) * 16);
        st_v4(dst + (size_t)v * 16, a0);
        st_v4(dst + (size_t)(v + 32) * 16, a1);
        st_v4(dst + (size_t)(v + 64) * 16, a2);
        st_v4(dst + (size_t)(v + 96) * 16, a3);
      }
      for (; v < nvec; v += 32) st_v4(dst + (size_t)v * 16, ld_nc_v4(src + (size_t)v * 16));
    }
    if (m_sm) {
      __threadfence();
      __syncwarp();
      if ((m_sm >> lane) & 1u) st_release_gpu(p.flags + q, epoch);
    }

    // bulk plane: lane 0 moves rows piecewise through the warp's two slots
    if (m_bk) {
      bool ok = true;
      for (uint32_t m = m_bk; m; m &= m - 1) {
        const int i = __ffs(m) - 1;
        const long long qi = __shfl_sync(0xffffffffu, q, i);
        if (lane == 0 && ok) {
          const uint8_t* src = eo + (row0 + i) * (long long)row_in;
          uint8_t* dst = win + qi * (long long)row_in;
          for (uint32_t off = 0; off < row_in && ok; off += kTpSlot) {
            const uint32_t bytes = row_in - off < (uint32_t)kTpSlot ? row_in - off : (uint32_t)kTpSlot;
            const int sl = (int)((uses[0] + uses[1]) & 1u);
            bulk_wait_read<1>();  // the copy that last read this slot has finished reading
            mbar_arrive_expect_tx(&bars[warp][sl], bytes);
            bulk_g2s(slots + sl * kTpSlot, src + off, bytes, &bars[warp][sl]);
            ok = mbar_wait_bounded(&bars[warp][sl], uses[sl] & 1u, p.status, p.timeout_ns);
            uses[sl] += 1;
            if (ok) {
              bulk_s2g(dst + off, slots + sl * kTpSlot, bytes);
              bulk_commit();
            }
          }
        }
      }
      if (lane == 0) {
        bulk_wait_all<0>();          // payload complete ...
        fence_proxy_async_global();  // ... and ordered before the generic-proxy flags
        __threadfence();
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      // flags of the bulk rows, after lane 0 saw their copies complete
      if (ok && ((m_bk >> lane) & 1u)) st_release_gpu(p.flags + q, epoch);
    }
  }

  // ---------------------------------------------------------- phase 2: reduce
  if (!p.put_only) {
    const int chunks = (nvec + 32 * kTpVpl - 1) / (32 * kTpVpl);
    const long long n_items = (long long)W * sh.bs * chunks;
    for (long long item = gwarp; item < n_items; item += nwarps) {
      const size_t tau = (size_t)(item / chunks);
      const int c = (int)(item % chunks);
      const uint8_t* src = nullptr;
      uint32_t w = 0;
      if (lane < sh.K) {
        const size_t pk = tau * sh.K + lane;
        w = reinterpret_cast<const uint32_t*>(p.scales)[pk];
        const int cls = classify_pick(p.ids, p.mask, sh, tau, lane);
        if (cls >= 0) {
          // the page: the source waits until every top-k status of its token is ready
          bool ready = ld_acquire_gpu(p.flags + pk) == epoch;
          if (!ready) {
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t it = 0; !ready; ++it) {
              ready = ld_acquire_gpu(p.flags + pk) == epoch;
              if (!ready && (it & 63u) == 63u && globaltimer_ns() - t0 > p.timeout_ns) {
                set_error(p.status, MOE_ERR_TIMEOUT);
                break;
              }
            }
          }
          if (ready) src = win + pk * (size_t)row_in;
        } else if (cls == kPickCopy) {
          src = static_cast<const uint8_t*>(p.x) + tau * (size_t)row_in;
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
      uint8_t* out = static_cast<uint8_t*>(p.x_out) + tau * (size_t)row_in;
      for (int i = 0; i < kTpVpl; ++i) {
        const int v = c * 32 * kTpVpl + i * 32 + lane;
        if (v >= nvec) break;
        const size_t off = (size_t)v * 16;
        if constexpr (DT == MOE_I32) {
          uint32_t acc[4] = {0u, 0u, 0u, 0u};
          for (int j = 0; j < n; ++j) {
            const int4 y = ld_v4(s_src[warp][j] + off);
            const uint32_t ww = s_w[warp][j];
            acc[0] += ww * (uint32_t)y.x;
            acc[1] += ww * (uint32_t)y.y;
            acc[2] += ww * (uint32_t)y.z;
            acc[3] += ww * (uint32_t)y.w;
          }
          st_v4(out + off, make_int4((int)acc[0], (int)acc[1], (int)acc[2], (int)acc[3]));
        } else {
          float acc[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = 0.f;
          for (int j = 0; j < n; j += 4) {
            int4 y[4];
#pragma unroll
            for (int g = 0; g < 4; ++g)
              if (j + g < n) y[g] = ld_v4(s_src[warp][j + g] + off);
#pragma unroll
            for (int g = 0; g < 4; ++g)
              if (j + g < n) fma16<DT>(acc, __uint_as_float(s_w[warp][j + g]), y[g]);
          }
          st_v4(out + off, pack16<DT>(acc));
        }
      }
      __syncwarp();
    }
  }

  // the last CTA publishes the epoch for the next call
  if (lane == 0) bulk_wait_all<0>();
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atomicAdd(&p.hdr->tp_done, 1u);
    s_last = prev == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last && tid == 0) {
    p.hdr->epoch = epoch;
    p.hdr->tp_done = 0;
    __threadfence();
  }
}

static size_t two_phase_smem(const Shape& sh) {
  return (size_t)kTpWarps * 2 * kTpSlot + (size_t)((sh.W + 2) & ~1) * sizeof(int) + (size_t)sh.W * 8 + 16;
}

cudaError_t launch_combine_two_phase(const CombineParams& p, cudaStream_t st, int num_sms) {
  const Shape& sh = p.sh;
  if (sh.row_in % 16 != 0) return cudaErrorNotSupported;  // 16-byte rows only
  const size_t smem = two_phase_smem(sh);
  void (*kern)(CombineParams) = sh.x_dtype == MOE_I32   ? two_phase_kernel<MOE_I32>
                                : sh.x_dtype == MOE_F16 ? two_phase_kernel<MOE_F16>
                                                        : two_phase_kernel<MOE_BF16>;
  int per_sm = 0;
  const cudaError_t e = resident_blocks((const void*)kern, kTpThreads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // rows per warp batch: up to 32 (one per lane), fewer when the call has
  // fewer picks than 32 per warp, so that every warp gets rows to move
  CombineParams q = p;
  const long long picks = (long long)sh.W * sh.bs * sh.K;
  const long long warps = (long long)num_sms * per_sm * kTpWarps;
  q.tp_rows = 32;
  while (q.tp_rows > 1 && picks < (long long)q.tp_rows * warps) q.tp_rows >>= 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(num_sms * per_sm);
  cfg.blockDim = dim3(kTpThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, q);
}

}  // namespace crs
