// Dispatch payload for per-group FP8 quantisation with per-expert smoothing
// (aclnnMoeDistributeDispatchV4, 参数说明 quantMode 3 and scalesOptional of
// shape (moeExpertNum, H), 约束说明 quantMode相关约束): every pick's row is
// quantised with the scales row of its own expert e,
//   x' = x * s[e], per 128-element group scale_g = amax_g / FMAX,
//   q = fp8_satfinite_rne(x' / scale_g).
//
// Expert-major, so that an expert's scales row is read once per run of its
// rows instead of once per pick:
//   * pe_rowmap_kernel (one warp per token) gives every routed pick its flat
//     receive row d*A + base + rank and writes the row's metadata (assist_info,
//     expand_scales, the pick -> row map); it also lists the receive rows of
//     all ranks back to back (rank 0's valid rows, then rank 1's, ...) as
//     {flat row, token, expert, plane} entries;
//   * scatter_pe_kernel (persistent) gives each CTA a contiguous run of that
//     list: rows of one expert follow each other, so each thread keeps its part
//     of the current expert's scales row in registers and reloads it only when
//     the expert changes. The list arrives in 256-entry chunks by TMA bulk
//     loads (two buffers), token rows by a 4-slot ring of TMA bulk loads, and
//     the CTA quantises one row at a time: thread tid takes vectors tid,
//     tid + nthreads (kPeVpt of them), keeps v = x * s as fp32 pairs, and writes
//     8 code bytes per vector, neighbouring threads adjacent (store plane), or
//     into a shared buffer that leaves by a TMA bulk copy (bulk plane). A
//     128-element group is 16 neighbouring lanes of one vector slot; its
//     maximum takes four shuffles and no CTA barrier.
// Codes through an approximate reciprocal r of scale_g (at most one fp32 unit
// in the last place off): y = v * r is within 1.5 * 2^-23 |q| of the exact
// quotient q and the IEEE quotient within 2^-24 |q|, so the two are less than
// 4 fp32 units in the last place apart and give the same FP8 code unless y
// lies within 16 units of a midpoint of two neighbouring codes (the fp32 bits
// below the format's mantissa within 16 of one half) or below the format's
// smallest normal; a vector with such an element takes the division.
// Inputs are finite (NaN elements give unspecified codes on this path).
//
// The token-major kernel of scatter_quant.cu keeps the other per-expert modes
// (static int8, per-token int8): measured on GB300 at 16 ranks x 256 tokens,
// h 7168, they ran slower in this form (per-token int8 192 vs 168 us, static
// int8 124 vs 104 us), per-group FP8 faster (184 vs 207 us).
#include <algorithm>

#include "quant_common.cuh"

namespace crs {

constexpr int kPeMaxThreads = 512;
constexpr int kPeVpt = 2;      // 16-byte vectors a thread: rows of up to 8192 elements
constexpr int kPeStages = 4;   // staged token rows
constexpr int kPeChunk = 256;  // list entries per chunk

// ---------------------------------------------------------------- row map

// One warp per token; lanes < K hold its picks. The running row offsets of the
// ranks (rank d's valid rows start at entry prefix[d] of the list) come from
// ep_recv_count, scanned by every CTA into shared memory.
__global__ void __launch_bounds__(256) pe_rowmap_kernel(ScatterParams p, const int32_t* ep, int4* list) {
  extern __shared__ __align__(16) int32_t s_prefix[];  // [W]
  __shared__ long long s_scan[32];
  const Shape sh = p.sh;
  const int LW = sh.L * sh.W;
  pdl_wait();
  pdl_launch_dependents();
  // prefix over ranks of the valid row counts (each thread a contiguous run)
  {
    const int per = (sh.W + 255) / 256;
    const int d0 = min(sh.W, (int)threadIdx.x * per), d1 = min(sh.W, d0 + per);
    long long local = 0;
    for (int d = d0; d < d1; ++d) local += min((long long)ep[(size_t)d * LW + LW - 1], (long long)sh.A);
    long long run = block_exclusive_scan(local, s_scan);
    for (int d = d0; d < d1; ++d) {
      s_prefix[d] = (int32_t)run;
      run += min((long long)ep[(size_t)d * LW + LW - 1], (long long)sh.A);
    }
    if (blockIdx.x == 0 && (int)threadIdx.x == 255) p.hdr->pe_rows = (uint32_t)run;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long n_tok = (long long)sh.W * sh.bs;
  const long long wstep = (long long)gridDim.x * 8;
  for (long long tau = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); tau < n_tok; tau += wstep) {
    if (lane >= sh.K) continue;
    const size_t pk = (size_t)tau * sh.K + lane;
    const int r = p.rank[pk];
    const int e = p.ids[pk];
    if (r < 0 || !MOE_IN_BOUNDS(p.status, e, sh.E)) continue;
    const int s = (int)(tau / sh.bs), t = (int)(tau % sh.bs);
    const int d = e / sh.L;
    const size_t g = (size_t)e * sh.W + s;
    const long long row = (long long)p.base[g] + r;
    if (row >= sh.A) {
      set_error(p.status, MOE_ERR_CAPACITY);
      continue;
    }
    const long long dst = (long long)d * sh.A + row;
    if (p.inv) p.inv[pk] = (int32_t)dst;
    int32_t* a = p.assist + dst * 3;
    a[0] = s;
    a[1] = t;
    a[2] = lane;
    if (p.expand_scales)
      reinterpret_cast<uint32_t*>(p.expand_scales)[dst] = reinterpret_cast<const uint32_t*>(p.scales)[pk];
    const long long li = (long long)s_prefix[d] + row;
    if (MOE_IN_BOUNDS(p.status, li, (long long)sh.W * sh.A))
      list[li] = make_int4((int)dst, (int)tau, e, (int)p.plane[g]);
  }
}

// ---------------------------------------------------------------- scales

// A thread's part of an expert's scales row, as fp32 pairs (all loads at once).
template <int VPT>
__device__ __forceinline__ void pe_load_scales(const float* srow, uint32_t nvec, f32x2 (&s)[VPT][4]) {
#pragma unroll
  for (int m = 0; m < VPT; ++m) {
    const uint32_t vi = threadIdx.x + m * blockDim.x;
    if (vi < nvec) {
      const ulonglong2 a = __ldg(reinterpret_cast<const ulonglong2*>(srow) + 2 * vi);
      const ulonglong2 b = __ldg(reinterpret_cast<const ulonglong2*>(srow) + 2 * vi + 1);
      s[m][0] = a.x;
      s[m][1] = a.y;
      s[m][2] = b.x;
      s[m][3] = b.y;
    }
  }
}

// 8 code bytes of vector vi: to global memory (store plane) or to the shared
// buffer of a bulk copy.
template <bool TO_SMEM>
__device__ __forceinline__ void put8(uint8_t* q, uint32_t vi, uint2 c) {
  if (TO_SMEM) {
    *reinterpret_cast<uint2*>(q + vi * 8) = c;
  } else {
    asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(q + vi * 8), "r"(c.x), "r"(c.y) : "memory");
  }
}

// 1/s from the hardware's approximate reciprocal (at most one unit in the
// last place off, per the PTX ISA): the reciprocal forms below only need
// y = v * r within a few fp32 units of the quotient, which their margins cover.
// s is normal and at most 2^121, so neither s nor 1/s is flushed.
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// The codes of one 8-element vector through the IEEE division: the rare
// vectors the reciprocal form leaves undecided, out of line so that the main
// path carries none of its instructions.
template <int YT>
__device__ __noinline__ uint2 fp8_codes_div(f32x2 v0, f32x2 v1, f32x2 v2, f32x2 v3, float scale, float gm) {
  const f32x2 v[4] = {v0, v1, v2, v3};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo, hi;
    f2_split(v[i], lo, hi);
    c[i] = gm == 0.f ? 0u : cvt_fp8x2<YT>(__fdiv_rn(lo, scale), __fdiv_rn(hi, scale));
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// Codes and group scales of one row from its products v.
template <int YT, bool TO_SMEM>
__device__ __forceinline__ void pe_codes(const f32x2 (&v)[kPeVpt][4], uint32_t nvec, int nthr, uint8_t* q,
                                         float* dyn_row) {
  const int tid = threadIdx.x;
  constexpr float kFmax = YT == MOE_Y_FP8_E4M3 ? 448.0f : 57344.0f;
  // fp32 bits below the FP8 mantissa (20 for E4M3, 21 for E5M2) without
  // their low 5, and their pattern at a midpoint after adding 16
  constexpr uint32_t kMidMask = YT == MOE_Y_FP8_E4M3 ? 0xFFFE0u : 0x1FFFE0u;
  constexpr uint32_t kMidHalf = YT == MOE_Y_FP8_E4M3 ? 0x80000u : 0x100000u;
  constexpr float kMinNormal = YT == MOE_Y_FP8_E4M3 ? 0.015625f : 6.103515625e-05f;  // 2^-6, 2^-14
#pragma unroll
  for (int m = 0; m < kPeVpt; ++m) {
    const uint32_t vi = tid + m * nthr;
    // a 128-element group is 16 neighbouring lanes of slot m
    float gm = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo, hi;
      f2_split(v[m][i], lo, hi);
      gm = fmax_abs3(gm, lo, hi);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
    if (vi >= nvec) continue;
    const float scale = __fdiv_rn(gm, kFmax);
    const bool fast = scale >= 1.17549435e-38f && scale <= 3.40282347e38f;
    const float r = rcp_approx(scale);
    const f32x2 rcp2 = f2_pack(r, r);
    uint32_t c[4];
    float ymin = 3.40282347e38f;
    bool near = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float yl, yh;
      f2_split(f2_mul(v[m][i], rcp2), yl, yh);
      c[i] = cvt_fp8x2<YT>(yl, yh);
      ymin = fmin_abs3(ymin, yl, yh);
      near |= ((__float_as_uint(yl) + 16u) & kMidMask) == kMidHalf;
      near |= ((__float_as_uint(yh) + 16u) & kMidMask) == kMidHalf;
    }
    uint2 w = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    if (!(fast && !near && ymin >= kMinNormal)) w = fp8_codes_div<YT>(v[m][0], v[m][1], v[m][2], v[m][3], scale, gm);
    put8<TO_SMEM>(q, vi, w);
    if ((vi & 15u) == 0) dyn_row[vi >> 4] = scale;
  }
}

// ---------------------------------------------------------------- payload

template <int DT, int YT>
__global__ void __launch_bounds__(kPeMaxThreads, 2) scatter_pe_kernel(ScatterParams p, const int4* list) {
  extern __shared__ __align__(128) uint8_t smem[];  // [kPeStages][slot_in] token rows, [2][slot_out] bulk rows
  __shared__ __align__(16) int4 s_list[2][kPeChunk];
  __shared__ __align__(8) uint64_t full_bar[kPeStages];
  __shared__ __align__(8) uint64_t list_bar[2];
  __shared__ int s_abort;  // written anywhere, read only right after a CTA barrier

  const Shape sh = p.sh;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const uint32_t row_in = (uint32_t)sh.row_in, row_out = (uint32_t)sh.row_out;
  const uint32_t slot_in = (uint32_t)align128(row_in), slot_out = (uint32_t)align128(row_out);
  uint8_t* xin = smem;
  uint8_t* qbuf = smem + kPeStages * slot_in;
  const uint8_t* x = static_cast<const uint8_t*>(p.x);
  uint8_t* out = static_cast<uint8_t*>(p.expand_x);
  float* dyn = static_cast<float*>(p.dyn_scales);
  const uint32_t nvec = (uint32_t)sh.h / 8;
  const int nd = sh.ngroups;
  const int n_tok = sh.W * sh.bs;           // < 2^31 (host check)
  const int n_rows = (int)(sh.W * sh.A);    // < 2^31 (host check)

  if (tid == 0) {
    for (int i = 0; i < kPeStages; ++i) mbar_init(&full_bar[i], 1);
    mbar_init(&list_bar[0], 1);
    mbar_init(&list_bar[1], 1);
    mbar_fence_init();
    s_abort = 0;
  }
  __syncthreads();
  pdl_wait();  // the row list and the metadata of the row map are visible from here on
  pdl_launch_dependents();
  if (p.perf && tid == 0) perf_begin(p);

  // this CTA's run [lo, hi) of the list
  const long long N = (long long)p.hdr->pe_rows;
  const long long lo = N * blockIdx.x / gridDim.x, hi = N * (blockIdx.x + 1) / gridDim.x;
  const int n = (int)(hi - lo);
  const int nchunks = (n + kPeChunk - 1) / kPeChunk;
  auto chunk_phase = [&](int c) { return (uint32_t)(c >> 1) & 1u; };
  auto load_chunk = [&](int c) {  // thread 0
    const int rows = min(kPeChunk, n - c * kPeChunk);
    mbar_arrive_expect_tx(&list_bar[c & 1], (uint32_t)rows * 16u);
    bulk_g2s(&s_list[c & 1][0], list + lo + (long long)c * kPeChunk, (uint32_t)rows * 16u, &list_bar[c & 1]);
  };
  // an entry of the list, clamped into range (a timed-out wait may leave a
  // stale one behind; its row is then never stored)
  auto entry = [&](int i) {
    int4 en = s_list[(i / kPeChunk) & 1][i % kPeChunk];
    en.x = min(max(en.x, 0), n_rows - 1);
    en.y = min(max(en.y, 0), n_tok - 1);
    en.z = min(max(en.z, 0), sh.E - 1);
    return en;
  };
  auto load_row = [&](int i) {  // thread 0, once the chunk of row i has landed
    const int st = i % kPeStages;
    mbar_arrive_expect_tx(&full_bar[st], row_in);
    bulk_g2s(xin + st * slot_in, x + (size_t)entry(i).y * row_in, row_in, &full_bar[st]);
  };
  if (tid == 0 && n > 0) {
    load_chunk(0);
    if (nchunks > 1) load_chunk(1);
    if (mbar_wait_bounded(&list_bar[0], 0u, p.status, p.timeout_ns)) {
      for (int i = 0; i < kPeStages && i < n; ++i) load_row(i);
    } else {
      s_abort = 1;
    }
  }
  __syncthreads();
  const int n_run = s_abort ? 0 : n;  // no row when the first chunk never landed

  // this thread's vectors tid + m * nthr of a row
  bool vok[kPeVpt];
#pragma unroll
  for (int m = 0; m < kPeVpt; ++m) vok[m] = (uint32_t)(tid + m * nthr) < nvec;
  const uint32_t xoff = (uint32_t)tid * 16u, xstep = (uint32_t)nthr * 16u;

  f32x2 sc[kPeVpt][4];  // this thread's part of the scales row of expert cur_e
  int cur_e = -1;
  int nb = 0;  // rows through the shared buffers so far
  int prev_seg = -1, prev_tau = -1;
  bool prev_bulk = false;
  int st = 0;
  uint32_t phase = 0;
  for (int i = 0; i < n_run; ++i) {
    bool ok = true;
    if (i % kPeChunk == 0)
      ok = mbar_wait_bounded(&list_bar[(i / kPeChunk) & 1], chunk_phase(i / kPeChunk), p.status, p.timeout_ns);
    if (ok) ok = mbar_wait_bounded(&full_bar[st], phase, p.status, p.timeout_ns);
    if (!ok) s_abort = 1;
    const int4 en = entry(i);
    const int e = en.z;
    const bool bulk = en.w != 0;
    if (e != cur_e) {
      pe_load_scales<kPeVpt>(p.qscales + (size_t)e * sh.h, nvec, sc);
      cur_e = e;
    }
    // v = x * s
    const uint8_t* row = xin + st * slot_in + xoff;
    f32x2 v[kPeVpt][4];
#pragma unroll
    for (int m = 0; m < kPeVpt; ++m) {
      if (vok[m]) {
        f32x2 xp[4];
        unpack8x2<DT>(*reinterpret_cast<const int4*>(row + m * xstep), xp);
#pragma unroll
        for (int q = 0; q < 4; ++q) v[m][q] = f2_mul(xp[q], sc[m][q]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) v[m][q] = 0ull;
      }
    }
    // the bulk buffer this row uses was last read by the bulk copy two bulk rows back
    if (bulk && tid == 0) bulk_wait_read<1>();
    // row i's slot is read and every thread's stores of row i-1 are issued
    __syncthreads();
    if (s_abort) break;
    if (tid == 0) {
      const int j = i + kPeStages;
      if (j < n) {
        if (j % kPeChunk != 0 ||
            mbar_wait_bounded(&list_bar[(j / kPeChunk) & 1], chunk_phase(j / kPeChunk), p.status, p.timeout_ns))
          load_row(j);
        else
          s_abort = 1;
      }
      // the last entry of a chunk has been read by everyone: refill its buffer
      if ((i + 1) % kPeChunk == 0 && i / kPeChunk + 2 < nchunks) load_chunk(i / kPeChunk + 2);
      if (i >= 1) {
        if (p.seg_ready) {
          if (prev_bulk) {
            bulk_wait_all<0>();
            fence_proxy_async_global();
          }
          __threadfence();
          publish_row(p, prev_seg);
        }
        if (p.perf) perf_mark(p, (size_t)prev_tau);
      }
    }
    const long long dst = en.x;
    float* dyn_row = dyn + dst * nd;
    if (!bulk) {
      pe_codes<YT, false>(v, nvec, nthr, out + dst * row_out, dyn_row);
    } else {
      uint8_t* qb = qbuf + (nb & 1) * slot_out;
      ++nb;
      pe_codes<YT, true>(v, nvec, nthr, qb, dyn_row);
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        bulk_s2g(out + dst * row_out, qb, row_out);
        bulk_commit();
      }
    }
    if (tid == 0 && (p.seg_ready || p.perf)) {
      prev_seg = e * sh.W + en.y / sh.bs;
      prev_tau = en.y;
      prev_bulk = bulk;
    }
    if (++st == kPeStages) {
      st = 0;
      phase ^= 1u;
    }
  }
  __syncthreads();  // every thread's stores of the last row are issued
  if (tid == 0) {
    bulk_wait_all<0>();
    if (prev_seg >= 0 && !s_abort) {
      if (p.seg_ready) {
        fence_proxy_async_global();
        __threadfence();
        publish_row(p, prev_seg);
      }
      if (p.perf) perf_mark(p, (size_t)prev_tau);
    }
  }
  if (p.perf) {
    __shared__ int s_last;
    perf_finish(p, &s_last);
  }
}

static size_t pe_smem(const Shape& sh) {
  return kPeStages * align128((size_t)sh.row_in) + 2 * align128((size_t)sh.row_out);
}

bool uses_scatter_pe(const Shape& sh) {
  return sh.quant == 3 && sh.scales_kind == MOE_SCALES_EXPERT && sh.row_in % 16 == 0 &&
         sh.row_out % 16 == 0 && sh.h / 8 <= kPeVpt * kPeMaxThreads && pe_smem(sh) <= 180 * 1024;
}

template <int DT, int YT>
static cudaError_t launch_pe_t(const ScatterParams& p, const int4* list, cudaStream_t st, int num_sms) {
  const size_t smem = pe_smem(p.sh);
  // whole warps with kPeVpt vectors a thread where the row allows (14 warps at h = 7168)
  const int nvec = p.sh.h / 8;
  const int threads = std::min(kPeMaxThreads, std::max(1, (nvec + 32 * kPeVpt - 1) / (32 * kPeVpt)) * 32);
  int per_sm = 0;
  const cudaError_t e = resident_blocks((const void*)scatter_pe_kernel<DT, YT>, threads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  PdlLaunch L(dim3(num_sms * per_sm), dim3(threads), smem, st);
  return cudaLaunchKernelEx(&L.cfg, scatter_pe_kernel<DT, YT>, p, list);
}

template <int DT>
static cudaError_t launch_pe_dt(const ScatterParams& p, const int4* list, cudaStream_t st, int num_sms) {
  return p.sh.ytype == MOE_Y_FP8_E4M3 ? launch_pe_t<DT, MOE_Y_FP8_E4M3>(p, list, st, num_sms)
                                      : launch_pe_t<DT, MOE_Y_FP8_E5M2>(p, list, st, num_sms);
}

cudaError_t launch_scatter_pe(const ScatterParams& p, const int32_t* ep_recv_count, int4* list, cudaStream_t st,
                              int num_sms, int* launches) {
  const Shape& sh = p.sh;
  *launches = 0;
  const long long n_tok = (long long)sh.W * sh.bs;
  if (n_tok == 0) return cudaSuccess;
  if (p.hdr == nullptr) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>((n_tok + 7) / 8, (long long)num_sms * 8);  // a warp a token
  PdlLaunch L(dim3(grid), dim3(256), (size_t)sh.W * sizeof(int32_t), st);
  cudaError_t e = cudaLaunchKernelEx(&L.cfg, pe_rowmap_kernel, p, ep_recv_count, list);
  if (e != cudaSuccess) return e;
  *launches = 1;
  e = sh.x_dtype == MOE_F16 ? launch_pe_dt<MOE_F16>(p, list, st, num_sms) : launch_pe_dt<MOE_BF16>(p, list, st, num_sms);
  if (e == cudaSuccess) *launches = 2;
  return e;
}

}  // namespace crs
