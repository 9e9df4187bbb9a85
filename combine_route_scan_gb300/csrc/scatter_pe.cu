// Dispatch payload for the quantisations with per-expert smoothing whose
// scale depends on the data (aclnnMoeDistributeDispatchV4, 参数说明 quantMode 2
// and 3 with scalesOptional of shape (moeExpertNum, H), 约束说明
// quantMode相关约束): every pick's row is quantised with the scales row of its
// own expert e, x' = x * s[e], then
//   quantMode 2 (per-token int8): scale = amax(|x'|) / 127 over the row,
//               q = clamp(round(x' / scale), -127, 127);
//   quantMode 3 (per-group FP8):  scale_g = amax_g / FMAX per 128 elements,
//               q = fp8_satfinite_rne(x' / scale_g).
//
// Expert-major, so that an expert's scales row is read once per run of its
// rows instead of once per pick:
//   * pe_rowmap_kernel (one warp per token) gives every routed pick its flat
//     receive row d*A + base + rank and writes the row's metadata (assist_info,
//     expand_scales, the pick -> row map); it also lists the receive rows of
//     all ranks back to back (rank 0's valid rows, then rank 1's, ...) as
//     {flat row, token, expert, plane} entries;
//   * scatter_pe_kernel (persistent) gives each CTA a contiguous run of that
//     list: rows of one expert follow each other, so each quantising thread
//     keeps its part of the current expert's scales row in registers and
//     reloads it only when the expert changes. A producer warp reads the list
//     (256-entry chunks by TMA bulk loads, two buffers) and stages token rows
//     in a 4-slot ring of TMA bulk loads, each slot with its clamped list entry
//     beside it; the quantising warps take one row at a time, keep v = x * s
//     as fp32 pairs and write 8 code bytes per 16-byte input vector to global
//     memory (store plane) or into a shared buffer that leaves by a TMA bulk
//     copy (bulk plane). Per-token int8: thread tid takes vectors
//     tid + m * nthreads (m < 4), neighbouring threads adjacent; the row
//     maximum crosses the one CTA barrier a row (a warp maximum by redux.sync
//     on the bits of non-negative floats, whose unsigned order is their
//     numeric order). Per-group FP8: thread tid takes the 32 elements
//     32 tid .. 32 tid + 31, a quarter of a 128-element group, so a group's
//     maximum takes two shuffles and its codes leave as 16-byte stores, for
//     a store-plane row before the row's barrier (they need no other warp's
//     values). The barrier a row frees the ring slot. The producer warp also writes the
//     dynamic scales (so that one warp, not every lane, carries those
//     divisions) and publishes ready flags and times.
//
// Codes from two bracketing reciprocals. From the row's (or group's) maximum
// a, r = F / a with F = 127 or FMAX (the hardware's approximate reciprocal and
// one Newton step) is within 3 * 2^-24 of 1/scale, so rh = r * (1 + 2^-21)
// and rl = r * (1 - 2^-21), rounded once, lie above and below 1/scale by a
// factor of more than 1 + 2^-24, and v * rh and v * rl bracket the IEEE
// quotient Q = fl(v / scale). Rounding to an integer (int8: an FMA with
// 1.5 * 2^23, exact product, one rounding, the code in the low byte) and the
// FP8 conversion are monotone, so where both ends give the same code, Q
// gives it too. An all-zero row or group has zero codes. A thread whose
// vectors hold an element the bracket leaves undecided (a half-integer or
// FP8 midpoint within the bracket: about one warp-row in fifty at random
// data) or whose maximum lies outside [2^-100, 2^100] stores the bracket's
// codes and queues itself; after the CTA's last row (and its bulk copies)
// the warps recompute the queued threads' vectors from global memory with
// the IEEE division and overwrite them, and only then publish those rows'
// ready flags. When the queue is full, every row from the first one that
// did not fit is recomputed whole. The divisions stay out of the quantising
// loop: measured on GB300 at 16 ranks x 256 tokens, h 7168, per-token int8
// took 154 us with the division fallback called from the loop and 143 us
// with it inlined there, against 119 us queued. Inputs are finite (NaN
// elements give unspecified codes here).
//
// The token-major kernel of scatter_quant.cu keeps static int8 with
// per-expert scales: measured on GB300 at 16 ranks x 256 tokens, h 7168, it
// ran slower in an expert-major form (124 vs 104 us).
#include <algorithm>

#include "quant_common.cuh"

namespace crs {

constexpr int kPeMaxThreads = 480;  // quantising threads; with the producer warp, 512
constexpr int kPeVpt = 4;           // 16-byte vectors a thread: rows of up to 15360 elements
constexpr int kPeStages = 4;        // staged token rows
constexpr int kPeChunk = 256;       // list entries per chunk
constexpr int kPeMaxWarps = 16;     // quantising warps, rounded up to whole float4 reads
constexpr int kPeMaxGroups = kPeVpt * kPeMaxThreads * 8 / 128;  // 120
constexpr int kPeFixCap = 256;      // queued threads a CTA before the remaining rows are recomputed whole
constexpr float kBracketHi = 1.0f + 0x1p-21f;
constexpr float kBracketLo = 1.0f - 0x1p-21f;
// the bracket argument holds for maxima in [2^-100, 2^100]: the scale, its
// reciprocal and every product stay normal and finite
constexpr float kFastMin = 0x1p-100f;
constexpr float kFastMax = 0x1p100f;

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

// ---------------------------------------------------------------- helpers

// A thread's part (its vectors vidx[m]) of an expert's scales row, as fp32
// pairs (all loads at once); zero for vectors past the row's end, whose
// products (x * 0, or NaN from a non-finite x) every maximum below ignores
// and no store writes.
__device__ __forceinline__ void pe_load_scales(const float* srow, const uint32_t (&vidx)[kPeVpt], const bool (&vok)[kPeVpt],
                                               f32x2 (&s)[kPeVpt][4]) {
#pragma unroll
  for (int m = 0; m < kPeVpt; ++m) {
    const uint32_t vi = vidx[m];
    if (vok[m]) {
      const ulonglong2 a = __ldg(reinterpret_cast<const ulonglong2*>(srow) + 2 * vi);
      const ulonglong2 b = __ldg(reinterpret_cast<const ulonglong2*>(srow) + 2 * vi + 1);
      s[m][0] = a.x;
      s[m][1] = a.y;
      s[m][2] = b.x;
      s[m][3] = b.y;
    } else {
      s[m][0] = s[m][1] = s[m][2] = s[m][3] = 0ull;
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

// 16 code bytes of vectors vi, vi + 1 (vi even).
template <bool TO_SMEM>
__device__ __forceinline__ void put16(uint8_t* q, uint32_t vi, uint2 a, uint2 b) {
  if (TO_SMEM) {
    *reinterpret_cast<uint4*>(q + vi * 8) = make_uint4(a.x, a.y, b.x, b.y);
  } else {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(q + vi * 8), "r"(a.x), "r"(a.y), "r"(b.x), "r"(b.y)
                 : "memory");
  }
}

// 1/s from the hardware's approximate reciprocal (at most one unit in the
// last place off, per the PTX ISA); s is normal and at most 2^100 where the
// result is used, so neither s nor 1/s is flushed.
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// The maximum of non-negative floats over the warp: their bit patterns order
// as unsigned integers the way the values do.
__device__ __forceinline__ float warp_max_nonneg(float m) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(__float_as_uint(m)));
  return __uint_as_float(r);
}

// The bracketing reciprocals (rh, rl) of scale = a / F from the maximum a:
// the approximate reciprocal and one Newton step give 1/a within about half
// an ulp, so r = F / a is within 3 * 2^-24 of 1/scale and rh, rl (rounded
// once) lie beyond 1/scale by a factor of more than 1 + (2^-21 - 4 * 2^-24).
__device__ __forceinline__ void pe_brackets(float a, float F, f32x2& rh2, f32x2& rl2) {
  const float r0 = rcp_approx(a);
  const float r1 = __fmaf_rn(r0, __fmaf_rn(-a, r0, 1.0f), r0);
  const float r = __fmul_rn(F, r1);
  const float rh = __fmul_rn(r, kBracketHi), rl = __fmul_rn(r, kBracketLo);
  rh2 = f2_pack(rh, rh);
  rl2 = f2_pack(rl, rl);
}
__device__ __forceinline__ bool pe_fast(float a) { return a >= kFastMin && a <= kFastMax; }

// Per-token int8 codes of one vector, branch-free: t = fl(v * r + 1.5 * 2^23)
// holds round-to-nearest-even(v * r) in its low mantissa bits (|v * r| < 128),
// so the code is its low byte; the return value is non-zero where the two
// brackets disagree.
__device__ __forceinline__ uint32_t pe_int8_codes(const f32x2 (&v)[4], f32x2 rh2, f32x2 rl2, uint2& out) {
  const f32x2 shift2 = f2_pack(kRoundShift, kRoundShift);
  uint32_t c[8];
  uint32_t diff = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a, b, x, y;
    f2_split(f2_fma(v[i], rh2, shift2), a, b);
    f2_split(f2_fma(v[i], rl2, shift2), x, y);
    c[2 * i] = __float_as_uint(a);
    c[2 * i + 1] = __float_as_uint(b);
    diff |= (__float_as_uint(a) ^ __float_as_uint(x)) | (__float_as_uint(b) ^ __float_as_uint(y));
  }
  out = pack8_low(c);
  return diff;
}

// Per-group FP8 codes of one vector, branch-free, as above.
template <int YT>
__device__ __forceinline__ uint32_t pe_fp8_codes(const f32x2 (&v)[4], f32x2 rh2, f32x2 rl2, uint2& out) {
  uint32_t c[4];
  uint32_t diff = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a, b, x, y;
    f2_split(f2_mul(v[i], rh2), a, b);
    f2_split(f2_mul(v[i], rl2), x, y);
    c[i] = cvt_fp8x2<YT>(a, b);
    diff |= c[i] ^ cvt_fp8x2<YT>(x, y);
  }
  out = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  return diff;
}

// A row's clamped list entry {flat row, token, expert, plane}.
__device__ __forceinline__ int4 pe_entry(const ScatterParams& p, const int4* list, long long li) {
  int4 en = list[li];
  en.x = min(max(en.x, 0), (int)(p.sh.W * p.sh.A) - 1);
  en.y = min(max(en.y, 0), p.sh.W * p.sh.bs - 1);
  en.z = min(max(en.z, 0), p.sh.E - 1);
  return en;
}

// The exact code of element k of the row (x row xrow, scales row srow) from
// the row's or group's maximum a, through the IEEE division.
template <int MODE, int DT, int YT>
__device__ __forceinline__ uint8_t pe_exact_code(const void* xrow, const float* srow, int k, float a) {
  constexpr float kF = MODE == 2 ? 127.0f : (YT == MOE_Y_FP8_E4M3 ? 448.0f : 57344.0f);
  if (a == 0.f) return 0;
  const float v = __fmul_rn(load_elem(xrow, k, DT), srow[k]);
  const float scale = __fdiv_rn(a, kF);
  return (uint8_t)(MODE == 2 ? (uint32_t)token_q(v, scale) : cvt_fp8x2<YT>(__fdiv_rn(v, scale), 0.f));
}

// The maximum of |x * s| over elements [k0, k1) of a row, by one warp.
template <int DT>
__device__ __forceinline__ float pe_warp_amax(const void* xrow, const float* srow, int k0, int k1) {
  float a = 0.f;
  for (int k = k0 + (int)(threadIdx.x & 31); k < k1; k += 32)
    a = fmaxf(a, fabsf(__fmul_rn(load_elem(xrow, k, DT), srow[k])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
}

// One warp: the exact codes of quantising thread tf's 32 elements (a lane
// each) of the row with entry en, in global memory: per-token int8, vectors
// tf + m * nthr with the row's maximum amax; per-group FP8, vectors 4 tf ..
// 4 tf + 3 with their group's maximum again (max is order-free, so it equals
// the quantising warps').
template <int MODE, int DT, int YT>
__device__ __noinline__ void pe_fix_thread(const ScatterParams& p, int4 en, int tf, int nthr, float amax) {
  const int lane = threadIdx.x & 31;
  const int h = p.sh.h;
  const void* xrow = static_cast<const uint8_t*>(p.x) + (size_t)en.y * p.sh.row_in;
  const float* srow = p.qscales + (size_t)en.z * h;
  uint8_t* q = static_cast<uint8_t*>(p.expand_x) + (long long)en.x * p.sh.row_out;
  float a = amax;
  int k;
  if (MODE == 2) {
    k = (tf + (lane >> 3) * nthr) * 8 + (lane & 7);  // vectors tf + m * nthr, a lane an element
  } else {
    // elements 32 tf .. 32 tf + 31, one 128-element group: its maximum first
    k = 32 * tf + lane;
    const int g0 = (tf >> 2) * 128;
    float xv[4], sv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kg = g0 + lane * 4 + j;
      xv[j] = kg < h ? load_elem(xrow, kg, DT) : 0.f;
      sv[j] = kg < h ? srow[kg] : 0.f;
    }
    a = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) a = fmaxf(a, fabsf(__fmul_rn(xv[j], sv[j])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  }
  if (k < h) q[k] = pe_exact_code<MODE, DT, YT>(xrow, srow, k, a);
}

// One warp: the exact codes of every element of the row with entry en.
template <int MODE, int DT, int YT>
__device__ __noinline__ void pe_fix_row(const ScatterParams& p, int4 en) {
  const int lane = threadIdx.x & 31;
  const int h = p.sh.h;
  const void* xrow = static_cast<const uint8_t*>(p.x) + (size_t)en.y * p.sh.row_in;
  const float* srow = p.qscales + (size_t)en.z * h;
  uint8_t* q = static_cast<uint8_t*>(p.expand_x) + (long long)en.x * p.sh.row_out;
  const int span = MODE == 2 ? h : 128;  // the elements one maximum covers
  for (int k0 = 0; k0 < h; k0 += span) {
    const int k1 = min(k0 + span, h);
    const float a = pe_warp_amax<DT>(xrow, srow, k0, k1);
    for (int k = k0 + lane; k < k1; k += 32) q[k] = pe_exact_code<MODE, DT, YT>(xrow, srow, k, a);
  }
}

// Queues quantising thread tid of row i (row maximum amax for per-token int8)
// for its exact codes after the last row; an entry past the capacity marks
// the first such row instead, from which every row is recomputed.
__device__ __forceinline__ void pe_queue(int4* q, int* nq, int* ovf, int* rowfix, int i, int tid, float amax) {
  const int k = atomicAdd(nq, 1);
  if (k < kPeFixCap)
    q[k] = make_int4(i, tid, __float_as_int(amax), 0);
  else
    atomicMin(ovf, i);
  *rowfix = 1;
}

// ---------------------------------------------------------------- payload

// MODE: quantMode 2 or 3; DT: MOE_F16 / MOE_BF16; YT: MOE_Y_* of the output.
// Warps 0 .. nw-1 quantise (nthr = 32 * nw threads); the last warp is the
// producer: its lane 0 reads the list and issues the row loads and bulk
// stores, publishes ready flags and times, and the warp writes the dynamic
// scales and the exact codes of queued threads, so that the quantising warps
// carry equal work and no division between barriers.
template <int MODE, int DT, int YT>
__global__ void __launch_bounds__(kPeMaxThreads + 32, 1) scatter_pe_kernel(ScatterParams p, const int4* list) {
  extern __shared__ __align__(128) uint8_t smem[];  // [kPeStages][slot_in] token rows, [2][slot_out] bulk rows
  __shared__ __align__(16) int4 s_list[2][kPeChunk];
  __shared__ __align__(16) int4 s_desc[kPeStages];          // the clamped list entry of each staged row
  __shared__ __align__(16) float s_part[2][kPeMaxWarps];    // per-token int8: warp maxima, by row parity
  __shared__ float s_gm[MODE == 3 ? 4 : 1][kPeMaxGroups];   // per-group FP8: group maxima, by row % 4
  __shared__ __align__(16) int4 s_fixq[kPeFixCap];         // queued threads: {row, thread, row maximum}
  __shared__ int s_nfix;                                    // entries queued (may exceed the capacity)
  __shared__ int s_ovf;                                     // the first row whose entry did not fit
  __shared__ int s_rowfix[4];                               // the row (by row % 4) queued a thread
  __shared__ __align__(8) uint64_t full_bar[kPeStages];
  __shared__ __align__(8) uint64_t list_bar[2];
  __shared__ int s_abort;  // written anywhere, read only right after a CTA barrier

  const Shape sh = p.sh;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x - 32;  // quantising threads
  const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
  const bool producer = warp == nw;
  const bool leader = tid == nthr;  // lane 0 of the producer warp
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
  constexpr float kF = MODE == 2 ? 127.0f : (YT == MOE_Y_FP8_E4M3 ? 448.0f : 57344.0f);

  if (leader) {
    for (int i = 0; i < kPeStages; ++i) mbar_init(&full_bar[i], 1);
    mbar_init(&list_bar[0], 1);
    mbar_init(&list_bar[1], 1);
    mbar_fence_init();
    s_abort = 0;
    s_nfix = 0;
    s_ovf = 0x7fffffff;
    s_rowfix[0] = s_rowfix[1] = s_rowfix[2] = s_rowfix[3] = 0;
  }
  if (tid < kPeStages) s_desc[tid] = make_int4(0, 0, 0, 0);  // in range even if a wait times out
  if (tid < 2 * kPeMaxWarps) (&s_part[0][0])[tid] = 0.f;
  __syncthreads();
  pdl_wait();  // the row list and the metadata of the row map are visible from here on
  pdl_launch_dependents();
  if (p.perf && leader) perf_begin(p);

  // this CTA's run [lo, hi) of the list
  const long long N = (long long)p.hdr->pe_rows;
  const long long lo = N * blockIdx.x / gridDim.x, hi = N * (blockIdx.x + 1) / gridDim.x;
  const int n = (int)(hi - lo);
  const int nchunks = (n + kPeChunk - 1) / kPeChunk;
  auto chunk_phase = [&](int c) { return (uint32_t)(c >> 1) & 1u; };
  auto load_chunk = [&](int c) {  // leader
    const int rows = min(kPeChunk, n - c * kPeChunk);
    mbar_arrive_expect_tx(&list_bar[c & 1], (uint32_t)rows * 16u);
    bulk_g2s(&s_list[c & 1][0], list + lo + (long long)c * kPeChunk, (uint32_t)rows * 16u, &list_bar[c & 1]);
  };
  // leader, once the chunk of row i has landed: the row's list entry, clamped
  // into range (a timed-out wait may leave a stale one behind; its row is
  // then never stored), beside the row's slot, then the row itself
  auto load_row = [&](int i) {
    const int st = i % kPeStages;
    int4 en = s_list[(i / kPeChunk) & 1][i % kPeChunk];
    en.x = min(max(en.x, 0), n_rows - 1);
    en.y = min(max(en.y, 0), n_tok - 1);
    en.z = min(max(en.z, 0), sh.E - 1);
    s_desc[st] = en;
    mbar_arrive_expect_tx(&full_bar[st], row_in);  // releases the entry to the slot's waiters
    bulk_g2s(xin + st * slot_in, x + (size_t)en.y * row_in, row_in, &full_bar[st]);
  };
  if (leader && n > 0) {
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

  // a quantising thread's vectors of a row: per-token int8, tid + m * nthr
  // (neighbouring threads adjacent); per-group FP8, the four vectors 4 tid ..
  // 4 tid + 3 (a quarter of a group), their halves taken in swapped order by
  // every other pair of threads so that a warp's 16-byte shared loads fall on
  // at most two threads a bank group. One past the row's end reads the row's
  // first vector instead.
  uint32_t vidx[kPeVpt];
  bool vok[kPeVpt];
  uint32_t xo[kPeVpt];
#pragma unroll
  for (int m = 0; m < kPeVpt; ++m) {
    vidx[m] = MODE == 2 ? (uint32_t)(tid + m * nthr) : (uint32_t)(4 * tid) + ((uint32_t)m ^ ((uint32_t)tid & 2u));
    vok[m] = !producer && vidx[m] < nvec;
    xo[m] = vok[m] ? vidx[m] * 16u : 0u;
  }

  // per-group FP8: the codes of one row from its products v, to q (the row in
  // global memory, or the shared buffer of a bulk row)
  auto fp8_row = [&](int i, uint8_t* q, bool bulk, const f32x2 (&v)[kPeVpt][4]) {
    // a 128-element group is 4 neighbouring threads: the maximum over this
    // thread's 32 elements, then two shuffles
    float gm = 0.f;
#pragma unroll
    for (int m = 0; m < kPeVpt; ++m) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float a, b;
        f2_split(v[m][k], a, b);
        gm = fmax_abs3(gm, a, b);
      }
    }
    gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 1));
    gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 2));
    if ((tid & 3) == 0 && vok[0]) s_gm[i & 3][tid >> 2] = gm;
    f32x2 rh2, rl2;
    pe_brackets(gm, kF, rh2, rl2);
    uint2 c[kPeVpt];
    uint32_t diff = 0;
#pragma unroll
    for (int m = 0; m < kPeVpt; ++m) {
      const uint32_t d = pe_fp8_codes<YT>(v[m], rh2, rl2, c[m]);
      diff |= vok[m] ? d : 0u;
    }
    if (!pe_fast(gm) || diff != 0u) {  // rare: zero codes for an all-zero group, else recomputed after the last row
      if (gm == 0.f) {
#pragma unroll
        for (int m = 0; m < kPeVpt; ++m) c[m] = make_uint2(0u, 0u);
      } else if (vok[0] || vok[2]) {  // the thread holds a vector of the row
        pe_queue(s_fixq, &s_nfix, &s_ovf, &s_rowfix[i & 3], i, tid, 0.f);
      }
    }
    // vectors vidx[2p], vidx[2p] + 1 are registers 2p, 2p + 1
#pragma unroll
    for (int m = 0; m < kPeVpt; m += 2) {
      if (vok[m + 1]) {
        if (bulk) put16<true>(q, vidx[m], c[m], c[m + 1]); else put16<false>(q, vidx[m], c[m], c[m + 1]);
      } else if (vok[m]) {
        if (bulk) put8<true>(q, vidx[m], c[m]); else put8<false>(q, vidx[m], c[m]);
      }
    }
  };
  f32x2 sc[kPeVpt][4];  // this thread's part of the scales row of expert cur_e
  int cur_e = -1;
  int nb = 0;         // rows through the shared buffers so far
  int4 pen = make_int4(0, 0, 0, 0);  // producer: the previous row's entry
  int st = 0;
  uint32_t phase = 0;
  for (int i = 0; i < n_run; ++i) {
    int4 en;
    f32x2 v[kPeVpt][4];
    if (!producer) {
      const bool landed = mbar_wait_bounded(&full_bar[st], phase, p.status, p.timeout_ns);
      if (!landed) s_abort = 1;
      en = s_desc[st];
      if (en.z != cur_e) {
        pe_load_scales(p.qscales + (size_t)en.z * sh.h, vidx, vok, sc);
        cur_e = en.z;
      }
      // v = x * s
      const uint8_t* row = xin + st * slot_in;
#pragma unroll
      for (int m = 0; m < kPeVpt; ++m) {
        f32x2 xp[4];
        unpack8x2<DT>(*reinterpret_cast<const int4*>(row + xo[m]), xp);
#pragma unroll
        for (int q = 0; q < 4; ++q) v[m][q] = f2_mul(xp[q], sc[m][q]);
      }
      if (MODE == 2) {
        float m0 = 0.f, m1 = 0.f;
#pragma unroll
        for (int m = 0; m < kPeVpt; ++m) {
#pragma unroll
          for (int q = 0; q < 4; q += 2) {
            float a0, a1, b0, b1;
            f2_split(v[m][q], a0, a1);
            f2_split(v[m][q + 1], b0, b1);
            m0 = fmax_abs3(m0, a0, a1);
            m1 = fmax_abs3(m1, b0, b1);
          }
        }
        const float wm = warp_max_nonneg(fmaxf(m0, m1));
        if (lane == 0) s_part[i & 1][warp] = wm;
      } else if (en.w == 0 && landed) {
        // per-group FP8, store plane: the codes need no other warp's values,
        // so they leave before the barrier (a row whose slot never landed is
        // not stored)
        fp8_row(i, out + (long long)en.x * row_out, false, v);
      }
    } else {
      en = s_desc[st];  // written by this warp's lane 0 rows ago
      // the bulk buffer this row uses was last read by the bulk copy two bulk rows back
      if (en.w != 0 && leader) bulk_wait_read<1>();
    }
    const bool bulk = en.w != 0;
    // row i's slot is read, every thread's stores of row i-1 (per-group FP8
    // store plane: of row i) are issued, the warp maxima of row i and the
    // group maxima and queue of row i-1 are visible
    __syncthreads();
    if (s_abort) break;
    const long long dst = en.x;
    uint8_t* q = bulk ? qbuf + (nb & 1) * slot_out : out + dst * row_out;
    float amax = 0.f;
    if (MODE == 2) {
#pragma unroll
      for (int k = 0; k < kPeMaxWarps / 4; ++k) {
        if (4 * k < nw) {
          const float4 a = reinterpret_cast<const float4*>(&s_part[i & 1][0])[k];
          amax = fmax_abs3(amax, a.x, a.y);
          amax = fmax_abs3(amax, a.z, a.w);
        }
      }
    }
    if (producer) {
      if (leader) {
        const int j = i + kPeStages;
        if (j < n) {
          if (j % kPeChunk != 0 ||
              mbar_wait_bounded(&list_bar[(j / kPeChunk) & 1], chunk_phase(j / kPeChunk), p.status, p.timeout_ns))
            load_row(j);
          else
            s_abort = 1;
        }
        // the last entry of a chunk has been read: refill its buffer
        if ((i + 1) % kPeChunk == 0 && i / kPeChunk + 2 < nchunks) load_chunk(i / kPeChunk + 2);
      }
      if (i >= 1) {
        // row i-1's ready flag and time, unless it queued a thread (then they
        // follow its exact codes after the last row)
        const bool later = s_rowfix[(i - 1) & 3] != 0 || i - 1 >= s_ovf;
        __syncwarp();
        if (lane == 0) s_rowfix[(i - 1) & 3] = 0;
        if (leader && !later) {
          if (p.seg_ready) {
            if (pen.w != 0) {
              bulk_wait_all<0>();
              fence_proxy_async_global();
            }
            __threadfence();
            publish_row(p, pen.z * sh.W + pen.y / sh.bs);
          }
          if (p.perf) perf_mark(p, (size_t)pen.y);
        }
        // the group scales of row i-1, from its group maxima
        if (MODE == 3) {
          for (int g = lane; g < nd; g += 32) dyn[(long long)pen.x * nd + g] = __fdiv_rn(s_gm[(i - 1) & 3][g], kF);
        }
      }
      if (MODE == 2 && leader) dyn[dst] = __fdiv_rn(amax, 127.0f);
      pen = en;
    } else if (MODE == 2) {
      f32x2 rh2, rl2;
      pe_brackets(amax, kF, rh2, rl2);
      uint2 c[kPeVpt];
      uint32_t diff = 0;
#pragma unroll
      for (int m = 0; m < kPeVpt; ++m) {
        const uint32_t d = pe_int8_codes(v[m], rh2, rl2, c[m]);
        diff |= vok[m] ? d : 0u;
      }
      if (amax == 0.f) {
#pragma unroll
        for (int m = 0; m < kPeVpt; ++m) c[m] = make_uint2(0u, 0u);
      } else if (!pe_fast(amax) || diff != 0u) {  // rare: recomputed exactly after the last row
        pe_queue(s_fixq, &s_nfix, &s_ovf, &s_rowfix[i & 3], i, tid, amax);
      }
      if (bulk) {
#pragma unroll
        for (int m = 0; m < kPeVpt; ++m)
          if (vok[m]) put8<true>(q, tid + m * nthr, c[m]);
      } else {
#pragma unroll
        for (int m = 0; m < kPeVpt; ++m)
          if (vok[m]) put8<false>(q, tid + m * nthr, c[m]);
      }
    } else if (bulk) {
      fp8_row(i, q, true, v);
    }
    if (bulk) {
      ++nb;
      fence_proxy_async_smem();
      __syncthreads();  // the row's codes and queue are in shared memory
      if (leader) {
        bulk_s2g(out + dst * row_out, q, row_out);
        bulk_commit();
      }
    }
    if (++st == kPeStages) {
      st = 0;
      phase ^= 1u;
    }
  }
  __syncthreads();  // every thread's stores of the last row are issued, its group maxima and queue visible
  const bool ran = n_run > 0 && !s_abort;
  if (producer && ran) {
    if (MODE == 3) {
      for (int g = lane; g < nd; g += 32) dyn[(long long)pen.x * nd + g] = __fdiv_rn(s_gm[(n_run - 1) & 3][g], kF);
    }
  }
  if (leader) {  // the bulk rows have landed: the exact codes below overwrite theirs
    bulk_wait_all<0>();
    fence_proxy_async_global();
  }
  __syncthreads();
  const int nq = min(s_nfix, kPeFixCap), ovf = s_ovf;
  const int nwarps = nw + 1;
  if (ran && nq > 0) {
    // the queued threads' exact codes, a warp an entry
    for (int k = warp; k < nq; k += nwarps) {
      const int4 f = s_fixq[k];
      if (f.x < ovf) pe_fix_thread<MODE, DT, YT>(p, pe_entry(p, list, lo + f.x), f.y, nthr, __int_as_float(f.z));
    }
    // the rows from the first one whose entry did not fit: every code again
    if (ovf < n_run) {
      for (int r = ovf + warp; r < n_run; r += nwarps) pe_fix_row<MODE, DT, YT>(p, pe_entry(p, list, lo + r));
    }
  }
  __syncthreads();  // every exact code is stored
  if (leader && ran) {
    // ready flags and times: the last row (unless queued), the queued rows
    // once each (a row's entries are adjacent), the rows from the overflow on
    auto publish = [&](const int4& en) {
      if (p.seg_ready) {
        fence_proxy_async_global();
        __threadfence();
        publish_row(p, en.z * sh.W + en.y / sh.bs);
      }
      if (p.perf) perf_mark(p, (size_t)en.y);
    };
    if (s_rowfix[(n_run - 1) & 3] == 0 && n_run - 1 < ovf) publish(pen);
    int last = -1;
    for (int k = 0; k < nq; ++k) {
      const int r = s_fixq[k].x;
      if (r != last && r < ovf) publish(pe_entry(p, list, lo + r));
      last = r;
    }
    for (int r = min(ovf, n_run); r < n_run; ++r) publish(pe_entry(p, list, lo + r));
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
  return (sh.quant == 2 || sh.quant == 3) && sh.scales_kind == MOE_SCALES_EXPERT && sh.row_in % 16 == 0 &&
         sh.row_out % 16 == 0 && sh.h / 8 <= kPeVpt * kPeMaxThreads && pe_smem(sh) <= 180 * 1024;
}

template <int MODE, int DT, int YT>
static cudaError_t launch_pe_t(const ScatterParams& p, const int4* list, cudaStream_t st, int num_sms) {
  const size_t smem = pe_smem(p.sh);
  // whole warps with kPeVpt vectors a thread where the row allows (7 warps at
  // h = 7168), and the producer warp
  const int nvec = p.sh.h / 8;
  const int threads = std::min(kPeMaxThreads, std::max(1, (nvec + 32 * kPeVpt - 1) / (32 * kPeVpt)) * 32) + 32;
  int per_sm = 0;
  const cudaError_t e = resident_blocks((const void*)scatter_pe_kernel<MODE, DT, YT>, threads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  PdlLaunch L(dim3(num_sms * per_sm), dim3(threads), smem, st);
  return cudaLaunchKernelEx(&L.cfg, scatter_pe_kernel<MODE, DT, YT>, p, list);
}

template <int DT>
static cudaError_t launch_pe_dt(const ScatterParams& p, const int4* list, cudaStream_t st, int num_sms) {
  if (p.sh.quant == 2) return launch_pe_t<2, DT, MOE_Y_DEFAULT>(p, list, st, num_sms);
  return p.sh.ytype == MOE_Y_FP8_E4M3 ? launch_pe_t<3, DT, MOE_Y_FP8_E4M3>(p, list, st, num_sms)
                                      : launch_pe_t<3, DT, MOE_Y_FP8_E5M2>(p, list, st, num_sms);
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
