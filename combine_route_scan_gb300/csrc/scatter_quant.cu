// Dispatch payload for the quantised modes of aclnnMoeDistributeDispatchV4
// (参数说明 quantMode / scalesOptional, 约束说明 quantMode相关约束) other than
// the unquantised copy of scatter.cu:
//   quantMode 1   static int8: q = clamp(rne(x * s), -128, 127), s of shape
//                 (1,), (h,) or (E, h) (the pick's expert's row);
//   quantMode 2   per-token int8, optionally after per-expert smoothing
//                 x' = x * s[e]: scale = amax / 127, q = clamp(rne(x' / scale), -127, 127);
//   quantMode 3   per-group FP8: groups of 128, scale_g = amax_g / FMAX,
//                 q = fp8(x' / scale_g), optional smoothing as for 2;
//   quantMode 4   MX (OCP Microscaling v1.0): blocks of 32 share the E8M0
//                 scale X = 2^(floor(log2 amax) - emax), q = x / X in FP8 E4M3,
//                 FP8 E5M2 or FP4 E2M1 (two codes a byte, even element low).
// Conversions are the sm_100-family cvt.rn.satfinite instructions (round to
// nearest even, saturating at the largest finite value).
//
// Same skeleton as the plain dispatch: persistent token-major CTAs, the source
// row staged in shared memory by a TMA bulk load, warp 0 building the
// destination list. A quantised row ("variant") is computed once per token,
// or once per pick when per-expert scales make every pick's row different.
// When no pick of it goes by bulk copies, each thread stores its codes straight
// from registers to every destination; otherwise the variant is written to one
// of two shared buffers and leaves by TMA bulk copies (bulk-plane segments)
// and 16-byte stores (store-plane segments). Each thread quantises 16-byte
// vectors of 8 elements; a 128-element group is 16 neighbouring lanes and a
// 32-element MX block 4, reduced with shuffles.
#include "quant_common.cuh"

namespace crs {

constexpr int kQStages = 2;  // staged source rows
constexpr int kQSlots = 2;   // quantised-row buffers: one is written while bulk copies read the other

// Rows of token i-1 are complete: warp 0 counts them toward their segments'
// flags, after lane 0 (which issued the bulk copies) saw them complete.
__device__ __forceinline__ void publish_token(const ScatterParams& p, const PickTable& a) {
  if ((threadIdx.x & 31) == 0) {
    bulk_wait_all<0>();
    fence_proxy_async_global();
  }
  __syncwarp();
  publish_rows_warp(p, a.sm_seg, a.n_sm);
  publish_rows_warp(p, a.bulk_seg, a.n_bulk);
}

// Where a quantised row goes: the shared buffers q (codes) and dq (dynamic
// scales) that bulk copies and 16-byte stores read afterwards, or
// straight from registers to the global destination rows dst[0..n), 8-byte
// stores (4 for FP4) coalesced across the warp.
struct RowSink {
  uint8_t* q;
  uint8_t* dq;
  const long long* dst;
  int n;
  uint8_t* out;
  uint8_t* dyn;
  uint32_t row_out;
  int nd;
};

// Per-token int8 with per-expert smoothing for one pick, by one warp: the
// maximum of |x * s[e]| over the row by the warp's shuffles (no CTA barrier,
// so the warps of a CTA quantise different picks at once), then the codes
// straight to the pick's row. Same arithmetic, same order-free maximum, same
// bytes as the CTA-wide form.
// MX FP8 with each 32-element block on a lane pair: a thread takes two
// 16-byte vectors (read in an order rotated by (lane / 4) % 2, so that the
// eight lanes of a shared-memory phase hit distinct banks), the pair's
// maximum comes from one shuffle, and the thread's 16 bytes of codes leave by
// one 16-byte store per destination, neighbouring threads adjacent. The even
// lane writes the block's E8M0 byte. Same arithmetic as the vector-per-thread
// form. Needs whole blocks (h a multiple of 32).
template <int DT, int YT>
__device__ __forceinline__ void quantize_mx8_half_blocks(const uint8_t* row, const RowSink& k, uint32_t nhalf) {
  const uint32_t rot = (threadIdx.x >> 2) & 1u;
  for (uint32_t base = 0; base < nhalf; base += kScatterThreads) {
    const uint32_t hb = base + threadIdx.x;
    const bool valid = hb < nhalf;  // nhalf is even: a pair is valid or not as a whole
    int4 raw[2] = {make_int4(0, 0, 0, 0), make_int4(0, 0, 0, 0)};  // raw[j] = vector 2hb + (j ^ rot)
    if (valid) {
#pragma unroll
      for (int j = 0; j < 2; ++j) raw[j] = *reinterpret_cast<const int4*>(row + (hb * 2 + (j ^ rot)) * 16);
    }
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float f[8];
      unpack8<DT>(raw[j], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    if (!valid) continue;
    const int se = mx_exponent(m, elem_emax(YT));
    const float inv = exp2_exact(-se);
    uint32_t w[4];  // w[2j], w[2j+1]: the codes of raw[j]
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float f[8];
      unpack8<DT>(raw[j], f);
      uint32_t c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] = cvt_fp8x2<YT>(__fmul_rn(f[2 * i], inv), __fmul_rn(f[2 * i + 1], inv));
      w[2 * j] = c[0] | (c[1] << 16);
      w[2 * j + 1] = c[2] | (c[3] << 16);
    }
    const int4 val = rot ? make_int4((int)w[2], (int)w[3], (int)w[0], (int)w[1])
                         : make_int4((int)w[0], (int)w[1], (int)w[2], (int)w[3]);
    for (int d = 0; d < k.n; ++d) {
      st_v4(k.out + k.dst[d] * k.row_out + hb * 16, val);
      if ((hb & 1u) == 0) k.dyn[k.dst[d] * k.nd + (hb >> 1)] = (uint8_t)(se + 127);
    }
  }
}

template <int DT>
__device__ __forceinline__ void quantize_pick_warp_mode2(const uint8_t* row, const float* srow, uint8_t* out,
                                                         uint8_t* dyn, long long dst, uint32_t row_out,
                                                         uint32_t nvec);

// SINK: kShared (the shared buffers), kOne (the single destination dst[0]),
// kMany (destinations dst[0..n)).
enum { kShared = 0, kOne = 1, kMany = 2 };

template <int SINK, typename V>
__device__ __forceinline__ void put(const RowSink& k, uint32_t off, V v) {
  if (SINK == kShared) {
    *reinterpret_cast<V*>(k.q + off) = v;
  } else if (SINK == kOne) {
    *reinterpret_cast<V*>(k.out + k.dst[0] * k.row_out + off) = v;
  } else {
    for (int b = 0; b < k.n; ++b) *reinterpret_cast<V*>(k.out + k.dst[b] * k.row_out + off) = v;
  }
}
template <int SINK, typename T>
__device__ __forceinline__ void put_dyn(const RowSink& k, int g, T v) {
  if (SINK == kShared) {
    reinterpret_cast<T*>(k.dq)[g] = v;
  } else if (SINK == kOne) {
    reinterpret_cast<T*>(k.dyn)[k.dst[0] * k.nd + g] = v;
  } else {
    for (int b = 0; b < k.n; ++b) reinterpret_cast<T*>(k.dyn)[k.dst[b] * k.nd + g] = v;
  }
}

// Per-token int8, first pass: the maximum of |x| (times srow when smoothing)
// over this thread's vectors of the row (the CTA's threads share them out),
// reduced over the warp; max is order-free, so any split gives the same value.
template <int DT>
__device__ __forceinline__ float token_amax_warp(const uint8_t* row, const float* srow, uint32_t nvec) {
  float m = 0.f;
  for (uint32_t v = threadIdx.x; v < nvec; v += kScatterThreads) {
    float f[8];
    unpack8<DT>(*reinterpret_cast<const int4*>(row + v * 16), f);
    if (srow) {
      float sc[8];
      load_scales8(srow, v, sc);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], sc[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// Per-token int8, second pass: scale = amax / 127 and the codes
// round(x / scale) clamped to [-127, 127] (all zeros for an all-zero row).
// RCP: through the reciprocal (token_code). Measured on GB300, it pays where
// the arithmetic bounds the kernel (per-expert smoothing: one quantisation a
// pick) and not on the per-token form, whose HBM traffic hides the divisions.
template <int SINK, int DT, bool RCP>
__device__ __forceinline__ void token_codes(const uint8_t* row, const float* srow, const RowSink& k, uint32_t nvec,
                                            float amax) {
  const float scale = __fdiv_rn(amax, 127.0f);
  const bool fast = RCP && token_rcp_ok(scale);
  const float rcp = fast ? __frcp_rn(scale) : 0.f;
  for (uint32_t v = threadIdx.x; v < nvec; v += kScatterThreads) {
    float f[8];
    unpack8<DT>(*reinterpret_cast<const int4*>(row + v * 16), f);
    if (srow) {
      float sc[8];
      load_scales8(srow, v, sc);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], sc[i]);
    }
    uint32_t c[8];
    if (fast) {
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = token_code(f[i], scale, rcp);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = amax == 0.f ? 0u : (uint32_t)token_q(f[i], scale);
    }
    put<SINK>(k, v * 8, pack8_low(c));
  }
  if (threadIdx.x == 0) put_dyn<SINK, float>(k, 0, scale);
}

// Quantises the staged row (elements times srow, or s0 for a (1,) coefficient)
// into the sink. Threads t0, t0 + nt, ... take the row's 16-byte vectors: the
// whole CTA (t0 = threadIdx.x, nt = the CTA size), or for modes 1 and 3, whose
// groups lie within a warp, one warp (t0 = its lane, nt = 32). Per-token int8
// is CTA-wide only: it reduces the row maximum through s_red with a barrier.
template <int MODE, int DT, int YT, int SINK>
__device__ __forceinline__ void quantize_variant(const uint8_t* row, const float* srow, float s0, const RowSink& k,
                                                 uint32_t nvec, float* s_red, int t0 = threadIdx.x,
                                                 int nt = kScatterThreads) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (MODE == 1) {
    for (uint32_t v = t0; v < nvec; v += nt) {
      float f[8], sc[8];
      unpack8<DT>(*reinterpret_cast<const int4*>(row + v * 16), f);
      if (srow) {
        load_scales8(srow, v, sc);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) sc[i] = s0;
      }
      int qv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] = static_q(__fmul_rn(f[i], sc[i]));
      put<SINK>(k, v * 8, pack8(qv));
    }
  } else if (MODE == 2) {
    const float m = token_amax_warp<DT>(row, srow, nvec);
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float amax = 0.f;
#pragma unroll
    for (int w = 0; w < kScatterWarps; ++w) amax = fmaxf(amax, s_red[w]);
    token_codes<SINK, DT, true>(row, srow, k, nvec, amax);
  } else {
    // a group (mode 3: 16 vectors) or block (mode 4: 4 vectors) is a run of
    // neighbouring lanes; every lane of a warp takes part in the shuffles,
    // past-the-end lanes with zeros
    constexpr int kLanes = MODE == 3 ? 16 : 4;
    for (uint32_t base = 0; base < nvec; base += nt) {
      const uint32_t v = base + t0;
      const bool valid = v < nvec;
      float f[8];
      if (valid) {
        unpack8<DT>(*reinterpret_cast<const int4*>(row + v * 16), f);
        if (srow) {
          float sc[8];
          load_scales8(srow, v, sc);
#pragma unroll
          for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], sc[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
#pragma unroll
      for (int o = kLanes / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (MODE == 3) {
        const float scale = __fdiv_rn(m, fp8_max(YT));
        if (valid) {
          uint32_t c[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            c[i] = m == 0.f ? 0u : cvt_fp8x2<YT>(__fdiv_rn(f[2 * i], scale), __fdiv_rn(f[2 * i + 1], scale));
          put<SINK>(k, v * 8, make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16)));
          if ((v & 15u) == 0) put_dyn<SINK, float>(k, (int)(v >> 4), scale);
        }
      } else {
        const int se = mx_exponent(m, elem_emax(YT));
        const float inv = exp2_exact(-se);
        if (valid) {
          uint32_t c[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) c[i] = cvt_y_pair(YT, __fmul_rn(f[2 * i], inv), __fmul_rn(f[2 * i + 1], inv));
          if (YT == MOE_Y_FP4_E2M1)
            put<SINK>(k, v * 4, c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24));
          else
            put<SINK>(k, v * 8, make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16)));
          if ((v & 3u) == 0) put_dyn<SINK, uint8_t>(k, (int)(v >> 2), (uint8_t)(se + 127));
        }
      }
    }
  }
}

// int8 codes straight to every destination of k, two neighbouring 16-byte
// vectors a thread (read in an order rotated by (lane / 4) % 2, so that the
// eight lanes of a shared-memory phase hit distinct banks) and one 16-byte
// store per destination, neighbouring threads adjacent. codes8(f, v) gives
// the 8 code bytes of vector v from its elements f. nvec must be even.
template <int DT, typename Codes8>
__device__ __forceinline__ void int8_codes_pairs(const uint8_t* row, const RowSink& k, uint32_t nvec,
                                                 Codes8 codes8) {
  const uint32_t rot = (threadIdx.x >> 2) & 1u;
  for (uint32_t pv = threadIdx.x; pv < nvec / 2; pv += kScatterThreads) {
    const uint32_t va = 2 * pv + rot, vb = 2 * pv + (rot ^ 1u);
    float f[8];
    unpack8<DT>(*reinterpret_cast<const int4*>(row + va * 16), f);
    const uint2 ca = codes8(f, va);
    unpack8<DT>(*reinterpret_cast<const int4*>(row + vb * 16), f);
    const uint2 cb = codes8(f, vb);
    const int4 val = rot ? make_int4((int)cb.x, (int)cb.y, (int)ca.x, (int)ca.y)
                         : make_int4((int)ca.x, (int)ca.y, (int)cb.x, (int)cb.y);
    for (int d = 0; d < k.n; ++d) st_v4(k.out + k.dst[d] * k.row_out + pv * 16, val);
  }
}

// Per-group FP8 with two neighbouring vectors a thread (read in an order
// rotated by (lane / 4) % 2 for distinct shared-memory banks): a 128-element
// group lies on 8 aligned lanes, its maximum comes from three shuffles, the
// thread's 16 bytes of codes leave by one 16-byte store per destination and
// the group's first lane writes its fp32 scale. Past-the-end lanes take part
// in the shuffles with zeros. Same arithmetic as the vector-a-thread form.
// nvec must be even.
template <int DT, int YT>
__device__ __forceinline__ void quantize_group_fp8_pairs(const uint8_t* row, const RowSink& k, uint32_t nvec) {
  const uint32_t rot = (threadIdx.x >> 2) & 1u;
  const uint32_t npair = nvec / 2;
  for (uint32_t base = 0; base < npair; base += kScatterThreads) {
    const uint32_t pv = base + threadIdx.x;
    const bool valid = pv < npair;
    float fa[8], fb[8];  // vectors 2pv + rot and 2pv + (rot ^ 1)
    if (valid) {
      unpack8<DT>(*reinterpret_cast<const int4*>(row + (2 * pv + rot) * 16), fa);
      unpack8<DT>(*reinterpret_cast<const int4*>(row + (2 * pv + (rot ^ 1u)) * 16), fb);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) fa[i] = fb[i] = 0.f;
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(fa[i]), fabsf(fb[i])));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (!valid) continue;
    const float scale = __fdiv_rn(m, fp8_max(YT));
    uint32_t ca[4], cb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ca[i] = m == 0.f ? 0u : cvt_fp8x2<YT>(__fdiv_rn(fa[2 * i], scale), __fdiv_rn(fa[2 * i + 1], scale));
      cb[i] = m == 0.f ? 0u : cvt_fp8x2<YT>(__fdiv_rn(fb[2 * i], scale), __fdiv_rn(fb[2 * i + 1], scale));
    }
    const uint32_t a0 = ca[0] | (ca[1] << 16), a1 = ca[2] | (ca[3] << 16);
    const uint32_t b0 = cb[0] | (cb[1] << 16), b1 = cb[2] | (cb[3] << 16);
    const int4 val = rot ? make_int4((int)b0, (int)b1, (int)a0, (int)a1) : make_int4((int)a0, (int)a1, (int)b0, (int)b1);
    for (int d = 0; d < k.n; ++d) {
      st_v4(k.out + k.dst[d] * k.row_out + pv * 16, val);
      if ((pv & 7u) == 0) reinterpret_cast<float*>(k.dyn)[k.dst[d] * k.nd + (pv >> 3)] = scale;
    }
  }
}

// MX FP4 with each 32-element block in one thread: its four 16-byte vectors
// are read from the staged row (in an order rotated by (lane / 2) % 4, so
// that the eight lanes of a shared-memory phase hit distinct banks), the
// block maximum gives the E8M0 exponent, and the 16 bytes of codes leave by
// one 16-byte store per destination, neighbouring threads' blocks adjacent.
// Same arithmetic, element by element, as the vector-per-thread form.
template <int DT>
__device__ __forceinline__ void quantize_fp4_blocks(const uint8_t* row, const RowSink& k, uint32_t nblk) {
  const uint32_t rot = (threadIdx.x >> 1) & 3u;
  for (uint32_t b = threadIdx.x; b < nblk; b += kScatterThreads) {
    int4 raw[4];  // raw[j] = vector 4b + ((j + rot) & 3)
#pragma unroll
    for (int j = 0; j < 4; ++j) raw[j] = *reinterpret_cast<const int4*>(row + (b * 4 + ((j + rot) & 3u)) * 16);
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float f[8];
      unpack8<DT>(raw[j], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    }
    const int se = mx_exponent(m, elem_emax(MOE_Y_FP4_E2M1));
    const float inv = exp2_exact(-se);
    uint32_t w[4];  // w[j]: the codes of raw[j]
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float f[8];
      unpack8<DT>(raw[j], f);
      uint32_t c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] = cvt_fp4x2(__fmul_rn(f[2 * i], inv), __fmul_rn(f[2 * i + 1], inv));
      w[j] = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
    }
    // back to vector order: word v holds w[(v - rot) & 3]
    if (rot & 1u) {
      const uint32_t t = w[3];
      w[3] = w[2]; w[2] = w[1]; w[1] = w[0]; w[0] = t;
    }
    if (rot & 2u) {
      uint32_t t = w[0]; w[0] = w[2]; w[2] = t;
      t = w[1]; w[1] = w[3]; w[3] = t;
    }
    const int4 val = make_int4((int)w[0], (int)w[1], (int)w[2], (int)w[3]);
    for (int d = 0; d < k.n; ++d) {
      st_v4(k.out + k.dst[d] * k.row_out + b * 16, val);
      k.dyn[k.dst[d] * k.nd + b] = (uint8_t)(se + 127);
    }
  }
}

template <int DT>
__device__ __forceinline__ void quantize_pick_warp_mode2(const uint8_t* row, const float* srow, uint8_t* out,
                                                         uint8_t* dyn, long long dst, uint32_t row_out,
                                                         uint32_t nvec) {
  const int lane = threadIdx.x & 31;
  // products v = x * s as fp32 pairs (packed multiplies), x from the staged
  // row and s from the expert's scales row, recomputed in the second pass
  auto products = [&](uint32_t v, f32x2 (&p)[4]) {
    f32x2 xp[4];
    unpack8x2<DT>(*reinterpret_cast<const int4*>(row + v * 16), xp);
    const ulonglong2 a = __ldg(reinterpret_cast<const ulonglong2*>(srow) + 2 * v);
    const ulonglong2 b = __ldg(reinterpret_cast<const ulonglong2*>(srow) + 2 * v + 1);
    p[0] = f2_mul(xp[0], a.x);
    p[1] = f2_mul(xp[1], a.y);
    p[2] = f2_mul(xp[2], b.x);
    p[3] = f2_mul(xp[3], b.y);
  };
  float m0 = 0.f, m1 = 0.f;
  for (uint32_t v = lane; v < nvec; v += 32) {
    f32x2 p[4];
    products(v, p);
    float a0, a1, b0, b1;
    f2_split(p[0], a0, a1);
    f2_split(p[1], b0, b1);
    m0 = fmax_abs3(m0, a0, a1);
    m1 = fmax_abs3(m1, b0, b1);
    f2_split(p[2], a0, a1);
    f2_split(p[3], b0, b1);
    m0 = fmax_abs3(m0, a0, a1);
    m1 = fmax_abs3(m1, b0, b1);
  }
  float m = fmaxf(m0, m1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float scale = __fdiv_rn(m, 127.0f);
  const bool fast = token_rcp_ok(scale);
  const float rcp = fast ? __frcp_rn(scale) : 0.f;
  const f32x2 rcp2 = f2_pack(rcp, rcp);
  uint8_t* q = out + dst * row_out;
  for (uint32_t v = lane; v < nvec; v += 32) {
    f32x2 p[4];
    products(v, p);
    *reinterpret_cast<uint2*>(q + v * 8) = token_codes8(p, scale, m, fast, rcp2);
  }
  if (lane == 0) reinterpret_cast<float*>(dyn)[dst] = scale;
}

// MODE: quantMode (1..4); DT: MOE_F16 / MOE_BF16; YT: MOE_Y_* of the output;
// PE: per-expert scales (every pick's row is different).
template <int MODE, int DT, int YT, bool PE>
__global__ void __launch_bounds__(kScatterThreads, (MODE == 2 || (MODE != 1 && !PE)) ? 5 : 0) scatter_quant_kernel(ScatterParams p) {
  MOE_PHASE_BEGIN(p, kPhaseScatter);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kQStages];
  __shared__ PickTable tabs[2];
  __shared__ float s_red[2][kScatterWarps];  // alternate by variant: a fast warp never overwrites a maximum still read
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
  const int my_n = (int)blockIdx.x < n_tok ? (n_tok - 1 - (int)blockIdx.x) / G + 1 : 0;
  const uint32_t row_in = (uint32_t)sh.row_in, row_out = (uint32_t)sh.row_out;
  const size_t slot_in = align128(row_in), slot_out = align128(row_out);
  const size_t slot_dyn = align128((size_t)sh.ngroups * 4);
  uint8_t* xin = smem;
  uint8_t* qbuf = smem + kQStages * slot_in;
  uint8_t* dbuf = qbuf + kQSlots * slot_out;
  const uint8_t* x = static_cast<const uint8_t*>(p.x);
  uint8_t* out = static_cast<uint8_t*>(p.expand_x);
  uint8_t* dyn = static_cast<uint8_t*>(p.dyn_scales);
  const uint32_t nvec = (uint32_t)sh.h / 8;
  const int nd = sh.ngroups;
  const int dyn_es = MODE == 4 ? 1 : 4;  // bytes of one dynamic-scale entry
  const float s0 = (MODE == 1 && sh.scales_kind == MOE_SCALES_SCALAR) ? __ldg(p.qscales) : 1.f;
  const float* chan = (MODE == 1 && sh.scales_kind == MOE_SCALES_CHANNEL) ? p.qscales : nullptr;

  if (tid == 0) {
    for (int i = 0; i < kQStages; ++i) mbar_init(&full_bar[i], 1);
    mbar_fence_init();
    s_abort = 0;
  }
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < kQStages && i < my_n; ++i) {
      const size_t tau = blockIdx.x + (size_t)i * G;
      mbar_arrive_expect_tx(&full_bar[i], row_in);
      bulk_g2s(xin + i * slot_in, x + tau * row_in, row_in, &full_bar[i]);
    }
  }
  pdl_wait();  // routing results are visible from here on
  MOE_PHASE_PAST_WAIT();
  pdl_launch_dependents();
  if (p.perf && tid == 0) perf_begin(p);

  int nv = 0;   // variants through the shared buffers so far (selects the buffer)
  int nvr = 0;  // variants so far (selects the s_red half)
  // warp 0: the destination-list loads of token i (both levels) and i + 1
  // (first level), so that building a list never waits on memory. Measured on
  // GB300 for the per-token and per-block modes (the registers it takes are
  // capped at five CTAs per SM); the static-scale and per-expert forms,
  // whose tokens cost little or a great deal, keep loading on the spot.
  constexpr bool kAhead = MODE != 1 && !PE;
  // per-token int8 without smoothing: one CTA barrier a token (s_red
  // alternates by token: a half is written again only after the next token's
  // barrier, which every thread passes after reading it)
  constexpr bool kMerge = MODE == 2 && !PE;
  PickAhead cur{}, nxt{};
  if (kAhead && warp == 0 && my_n > 0) {
    pick_load_first(p, blockIdx.x, cur);
    if (my_n > 1) pick_load_first(p, blockIdx.x + (size_t)G, nxt);
    pick_load_second(p, (int)(blockIdx.x / sh.bs), cur);
  }
  for (int i = 0; i < my_n; ++i) {
    const size_t tau = blockIdx.x + (size_t)i * G;
    const int s = (int)(tau / sh.bs), t = (int)(tau % sh.bs);
    const int stage = i % kQStages;
    const uint32_t parity = (uint32_t)(i / kQStages) & 1u;
    PickTable& tab = tabs[i & 1];
    const uint8_t* row = xin + stage * slot_in;

    const bool ok = mbar_wait_bounded(&full_bar[stage], parity, p.status, p.timeout_ns);
    if (!ok) s_abort = 1;
    // the buffer of this token's first shared variant was last read by the
    // bulk group two variants back: at most one newer group may still read
    if (tid == 0) bulk_wait_read<1>();
    if constexpr (kMerge) {
      // per-token int8: the row maximum's first pass goes before the token's
      // barrier, which then publishes the warps' maxima with the pick table
      const float m = token_amax_warp<DT>(row, nullptr, nvec);
      if ((tid & 31) == 0) s_red[i & 1][warp] = m;
    }
    if (warp == 0) {
      if constexpr (kAhead) {
        build_picks_from(p, tau, s, t, tab, cur);
        PickAhead n2{};
        if (i + 1 < my_n) pick_load_second(p, (int)((tau + G) / sh.bs), nxt);
        if (i + 2 < my_n) pick_load_first(p, tau + 2 * (size_t)G, n2);
        cur = nxt;
        nxt = n2;
      } else {
        build_picks(p, tau, s, t, tab);
      }
    }
    __syncthreads();
    if (s_abort) break;
    if (p.seg_ready && warp == 0 && i >= 1) publish_token(p, tabs[(i - 1) & 1]);
    if (tid == 0 && i >= 1) {
      if (p.perf) perf_mark(p, tau - G);
      // the previous token's source slot is free: its reads were generic loads
      // that all finished before the barrier above
      const int nxt = i - 1 + kQStages;
      if (nxt < my_n) {
        const int ps = (i - 1) % kQStages;
        const size_t tn = blockIdx.x + (size_t)nxt * G;
        mbar_arrive_expect_tx(&full_bar[ps], row_in);
        bulk_g2s(xin + ps * slot_in, x + tn * row_in, row_in, &full_bar[ps]);
      }
    }
    const int nsm = tab.n_sm, nbk = tab.n_bulk;
    // Tokens with no bulk-plane pick store their codes straight from
    // registers. Measured on GB300: with a vector a thread (8-byte stores, 4
    // for FP4), FP4 and per-group rows leave faster through the shared buffer
    // as 16-byte stores; with 16-byte stores from registers they leave faster
    // still: MX rows of whole blocks with a block (FP4) or half a block (FP8)
    // a thread (direct4: FP4 47 -> 39 us, MX FP8 54 -> 52 us at the bench
    // shape), per-group FP8 rows with two vectors a thread (direct3: 57.5 ->
    // 53.3 us), per-token int8 rows likewise (53.2 -> 52.0 us; static int8
    // was 1% slower that way).
    const bool direct = nbk == 0 && YT != MOE_Y_FP4_E2M1 && MODE != 3;
    const bool direct4 = MODE == 4 && !PE && nbk == 0 && sh.h % 32 == 0;
    const bool direct3 = MODE == 3 && !PE && nbk == 0 && nvec % 2 == 0;
    float amax = 0.f;
    if constexpr (kMerge) {
#pragma unroll
      for (int w = 0; w < kScatterWarps; ++w) amax = fmaxf(amax, s_red[i & 1][w]);
    }

    // store-plane picks straight from registers: each pick on its own with
    // per-expert scales, else one pass for all of them when the token has no
    // bulk-plane pick (no shared buffer, no barrier)
    if constexpr (PE) {
      // one store-plane pick per warp (no CTA barrier; each lane keeps many
      // scales loads in flight)
      for (int j = warp; j < nsm; j += kScatterWarps) {
        const float* srow = p.qscales + (size_t)(tab.sm_seg[j] / sh.W) * sh.h;
        if constexpr (MODE == 2) {
          quantize_pick_warp_mode2<DT>(row, srow, out, dyn, tab.sm_dst[j], row_out, nvec);
        } else {
          const RowSink k{nullptr, nullptr, &tab.sm_dst[j], 1, out, dyn, row_out, nd};
          quantize_variant<MODE, DT, YT, kOne>(row, srow, s0, k, nvec, nullptr, tid & 31, 32);
        }
      }
    } else if (direct4) {
      if (nsm > 0) {
        const RowSink k{nullptr, nullptr, tab.sm_dst, nsm, out, dyn, row_out, nd};
        if constexpr (YT == MOE_Y_FP4_E2M1)
          quantize_fp4_blocks<DT>(row, k, (uint32_t)nd);
        else
          quantize_mx8_half_blocks<DT, YT>(row, k, (uint32_t)nd * 2);
      }
    } else if (direct3) {
      if (nsm > 0) {
        const RowSink k{nullptr, nullptr, tab.sm_dst, nsm, out, dyn, row_out, nd};
        quantize_group_fp8_pairs<DT, YT>(row, k, nvec);
      }
    } else if (direct && nsm > 0) {
      const RowSink k{nullptr, nullptr, tab.sm_dst, nsm, out, dyn, row_out, nd};
      if constexpr (kMerge) {
        if (nvec % 2 == 0) {
          const float scale = __fdiv_rn(amax, 127.0f);
          int8_codes_pairs<DT>(row, k, nvec, [&](const float(&f)[8], uint32_t) {
            int qv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) qv[i] = amax == 0.f ? 0 : token_q(f[i], scale);
            return pack8(qv);
          });
          if (tid == 0) put_dyn<kMany, float>(k, 0, scale);
        } else {
          token_codes<kMany, DT, false>(row, nullptr, k, nvec, amax);
        }
      } else {
        quantize_variant<MODE, DT, YT, kMany>(row, chan, s0, k, nvec, s_red[nvr++ & 1]);
      }
    }

    // variants through the shared buffers: one per bulk-plane pick (per-expert
    // scales), or one for all picks when some go by bulk copies
    const int j0 = PE ? nsm : 0;
    const int j1 = PE ? nsm + nbk : (!direct && !direct4 && !direct3 && nsm + nbk > 0 ? 1 : 0);
    for (int j = j0; j < j1; ++j) {
      const int qs = nv & 1;
      ++nv;
      uint8_t* q = qbuf + qs * slot_out;
      uint8_t* dq = dbuf + qs * slot_dyn;
      if (j > j0) {
        if (tid == 0) bulk_wait_read<1>();
        __syncthreads();
      }
      const float* srow = PE ? p.qscales + (size_t)(tab.bulk_seg[j - nsm] / sh.W) * sh.h : chan;
      const RowSink k{q, dq, nullptr, 0, out, dyn, row_out, nd};
      if constexpr (kMerge)
        token_codes<kShared, DT, false>(row, nullptr, k, nvec, amax);
      else
        quantize_variant<MODE, DT, YT, kShared>(row, srow, s0, k, nvec, s_red[nvr++ & 1]);
      fence_proxy_async_smem();
      __syncthreads();

      // destinations: the bulk pick (per-expert scales) or every pick
      const int bk0 = PE ? j - nsm : 0, bk1 = PE ? j - nsm + 1 : nbk;
      const int ns = PE ? 0 : nsm;
      if (tid == 0) {
        for (int b = bk0; b < bk1; ++b) bulk_s2g(out + tab.bulk_dst[b] * row_out, q, row_out);
        bulk_commit();
      }
      if (ns > 0) {
        for (uint32_t u = tid; u < row_out / 16; u += kScatterThreads) {
          const int4 val = *reinterpret_cast<const int4*>(q + u * 16);
          for (int b = 0; b < ns; ++b) st_v4(out + tab.sm_dst[b] * row_out + u * 16, val);
        }
      }
      if (MODE != 1) {
        const int ndst = ns + (bk1 - bk0);
        for (int idx = tid; idx < ndst * nd; idx += kScatterThreads) {
          const int b = idx / nd, g = idx % nd;
          const long long dst = b < ns ? tab.sm_dst[b] : tab.bulk_dst[bk0 + b - ns];
          if (dyn_es == 4)
            reinterpret_cast<float*>(dyn)[dst * nd + g] = reinterpret_cast<const float*>(dq)[g];
          else
            dyn[dst * nd + g] = dq[g];
        }
      }
    }
  }
  __syncthreads();  // every thread's stores of the last token are issued
  if (warp == 0 && !s_abort && my_n > 0) {
    if (p.seg_ready) publish_token(p, tabs[(my_n - 1) & 1]);
    if (tid == 0) {
      bulk_wait_all<0>();
      if (p.perf) perf_mark(p, blockIdx.x + (size_t)(my_n - 1) * G);
    }
  }
  if (tid == 0) bulk_wait_all<0>();
#ifdef MOE_FLAG_OBSERVER
  observer_producer_end(p);
#endif
  if (p.perf) {
    __shared__ int s_last;
    perf_finish(p, &s_last);
  }
}

// Rows that are not 16-byte multiples: element-wise, one token per CTA at a
// time, every row by plain stores. Groups / blocks go one per warp.
template <int MODE>
__global__ void __launch_bounds__(kScatterThreads) scatter_quant_plain_kernel(ScatterParams p) {
  __shared__ PickTable tab;
  __shared__ float s_red[kScatterWarps];
  const Shape sh = p.sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_tok = sh.W * sh.bs;
  const int h = sh.h, dt = sh.x_dtype, yt = sh.ytype;
  const bool pe = sh.scales_kind == MOE_SCALES_EXPERT;
  pdl_wait();
  pdl_launch_dependents();
  if (p.perf && tid == 0) perf_begin(p);
  for (size_t tau = blockIdx.x; tau < (size_t)n_tok; tau += gridDim.x) {
    const int s = (int)(tau / sh.bs), t = (int)(tau % sh.bs);
    if (warp == 0) {
      build_picks(p, tau, s, t, tab);
      __syncwarp();
      if (lane == 0) {  // both planes are carried by plain stores here
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
    const int nvar = pe ? ns : 1;
    const size_t xrow = tau * (size_t)h;
    for (int j = 0; j < nvar; ++j) {
      const int d0 = pe ? j : 0, d1 = pe ? j + 1 : ns;
      const float* srow = nullptr;
      float s0 = 1.f;
      if (pe) srow = p.qscales + (size_t)(tab.sm_seg[j] / sh.W) * h;
      else if (sh.scales_kind == MOE_SCALES_CHANNEL) srow = p.qscales;
      else if (sh.scales_kind == MOE_SCALES_SCALAR) s0 = p.qscales[0];
      auto elem = [&](int jx) {
        const float v = load_elem(p.x, xrow + jx, dt);
        return srow ? __fmul_rn(v, srow[jx]) : (sh.scales_kind == MOE_SCALES_SCALAR ? __fmul_rn(v, s0) : v);
      };
      if (MODE == 1) {
        int8_t* o = static_cast<int8_t*>(p.expand_x);
        for (int jx = tid; jx < h; jx += kScatterThreads) {
          const int8_t qv = (int8_t)static_q(elem(jx));
          for (int b = d0; b < d1; ++b) o[tab.sm_dst[b] * h + jx] = qv;
        }
      } else if (MODE == 2) {
        float m = 0.f;
        for (int jx = tid; jx < h; jx += kScatterThreads) m = fmaxf(m, fabsf(elem(jx)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) s_red[warp] = m;
        __syncthreads();
        float amax = 0.f;
        for (int w = 0; w < kScatterWarps; ++w) amax = fmaxf(amax, s_red[w]);
        const float scale = __fdiv_rn(amax, 127.0f);
        int8_t* o = static_cast<int8_t*>(p.expand_x);
        for (int jx = tid; jx < h; jx += kScatterThreads) {
          const int8_t qv = amax == 0.f ? (int8_t)0 : (int8_t)token_q(elem(jx), scale);
          for (int b = d0; b < d1; ++b) o[tab.sm_dst[b] * h + jx] = qv;
        }
        if (tid == 0)
          for (int b = d0; b < d1; ++b) static_cast<float*>(p.dyn_scales)[tab.sm_dst[b]] = scale;
        __syncthreads();  // s_red is reused by the next variant
      } else {
        const int gsz = MODE == 3 ? 128 : 32;
        const int ng = sh.ngroups;
        const bool fp4 = yt == MOE_Y_FP4_E2M1;
        const int rob = sh.row_out;
        uint8_t* o = static_cast<uint8_t*>(p.expand_x);
        for (int g = warp; g < ng; g += kScatterWarps) {
          const int j0 = g * gsz, j1 = min(h, j0 + gsz);
          float m = 0.f;
          for (int jx = j0 + lane; jx < j1; jx += 32) m = fmaxf(m, fabsf(elem(jx)));
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
          if (MODE == 3) {
            const float scale = __fdiv_rn(m, fp8_max(yt));
            for (int jx = j0 + lane; jx < j1; jx += 32) {
              const uint8_t c = m == 0.f ? (uint8_t)0
                                         : (uint8_t)(cvt_y_pair(yt, __fdiv_rn(elem(jx), scale), 0.f) & 0xffu);
              for (int b = d0; b < d1; ++b) o[tab.sm_dst[b] * rob + jx] = c;
            }
            if (lane == 0)
              for (int b = d0; b < d1; ++b) static_cast<float*>(p.dyn_scales)[tab.sm_dst[b] * ng + g] = scale;
          } else {
            const int se = mx_exponent(m, elem_emax(yt));
            const float inv = exp2_exact(-se);
            if (fp4) {
              for (int jp = j0 / 2 + lane; jp < j1 / 2; jp += 32) {
                const uint8_t c = (uint8_t)cvt_fp4x2(__fmul_rn(elem(2 * jp), inv), __fmul_rn(elem(2 * jp + 1), inv));
                for (int b = d0; b < d1; ++b) o[tab.sm_dst[b] * rob + jp] = c;
              }
            } else {
              for (int jx = j0 + lane; jx < j1; jx += 32) {
                const uint8_t c = (uint8_t)(cvt_y_pair(yt, __fmul_rn(elem(jx), inv), 0.f) & 0xffu);
                for (int b = d0; b < d1; ++b) o[tab.sm_dst[b] * rob + jx] = c;
              }
            }
            if (lane == 0)
              for (int b = d0; b < d1; ++b) static_cast<uint8_t*>(p.dyn_scales)[tab.sm_dst[b] * ng + g] = (uint8_t)(se + 127);
          }
        }
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

static size_t quant_smem(const Shape& sh) {
  return kQStages * align128((size_t)sh.row_in) + kQSlots * align128((size_t)sh.row_out) +
         kQSlots * align128((size_t)sh.ngroups * 4);
}

bool scatter_quant_tma_fits(const Shape& sh) { return quant_smem(sh) <= 200 * 1024; }

template <typename KernelT>
static cudaError_t launch_quant_persistent(KernelT kernel, const ScatterParams& p, cudaStream_t st, int num_sms) {
  const size_t smem = quant_smem(p.sh);
  int per_sm = 0;
  const cudaError_t e = resident_blocks((const void*)kernel, kScatterThreads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int n_tok = p.sh.W * p.sh.bs;
#ifdef MOE_FLAG_OBSERVER
  if (p.observe) return launch_observed(kernel, p, st, min(n_tok, num_sms * per_sm - 1) + 1, smem);
#endif
  const int grid = max(1, min(n_tok, num_sms * per_sm));
  PdlLaunch L(dim3(grid), dim3(kScatterThreads), smem, st);
  return cudaLaunchKernelEx(&L.cfg, kernel, p);
}

template <int DT>
static cudaError_t launch_quant_dt(const ScatterParams& p, cudaStream_t st, int nsm) {
  const Shape& sh = p.sh;
  const bool pe = sh.scales_kind == MOE_SCALES_EXPERT;
  switch (sh.quant) {
    case 1:
      return pe ? launch_quant_persistent(scatter_quant_kernel<1, DT, MOE_Y_DEFAULT, true>, p, st, nsm)
                : launch_quant_persistent(scatter_quant_kernel<1, DT, MOE_Y_DEFAULT, false>, p, st, nsm);
    case 2:
      return pe ? launch_quant_persistent(scatter_quant_kernel<2, DT, MOE_Y_DEFAULT, true>, p, st, nsm)
                : launch_quant_persistent(scatter_quant_kernel<2, DT, MOE_Y_DEFAULT, false>, p, st, nsm);
    case 3:
      if (sh.ytype == MOE_Y_FP8_E4M3)
        return pe ? launch_quant_persistent(scatter_quant_kernel<3, DT, MOE_Y_FP8_E4M3, true>, p, st, nsm)
                  : launch_quant_persistent(scatter_quant_kernel<3, DT, MOE_Y_FP8_E4M3, false>, p, st, nsm);
      return pe ? launch_quant_persistent(scatter_quant_kernel<3, DT, MOE_Y_FP8_E5M2, true>, p, st, nsm)
                : launch_quant_persistent(scatter_quant_kernel<3, DT, MOE_Y_FP8_E5M2, false>, p, st, nsm);
    default:
      if (sh.ytype == MOE_Y_FP8_E4M3)
        return launch_quant_persistent(scatter_quant_kernel<4, DT, MOE_Y_FP8_E4M3, false>, p, st, nsm);
      if (sh.ytype == MOE_Y_FP8_E5M2)
        return launch_quant_persistent(scatter_quant_kernel<4, DT, MOE_Y_FP8_E5M2, false>, p, st, nsm);
      return launch_quant_persistent(scatter_quant_kernel<4, DT, MOE_Y_FP4_E2M1, false>, p, st, nsm);
  }
}

cudaError_t launch_scatter_quant(const ScatterParams& p, cudaStream_t st, int num_sms, bool tma) {
  const Shape& sh = p.sh;
  if (sh.W * sh.bs == 0) return cudaSuccess;
  if (!tma) {
    const int grid = max(1, min(sh.W * sh.bs, num_sms * 4));
    PdlLaunch L(dim3(grid), dim3(kScatterThreads), 0, st);
    switch (sh.quant) {
      case 1: return cudaLaunchKernelEx(&L.cfg, scatter_quant_plain_kernel<1>, p);
      case 2: return cudaLaunchKernelEx(&L.cfg, scatter_quant_plain_kernel<2>, p);
      case 3: return cudaLaunchKernelEx(&L.cfg, scatter_quant_plain_kernel<3>, p);
      default: return cudaLaunchKernelEx(&L.cfg, scatter_quant_plain_kernel<4>, p);
    }
  }
  return sh.x_dtype == MOE_F16 ? launch_quant_dt<MOE_F16>(p, st, num_sms) : launch_quant_dt<MOE_BF16>(p, st, num_sms);
}

}  // namespace crs
