// Element conversions and code arithmetic shared by the quantising dispatch
// kernels (scatter_quant.cu: token-major; scatter_pe.cu: expert-major for
// per-expert scales). aclnnMoeDistributeDispatchV4, 参数说明 quantMode /
// scalesOptional and 约束说明 quantMode相关约束: static int8, per-token int8,
// per-group FP8 and MX FP8 / FP4 codes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "scatter_common.cuh"

namespace crs {

template <int DT>
__device__ __forceinline__ void unpack8(int4 v, float (&f)[8]) {
  const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (DT == MOE_F16) {
      const __half2 h2 = *reinterpret_cast<const __half2*>(&w[i]);
      f[2 * i] = __low2float(h2);
      f[2 * i + 1] = __high2float(h2);
    } else {
      const __nv_bfloat162 h2 = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      f[2 * i] = __low2float(h2);
      f[2 * i + 1] = __high2float(h2);
    }
  }
}

__device__ __forceinline__ float load_elem(const void* x, size_t i, int dt) {
  const uint16_t b = static_cast<const uint16_t*>(x)[i];
  return dt == MOE_F16 ? __half2float(__ushort_as_half(b)) : __bfloat162float(__ushort_as_bfloat16(b));
}

// Two fp32 values -> two FP8 codes, the first in the low byte.
template <int YT>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
  uint16_t r;
  if (YT == MOE_Y_FP8_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 values -> two FP4 E2M1 codes in one byte, the first in the low nibble.
__device__ __forceinline__ uint32_t cvt_fp4x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t cvt_y_pair(int yt, float lo, float hi) {
  if (yt == MOE_Y_FP8_E4M3) return cvt_fp8x2<MOE_Y_FP8_E4M3>(lo, hi);
  if (yt == MOE_Y_FP8_E5M2) return cvt_fp8x2<MOE_Y_FP8_E5M2>(lo, hi);
  return cvt_fp4x2(lo, hi);
}

__device__ __forceinline__ float fp8_max(int yt) { return yt == MOE_Y_FP8_E4M3 ? 448.0f : 57344.0f; }
__device__ __forceinline__ int elem_emax(int yt) {
  return yt == MOE_Y_FP8_E4M3 ? 8 : yt == MOE_Y_FP8_E5M2 ? 15 : 2;
}

// floor(log2(a)) of a finite a > 0, subnormals included (from the bit fields).
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t b = __float_as_uint(a);
  const int e = (int)((b >> 23) & 0xffu);
  if (e) return e - 127;
  return (31 - __clz(b & 0x7fffffu)) - 149;
}

// MX shared exponent of a block: floor(log2 amax) - emax clamped to [-127, 127];
// -127 for an all-zero block.
__device__ __forceinline__ int mx_exponent(float amax, int emax) {
  if (!(amax > 0.f)) return -127;
  return max(-127, min(127, floor_log2(amax) - emax));
}

// 2^k for k in [-127, 127], exactly (2^-127 is subnormal).
__device__ __forceinline__ float exp2_exact(int k) {
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ int static_q(float v) { return max(-128, min(127, __float2int_rn(v))); }
__device__ __forceinline__ int token_q(float v, float scale) {
  return max(-127, min(127, __float2int_rn(__fdiv_rn(v, scale))));
}

// Per-token int8 code from the reciprocal r = 1/scale (rounded once): y = v*r
// is within 2^-23 |y| of v/scale and the IEEE quotient within half an ulp of
// it, so y rounded to the nearest integer (adding 1.5 * 2^23 leaves it, ties to
// even, in the low mantissa bits) is the code of the quotient unless y lies
// within 2^-14 of a half-integer: those, and NaN, take the division. For
// |v| <= amax and a normal scale, |y| <= 127.00003 needs no clamp. The code is
// the low byte of the returned word.
constexpr float kRoundShift = 12582912.0f;  // 1.5 * 2^23
constexpr float kNearHalf = 0.5f - 0.00006103515625f;  // 0.5 - 2^-14
__device__ __forceinline__ uint32_t token_code(float v, float scale, float rcp) {
  const float y = __fmul_rn(v, rcp);
  const float t = __fadd_rn(y, kRoundShift);
  const float d = fabsf(__fsub_rn(y, __fsub_rn(t, kRoundShift)));
  return d <= kNearHalf ? __float_as_uint(t) : (uint32_t)token_q(v, scale);
}
// the reciprocal form holds for a normal, finite scale (an all-zero row, a
// subnormal or infinite scale quantise through the division)
__device__ __forceinline__ bool token_rcp_ok(float scale) { return scale >= 1.17549435e-38f && scale <= 3.40282347e38f; }

// low bytes of c[0..8) as 8 consecutive bytes
__device__ __forceinline__ uint2 pack8_low(const uint32_t (&c)[8]) {
  const uint32_t a = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
  const uint32_t b = __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
  return make_uint2(a, b);
}

__device__ __forceinline__ uint2 pack8(const int (&q)[8]) {
  uint32_t a = 0, b = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a |= ((uint32_t)q[i] & 0xffu) << (8 * i);
    b |= ((uint32_t)q[i + 4] & 0xffu) << (8 * i);
  }
  return make_uint2(a, b);
}

// Coefficient / smoothing weights of 8 elements starting at v*8 (16-byte
// aligned loads: the scales array is 16-byte aligned and h % 8 == 0 here).
__device__ __forceinline__ void load_scales8(const float* srow, uint32_t v, float (&s)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(srow) + 2 * v);
  const float4 b = __ldg(reinterpret_cast<const float4*>(srow) + 2 * v + 1);
  s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w;
  s[4] = b.x; s[5] = b.y; s[6] = b.z; s[7] = b.w;
}

// ---------------------------------------------------------------- f32x2
// Two fp32 values in one 64-bit register, the first in the low word, and the
// sm_100-family packed instructions that round each lane to nearest even as
// the scalar forms do (one issue slot for two results).
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_sub(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// max(a, |b|, |c|) and min(a, |b|, |c|), one three-input instruction each
__device__ __forceinline__ float fmax_abs3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(fabsf(b)), "f"(fabsf(c)));
  return d;
}
__device__ __forceinline__ float fmin_abs3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(fabsf(b)), "f"(fabsf(c)));
  return d;
}

// The 8 elements of a 16-byte vector as four fp32 pairs (exact conversions).
template <int DT>
__device__ __forceinline__ void unpack8x2(int4 v, f32x2 (&o)[4]) {
  const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (DT == MOE_BF16) {
      o[i] = f2_pack(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      o[i] = f2_pack(f.x, f.y);
    }
  }
}

// The per-token int8 codes of one 8-element vector through the IEEE division
// (the rare vectors whose reciprocal form is undecided), out of line so that
// the main path carries none of its instructions.
static __device__ __noinline__ uint2 token_codes_div8(f32x2 v0, f32x2 v1, f32x2 v2, f32x2 v3, float scale, float amax) {
  const f32x2 v[4] = {v0, v1, v2, v3};
  int qv[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo, hi;
    f2_split(v[i], lo, hi);
    qv[2 * i] = amax == 0.f ? 0 : token_q(lo, scale);
    qv[2 * i + 1] = amax == 0.f ? 0 : token_q(hi, scale);
  }
  return pack8(qv);
}

// Per-token int8 codes of 8 products v through the reciprocal r = fl(1/scale):
// rounding y = v * r to an integer (adding 1.5 * 2^23, the code then in the
// low byte) gives the code of the IEEE quotient unless y lies within 2^-14 of
// a half-integer (the argument at token_code); one test for the vector, whose
// rare failures take the division.
__device__ __forceinline__ uint2 token_codes8(const f32x2 (&v)[4], float scale, float amax, bool fast, f32x2 rcp2) {
  const f32x2 shift2 = f2_pack(kRoundShift, kRoundShift);
  uint32_t c[8];
  float dm = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const f32x2 y = f2_mul(v[i], rcp2);
    const f32x2 t = f2_add(y, shift2);
    const f32x2 d = f2_sub(y, f2_sub(t, shift2));
    float dl, dh, tl, th;
    f2_split(d, dl, dh);
    f2_split(t, tl, th);
    dm = fmax_abs3(dm, dl, dh);
    c[2 * i] = __float_as_uint(tl);
    c[2 * i + 1] = __float_as_uint(th);
  }
  if (!(fast && dm <= kNearHalf)) return token_codes_div8(v[0], v[1], v[2], v[3], scale, amax);
  return pack8_low(c);
}

}  // namespace crs
