/*
 * CPU oracle for MoE token dispatch / combine. TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded statement of what the method computes. Only
 * the tests, the smoke check and the benchmark's CPU-baseline leg load it; the
 * CUDA library never does, and the two share no code, header or table.
 *
 * Sources (web pages; garbled tables are read as stated below):
 *   [SHMEM]  "双平面 MoE Combine 示例" (cann/shmem examples/combine/combine_doubleplane
 *            README): sections 功能说明 (inputs/outputs, check formula),
 *            方案设计 (the SDMA / MTE plane choice), 实现逻辑.
 *   [DISP]   "aclnnMoeDistributeDispatchV4" (CANN API doc): 接口功能 (AllToAllV),
 *            参数说明 (masks, zero / copy expert id ranges, quantMode,
 *            epRecvCountsOut shape), 约束说明 (determinism; "/" is integer
 *            division).
 *   [MEGA]   xLLM pull request "MegaMoe" (接入方案): dispatch, expert FFN and
 *            activation, combine in one operator; A3 intermediate_hidden = 512.
 *
 * Readings where the pages are silent or garbled:
 *   - expert e lives on rank d = e / L, local expert le = e % L (L = E / W);
 *   - ep_recv_count[d][le*W + s] is the running (inclusive) count over the
 *     (local_expert, src_rank) segments of rank d, local expert major;
 *   - inside a segment, rows follow the source order (t ascending, then k);
 *   - capacity A = bs * W * min(L, K) rows per rank; routed ids of one token
 *     must be distinct;
 *   - masked picks, zero experts: contribute nothing; copy experts contribute
 *     w * x (the weight is applied like every other top-k output);
 *   - combine accumulates in fp32, k ascending, one fused multiply-add per pick
 *     (int32 data: exact integer sum, wrapped to 32 bits), then rounds to
 *     nearest-even into the data type;
 *   - quantMode 2: per token amax = max |x| (fp32), scale = amax / 127 (IEEE
 *     fp32 division), q = clamp(round_half_even(x / scale), -127, 127); amax 0
 *     gives scale 0 and q 0;
 *   - the optional scales input ([DISP] 参数说明 scalesOptional and the
 *     quantMode constraints): one fp32 per element, shaped (1,), (H,) or
 *     (E, H); for quantMode 1 it is the static quantisation coefficient,
 *     q = clamp(round_half_even(x * s), -128, 127) (a saturating int8 cast);
 *     for quantMode 2 and 3 it is the smoothing weight of the pick's expert
 *     (shape (E, H)), applied as x' = x * s[e] (fp32) before the dynamic
 *     quantisation, so rows of one token sent to different experts differ;
 *   - quantMode 3 (per-group dynamic): groups of 128 consecutive elements of a
 *     row (the last one may be shorter), scale_g = amax_g / FMAX (FMAX = 448
 *     for FP8 E4M3, 57344 for FP8 E5M2), q = fp8(x / scale_g) rounded to
 *     nearest even with saturation to +-FMAX; amax_g 0 gives scale 0 and +0;
 *   - quantMode 4 (MX, the OCP Microscaling v1.0 conversion): blocks of 32
 *     elements share X = 2^(floor(log2 amax_b) - emax_elem), clamped to
 *     [2^-127, 2^127] and stored as an E8M0 byte (exponent + 127); elements
 *     are x / X rounded to nearest even in the element format (FP8 E4M3,
 *     emax 8; FP8 E5M2, emax 15; FP4 E2M1, emax 2; two FP4 codes per byte,
 *     the even element in the low nibble) with saturation to the largest
 *     finite value; a zero block gets byte 0;
 *   - FFN variant: SwiGLU, y = (silu(x Wg^T) * (x Wu^T)) Wd^T with weights stored
 *     out-major (w_gate, w_up [E][I][h], w_down [E][h][I]), evaluated in fp64.
 *
 * Parity pins: every function here is checked in tests/test_oracle_*.py against
 * brute force, closed forms, hand-worked fixtures or library routines.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status codes: the same numbers the public C ABI documents, written down here
 * independently so the tests can compare outcomes by name. */
enum {
  ORC_OK = 0,
  ORC_ERR_INVALID_ARG = 1,
  ORC_ERR_UNSUPPORTED = 2,
  ORC_ERR_BAD_EXPERT_ID = 4,
  ORC_ERR_MASK_ORDER = 5,
  ORC_ERR_CAPACITY = 8,
  ORC_ERR_BAD_ASSIST = 9,
};

enum { ORC_X_INT32 = 0, ORC_X_FP16 = 1, ORC_X_BF16 = 2 };
/* Element type of a quantised expand_x row. */
enum { ORC_Y_INT8 = 0, ORC_Y_FP8_E4M3 = 1, ORC_Y_FP8_E5M2 = 2, ORC_Y_FP4_E2M1 = 3 };
/* Shape of the scales input: none, (1,), (H,), (E, H). */
enum { ORC_SC_NONE = 0, ORC_SC_SCALAR = 1, ORC_SC_CHANNEL = 2, ORC_SC_EXPERT = 3 };
enum { PICK_BAD = -1, PICK_INACTIVE = 0, PICK_ZERO = 1, PICK_COPY = 2, PICK_ROUTED = 3 };

typedef struct {
  int32_t W;           /* epWorldSize: number of EP ranks */
  int32_t bs;          /* tokens per rank */
  int32_t h;           /* hidden size */
  int32_t K;           /* top-k */
  int32_t E;           /* moeExpertNum (routed experts) */
  int32_t Z;           /* zeroExpertNum */
  int32_t C;           /* copyExpertNum */
  int32_t quant_mode;  /* 0 none, 1 static int8, 2 per-token int8, 3 per-group fp8, 4 MX */
  int32_t mask_kind;   /* 0 none, 1 (bs,), 2 (bs, K) */
  int32_t x_kind;      /* ORC_X_* */
  int64_t bulk_min_bytes; /* plane-2 size threshold (2 MB on the page) */
  int32_t y_kind;      /* ORC_Y_*: element type of quantised rows (modes 3, 4) */
  int32_t scales_kind; /* ORC_SC_*: shape of the scales input */
} orc_cfg;

/* ---------------------------------------------------------------- scalars */

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round to nearest, ties to even, by the bit pattern of the fp32 value. */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static float fp16_to_f32(uint16_t b) {
  _Float16 v;
  memcpy(&v, &b, 2);
  return (float)v;
}

static uint16_t f32_to_fp16(float f) {
  _Float16 v = (_Float16)f; /* IEEE conversion, round to nearest even */
  uint16_t b;
  memcpy(&b, &v, 2);
  return b;
}

static int elem_bytes(const orc_cfg* c) { return c->x_kind == ORC_X_INT32 ? 4 : 2; }

static float load_f(const orc_cfg* c, const void* base, size_t i) {
  const uint16_t* p = (const uint16_t*)base;
  return c->x_kind == ORC_X_FP16 ? fp16_to_f32(p[i]) : bf16_to_f32(p[i]);
}

static void store_f(const orc_cfg* c, void* base, size_t i, float v) {
  uint16_t* p = (uint16_t*)base;
  p[i] = c->x_kind == ORC_X_FP16 ? f32_to_fp16(v) : f32_to_bf16(v);
}

/* ------------------------------------------------------------ config rules */

int orc_check_cfg(const orc_cfg* c) {
  /* epWorldSize in [2, 768]; moeExpertNum in (0, 1024] and a multiple of W. */
  if (c->W < 2 || c->W > 768) return ORC_ERR_INVALID_ARG;
  if (c->E <= 0 || c->E > 1024 || c->E % c->W) return ORC_ERR_INVALID_ARG;
  if (c->bs < 0 || c->h <= 0 || c->K <= 0 || c->K > 32) return ORC_ERR_INVALID_ARG;
  if (c->Z < 0 || c->C < 0) return ORC_ERR_INVALID_ARG;
  if ((int64_t)c->E + c->Z + c->C >= 2147483647LL) return ORC_ERR_INVALID_ARG;
  if (c->mask_kind < 0 || c->mask_kind > 2) return ORC_ERR_INVALID_ARG;
  if (c->x_kind < 0 || c->x_kind > 2) return ORC_ERR_INVALID_ARG;
  if (c->quant_mode < 0 || c->quant_mode > 4) return ORC_ERR_UNSUPPORTED;
  if (c->y_kind < 0 || c->y_kind > 3 || c->scales_kind < 0 || c->scales_kind > 3) return ORC_ERR_INVALID_ARG;
  if (c->quant_mode == 0) {
    if (c->y_kind != ORC_Y_INT8 || c->scales_kind != ORC_SC_NONE) return ORC_ERR_INVALID_ARG;
    return ORC_OK;
  }
  if (c->x_kind == ORC_X_INT32) return ORC_ERR_UNSUPPORTED;
  switch (c->quant_mode) {
    case 1: /* static: int8 out, a coefficient of any of the three shapes */
      if (c->y_kind != ORC_Y_INT8 || c->scales_kind == ORC_SC_NONE) return ORC_ERR_INVALID_ARG;
      break;
    case 2: /* per token: int8 out, optional per-expert smoothing */
      if (c->y_kind != ORC_Y_INT8) return ORC_ERR_INVALID_ARG;
      if (c->scales_kind != ORC_SC_NONE && c->scales_kind != ORC_SC_EXPERT) return ORC_ERR_INVALID_ARG;
      break;
    case 3: /* per group: fp8 out, optional per-expert smoothing */
      if (c->y_kind != ORC_Y_FP8_E4M3 && c->y_kind != ORC_Y_FP8_E5M2) return ORC_ERR_INVALID_ARG;
      if (c->scales_kind != ORC_SC_NONE && c->scales_kind != ORC_SC_EXPERT) return ORC_ERR_INVALID_ARG;
      break;
    default: /* MX: fp8 or fp4 out, no scales input; fp4 rows pack two codes a byte */
      if (c->y_kind == ORC_Y_INT8 || c->scales_kind != ORC_SC_NONE) return ORC_ERR_INVALID_ARG;
      if (c->y_kind == ORC_Y_FP4_E2M1 && c->h % 2) return ORC_ERR_INVALID_ARG;
      break;
  }
  return ORC_OK;
}

/* Bytes of one expand_x row. */
static int64_t row_out_bytes(const orc_cfg* c) {
  if (c->quant_mode == 0) return (int64_t)c->h * elem_bytes(c);
  if (c->quant_mode == 4 && c->y_kind == ORC_Y_FP4_E2M1) return c->h / 2;
  return c->h;
}

int64_t orc_capacity(const orc_cfg* c) {
  int64_t L = c->E / c->W;
  return (int64_t)c->bs * c->W * (L < c->K ? L : c->K);
}

/* Is pick (s, t, k) active? 1D mask: per token; 2D mask: per pick. */
static int pick_active(const orc_cfg* c, const uint8_t* mask, int s, int t, int k) {
  if (c->mask_kind == 0 || mask == NULL) return 1;
  if (c->mask_kind == 1) return mask[(size_t)s * c->bs + t] != 0;
  return mask[((size_t)s * c->bs + t) * c->K + k] != 0;
}

/* Class of one pick: inactive, zero expert [E, E+Z), copy expert
 * [E+Z, E+Z+C), routed [0, E), or bad. */
static int classify(const orc_cfg* c, const int32_t* ids, const uint8_t* mask,
                    int s, int t, int k, int32_t* e_out) {
  if (!pick_active(c, mask, s, t, k)) return PICK_INACTIVE;
  int32_t e = ids[((size_t)s * c->bs + t) * c->K + k];
  *e_out = e;
  if (e < 0) return PICK_BAD;
  if (e < c->E) return PICK_ROUTED;
  if ((int64_t)e < (int64_t)c->E + c->Z) return PICK_ZERO;
  if ((int64_t)e < (int64_t)c->E + c->Z + c->C) return PICK_COPY;
  return PICK_BAD;
}

/* The 1D mask must list its trues before its falses. */
static int check_mask_order(const orc_cfg* c, const uint8_t* mask) {
  if (c->mask_kind != 1 || mask == NULL) return ORC_OK;
  for (int s = 0; s < c->W; ++s) {
    int seen_false = 0;
    for (int t = 0; t < c->bs; ++t) {
      int a = mask[(size_t)s * c->bs + t] != 0;
      if (!a) seen_false = 1;
      else if (seen_false) return ORC_ERR_MASK_ORDER;
    }
  }
  return ORC_OK;
}

/* Format of a small binary float: exponent / mantissa widths, bias, largest
 * finite magnitude and its code (FP8 E4M3 keeps S.1111.111 for NaN; E5M2 and
 * E2M1 follow the IEEE pattern; E2M1 has no inf or NaN). */
typedef struct { int mb, bias; double maxv; int max_code, sign_bit; } minifloat_fmt;

static minifloat_fmt fmt_of(int y_kind) {
  minifloat_fmt f;
  if (y_kind == ORC_Y_FP8_E4M3) { f.mb = 3; f.bias = 7; f.maxv = 448.0; f.max_code = 0x7E; f.sign_bit = 0x80; }
  else if (y_kind == ORC_Y_FP8_E5M2) { f.mb = 2; f.bias = 15; f.maxv = 57344.0; f.max_code = 0x7B; f.sign_bit = 0x80; }
  else { f.mb = 1; f.bias = 1; f.maxv = 6.0; f.max_code = 0x7; f.sign_bit = 0x8; }
  return f;
}

/* Finite fp32 -> the nearest value of the format, ties to the even code,
 * magnitudes at or above the largest finite value saturate to it. The sign
 * is kept (a negative value that rounds to zero gives the negative zero). */
static uint8_t f32_to_minifloat(float v, int y_kind) {
  minifloat_fmt f = fmt_of(y_kind);
  int neg = signbit(v) != 0;
  double a = fabs((double)v);
  int code;
  if (a >= f.maxv) {
    code = f.max_code;
  } else {
    int emin = 1 - f.bias;   /* exponent of the smallest normal */
    int e;
    if (a < ldexp(1.0, emin)) e = emin;                 /* subnormal: fixed quantum */
    else { int ex; frexp(a, &ex); e = ex - 1; }          /* a in [2^e, 2^(e+1)) */
    double quantum = ldexp(1.0, e - f.mb);
    double n = nearbyint(a / quantum);                  /* exact quotient, RNE */
    /* subnormals: the code is n itself; normals: biased exponent field plus
     * the mantissa, and a carry out of the mantissa moves to the next binade */
    if (e == emin && a < ldexp(1.0, emin)) code = (int)n;
    else code = ((e + f.bias) << f.mb) + (int)n - (1 << f.mb);
    if (code > f.max_code) code = f.max_code;
  }
  return (uint8_t)(code | (neg ? f.sign_bit : 0));
}

/* Element j of a row, multiplied by the smoothing / static coefficient that
 * applies to it (quant_scales is NULL or shaped as scales_kind says). */
static float scaled_elem(const orc_cfg* c, const void* x, size_t row, int j, int32_t e,
                         const float* quant_scales) {
  float v = load_f(c, x, row * c->h + j);
  switch (c->scales_kind) {
    case ORC_SC_SCALAR: return v * quant_scales[0];
    case ORC_SC_CHANNEL: return v * quant_scales[j];
    case ORC_SC_EXPERT: return v * quant_scales[(size_t)e * c->h + j];
    default: return v;
  }
}

/* Quantise row `row` of x for a pick of expert e (quantMode 1..4). Writes the
 * row's row_out_bytes(c) bytes to q and its dynamic scales to dyn (mode 2: one
 * fp32; mode 3: ceil(h/128) fp32; mode 4: ceil(h/32) E8M0 bytes; mode 1:
 * nothing). */
static void quantize_pick(const orc_cfg* c, const void* x, size_t row, int32_t e, const float* quant_scales,
                          uint8_t* q, void* dyn) {
  const int h = c->h;
  float* xs = (float*)malloc((size_t)h * sizeof(float));
  for (int j = 0; j < h; ++j) xs[j] = scaled_elem(c, x, row, j, e, quant_scales);
  if (c->quant_mode == 1) {
    for (int j = 0; j < h; ++j) {
      float r = nearbyintf(xs[j]);
      if (r > 127.0f) r = 127.0f;
      if (r < -128.0f) r = -128.0f;
      q[j] = (uint8_t)(int8_t)r;
    }
  } else if (c->quant_mode == 2) {
    float amax = 0.0f;
    for (int j = 0; j < h; ++j) if (fabsf(xs[j]) > amax) amax = fabsf(xs[j]);
    float scale = amax / 127.0f;
    for (int j = 0; j < h; ++j) {
      float r = amax == 0.0f ? 0.0f : nearbyintf(xs[j] / scale);
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
      q[j] = (uint8_t)(int8_t)r;
    }
    if (dyn) ((float*)dyn)[0] = scale;
  } else if (c->quant_mode == 3) {
    const float fmax = c->y_kind == ORC_Y_FP8_E4M3 ? 448.0f : 57344.0f;
    for (int g0 = 0; g0 < h; g0 += 128) {
      int g1 = g0 + 128 < h ? g0 + 128 : h;
      float amax = 0.0f;
      for (int j = g0; j < g1; ++j) if (fabsf(xs[j]) > amax) amax = fabsf(xs[j]);
      float scale = amax / fmax;
      for (int j = g0; j < g1; ++j) q[j] = amax == 0.0f ? 0 : f32_to_minifloat(xs[j] / scale, c->y_kind);
      if (dyn) ((float*)dyn)[g0 / 128] = scale;
    }
  } else {
    const int emax = c->y_kind == ORC_Y_FP8_E4M3 ? 8 : c->y_kind == ORC_Y_FP8_E5M2 ? 15 : 2;
    if (c->y_kind == ORC_Y_FP4_E2M1) memset(q, 0, (size_t)h / 2);
    for (int b0 = 0; b0 < h; b0 += 32) {
      int b1 = b0 + 32 < h ? b0 + 32 : h;
      float amax = 0.0f;
      for (int j = b0; j < b1; ++j) if (fabsf(xs[j]) > amax) amax = fabsf(xs[j]);
      int se = -127;
      if (amax > 0.0f) {
        int ex;
        frexpf(amax, &ex);          /* amax in [2^(ex-1), 2^ex) */
        se = (ex - 1) - emax;
        if (se < -127) se = -127;
        if (se > 127) se = 127;
      }
      float X = ldexpf(1.0f, se);
      for (int j = b0; j < b1; ++j) {
        uint8_t code = f32_to_minifloat(xs[j] / X, c->y_kind);
        if (c->y_kind == ORC_Y_FP4_E2M1) q[j / 2] |= (uint8_t)(code << (4 * (j % 2)));
        else q[j] = code;
      }
      if (dyn) ((uint8_t*)dyn)[b0 / 32] = (uint8_t)(se + 127);
    }
  }
  free(xs);
}

/* Entries of dynamic scales per expand_x row (and their bytes). */
static int64_t dyn_per_row(const orc_cfg* c) {
  if (c->quant_mode == 2) return 1;
  if (c->quant_mode == 3) return (c->h + 127) / 128;
  if (c->quant_mode == 4) return (c->h + 31) / 32;
  return 0;
}
static int dyn_elem_bytes(const orc_cfg* c) { return c->quant_mode == 4 ? 1 : 4; }

/* ------------------------------------------------------------------ dispatch
 *
 * expandXOut = AllToAllV(X) over the EP ranks, with the rows of each receiving
 * rank grouped by local expert and then by source rank, and the per-segment
 * running receive counts in ep_recv_count.
 *
 *   x             [W][bs][h]          expert_ids [W][bs][K]
 *   mask          [W][bs] / [W][bs][K] or NULL
 *   scales        [W][bs][K] (int32 for int32 x, else fp32), may be NULL
 *   quant_scales  fp32 (1,), (h,) or (E, h) as scales_kind says, or NULL
 *   expand_x      [W][A][row_out_bytes] (x's type unquantised; int8, fp8 or
 *                 packed fp4 codes otherwise)
 *   dyn_scales    [W][A][dyn_per_row] (fp32; E8M0 bytes for quantMode 4), or
 *                 NULL; quantMode 0 and 1 have none
 *   assist        [W][A][3] int32 = (src_rank, src_token, src_topk)
 *   ep_recv_count [W][L*W] int32
 *   expand_scales [W][A] (the pick's weight), may be NULL
 * Rows at or beyond ep_recv_count[d][L*W-1] are left untouched.
 */
int orc_dispatch(const orc_cfg* c, const void* x, const int32_t* ids, const uint8_t* mask,
                 const void* scales, const float* quant_scales, void* expand_x, void* dyn_scales,
                 int32_t* assist, int32_t* ep_recv_count, void* expand_scales) {
  int st = orc_check_cfg(c);
  if (st) return st;
  if (c->scales_kind != ORC_SC_NONE && quant_scales == NULL) return ORC_ERR_INVALID_ARG;
  const int W = c->W, bs = c->bs, h = c->h, K = c->K, E = c->E, L = E / W;
  const int64_t A = orc_capacity(c);
  const int es = elem_bytes(c);

  st = check_mask_order(c, mask);
  if (st) return st;

  /* 1. classify every pick; count the rows of each (expert, source) segment */
  int64_t* cnt = (int64_t*)calloc((size_t)E * W, sizeof(int64_t));
  int64_t* next = (int64_t*)calloc((size_t)E * W, sizeof(int64_t));
  if (!cnt || !next) { free(cnt); free(next); return ORC_ERR_INVALID_ARG; }
  for (int s = 0; s < W && !st; ++s)
    for (int t = 0; t < bs && !st; ++t)
      for (int k = 0; k < K; ++k) {
        int32_t e = -1;
        int cls = classify(c, ids, mask, s, t, k, &e);
        if (cls == PICK_BAD) { st = ORC_ERR_BAD_EXPERT_ID; break; }
        if (cls != PICK_ROUTED) continue;
        for (int k2 = 0; k2 < k; ++k2) { /* routed ids of a token are distinct */
          int32_t e2 = -1;
          if (classify(c, ids, mask, s, t, k2, &e2) == PICK_ROUTED && e2 == e) {
            st = ORC_ERR_BAD_EXPERT_ID;
            break;
          }
        }
        if (st) break;
        cnt[(size_t)e * W + s] += 1;
      }
  if (st) { free(cnt); free(next); return st; }

  /* 2. running receive counts per rank, local expert major, source minor.
   *    Segment (d, le, s) has flat index (d*L + le)*W + s = e*W + s. */
  for (int d = 0; d < W; ++d) {
    int64_t run = 0;
    for (int le = 0; le < L; ++le)
      for (int s = 0; s < W; ++s) {
        size_t g = ((size_t)d * L + le) * W + s;
        next[g] = run;           /* first row of the segment */
        run += cnt[g];
        ep_recv_count[g] = (int32_t)run;
      }
    if (run > A) { free(cnt); free(next); return ORC_ERR_CAPACITY; }
  }

  /* 3. place every routed pick: rows of a segment in (t, k) order */
  const int64_t rob = row_out_bytes(c), nd = dyn_per_row(c), db = dyn_elem_bytes(c);
  for (int s = 0; s < W; ++s)
    for (int t = 0; t < bs; ++t) {
      size_t src = (size_t)s * bs + t;
      for (int k = 0; k < K; ++k) {
        int32_t e = -1;
        if (classify(c, ids, mask, s, t, k, &e) != PICK_ROUTED) continue;
        int d = e / L;
        size_t g = (size_t)e * W + s;
        size_t row = (size_t)d * A + (size_t)next[g]++;
        if (c->quant_mode != 0) {
          quantize_pick(c, x, src, e, quant_scales, (uint8_t*)expand_x + row * rob,
                        dyn_scales ? (char*)dyn_scales + row * nd * db : NULL);
        } else {
          memcpy((char*)expand_x + row * h * es, (const char*)x + src * h * es, (size_t)h * es);
        }
        assist[row * 3 + 0] = s;
        assist[row * 3 + 1] = t;
        assist[row * 3 + 2] = k;
        if (expand_scales && scales)
          memcpy((char*)expand_scales + row * 4, (const char*)scales + (src * K + k) * 4, 4);
      }
    }
  free(cnt);
  free(next);
  return ORC_OK;
}

/* Rows of segment g = (d*L + le)*W + s, from the running counts. */
static int64_t seg_rows(const orc_cfg* c, const int32_t* ep_recv_count, size_t g) {
  int LW = (c->E / c->W) * c->W;
  return (g % LW == 0) ? ep_recv_count[g] : (int64_t)ep_recv_count[g] - ep_recv_count[g - 1];
}

/* ----------------------------------------------------------- plane choice
 *
 * [SHMEM] 方案设计: a segment goes over the bulk (SDMA) plane iff it is remote,
 * non-empty, at least bulk_min_bytes, and larger than the mean remote segment of
 * the rank doing the writing, tested by the cross multiply
 *     segment_bytes * threshold_den > threshold_num,
 *     threshold_num = remote_tokens * h * sizeof(T),
 *     threshold_den = max(W - 1, 1) * local_expert_num.
 * plane[g] = 1 for the bulk plane, 0 for plain stores; g indexes segments like
 * ep_recv_count.
 *
 * Combine: the writer is rank d (it holds the expert outputs and writes them
 * back to source s); remote_tokens = rows of d that came from s != d.
 */
int orc_combine_plane(const orc_cfg* c, const int32_t* ep_recv_count, uint8_t* plane) {
  int st = orc_check_cfg(c);
  if (st) return st;
  const int W = c->W, L = c->E / c->W;
  const int64_t row_bytes = (int64_t)c->h * elem_bytes(c);
  const int64_t den = (int64_t)(W - 1 > 1 ? W - 1 : 1) * L;
  for (int d = 0; d < W; ++d) {
    int64_t remote = 0;
    for (int le = 0; le < L; ++le)
      for (int s = 0; s < W; ++s)
        if (s != d) remote += seg_rows(c, ep_recv_count, ((size_t)d * L + le) * W + s);
    int64_t num = remote * row_bytes;
    for (int le = 0; le < L; ++le)
      for (int s = 0; s < W; ++s) {
        size_t g = ((size_t)d * L + le) * W + s;
        int64_t n = seg_rows(c, ep_recv_count, g);
        int64_t bytes = n * row_bytes;
        plane[g] = (uint8_t)(s != d && n > 0 && bytes >= c->bulk_min_bytes && bytes * den > num);
      }
  }
  return ORC_OK;
}

/* Dispatch, by symmetry: the writer is source s; remote_tokens = rows that s
 * sends to ranks d != s; sizeof(T) * h is the size of the row written (h bytes
 * for int8 and fp8, h / 2 for packed fp4). */
int orc_dispatch_plane(const orc_cfg* c, const int32_t* ep_recv_count, uint8_t* plane) {
  int st = orc_check_cfg(c);
  if (st) return st;
  const int W = c->W, L = c->E / c->W;
  const int64_t row_bytes = row_out_bytes(c);
  const int64_t den = (int64_t)(W - 1 > 1 ? W - 1 : 1) * L;
  for (int s = 0; s < W; ++s) {
    int64_t remote = 0;
    for (int d = 0; d < W; ++d)
      if (d != s)
        for (int le = 0; le < L; ++le) remote += seg_rows(c, ep_recv_count, ((size_t)d * L + le) * W + s);
    int64_t num = remote * row_bytes;
    for (int d = 0; d < W; ++d)
      for (int le = 0; le < L; ++le) {
        size_t g = ((size_t)d * L + le) * W + s;
        int64_t n = seg_rows(c, ep_recv_count, g);
        int64_t bytes = n * row_bytes;
        plane[g] = (uint8_t)(s != d && n > 0 && bytes >= c->bulk_min_bytes && bytes * den > num);
      }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------ combine
 *
 * [SHMEM] 功能说明, check formula:
 *     x_out[token] = sum_k topk_output[token, k] * expert_scales[token, k]
 * topk_output of a routed pick is the expert-output row that assist_info names
 * for it (rows [0, ep_recv_count[d][L*W-1]) of every rank d); copy experts give
 * x[token], zero experts and masked picks give nothing.
 *
 *   expert_out [W][A][h] (x's type)   x_out [W][bs][h]
 */
int orc_combine(const orc_cfg* c, const void* expert_out, const int32_t* assist,
                const int32_t* ep_recv_count, const int32_t* ids, const void* scales,
                const uint8_t* mask, const void* x, void* x_out) {
  int st = orc_check_cfg(c);
  if (st) return st;
  const int W = c->W, bs = c->bs, h = c->h, K = c->K, L = c->E / c->W;
  const int64_t A = orc_capacity(c);
  st = check_mask_order(c, mask);
  if (st) return st;

  /* 1. which expert-output row holds each routed pick */
  size_t npick = (size_t)W * bs * K;
  int64_t* where = (int64_t*)malloc(npick * sizeof(int64_t));
  for (size_t i = 0; i < npick; ++i) where[i] = -1;
  for (int d = 0; d < W && !st; ++d) {
    int64_t rows = ep_recv_count[(size_t)d * L * W + (size_t)L * W - 1];
    if (rows < 0 || rows > A) { st = ORC_ERR_BAD_ASSIST; break; }
    for (int64_t r = 0; r < rows; ++r) {
      size_t row = (size_t)d * A + (size_t)r;
      int32_t s = assist[row * 3 + 0], t = assist[row * 3 + 1], k = assist[row * 3 + 2];
      if (s < 0 || s >= W || t < 0 || t >= bs || k < 0 || k >= K) { st = ORC_ERR_BAD_ASSIST; break; }
      size_t p = ((size_t)s * bs + t) * K + k;
      if (where[p] >= 0) { st = ORC_ERR_BAD_ASSIST; break; }
      where[p] = (int64_t)row;
    }
  }

  /* 2. weighted sum per token, k ascending */
  for (int s = 0; s < W && !st; ++s)
    for (int t = 0; t < bs && !st; ++t) {
      size_t tok = (size_t)s * bs + t;
      int cls[32];
      for (int k = 0; k < K; ++k) {
        int32_t e = -1;
        cls[k] = classify(c, ids, mask, s, t, k, &e);
        if (cls[k] == PICK_BAD) { st = ORC_ERR_BAD_EXPERT_ID; break; }
        if (cls[k] == PICK_ROUTED && where[tok * K + k] < 0) { st = ORC_ERR_BAD_ASSIST; break; }
        if (cls[k] != PICK_ROUTED && where[tok * K + k] >= 0) { st = ORC_ERR_BAD_ASSIST; break; }
      }
      if (st) break;
      for (int j = 0; j < h; ++j) {
        if (c->x_kind == ORC_X_INT32) {
          int64_t acc = 0;
          for (int k = 0; k < K; ++k) {
            int64_t w = ((const int32_t*)scales)[tok * K + k];
            if (cls[k] == PICK_ROUTED)
              acc += w * ((const int32_t*)expert_out)[(size_t)where[tok * K + k] * h + j];
            else if (cls[k] == PICK_COPY)
              acc += w * ((const int32_t*)x)[tok * h + j];
          }
          ((int32_t*)x_out)[tok * h + j] = (int32_t)(uint32_t)(uint64_t)acc;
        } else {
          float acc = 0.0f;
          for (int k = 0; k < K; ++k) {
            float w = ((const float*)scales)[tok * K + k];
            if (cls[k] == PICK_ROUTED)
              acc = fmaf(w, load_f(c, expert_out, (size_t)where[tok * K + k] * h + j), acc);
            else if (cls[k] == PICK_COPY)
              acc = fmaf(w, load_f(c, x, tok * h + j), acc);
          }
          store_f(c, x_out, tok * h + j, acc);
        }
      }
    }
  free(where);
  return st;
}

/* ---------------------------------------------------------- expert FFN
 *
 * [MEGA] fuses the expert FFN and its activation between dispatch and combine;
 * the activation is SwiGLU: y = (silu(x Wg^T) * (x Wu^T)) Wd^T,
 * silu(a) = a/(1+e^-a). Weights are stored out-major, like a linear layer (the
 * pages leave the layout open): w_gate, w_up [E][I][h], w_down [E][h][I].
 * Evaluated in fp64 from bf16 operands.
 *   x_rows [n][h] bf16 bits, expert [n] (global expert id per row); y [n][h] fp64
 */
int orc_swiglu_rows(int h, int I, int E, int64_t n, const uint16_t* x_rows, const int32_t* expert,
                    const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                    double* y) {
  if (h <= 0 || I <= 0 || E <= 0 || n < 0) return ORC_ERR_INVALID_ARG;
  double* xv = (double*)malloc(sizeof(double) * h);
  double* a = (double*)malloc(sizeof(double) * I);
  for (int64_t r = 0; r < n; ++r) {
    int32_t e = expert[r];
    if (e < 0 || e >= E) { free(xv); free(a); return ORC_ERR_BAD_EXPERT_ID; }
    const uint16_t* xr = x_rows + (size_t)r * h;
    const uint16_t* wg = w_gate + (size_t)e * I * h;
    const uint16_t* wu = w_up + (size_t)e * I * h;
    const uint16_t* wd = w_down + (size_t)e * h * I;
    for (int j = 0; j < h; ++j) xv[j] = bf16_to_f32(xr[j]);
    for (int i = 0; i < I; ++i) {
      double g = 0.0, u = 0.0;
      for (int j = 0; j < h; ++j) {
        g += xv[j] * bf16_to_f32(wg[(size_t)i * h + j]);
        u += xv[j] * bf16_to_f32(wu[(size_t)i * h + j]);
      }
      a[i] = g / (1.0 + exp(-g)) * u;
    }
    double* yr = y + (size_t)r * h;
    for (int j = 0; j < h; ++j) {
      double acc = 0.0;
      for (int i = 0; i < I; ++i) acc += a[i] * bf16_to_f32(wd[(size_t)j * I + i]);
      yr[j] = acc;
    }
  }
  free(xv);
  free(a);
  return ORC_OK;
}

/* The whole FFN variant for a set of tokens (dispatch -> expert -> combine):
 *   x_out[token] = sum_k w_k * FFN_{e_k}(x[token])   for routed picks,
 *                + w_k * x[token]                     for copy experts,
 * in fp64. tokens[i] = s*bs + t; out [n_tok][h]. Only bf16 x; weights as in
 * orc_swiglu_rows. */
int orc_moe_ffn_tokens(const orc_cfg* c, int I, int64_t n_tok, const int64_t* tokens,
                       const uint16_t* x, const int32_t* ids, const uint8_t* mask,
                       const float* scales, const uint16_t* w_gate, const uint16_t* w_up,
                       const uint16_t* w_down, double* out) {
  int st = orc_check_cfg(c);
  if (st) return st;
  if (c->x_kind != ORC_X_BF16) return ORC_ERR_UNSUPPORTED;
  const int bs = c->bs, h = c->h, K = c->K;
  double* y = (double*)malloc(sizeof(double) * h);
  for (int64_t i = 0; i < n_tok && !st; ++i) {
    int64_t tok = tokens[i];
    int s = (int)(tok / bs), t = (int)(tok % bs);
    double* o = out + (size_t)i * h;
    for (int j = 0; j < h; ++j) o[j] = 0.0;
    for (int k = 0; k < K; ++k) {
      int32_t e = -1;
      int cls = classify(c, ids, mask, s, t, k, &e);
      if (cls == PICK_BAD) { st = ORC_ERR_BAD_EXPERT_ID; break; }
      double w = scales[(size_t)tok * K + k];
      if (cls == PICK_ROUTED) {
        st = orc_swiglu_rows(h, I, c->E, 1, x + (size_t)tok * h, &e, w_gate, w_up, w_down, y);
        if (st) break;
        for (int j = 0; j < h; ++j) o[j] += w * y[j];
      } else if (cls == PICK_COPY) {
        for (int j = 0; j < h; ++j) o[j] += w * bf16_to_f32(x[(size_t)tok * h + j]);
      }
    }
  }
  free(y);
  return st;
}

/* Scalar conversions, exported so the tests can pin them to library routines. */
uint16_t orc_f32_to_bf16(float f) { return f32_to_bf16(f); }
float orc_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }
uint16_t orc_f32_to_fp16(float f) { return f32_to_fp16(f); }
float orc_fp16_to_f32(uint16_t b) { return fp16_to_f32(b); }

/* quantMode 2 on one row, exported for the hand-worked quantiser fixtures. */
float orc_quantize_row(const orc_cfg* c, const void* x_row, int8_t* q) {
  float scale = 0.0f;
  if (c->quant_mode != 2 || c->scales_kind != ORC_SC_NONE) return -1.0f;
  quantize_pick(c, x_row, 0, 0, NULL, (uint8_t*)q, &scale);
  return scale;
}

/* One fp32 value in a small float format (ORC_Y_FP8_E4M3 / _E5M2 / FP4_E2M1). */
uint8_t orc_f32_to_minifloat(float v, int y_kind) { return f32_to_minifloat(v, y_kind); }

/* quantMode 1..4 on one row for a pick of expert e (exported for the pins). */
int orc_quantize_pick(const orc_cfg* c, const void* x_row, int32_t e, const float* quant_scales,
                      uint8_t* q, void* dyn) {
  int st = orc_check_cfg(c);
  if (st) return st;
  if (c->quant_mode == 0) return ORC_ERR_INVALID_ARG;
  quantize_pick(c, x_row, 0, e, quant_scales, q, dyn);
  return ORC_OK;
}
