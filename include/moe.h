/*
 * moe.h - C ABI of the GB300 MoE token dispatch / combine library
 * (libcrs_moe.so, built from combine_route_scan_gb300/csrc).
 *
 * The W ranks of an expert-parallel (EP) group are emulated as W partitions of
 * one GPU's memory: every array carries a leading W axis, and a "remote put"
 * from rank s to rank d is a store into partition d. One call handles all W
 * ranks at once.
 *
 * Sources (web pages):
 *   [DISP]  "aclnnMoeDistributeDispatchV4" (CANN API doc): 接口功能
 *           (expandXOut = AllToAllV(X), optional quantisation first), 参数说明
 *           (active masks, zero / copy / const expert id ranges, quantMode,
 *           epRecvCountsOut and expandScalesOut shapes, value ranges), 约束说明
 *           (deterministic; dispatch outputs go unchanged into combine; "/" is
 *           integer division), the two-phase GetWorkspaceSize + execute
 *           contract, 环境变量约束 (receive buffer of BS*W*min(L,K) rows).
 *   [SHMEM] "双平面 MoE Combine 示例" (cann/shmem combine_doubleplane README):
 *           功能说明 (combine inputs, check formula), 方案设计 (plane choice),
 *           实现逻辑 (bounded bulk backlog, status-after-payload protocol).
 *   [MEGA]  xLLM "MegaMoe" pull request: dispatch + expert FFN/activation +
 *           combine in one operator.
 *
 * Conventions, for every entry point:
 *   - Pointers named like arrays are DEVICE pointers (cudaMalloc or torch
 *     memory) unless the comment says host. The caller owns every buffer; the
 *     library never allocates, frees or keeps a pointer past the call (it
 *     remembers which buffers a workspace's row map was written for, as
 *     addresses that are compared but never dereferenced; see moe_combine).
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy stream.
 *     Every call only enqueues work and returns.
 *   - Argument errors return at once, before anything is launched.
 *   - Errors found on the device (bad expert id, 1D mask out of order, a
 *     capacity overflow, inconsistent assist_info, a flag wait that timed out)
 *     are recorded in the workspace's status word; read them with
 *     moe_get_device_status. Outputs are unspecified after such an error.
 *   - Rows of expand_x / assist_info / dynamic_scales / expand_scales at or
 *     beyond ep_recv_count[d][L*W-1] are left untouched (their content is
 *     unspecified and no one may depend on it, as [DISP] says).
 *   - Results do not depend on thread timing: same inputs, same bytes.
 */
#ifndef CRS_MOE_H
#define CRS_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* a value out of the ranges below, a NULL array, misalignment */
  MOE_ERR_UNSUPPORTED = 2,   /* const experts, quant_mode outside 0..4, int32 x with quant */
  MOE_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than moe_get_workspace_size */
  MOE_ERR_BAD_EXPERT_ID = 4, /* an active id outside [0, E+Z+C), or a routed id twice in a token */
  MOE_ERR_MASK_ORDER = 5,    /* a 1D active mask with a true after a false */
  MOE_ERR_TIMEOUT = 6,       /* a bounded flag / barrier wait ran out */
  MOE_ERR_CUDA = 7,          /* a CUDA runtime call failed */
  MOE_ERR_CAPACITY = 8,      /* a rank would receive more than A rows */
  MOE_ERR_BAD_ASSIST = 9,    /* assist_info / ep_recv_count do not match the routing */
  MOE_ERR_OUT_OF_BOUNDS = 10, /* bounds-checked builds only (-DMOE_BOUNDS_CHECK): a kernel
                                computed an index outside its buffer and skipped the access */
} moe_status_t;

typedef enum { MOE_I32 = 0, MOE_F16 = 1, MOE_BF16 = 2 } moe_dtype_t;

/* Element type of quantised expand_x rows (moe_config_t.expand_dtype; [DISP]
 * 约束说明 quantMode相关约束: per-group rows are FP8, MX rows FP8 or FP4). */
enum {
  MOE_Y_DEFAULT = 0,   /* x's type (quant_mode 0) or int8 (quant_mode 1, 2) */
  MOE_Y_FP8_E4M3 = 1,  /* OCP FP8 E4M3 (max 448, S.1111.111 = NaN) */
  MOE_Y_FP8_E5M2 = 2,  /* OCP FP8 E5M2 (max 57344) */
  MOE_Y_FP4_E2M1 = 3,  /* OCP FP4 E2M1 (max 6), two codes per byte, the even element
                          in the low nibble; quant_mode 4 only, h even */
};

/* Shape of the optional `scales` input of moe_dispatch (moe_config_t.scales_kind;
 * [DISP] 参数说明 scalesOptional and 约束说明 quantMode相关约束). fp32. */
enum {
  MOE_SCALES_NONE = 0,
  MOE_SCALES_SCALAR = 1,   /* (1,): quant_mode 1 only */
  MOE_SCALES_CHANNEL = 2,  /* (h,): quant_mode 1 only */
  MOE_SCALES_EXPERT = 3,   /* (E, h): the row of the pick's expert; quant_mode 1, 2, 3 */
};

/* Which plane carries each (local expert, source) segment ([SHMEM] 方案设计). */
enum {
  MOE_PLANE_RULE = 0,        /* the page's rule: bulk iff remote, non-empty, >= bulk_min_bytes
                                and larger than the writer's mean remote segment */
  MOE_PLANE_STORES_ONLY = 1, /* every segment by SM stores (the classic single plane) */
  MOE_PLANE_BULK_ALL = 2,    /* every non-empty remote segment by TMA bulk copies */
};

/* How moe_combine runs. */
enum {
  MOE_COMBINE_GATHER = 0,    /* one pass: gather each token's K expert rows and reduce */
  MOE_COMBINE_TWO_PHASE = 1, /* [SHMEM]: put expert rows into the source's window with
                                per-pick ready flags, then wait on the flags and reduce */
  MOE_COMBINE_PUT_ONLY = 2,  /* phase 1 of TWO_PHASE alone (the page's comm_only);
                                x_out is not written */
};

typedef struct {
  int32_t ep_world_size;    /* W: EP ranks, [2, 768] */
  int32_t bs;               /* BS: tokens per rank, >= 0, W*bs*topk < 2^31 */
  int32_t h;                /* H: hidden size, > 0 */
  int32_t topk;             /* K: picks per token, [1, 32] */
  int32_t moe_expert_num;   /* E: routed experts, (0, 1024], E % W == 0; L = E / W
                               experts live on each rank, expert e on rank e / L */
  int32_t zero_expert_num;  /* Z >= 0: ids [E, E+Z) contribute nothing */
  int32_t copy_expert_num;  /* C >= 0: ids [E+Z, E+Z+C) contribute w * x */
  int32_t const_expert_num; /* must be 0 (the page gives no formula) */
  int32_t quant_mode;       /* [DISP] quantMode; x must be fp16 / bf16 when != 0:
                               0: none;
                               1: static int8, q = clamp(rne(x * s), -128, 127), s from
                                  `scales` (any MOE_SCALES_* but NONE);
                               2: per-token dynamic int8, x' = x * s[e] when scales_kind
                                  is MOE_SCALES_EXPERT (per-expert smoothing), scale =
                                  amax|x'| / 127, q = clamp(rne(x' / scale), -127, 127);
                               3: per-group dynamic FP8 (expand_dtype E4M3 / E5M2):
                                  groups of 128 elements, scale_g = amax_g / FMAX,
                                  q = fp8_satfinite_rne(x' / scale_g); optional smoothing
                                  as for 2;
                               4: MX (OCP Microscaling v1.0): blocks of 32 share
                                  X = 2^(floor(log2 amax) - emax_elem), clamped to
                                  [2^-127, 2^127], stored as an E8M0 byte; q = x / X in
                                  expand_dtype (E4M3 / E5M2 / E2M1), RNE, saturating; no
                                  scales input. A zero group / block gets scale 0 (mode 3)
                                  or byte 0 (mode 4) and zero codes. */
  int32_t mask_kind;        /* 0: no mask; 1: (BS,) per token; 2: (BS, K) per pick */
  int32_t x_dtype;          /* moe_dtype_t of x, expand_x (quant 0), expert_out, x_out;
                               expert_scales are int32 for MOE_I32, fp32 otherwise */
  int32_t plane_policy;     /* MOE_PLANE_* */
  int64_t bulk_min_bytes;   /* bulk-plane size threshold; the page's "2MB" = 2097152 */
  int32_t combine_mode;     /* MOE_COMBINE_* */
  int32_t wait_timeout_us;  /* bound on every flag wait (two-phase combine), > 0 */
  int32_t ffn_intermediate; /* I for moe_dispatch_ffn_combine, else 0 */
  int32_t expand_dtype;     /* MOE_Y_*: 0 for quant_mode 0..2; E4M3 / E5M2 for 3;
                               E4M3 / E5M2 / E2M1 for 4 */
  void* const* prof_events; /* optional host array {start, stop} of cudaEvent_t: recorded
                               on `stream` around the call's main kernel (scatter for
                               dispatch, reduce for combine, the gate/up GEMM for
                               dispatch_ffn_combine); NULL for none */
  uint32_t* seg_ready;      /* optional device array [W][L*W] (moe_dispatch only): the
                               segment's ready flag ([SHMEM] 实现逻辑: status written only
                               after its payload is visible). Each entry is set to
                               seg_ready_ticket with a release store once every row of
                               segment (le, s) of rank d is in place in expand_x and its
                               metadata (bulk-plane rows: after their bulk copies completed
                               and an async-proxy fence); empty segments too. A consumer on
                               another stream may poll it with acquire loads. NULL: none */
  uint32_t seg_ready_ticket; /* value this call stores into seg_ready; pick one the array
                               does not hold yet (e.g. a per-call counter) */
  int32_t scales_kind;      /* MOE_SCALES_*: shape of moe_dispatch's `scales` input */
  int64_t* performance_info; /* optional device array [W] int64 (moe_dispatch only; [DISP]
                               参数说明 performanceInfoOptional): each call ADDS to entry s
                               rank s's communication time in nanoseconds (%globaltimer), from
                               the earliest payload-CTA start to the moment the stores of rank
                               s's last token were issued by every thread (for a CTA's final
                               token: completed). The caller clears it when it wants to.
                               8-byte aligned, else MOE_ERR_INVALID_ARG. NULL: off */
} moe_config_t;

/* Workspace bytes for `cfg` (first phase of [DISP]'s two-phase contract), and
 * the per-rank receive capacity A = bs * W * min(L, K) ([DISP] 环境变量约束).
 * Either output pointer (host) may be NULL. Validates cfg. */
moe_status_t moe_get_workspace_size(const moe_config_t* cfg, size_t* ws_bytes, int64_t* rows_per_rank);

/* Clears the workspace header (status word, call counters, flag epoch).
 * Required once before the first call that uses a workspace, and after
 * reallocating it. Enqueued on `stream`.
 * A workspace carries state from one call to the next (counters, the row map
 * a dispatch leaves for its combine): calls that use one workspace must run
 * one after another on the GPU (one stream, or streams ordered by events);
 * overlapping calls need a workspace each. */
moe_status_t moe_workspace_init(const moe_config_t* cfg, void* ws, size_t ws_bytes, void* stream);

/* Dispatch ([DISP] 接口功能: expandXOut = AllToAllV(X), quantised first when
 * quant_mode != 0).
 *
 * Inputs (device, row-major, leading W axis):
 *   x             [W][bs][h] of x_dtype
 *   expert_ids    [W][bs][K] int32
 *   active_mask   NULL, [W][bs] (mask_kind 1) or [W][bs][K] (mask_kind 2) bytes, 0 = false
 *   expert_scales NULL or [W][bs][K] (int32 / fp32); needed iff expand_scales != NULL
 *   scales        fp32 shaped as scales_kind says ((1,), (h,) or (E, h)), 16-byte
 *                 aligned; NULL iff scales_kind is MOE_SCALES_NONE
 * Outputs (device):
 *   expand_x       [W][A][row bytes]: rank d's received rows, grouped by local expert,
 *                  then by source rank, then in (token, k) order; x's type for quant_mode
 *                  0, int8 for 1 and 2, FP8 codes (h bytes) or packed FP4 (h/2 bytes)
 *   dynamic_scales per row: quant_mode 2: [W][A] fp32; 3: [W][A][ceil(h/128)] fp32;
 *                  4: [W][A][ceil(h/32)] E8M0 bytes; NULL for quant_mode 0 and 1
 *   assist_info    [W][A][3] int32: (src_rank, src_token, src_topk) of each row
 *   ep_recv_count  [W][L*W] int32: running row count over segments le*W + s of rank d
 *   expand_scales  NULL or [W][A]: the row's weight expert_scales[s][t][k]
 *   seg_plane      NULL or [W][L*W] uint8: 1 where the segment went by bulk copies
 * Alignment: every array 16-byte aligned; rows use TMA only when the input and
 * output row bytes are multiples of 16, else plain stores carry all rows. */
moe_status_t moe_dispatch(const moe_config_t* cfg, const void* x, const int32_t* expert_ids,
                          const uint8_t* active_mask, const void* expert_scales, const float* scales,
                          void* expand_x, void* dynamic_scales, int32_t* assist_info, int32_t* ep_recv_count,
                          void* expand_scales, uint8_t* seg_plane, void* ws, size_t ws_bytes,
                          void* stream);

/* Combine ([SHMEM] 功能说明, check formula):
 *   x_out[s][t] = sum over k ascending of expert_scales[s][t][k] * y_k
 * with y_k the expert-output row that assist_info names for pick (s,t,k), x[s][t]
 * for a copy expert, nothing for a zero expert or an inactive pick; fp32
 * accumulation by fused multiply-add, rounded to nearest-even into x_dtype
 * (int32: the exact sum modulo 2^32). A token with no contribution gets zeros.
 *
 *   expert_out    [W][A][h] of x_dtype (the expert outputs at dispatch's rows)
 *   assist_info, ep_recv_count: dispatch's outputs, unchanged ([DISP] 接口配套约束)
 *   expert_ids, expert_scales, active_mask: as given to dispatch
 *   x             [W][bs][h]; needed iff copy_expert_num > 0 (else may be NULL)
 *   x_out         [W][bs][h] of x_dtype (not written for MOE_COMBINE_PUT_ONLY)
 *   seg_plane     NULL or [W][L*W] uint8: two-phase plane per segment (writer = rank d)
 * combine_mode selects the gather or the two-phase window protocol; both give
 * the same bytes.
 * Gather mode reads each routed pick's row from a pick -> row map in the
 * workspace. moe_dispatch writes that map for the assist_info and
 * ep_recv_count it fills and records their addresses in the workspace; the
 * library also remembers (host side, per workspace) which two addresses the
 * last such call enqueued. When this call passes the same two and nothing can
 * have replaced the map since (no dispatch on this workspace was captured
 * into a CUDA graph, or this combine is captured in the same capture as that
 * dispatch), the map is used as it is; otherwise an inverse-map kernel first
 * rebuilds it from assist_info, or returns at once when the workspace's
 * record shows the map already belongs to these buffers. The reduce checks
 * every pick's row against assist_info and ep_recv_count: contents changed in
 * place, a pick that no row names, or a receive count above the capacity are
 * reported as MOE_ERR_BAD_ASSIST. moe_workspace_init forgets a workspace's
 * history. A caller that rewrites assist_info / ep_recv_count in place between
 * the dispatch and this call, even with another layout that dispatch could
 * make (rows permuted within a segment together with expert_out), must call
 * moe_workspace_init first or pass the layout in other buffers: otherwise the
 * dispatch's map is kept and the picks it no longer fits are reported as
 * MOE_ERR_BAD_ASSIST. A layout that dispatch cannot make (a pick named by two
 * rows, a row naming an unrouted pick) gives unspecified x_out. */
moe_status_t moe_combine(const moe_config_t* cfg, const void* expert_out, const int32_t* assist_info,
                         const int32_t* ep_recv_count, const int32_t* expert_ids,
                         const void* expert_scales, const uint8_t* active_mask, const void* x,
                         void* x_out, uint8_t* seg_plane, void* ws, size_t ws_bytes, void* stream);

/* Dispatch -> per-expert SwiGLU FFN -> combine in one call ([MEGA] 背景与目标 and
 * 依赖关系: one operator for dispatch, expert FFN with activation, and combine;
 * intermediate_hidden = 512 on A3):
 *   x_out[s][t] = sum_k w_k * ( silu(x Wg[e]^T) * (x Wu[e]^T) ) Wd[e]^T   (routed picks)
 *               + sum_k w_k * x                                             (copy experts)
 * bf16 only, quant_mode 0, combine_mode MOE_COMBINE_GATHER; I a multiple of
 * 128 and h a multiple of 256 (tensor-core tiles), else MOE_ERR_UNSUPPORTED.
 * The FFN runs on tcgen05 tensor cores with fp32 accumulation; the
 * intermediate and expert outputs are rounded to bf16.
 *   w_gate, w_up [E][I][h] bf16 and w_down [E][h][I] bf16, stored out-major like
 *   a linear layer's weight (each row is one output feature); expert_scales fp32.
 * The workspace holds the dispatch outputs and intermediates (size from
 * moe_get_workspace_size with ffn_intermediate = I). */
moe_status_t moe_dispatch_ffn_combine(const moe_config_t* cfg, const void* x, const int32_t* expert_ids,
                                      const uint8_t* active_mask, const float* expert_scales,
                                      const void* w_gate, const void* w_up, const void* w_down,
                                      void* x_out, void* ws, size_t ws_bytes, void* stream);

/* Gather combine without any caller-allocated workspace. The pages have no
 * counterpart of this entry point: it exists for callers that cannot allocate
 * device memory, such as a plugin or custom-op host that hands the library
 * only its input and output buffers, or a serving loop that must not allocate
 * after start-up (an allocation can synchronise the device or fail under
 * memory pressure mid-step).
 * Computes exactly what moe_combine does in MOE_COMBINE_GATHER mode (same
 * arguments, same bytes out); its pick -> row scratch is a fixed device array
 * inside the library (1 MiB per device, held until the process exits).
 *   - W * bs * topk must be <= 262144, else MOE_ERR_INVALID_ARG and nothing is
 *     enqueued; combine_mode must be MOE_COMBINE_GATHER and quant_mode 0.
 *   - status: device pointer to one int32 (required); the call sets it to 0
 *     and the kernels record the first device-side error in it.
 *   - The first call on a device looks up the scratch's device address with
 *     that device current; make it before any stream capture.
 *   - All calls on a device share the scratch: calls that overlap on the GPU
 *     race and must be serialised by the caller.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine. */
moe_status_t moe_combine_noalloc(const moe_config_t* cfg, const void* expert_out, const int32_t* assist_info,
                                 const int32_t* ep_recv_count, const int32_t* expert_ids,
                                 const void* expert_scales, const uint8_t* active_mask, const void* x,
                                 void* x_out, int32_t* status, void* stream);

/* Synchronises `stream`, returns in *status (host) the first device-side error
 * recorded in the workspace since the last read (MOE_OK if none), and clears it. */
moe_status_t moe_get_device_status(void* ws, void* stream, int32_t* status);

/* Static text for a status code. */
const char* moe_status_string(int32_t status);

/* Kernels this library has enqueued in this process so far (host-side count
 * of successful launches, every entry point and device; a launch captured
 * into a CUDA graph counts once, at capture). */
uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* CRS_MOE_H */
