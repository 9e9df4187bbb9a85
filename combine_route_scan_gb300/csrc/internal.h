// Internal declarations of the MoE dispatch / combine library: workspace
// layout, kernel parameter blocks and launchers. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace crs {

// Workspace header (first 256 bytes of the workspace).
struct WsHeader {
  int status;           // first device-side error (moe_status_t), sticky until read
  uint32_t epoch;       // two-phase combine flag epoch (last completed call)
  uint32_t route_done;  // route CTAs finished in the current dispatch
  uint32_t tp_done;     // two-phase combine CTAs finished in the current call
  unsigned long long perf_start_inv;  // ~(earliest scatter CTA start), kept with atomicMax
  uint32_t scatter_done;              // scatter CTAs finished (performance info)
  uint32_t inv_valid;                 // the inv region holds the pick -> row map of the last dispatch ...
  unsigned long long inv_assist;      // ... whose assist_info and ep_recv_count were these buffers
  unsigned long long inv_ep;
  uint32_t scatter_next;  // TMA scatter: next token ticket (zeroed by the routing kernel)
  uint32_t pe_rows;       // per-group FP8 with per-expert scales: receive rows of all ranks (the row list length)
  uint32_t pad[50];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Byte offsets of the workspace regions.
struct WsLayout {
  size_t cnt;      // int32 [E*W]     rows of segment g = e*W + s
  size_t base;     // int32 [E*W]     first row of segment g inside its rank
  size_t plane_d;  // uint8 [E*W]     dispatch plane per segment
  size_t landed;   // uint32 [E*W]    dispatch rows in place per segment (ready flags)
  size_t perf_end; // uint64 [W]      latest row-store time per source rank (performance info)
  size_t rank;     // int32 [W*bs*K]  position of a routed pick inside its segment
  size_t inv;      // int32 [W*bs*K]  combine: flat expert-output row of each pick
  size_t plane_c;  // uint8 [E*W]     two-phase combine plane per segment
  size_t flags;    // uint32 [W*bs*K] two-phase combine ready flags
  size_t window;   // [W*bs*K][h]     two-phase combine window
  size_t pe_list;  // int4 [W*A]      per-token int8 / per-group FP8 with per-expert scales: {row, token, expert, plane} of every receive row
  // moe_dispatch_ffn_combine only
  size_t ffn_expand_x;   // bf16 [W*A][h]
  size_t ffn_assist;     // int32 [W*A][3]
  size_t ffn_ep;         // int32 [W][L*W]
  size_t ffn_h1;         // bf16 [W*A][I]
  size_t ffn_y;          // bf16 [W*A][h]
  size_t ffn_done;       // uint32 [E] gate/up epilogue warps finished per expert
  size_t total;
};

struct Shape {
  int W, bs, h, K, E, L, Z, C;
  int mask_kind, quant, x_dtype;
  int ytype;         // MOE_Y_* of quantised rows
  int scales_kind;   // MOE_SCALES_* of the scales input
  int ngroups;       // dynamic-scale entries per row (mode 2: 1; 3: ceil(h/128); 4: ceil(h/32))
  int64_t A;         // rows per rank
  int es;            // element bytes of x
  int row_in;        // h * es
  int row_out;       // bytes of an expand_x row (h for int8)
};

struct RouteParams {
  const int32_t* ids;
  const uint8_t* mask;
  Shape sh;
  int32_t* cnt;
  int32_t* rank;
  int32_t* base;
  int32_t* ep_recv_count;
  uint8_t* plane;
  uint8_t* seg_plane_out;  // optional user copy of plane
  int plane_policy;
  int bulk_ok;             // rows and pointers allow TMA bulk copies
  int64_t bulk_min_bytes;
  uint32_t* done;
  int* status;
  uint32_t* landed;        // per-segment rows in place (zeroed here when flags are on)
  uint32_t* seg_ready;     // optional ready flags
  uint32_t ticket;
  WsHeader* hdr;           // records which assist_info / ep_recv_count the pick -> row map belongs to
  const int32_t* assist_out;
  uint32_t* zero_words;    // optional: words the routing kernel clears for the kernels after it
  int n_zero_words;
#ifdef MOE_PHASE_TIMES
  unsigned long long* phase;  // test builds: per-kernel phase times
#endif
};

#ifdef MOE_FLAG_OBSERVER
// Test builds only (-DMOE_FLAG_OBSERVER): where the flag observer of the
// dispatch payload kernels copies each segment the moment its ready flag shows
// the call's ticket (see observe_flags in scatter_common.cuh).
struct FlagObserver {
  uint8_t* rows;                        // [W][A][row bytes], like expand_x
  int32_t* assist;                      // [W][A][3], like assist_info
  uint8_t* dyn;                         // like dynamic_scales (quantised modes), or null
  unsigned long long* seen_ns;          // [E*W] %globaltimer once the segment's copy was taken
  unsigned long long* producer_end_ns;  // latest end of a storing CTA
  uint32_t* n_seen;                     // segments seen
};
#endif

struct ScatterParams {
  const void* x;
  const int32_t* ids;
  const uint8_t* mask;
  const void* scales;      // may be null
  void* expand_x;
  void* dyn_scales;        // per-row dynamic scales (fp32; E8M0 bytes for quant 4)
  const float* qscales;    // scales input (static coefficients / smoothing weights), or null
  int32_t* assist;
  void* expand_scales;     // may be null
  const int32_t* rank;
  const int32_t* base;
  const uint8_t* plane;
  const int32_t* cnt;      // rows per segment
  uint32_t* landed;        // per-segment rows in place
  uint32_t* seg_ready;     // optional ready flags
  uint32_t ticket;
  int32_t* inv;                    // pick -> flat row map (workspace), written for every routed pick
  int stream_below;                // TMA scatter with streaming stores: tokens below this index use them
  int64_t* perf;                   // per-rank communication time (user array [W]), or null
  unsigned long long* perf_end;    // [W] workspace
  WsHeader* hdr;
  Shape sh;
  int* status;
  uint64_t timeout_ns;
#ifdef MOE_FLAG_OBSERVER
  FlagObserver obs;
  int observe;  // the grid's last CTA observes instead of storing
#endif
#ifdef MOE_PHASE_TIMES
  unsigned long long* phase;  // test builds: per-kernel phase times
#endif
};

struct CombineParams {
  const void* expert_out;
  const int32_t* assist;
  const int32_t* ep_recv_count;
  const int32_t* ids;
  const void* scales;
  const uint8_t* mask;
  const void* x;
  void* x_out;
  int32_t* inv;
  Shape sh;
  int* status;
  // two-phase
  void* window;
  uint32_t* flags;
  uint8_t* plane;
  uint8_t* seg_plane_out;
  WsHeader* hdr;
  int plane_policy;
  int bulk_ok;
  int64_t bulk_min_bytes;
  int put_only;
  int tp_rows;             // two-phase: rows per warp batch (1..32)
  uint64_t timeout_ns;
#ifdef MOE_PHASE_TIMES
  unsigned long long* phase;  // test builds: per-kernel phase times
#endif
};

// Everything the expert-FFN grouped GEMMs need.
struct FfnLaunch {
  Shape sh;
  int I;                   // intermediate size
  const void* w_gate;      // [E][I][h] bf16
  const void* w_up;        // [E][I][h] bf16
  const void* w_down;      // [E][h][I] bf16
  const void* expand_x;    // [W*A][h] bf16 (dispatch output)
  void* h1;                // [W*A][I] bf16
  void* y;                 // [W*A][h] bf16 (expert outputs)
  const int32_t* ep;       // [W][L*W] running receive counts
  uint32_t* done;          // [E] per-expert gate/up completion counters (cleared by the routing kernel)
  int* status;
  uint64_t timeout_ns;
};

// CTAs of `kernel` resident per SM with `threads` threads and `smem` bytes of
// dynamic shared memory on the current device, after raising the kernel's
// dynamic shared-memory limit to `smem`. Both steps are host calls of a few
// microseconds; the answer is cached per (device, kernel, threads, smem).
cudaError_t resident_blocks(const void* kernel, int threads, size_t smem, int* per_sm);

// True when the TMA scatter's shared-memory ring fits for this shape.
bool scatter_tma_fits(const Shape& sh);
// The quantising scatter (every quant_mode but 0) and its fit test.
bool scatter_quant_tma_fits(const Shape& sh);
cudaError_t launch_scatter_quant(const ScatterParams& p, cudaStream_t st, int num_sms, bool tma);
inline bool uses_scatter_quant(const Shape& sh) { return sh.quant != 0; }
// The expert-major payload of per-group FP8 with per-expert scales (row map kernel +
// payload kernel); `launches` receives the number of kernels enqueued.
bool uses_scatter_pe(const Shape& sh);
cudaError_t launch_scatter_pe(const ScatterParams& p, const int32_t* ep_recv_count, int4* list, cudaStream_t st,
                              int num_sms, int* launches);

// Launchers (each returns the launch error, if any).
cudaError_t launch_route(const RouteParams& p, cudaStream_t st);
cudaError_t launch_scatter(const ScatterParams& p, cudaStream_t st, int num_sms, bool tma);
cudaError_t launch_combine_inverse(const CombineParams& p, cudaStream_t st);
cudaError_t launch_combine_reduce(const CombineParams& p, cudaStream_t st, int num_sms);
cudaError_t launch_combine_two_phase(const CombineParams& p, cudaStream_t st, int num_sms);
cudaError_t launch_ffn(const FfnLaunch& f, cudaStream_t st, int num_sms, void* const* prof_events);

// Launch config helper: programmatic dependent launch on `st`.
struct PdlLaunch {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t st) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
};

}  // namespace crs
