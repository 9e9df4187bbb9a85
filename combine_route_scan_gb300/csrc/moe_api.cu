// Host side of the C ABI declared in include/moe.h: argument validation
// (value ranges of aclnnMoeDistributeDispatchV4, 参数说明), the workspace
// layout (first phase of its GetWorkspaceSize + execute contract) and the
// kernel launches, chained on the caller's stream with programmatic
// dependent launch.
#include <string.h>

#include <atomic>
#include <mutex>

#include "internal.h"

namespace crs {

namespace {
std::atomic<uint64_t> g_launches{0};
}
// n more kernels were enqueued (moe_launch_count)
void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

cudaError_t resident_blocks(const void* kernel, int threads, size_t smem, int* per_sm) {
  // The dynamic shared-memory limit is state of the kernel, not of one call:
  // it is only ever raised (to the largest size asked for so far), so a call
  // with a smaller size never lowers it under a later, larger one.
  struct Limit {
    const void* kernel;
    int dev;
    size_t smem;
  };
  struct Occupancy {
    const void* kernel;
    int dev, threads;
    size_t smem;
    int per_sm;
  };
  static Limit limits[128];
  static Occupancy occ[256];
  static int n_limits = 0, n_occ = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  Limit* lim = nullptr;
  for (int i = 0; i < n_limits; ++i)
    if (limits[i].kernel == kernel && limits[i].dev == dev) lim = &limits[i];
  if (!lim || lim->smem < smem) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (lim) lim->smem = smem;
    else if (n_limits < 128) limits[n_limits++] = Limit{kernel, dev, smem};
  }
  for (int i = 0; i < n_occ; ++i) {
    const Occupancy& t = occ[i];
    if (t.kernel == kernel && t.dev == dev && t.threads == threads && t.smem == smem) {
      *per_sm = t.per_sm;
      return cudaSuccess;
    }
  }
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  if (n_occ < 256) occ[n_occ++] = Occupancy{kernel, dev, threads, smem, n};
  *per_sm = n;
  return cudaSuccess;
}

}  // namespace crs

using namespace crs;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int elem_bytes(int dt) { return dt == MOE_I32 ? 4 : 2; }

moe_status_t make_shape(const moe_config_t* c, Shape* sh) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->ep_world_size < 2 || c->ep_world_size > 768) return MOE_ERR_INVALID_ARG;
  if (c->moe_expert_num <= 0 || c->moe_expert_num > 1024 || c->moe_expert_num % c->ep_world_size)
    return MOE_ERR_INVALID_ARG;
  if (c->bs < 0 || c->h <= 0 || c->topk < 1 || c->topk > 32) return MOE_ERR_INVALID_ARG;
  if (c->zero_expert_num < 0 || c->copy_expert_num < 0 || c->const_expert_num < 0) return MOE_ERR_INVALID_ARG;
  if ((long long)c->moe_expert_num + c->zero_expert_num + c->copy_expert_num + c->const_expert_num >=
      2147483647LL)
    return MOE_ERR_INVALID_ARG;
  if (c->const_expert_num != 0) return MOE_ERR_UNSUPPORTED;
  if (c->mask_kind < 0 || c->mask_kind > 2) return MOE_ERR_INVALID_ARG;
  if (c->x_dtype < MOE_I32 || c->x_dtype > MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->quant_mode < 0 || c->quant_mode > 4) return MOE_ERR_UNSUPPORTED;
  if (c->expand_dtype < MOE_Y_DEFAULT || c->expand_dtype > MOE_Y_FP4_E2M1 ||
      c->scales_kind < MOE_SCALES_NONE || c->scales_kind > MOE_SCALES_EXPERT)
    return MOE_ERR_INVALID_ARG;
  if (c->quant_mode == 0) {
    if (c->expand_dtype != MOE_Y_DEFAULT || c->scales_kind != MOE_SCALES_NONE) return MOE_ERR_INVALID_ARG;
  } else {
    if (c->x_dtype == MOE_I32) return MOE_ERR_UNSUPPORTED;
    const int y = c->expand_dtype, k = c->scales_kind;
    const bool smooth_ok = k == MOE_SCALES_NONE || k == MOE_SCALES_EXPERT;
    bool ok;
    switch (c->quant_mode) {
      case 1: ok = y == MOE_Y_DEFAULT && k != MOE_SCALES_NONE; break;
      case 2: ok = y == MOE_Y_DEFAULT && smooth_ok; break;
      case 3: ok = (y == MOE_Y_FP8_E4M3 || y == MOE_Y_FP8_E5M2) && smooth_ok; break;
      default: ok = y != MOE_Y_DEFAULT && k == MOE_SCALES_NONE && (y != MOE_Y_FP4_E2M1 || c->h % 2 == 0); break;
    }
    if (!ok) return MOE_ERR_INVALID_ARG;
  }
  if (c->plane_policy < MOE_PLANE_RULE || c->plane_policy > MOE_PLANE_BULK_ALL) return MOE_ERR_INVALID_ARG;
  if (c->bulk_min_bytes < 0) return MOE_ERR_INVALID_ARG;
  if (c->combine_mode < MOE_COMBINE_GATHER || c->combine_mode > MOE_COMBINE_PUT_ONLY) return MOE_ERR_INVALID_ARG;
  if (c->wait_timeout_us <= 0) return MOE_ERR_INVALID_ARG;
  if (c->ffn_intermediate < 0) return MOE_ERR_INVALID_ARG;
  const long long picks = (long long)c->ep_world_size * c->bs * c->topk;
  if (picks >= 2147483647LL) return MOE_ERR_INVALID_ARG;
  sh->W = c->ep_world_size;
  sh->bs = c->bs;
  sh->h = c->h;
  sh->K = c->topk;
  sh->E = c->moe_expert_num;
  sh->L = c->moe_expert_num / c->ep_world_size;
  sh->Z = c->zero_expert_num;
  sh->C = c->copy_expert_num;
  sh->mask_kind = c->mask_kind;
  sh->quant = c->quant_mode;
  sh->x_dtype = c->x_dtype;
  sh->A = (int64_t)c->bs * c->ep_world_size * (sh->L < sh->K ? sh->L : sh->K);
  sh->es = elem_bytes(c->x_dtype);
  const long long row_in = (long long)c->h * sh->es;
  if (row_in > (1LL << 30)) return MOE_ERR_INVALID_ARG;
  sh->row_in = (int)row_in;
  sh->ytype = c->expand_dtype;
  sh->scales_kind = c->scales_kind;
  sh->ngroups = c->quant_mode == 2 ? 1 : c->quant_mode == 3 ? (c->h + 127) / 128
              : c->quant_mode == 4 ? (c->h + 31) / 32 : 0;
  if (c->quant_mode == 0) sh->row_out = sh->row_in;
  else if (c->quant_mode == 4 && c->expand_dtype == MOE_Y_FP4_E2M1) sh->row_out = c->h / 2;
  else sh->row_out = c->h;
  if ((long long)sh->W * sh->A >= 2147483647LL) return MOE_ERR_INVALID_ARG;  // flat rows fit int32
  return MOE_OK;
}

WsLayout make_layout(const moe_config_t* c, const Shape& sh) {
  WsLayout L{};
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  const size_t segs = (size_t)sh.E * sh.W;
  const size_t picks = (size_t)sh.W * sh.bs * sh.K;
  L.cnt = take(segs * 4);
  L.base = take(segs * 4);
  L.plane_d = take(segs);
  L.landed = take(segs * 4);
  L.perf_end = take((size_t)sh.W * 8);
  L.rank = take(picks * 4);
  L.inv = take(picks * 4);
  if ((c->quant_mode == 2 || c->quant_mode == 3) && c->scales_kind == MOE_SCALES_EXPERT) L.pe_list = take((size_t)sh.W * sh.A * 16);
  if (c->combine_mode != MOE_COMBINE_GATHER) {
    L.plane_c = take(segs);
    L.flags = take(picks * 4);
    L.window = take(picks * (size_t)sh.row_in);
  }
  if (c->ffn_intermediate > 0) {
    const size_t rows = (size_t)sh.W * sh.A;
    L.ffn_expand_x = take(rows * sh.h * 2);
    L.ffn_assist = take(rows * 12);
    L.ffn_ep = take(segs * 4);
    L.ffn_h1 = take(rows * (size_t)c->ffn_intermediate * 2);
    L.ffn_y = take(rows * sh.h * 2);
    L.ffn_done = take((size_t)sh.E * 4);
  }
  L.total = off;
  return L;
}

int num_sms_of_current_device() {
  static std::atomic<int> cache[64] = {};  // callers may be on several host threads
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

uint64_t timeout_ns(const moe_config_t* c) { return (uint64_t)c->wait_timeout_us * 1000ull; }

moe_status_t check_ws(const moe_config_t* c, const Shape& sh, void* ws, size_t ws_bytes, WsLayout* L) {
  *L = make_layout(c, sh);
  if (!ws || ws_bytes < L->total || !aligned(ws, kAlign)) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status_t record(void* const* ev, int which, cudaStream_t st) {
  if (!ev || !ev[which]) return MOE_OK;
  return cudaEventRecord(static_cast<cudaEvent_t>(ev[which]), st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

extern "C" {

moe_status_t moe_get_workspace_size(const moe_config_t* cfg, size_t* ws_bytes, int64_t* rows_per_rank) {
  Shape sh;
  moe_status_t st = make_shape(cfg, &sh);
  if (st != MOE_OK) return st;
  const WsLayout L = make_layout(cfg, sh);
  if (ws_bytes) *ws_bytes = L.total;
  if (rows_per_rank) *rows_per_rank = sh.A;
  return MOE_OK;
}

// Which assist_info / ep_recv_count the pick -> row map in each workspace was
// last written for, as far as this process enqueued it, so that a combine of
// those very buffers can skip the inverse-map pass. The addresses are
// compared, never dereferenced. A dispatch captured into a CUDA graph may be
// replayed at any later time and overwrite the map unseen, so it marks the
// workspace: from then on only a combine captured in the same capture
// sequence as the dispatch (the graph replays the two in order) skips the
// pass; every other combine on that workspace runs it, and the inverse kernel
// itself returns at once when the routing kernel's record in the workspace
// header shows the map already belongs to its buffers. moe_workspace_init
// clears the mark.
namespace {
struct MapOwner {
  const void* ws;
  const void* assist;
  const void* ep;
  unsigned long long capture;  // capture sequence of the dispatch, 0 = not captured
  bool graphed;                // some dispatch on this workspace was captured
};
std::mutex g_owner_mu;
MapOwner g_owner[256];
int g_owner_next = 0;

// Capture sequence of `s` (0 when the stream is not capturing).
unsigned long long capture_id(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  unsigned long long id = 0;
  if (cudaStreamGetCaptureInfo(s, &st, &id) != cudaSuccess) {
    cudaGetLastError();
    return ~0ull;  // unknown: treated as a capture that matches nothing
  }
  return st == cudaStreamCaptureStatusNone ? 0ull : id;
}

MapOwner* owner_slot(const void* ws) {
  for (MapOwner& o : g_owner)
    if (o.ws == ws) return &o;
  MapOwner* o = &g_owner[g_owner_next];
  g_owner_next = (g_owner_next + 1) % 256;
  *o = MapOwner{ws, nullptr, nullptr, 0ull, false};
  return o;
}

void set_map_owner(const void* ws, const void* assist, const void* ep, cudaStream_t s) {
  const unsigned long long cap = capture_id(s);
  std::lock_guard<std::mutex> lock(g_owner_mu);
  MapOwner* o = owner_slot(ws);
  o->assist = assist;
  o->ep = ep;
  o->capture = cap;
  if (cap != 0) o->graphed = true;
}

void reset_map_owner(const void* ws) {
  std::lock_guard<std::mutex> lock(g_owner_mu);
  *owner_slot(ws) = MapOwner{ws, nullptr, nullptr, 0ull, false};
}

bool map_owned_by(const void* ws, const void* assist, const void* ep, cudaStream_t s) {
  const unsigned long long cap = capture_id(s);
  std::lock_guard<std::mutex> lock(g_owner_mu);
  for (const MapOwner& o : g_owner)
    if (o.ws == ws)
      return assist != nullptr && o.assist == assist && o.ep == ep && o.capture == cap && cap != ~0ull &&
             (cap != 0 || !o.graphed);
  return false;
}
}  // namespace

moe_status_t moe_workspace_init(const moe_config_t* cfg, void* ws, size_t ws_bytes, void* stream) {
  Shape sh;
  moe_status_t st = make_shape(cfg, &sh);
  if (st != MOE_OK) return st;
  WsLayout L;
  st = check_ws(cfg, sh, ws, ws_bytes, &L);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), s) != cudaSuccess) return MOE_ERR_CUDA;
  reset_map_owner(ws);
  if (cudaMemsetAsync(static_cast<uint8_t*>(ws) + L.perf_end, 0, (size_t)sh.W * 8, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (L.flags && cudaMemsetAsync(static_cast<uint8_t*>(ws) + L.flags, 0,
                                 (size_t)sh.W * sh.bs * sh.K * 4, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

#ifdef MOE_PHASE_TIMES
namespace {
std::atomic<unsigned long long*> g_phase{nullptr};
}  // namespace

// Test builds only (not declared in include/moe.h): the kernels of the next
// calls record their phase times into `buf`, a device array of 16 words
// (4 a kernel: routing, scatter, inverse map, reduce; see PhaseScope), which
// the caller zeroes before a call. NULL turns the recording off.
moe_status_t moe_test_set_phase_buffer(void* buf) {
  g_phase.store(static_cast<unsigned long long*>(buf));
  return MOE_OK;
}
#endif

#ifdef MOE_FLAG_OBSERVER
namespace {
std::mutex g_observer_mu;
bool g_observer_on = false;
FlagObserver g_observer{};
}  // namespace

// Test builds only (not declared in include/moe.h): the next dispatches with
// ready flags run the flag observer of their payload grid, which copies each
// segment the moment its flag shows the call's ticket into these device
// buffers (rows like expand_x, assist like assist_info, dyn like
// dynamic_scales or NULL; seen_ns [E*W] and producer_end_ns, n_seen single
// words). rows == NULL turns the observer off.
moe_status_t moe_test_set_flag_observer(void* rows, void* assist, void* dyn, void* seen_ns, void* producer_end_ns,
                                        void* n_seen) {
  std::lock_guard<std::mutex> lock(g_observer_mu);
  g_observer_on = rows != nullptr;
  if (g_observer_on && (!assist || !seen_ns || !producer_end_ns || !n_seen || !aligned(rows, 16)))
    return MOE_ERR_INVALID_ARG;
  g_observer = FlagObserver{static_cast<uint8_t*>(rows), static_cast<int32_t*>(assist), static_cast<uint8_t*>(dyn),
                            static_cast<unsigned long long*>(seen_ns),
                            static_cast<unsigned long long*>(producer_end_ns), static_cast<uint32_t*>(n_seen)};
  return MOE_OK;
}
#endif

moe_status_t moe_dispatch(const moe_config_t* cfg, const void* x, const int32_t* expert_ids,
                          const uint8_t* active_mask, const void* expert_scales, const float* scales,
                          void* expand_x, void* dynamic_scales, int32_t* assist_info, int32_t* ep_recv_count,
                          void* expand_scales, uint8_t* seg_plane, void* ws, size_t ws_bytes, void* stream) {
  Shape sh;
  moe_status_t st = make_shape(cfg, &sh);
  if (st != MOE_OK) return st;
  const bool empty = sh.W * (long long)sh.bs == 0;
  if (!empty && (!x || !expert_ids || !expand_x || !assist_info)) return MOE_ERR_INVALID_ARG;
  if (!ep_recv_count) return MOE_ERR_INVALID_ARG;
  if (sh.mask_kind != 0 && !active_mask && !empty) return MOE_ERR_INVALID_ARG;
  if (expand_scales && !expert_scales) return MOE_ERR_INVALID_ARG;
  if (sh.ngroups > 0 && !dynamic_scales && !empty) return MOE_ERR_INVALID_ARG;
  if ((sh.scales_kind != MOE_SCALES_NONE) != (scales != nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(expand_x, 16) || !aligned(expert_ids, 4) || !aligned(expert_scales, 4) ||
      !aligned(assist_info, 4) || !aligned(ep_recv_count, 4) || !aligned(expand_scales, 4) ||
      !aligned(dynamic_scales, 4) || !aligned(scales, 16) || !aligned(cfg->seg_ready, 4) ||
      !aligned(cfg->performance_info, 8))
    return MOE_ERR_INVALID_ARG;
  WsLayout L;
  st = check_ws(cfg, sh, ws, ws_bytes, &L);
  if (st != MOE_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(ws);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nsm = num_sms_of_current_device();
  if (nsm <= 0) return MOE_ERR_CUDA;

  const bool quant_kernel = uses_scatter_quant(sh);
  const bool tma = sh.row_in % 16 == 0 && sh.row_out % 16 == 0 &&
                   (quant_kernel ? scatter_quant_tma_fits(sh) : scatter_tma_fits(sh));

  RouteParams rp{};
  rp.ids = expert_ids;
  rp.mask = sh.mask_kind ? active_mask : nullptr;
  rp.sh = sh;
  rp.cnt = reinterpret_cast<int32_t*>(w + L.cnt);
  rp.rank = reinterpret_cast<int32_t*>(w + L.rank);
  rp.base = reinterpret_cast<int32_t*>(w + L.base);
  rp.ep_recv_count = ep_recv_count;
  rp.plane = w + L.plane_d;
  rp.seg_plane_out = seg_plane;
  rp.plane_policy = cfg->plane_policy;
  rp.bulk_ok = tma ? 1 : 0;
  rp.bulk_min_bytes = cfg->bulk_min_bytes;
  rp.done = &hdr->route_done;
  rp.status = &hdr->status;
  rp.landed = reinterpret_cast<uint32_t*>(w + L.landed);
  rp.seg_ready = cfg->seg_ready;
  rp.ticket = cfg->seg_ready_ticket;
  rp.hdr = hdr;
  rp.assist_out = assist_info;
#ifdef MOE_PHASE_TIMES
  rp.phase = g_phase.load();
#endif
  if (launch_route(rp, s) != cudaSuccess) return MOE_ERR_CUDA;
  note_launches(1);

  ScatterParams sp{};
  sp.cnt = rp.cnt;
  sp.landed = rp.landed;
  sp.seg_ready = cfg->seg_ready;
  sp.ticket = cfg->seg_ready_ticket;
  sp.inv = reinterpret_cast<int32_t*>(w + L.inv);
  sp.perf = cfg->performance_info;
  sp.perf_end = reinterpret_cast<unsigned long long*>(w + L.perf_end);
  sp.hdr = hdr;
  sp.x = x;
  sp.ids = expert_ids;
  sp.mask = rp.mask;
  sp.scales = expert_scales;
  sp.expand_x = expand_x;
  sp.dyn_scales = dynamic_scales;
  sp.qscales = scales;
  sp.assist = assist_info;
  sp.expand_scales = expand_scales;
  sp.rank = rp.rank;
  sp.base = rp.base;
  sp.plane = rp.plane;
  sp.sh = sh;
  sp.status = &hdr->status;
  sp.timeout_ns = timeout_ns(cfg);
#ifdef MOE_PHASE_TIMES
  sp.phase = g_phase.load();
#endif
#ifdef MOE_FLAG_OBSERVER
  {
    std::lock_guard<std::mutex> lock(g_observer_mu);
    // observed: 16-byte rows on the token-major kernels, flags on, at most 64
    // segments a thread of the observing CTA
    sp.observe = g_observer_on && cfg->seg_ready && tma && !(quant_kernel && uses_scatter_pe(sh)) &&
                 (long long)sh.E * sh.W <= 64LL * 256 && !cfg->performance_info;
    sp.obs = g_observer;
  }
#endif
  if (record(cfg->prof_events, 0, s) != MOE_OK) return MOE_ERR_CUDA;
  if (quant_kernel && tma && uses_scatter_pe(sh)) {
    int launched = 0;
    const cudaError_t e =
        launch_scatter_pe(sp, ep_recv_count, reinterpret_cast<int4*>(w + L.pe_list), s, nsm, &launched);
    note_launches(launched);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    const cudaError_t e = quant_kernel ? launch_scatter_quant(sp, s, nsm, tma) : launch_scatter(sp, s, nsm, tma);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (!empty) note_launches(1);
  }
  set_map_owner(ws, assist_info, ep_recv_count, s);  // the scatter writes the map for these buffers
  if (record(cfg->prof_events, 1, s) != MOE_OK) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* expert_out, const int32_t* assist_info,
                         const int32_t* ep_recv_count, const int32_t* expert_ids, const void* expert_scales,
                         const uint8_t* active_mask, const void* x, void* x_out, uint8_t* seg_plane, void* ws,
                         size_t ws_bytes, void* stream) {
  Shape sh;
  moe_status_t st = make_shape(cfg, &sh);
  if (st != MOE_OK) return st;
  if (cfg->quant_mode != 0) return MOE_ERR_UNSUPPORTED;  // expert outputs are in x's type
  const bool empty = sh.W * (long long)sh.bs == 0;
  if (!ep_recv_count) return MOE_ERR_INVALID_ARG;
  if (!empty && (!expert_out || !assist_info || !expert_ids || !expert_scales)) return MOE_ERR_INVALID_ARG;
  if (!empty && cfg->combine_mode != MOE_COMBINE_PUT_ONLY && !x_out) return MOE_ERR_INVALID_ARG;
  if (sh.mask_kind != 0 && !active_mask && !empty) return MOE_ERR_INVALID_ARG;
  if (sh.C > 0 && !x && !empty) return MOE_ERR_INVALID_ARG;
  if (!aligned(expert_out, 16) || !aligned(x, 16) || !aligned(x_out, 16) || !aligned(assist_info, 4) ||
      !aligned(ep_recv_count, 4) || !aligned(expert_ids, 4) || !aligned(expert_scales, 4))
    return MOE_ERR_INVALID_ARG;
  WsLayout L;
  st = check_ws(cfg, sh, ws, ws_bytes, &L);
  if (st != MOE_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(ws);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nsm = num_sms_of_current_device();
  if (nsm <= 0) return MOE_ERR_CUDA;

  CombineParams cp{};
  cp.expert_out = expert_out;
  cp.assist = assist_info;
  cp.ep_recv_count = ep_recv_count;
  cp.ids = expert_ids;
  cp.scales = expert_scales;
  cp.mask = sh.mask_kind ? active_mask : nullptr;
  cp.x = x;
  cp.x_out = x_out;
  cp.inv = reinterpret_cast<int32_t*>(w + L.inv);
  cp.sh = sh;
  cp.status = &hdr->status;
  cp.hdr = hdr;
  cp.plane_policy = cfg->plane_policy;
  cp.bulk_min_bytes = cfg->bulk_min_bytes;
  cp.timeout_ns = timeout_ns(cfg);
#ifdef MOE_PHASE_TIMES
  cp.phase = g_phase.load();
#endif
  cp.seg_plane_out = seg_plane;
  if (empty) return MOE_OK;
  if (cfg->combine_mode == MOE_COMBINE_GATHER) {
    // the map of the dispatch that wrote these buffers on this workspace is
    // used as it is; otherwise it is rebuilt from assist_info first
    if (!map_owned_by(ws, assist_info, ep_recv_count, s)) {
      if (launch_combine_inverse(cp, s) != cudaSuccess) return MOE_ERR_CUDA;
      note_launches(1);
    }
    if (record(cfg->prof_events, 0, s) != MOE_OK) return MOE_ERR_CUDA;
    if (launch_combine_reduce(cp, s, nsm) != cudaSuccess) return MOE_ERR_CUDA;
    note_launches(1);
  } else {
    cp.window = w + L.window;
    cp.flags = reinterpret_cast<uint32_t*>(w + L.flags);
    cp.plane = w + L.plane_c;
    cp.bulk_ok = sh.row_in % 16 == 0 && aligned(expert_out, 16);
    cp.put_only = cfg->combine_mode == MOE_COMBINE_PUT_ONLY;
    if (record(cfg->prof_events, 0, s) != MOE_OK) return MOE_ERR_CUDA;
    cudaError_t e = launch_combine_two_phase(cp, s, nsm);
    if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    note_launches(1);
  }
  if (record(cfg->prof_events, 1, s) != MOE_OK) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_dispatch_ffn_combine(const moe_config_t* cfg, const void* x, const int32_t* expert_ids,
                                      const uint8_t* active_mask, const float* expert_scales, const void* w_gate,
                                      const void* w_up, const void* w_down, void* x_out, void* ws, size_t ws_bytes,
                                      void* stream) {
  Shape sh;
  moe_status_t st = make_shape(cfg, &sh);
  if (st != MOE_OK) return st;
  const int I = cfg->ffn_intermediate;
  if (cfg->x_dtype != MOE_BF16 || cfg->quant_mode != 0 || cfg->combine_mode != MOE_COMBINE_GATHER)
    return MOE_ERR_UNSUPPORTED;
  // tensor-core tiles: 128 intermediate rows per gate/up tile, 256 output rows
  // per down tile, 64-element K blocks
  if (I <= 0 || I % 128 != 0 || sh.h % 256 != 0) return MOE_ERR_UNSUPPORTED;
  const bool empty = sh.W * (long long)sh.bs == 0;
  if (!empty && (!x || !expert_ids || !expert_scales || !w_gate || !w_up || !w_down || !x_out))
    return MOE_ERR_INVALID_ARG;
  if (sh.mask_kind != 0 && !active_mask && !empty) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(x_out, 16) || !aligned(w_gate, 16) || !aligned(w_up, 16) ||
      !aligned(w_down, 16) || !aligned(expert_ids, 4) || !aligned(expert_scales, 4))
    return MOE_ERR_INVALID_ARG;
  WsLayout L;
  st = check_ws(cfg, sh, ws, ws_bytes, &L);
  if (st != MOE_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(ws);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nsm = num_sms_of_current_device();
  if (nsm <= 0) return MOE_ERR_CUDA;
  int32_t* ep = reinterpret_cast<int32_t*>(w + L.ffn_ep);
  int32_t* assist = reinterpret_cast<int32_t*>(w + L.ffn_assist);
  void* ex = w + L.ffn_expand_x;

  // 1. dispatch into the workspace
  const bool tma = sh.row_in % 16 == 0 && scatter_tma_fits(sh);
  RouteParams rp{};
  rp.ids = expert_ids;
  rp.mask = sh.mask_kind ? active_mask : nullptr;
  rp.sh = sh;
  rp.cnt = reinterpret_cast<int32_t*>(w + L.cnt);
  rp.rank = reinterpret_cast<int32_t*>(w + L.rank);
  rp.base = reinterpret_cast<int32_t*>(w + L.base);
  rp.ep_recv_count = ep;
  rp.plane = w + L.plane_d;
  rp.plane_policy = cfg->plane_policy;
  rp.bulk_ok = tma ? 1 : 0;
  rp.bulk_min_bytes = cfg->bulk_min_bytes;
  rp.done = &hdr->route_done;
  rp.status = &hdr->status;
  rp.hdr = hdr;
  rp.assist_out = assist;
#ifdef MOE_PHASE_TIMES
  rp.phase = g_phase.load();
#endif
  rp.zero_words = reinterpret_cast<uint32_t*>(w + L.ffn_done);
  rp.n_zero_words = sh.E;
  if (launch_route(rp, s) != cudaSuccess) return MOE_ERR_CUDA;
  note_launches(1);
  ScatterParams sp{};
  sp.x = x;
  sp.ids = expert_ids;
  sp.mask = rp.mask;
  sp.expand_x = ex;
  sp.assist = assist;
  sp.inv = reinterpret_cast<int32_t*>(w + L.inv);
  sp.rank = rp.rank;
  sp.base = rp.base;
  sp.plane = rp.plane;
  sp.sh = sh;
  sp.status = &hdr->status;
  sp.hdr = hdr;
  sp.timeout_ns = timeout_ns(cfg);
#ifdef MOE_PHASE_TIMES
  sp.phase = g_phase.load();
#endif
  if (!empty && launch_scatter(sp, s, nsm, tma) != cudaSuccess) return MOE_ERR_CUDA;
  if (empty) return MOE_OK;
  note_launches(1);
  set_map_owner(ws, assist, ep, s);  // the map now belongs to this call's own buffers

  // 2. expert FFN on the tensor cores: h1 = silu(x Wg^T) * (x Wu^T), y = h1 Wd^T
  FfnLaunch f{};
  f.sh = sh;
  f.I = I;
  f.w_gate = w_gate;
  f.w_up = w_up;
  f.w_down = w_down;
  f.expand_x = ex;
  f.h1 = w + L.ffn_h1;
  f.y = w + L.ffn_y;
  f.ep = ep;
  f.done = reinterpret_cast<uint32_t*>(w + L.ffn_done);
  f.status = &hdr->status;
  f.timeout_ns = timeout_ns(cfg);
  if (launch_ffn(f, s, nsm, cfg->prof_events) != cudaSuccess) return MOE_ERR_CUDA;
  note_launches(1);

  // 3. combine the expert outputs
  CombineParams cp{};
  cp.expert_out = f.y;
  cp.assist = assist;
  cp.ep_recv_count = ep;
  cp.ids = expert_ids;
  cp.scales = expert_scales;
  cp.mask = rp.mask;
  cp.x = x;
  cp.x_out = x_out;
  cp.inv = reinterpret_cast<int32_t*>(w + L.inv);
  cp.sh = sh;
  cp.status = &hdr->status;
  cp.hdr = hdr;
  // the scatter above wrote the pick -> row map: no inverse pass
  if (launch_combine_reduce(cp, s, nsm) != cudaSuccess) return MOE_ERR_CUDA;
  note_launches(1);
  return MOE_OK;
}

moe_status_t moe_get_device_status(void* ws, void* stream, int32_t* status) {
  if (!ws || !status) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  *status = v;
  return MOE_OK;
}

uint64_t moe_launch_count(void) { return crs::g_launches.load(std::memory_order_relaxed); }

const char* moe_status_string(int32_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MOE_ERR_BAD_EXPERT_ID: return "expert id out of range or repeated in a token";
    case MOE_ERR_MASK_ORDER: return "1D active mask has a true after a false";
    case MOE_ERR_TIMEOUT: return "bounded wait timed out";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_CAPACITY: return "receive capacity exceeded";
    case MOE_ERR_BAD_ASSIST: return "assist_info / ep_recv_count do not match the routing";
    case MOE_ERR_OUT_OF_BOUNDS: return "index outside its buffer (bounds-checked build)";
    default: return "unknown status";
  }
}

}  // extern "C"
