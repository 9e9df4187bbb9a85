// moe_combine_noalloc: the gather combine for callers that cannot allocate
// device memory. Same kernels and results as moe_combine in
// MOE_COMBINE_GATHER mode; the only difference is where the scratch lives.
//
// moe_combine needs a caller-allocated workspace for its pick -> row map.
// Some callers have no way to provide one: a plugin or custom-op host that
// hands the library only its input and output buffers, or a serving loop that
// must not allocate after start-up (an allocation can synchronise the device
// or fail under memory pressure in the middle of a step). For them the map
// lives here, in a fixed device array that every GPU loading this library
// holds until the process exits.
//
// Limits and rules:
//   * at most kNoAllocMaxPicks = 262144 picks (W * bs * topk) per call, i.e.
//     1 MiB of scratch per device; larger calls are rejected with
//     MOE_ERR_INVALID_ARG before anything is enqueued;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture;
//   * every call on a device shares the one array and it keeps the last call's
//     contents (nothing in it needs to start at zero: each call rewrites the
//     entries it reads). Calls that overlap on the GPU, on different streams,
//     race on it and must be serialised by the caller;
//   * device-side errors go to the caller's `status` word (set to 0 by the
//     call before its kernels run);
//   * nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "internal.h"

namespace crs {
void note_launches(int n);  // moe_api.cu: the library's launch count
}

namespace {

constexpr long long kNoAllocMaxPicks = 262144;

// The scratch: pick -> flat expert-output row. In host code this name is only
// a stand-in; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) int32_t g_noalloc_inv[kNoAllocMaxPicks];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_inv_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Device address of the scratch and the SM count of the current device,
// looked up once per device.
moe_status_t scratch_for_current_device(int32_t** inv, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_inv_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_inv) != cudaSuccess || !p) return MOE_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return MOE_ERR_CUDA;
    g_inv_ptr[dev] = static_cast<int32_t*>(p);
    g_num_sms[dev] = n;
  }
  *inv = g_inv_ptr[dev];
  *num_sms = g_num_sms[dev];
  return MOE_OK;
}

bool aligned_to(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" moe_status_t moe_combine_noalloc(const moe_config_t* cfg, const void* expert_out,
                                            const int32_t* assist_info, const int32_t* ep_recv_count,
                                            const int32_t* expert_ids, const void* expert_scales,
                                            const uint8_t* active_mask, const void* x, void* x_out, int32_t* status,
                                            void* stream) {
  // the configuration rules of every other entry point
  int64_t A = 0;
  moe_status_t st = moe_get_workspace_size(cfg, nullptr, &A);
  if (st != MOE_OK) return st;
  if (cfg->quant_mode != 0 || cfg->combine_mode != MOE_COMBINE_GATHER) return MOE_ERR_UNSUPPORTED;
  const long long picks = (long long)cfg->ep_world_size * cfg->bs * cfg->topk;
  if (picks > kNoAllocMaxPicks) return MOE_ERR_INVALID_ARG;
  const bool empty = picks == 0;
  if (!status || !ep_recv_count) return MOE_ERR_INVALID_ARG;
  if (!empty && (!expert_out || !assist_info || !expert_ids || !expert_scales || !x_out))
    return MOE_ERR_INVALID_ARG;
  if (cfg->mask_kind != 0 && !active_mask && !empty) return MOE_ERR_INVALID_ARG;
  if (cfg->copy_expert_num > 0 && !x && !empty) return MOE_ERR_INVALID_ARG;
  if (!aligned_to(expert_out, 16) || !aligned_to(x, 16) || !aligned_to(x_out, 16) ||
      !aligned_to(assist_info, 4) || !aligned_to(ep_recv_count, 4) || !aligned_to(expert_ids, 4) ||
      !aligned_to(expert_scales, 4) || !aligned_to(status, 4))
    return MOE_ERR_INVALID_ARG;

  int32_t* inv = nullptr;
  int nsm = 0;
  st = scratch_for_current_device(&inv, &nsm);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (empty) return MOE_OK;

  crs::Shape sh{};
  sh.W = cfg->ep_world_size;
  sh.bs = cfg->bs;
  sh.h = cfg->h;
  sh.K = cfg->topk;
  sh.E = cfg->moe_expert_num;
  sh.L = cfg->moe_expert_num / cfg->ep_world_size;
  sh.Z = cfg->zero_expert_num;
  sh.C = cfg->copy_expert_num;
  sh.mask_kind = cfg->mask_kind;
  sh.quant = 0;
  sh.x_dtype = cfg->x_dtype;
  sh.A = A;
  sh.es = cfg->x_dtype == MOE_I32 ? 4 : 2;
  sh.row_in = cfg->h * sh.es;
  sh.row_out = sh.row_in;

  crs::CombineParams cp{};
  cp.expert_out = expert_out;
  cp.assist = assist_info;
  cp.ep_recv_count = ep_recv_count;
  cp.ids = expert_ids;
  cp.scales = expert_scales;
  cp.mask = cfg->mask_kind ? active_mask : nullptr;
  cp.x = x;
  cp.x_out = x_out;
  cp.inv = inv;
  cp.sh = sh;
  cp.status = status;
  if (crs::launch_combine_inverse(cp, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (crs::launch_combine_reduce(cp, s, nsm) != cudaSuccess) return MOE_ERR_CUDA;
  crs::note_launches(2);
  return MOE_OK;
}
