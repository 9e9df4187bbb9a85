// Dispatch -> per-expert SwiGLU FFN -> combine in one call (xLLM MegaMoe pull
// request, 背景与目标: dispatch, expert FFN with activation and combine as one
// operator; intermediate_hidden = 512 on A3).
//
// The expert FFN is a grouped GEMM over the contiguous row ranges dispatch
// leaves for each expert (ep_recv_count is local-expert major, so one expert's
// rows from every source are adjacent). It runs on the 5th-generation tensor
// cores:
//   * swap-AB: the weights are the MMA's A operand (M = 128 weight rows per
//     tile), the expert's tokens are B (N <= 64 per pass), so the weights, the
//     streamed operand, fill the 128-lane tile whatever the token count;
//   * weights are stored out-major (w_gate, w_up [E][I][h], w_down [E][h][I]),
//     so A and B are both K-major; TMA tensor loads with 128-byte swizzle put
//     64-element K blocks into shared memory in the layout tcgen05 reads;
//   * warp 0 issues the TMA loads into a 5-stage ring (mbarrier complete_tx),
//     one thread of warp 1 issues tcgen05.mma (bf16 x bf16 -> fp32 in TMEM)
//     and tcgen05.commit to release each stage, warps 2..5 drain the
//     accumulator with tcgen05.ld; two accumulator sets in TMEM let the MMAs of
//     the next unit run while the epilogue drains the last one;
//   * first GEMM: a unit = (expert, 128 rows of gate and the same 128 rows of
//     up); its epilogue computes h1 = bf16(silu(g) * u);
//   * second GEMM: a unit = (expert, 2 x 128 rows of down); its epilogue writes
//     the bf16 expert output y, which the gather combine then reduces.
// Both GEMMs run in one persistent launch (one CTA per SM, all resident: a
// cooperative launch): every CTA walks its share of the gate/up units and then
// of the down units, and a down unit waits (bounded) until every gate/up unit
// of its expert has stored its h1 rows, counted per expert in the workspace.
// So the SMs that finish their gate/up share early stream down weights while
// the last gate/up units run. Every wait is bounded and a timeout leaves
// MOE_ERR_TIMEOUT in the status word instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"

namespace crs {

constexpr int kFfnThreads = 192;  // warp 0: TMA, warp 1: MMA + TMEM, warps 2..5: epilogue
// 5 x 40 KB in flight a CTA: measured on GB300 at 8 ranks x 64 tokens, h 2048,
// 128 experts, both GEMMs 141.5 us with 4 stages, 137.3 us with 5 (6 do not fit)
constexpr int kFfnStages = 5;
constexpr int kNP = 64;  // tokens per MMA pass (MMA N)
constexpr int kT = 2;    // weight tiles per unit
constexpr int kBK = 64;  // K elements per k-block: 128 bytes of bf16, one swizzle span
constexpr uint32_t kATile = 128 * 128;
constexpr uint32_t kBTile = kNP * 128;
constexpr uint32_t kStage = kBTile + kT * kATile;
constexpr uint32_t kTmemCols = 2 * kT * kNP;
constexpr size_t kFfnSmem = (size_t)kFfnStages * kStage + 1024;  // + alignment to 1024
static_assert(kStage % 1024 == 0, "stages stay 1024-byte aligned");

enum { FFN_GATE_UP = 0, FFN_DOWN = 1 };

struct FfnParams {
  const int32_t* ep;   // running receive counts [W][L*W]
  __nv_bfloat16* h1;   // [W*A][I]: gate/up output, down input
  __nv_bfloat16* y;    // [W*A][h]: down output
  uint32_t* done;      // [E] gate/up epilogue warps finished per expert (zeroed by the routing kernel)
  int W, L, E;
  long long A;
  int h, I;
  int tiles_gu, tiles_dn;  // units per expert: I / 128 (gate/up), h / 256 (down)
  int* status;
  uint64_t timeout_ns;
};

// ------------------------------------------------------------- tcgen05 / TMA

__device__ __forceinline__ void tma_load_2d(void* smem, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns of TMEM -> 16 registers per thread.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(const void* smem) {
  const uint64_t addr = smem_u32(smem);
  return ((addr >> 4) & 0x3FFFull)  // start address
         | (1ull << 16)             // leading byte offset (unused for swizzled K-major)
         | (64ull << 32)            // stride byte offset: 1024 B between 8-row groups
         | (1ull << 46)             // descriptor version
         | (2ull << 61);            // 128-byte swizzle
}

// Instruction descriptor: bf16 A and B, fp32 D, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// ------------------------------------------------------------- the kernel

// A unit: one expert's 2 x 128 weight rows against all of its tokens. Units
// [0, E*tiles_gu) are gate/up (the same 128 rows of gate and of up), the rest
// down (two 128-row slices of the down projection).
struct Unit {
  int mode, e, tile, n_e, K;
  long long row0;  // flat expand row of the expert's first token
};

__device__ __forceinline__ Unit unit_of(const FfnParams& p, int u) {
  Unit x;
  const int n_gu = p.E * p.tiles_gu;
  x.mode = u < n_gu ? FFN_GATE_UP : FFN_DOWN;
  if (x.mode == FFN_DOWN) u -= n_gu;
  const int tiles = x.mode == FFN_GATE_UP ? p.tiles_gu : p.tiles_dn;
  x.e = u / tiles;
  x.tile = u % tiles;
  x.K = x.mode == FFN_GATE_UP ? p.h : p.I;
  const int d = x.e / p.L, le = x.e % p.L, LW = p.L * p.W;
  const int32_t* epd = p.ep + (size_t)d * LW;
  const int start = le == 0 ? 0 : epd[le * p.W - 1];
  const int end = epd[le * p.W + p.W - 1];
  x.n_e = end > start ? end - start : 0;
  x.row0 = (long long)d * p.A + start;
  return x;
}

// First weight row of tile t of a unit (rows of w_gate / w_up: expert-major
// I rows; of w_down: expert-major h rows).
__device__ __forceinline__ int a_row(const FfnParams& p, const Unit& u, int t) {
  return u.mode == FFN_GATE_UP ? u.e * p.I + u.tile * 128 : u.e * p.h + u.tile * 256 + t * 128;
}

// A down unit may start once all gate/up units of its expert have stored their
// h1 rows: bounded acquire-spin on the expert's counter, then order those
// generic-proxy stores before this thread's TMA (async-proxy) reads of h1.
__device__ __forceinline__ bool wait_expert(const FfnParams& p, int e, volatile int* abort_flag) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p.done + e) : "memory");
    if (v >= 4u * (uint32_t)p.tiles_gu) break;  // every epilogue warp of every gate/up unit
    if ((it & 63u) == 63u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        set_error(p.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const FfnParams& p,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        set_error(p.status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__global__ void __launch_bounds__(kFfnThreads, 1)
    ffn_kernel(const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_u,
               const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_d,
               const __grid_constant__ CUtensorMap map_h, FfnParams p) {
  extern __shared__ __align__(1024) uint8_t fsm_raw[];
  __shared__ __align__(8) uint64_t full[kFfnStages], empty[kFfnStages], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* fsm = fsm_raw + ((1024u - (smem_u32(fsm_raw) & 1023u)) & 1023u);
  const int n_units = p.E * (p.tiles_gu + p.tiles_dn);

  pdl_wait();  // the expert rows are ready
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kFfnStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128);
    }
    mbar_fence_init();
    s_abort = 0;
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // Every role walks the same units: u = blockIdx.x, +grid, ... over gate/up
  // units first, down units after, so each CTA meets its down units only once
  // all of its own gate/up loads are issued, and CTAs whose gate/up share ran
  // out early start on down units while others finish theirs.
  if (warp == 0) {
    if (lane == 0) {
      // producer: B (tokens or h1 rows) and kT weight tiles per k-block
      uint32_t it = 0;
      for (int u = blockIdx.x; u < n_units && !s_abort; u += gridDim.x) {
        const Unit un = unit_of(p, u);
        const int passes = (un.n_e + kNP - 1) / kNP;
        if (passes == 0) continue;
        if (un.mode == FFN_DOWN && !wait_expert(p, un.e, &s_abort)) break;
        const CUtensorMap* mb = un.mode == FFN_GATE_UP ? &map_x : &map_h;
        const CUtensorMap* ma0 = un.mode == FFN_GATE_UP ? &map_g : &map_d;
        const CUtensorMap* ma1 = un.mode == FFN_GATE_UP ? &map_u : &map_d;
        const int KB = un.K / kBK;
        for (int ps = 0; ps < passes && !s_abort; ++ps) {
          for (int kb = 0; kb < KB; ++kb, ++it) {
            const uint32_t stage = it % kFfnStages, round = it / kFfnStages;
            if (round > 0 && !wait_or_abort(&empty[stage], (round - 1) & 1u, p, &s_abort)) break;
            uint8_t* st = fsm + stage * kStage;
            mbar_arrive_expect_tx(&full[stage], kStage);
            tma_load_2d(st, mb, kb * kBK, (int)(un.row0 + (long long)ps * kNP), &full[stage]);
#pragma unroll
            for (int t = 0; t < kT; ++t)
              tma_load_2d(st + kBTile + t * kATile, t == 1 ? ma1 : ma0, kb * kBK, a_row(p, un, t), &full[stage]);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer
      uint32_t it = 0, acc = 0;
      for (int u = blockIdx.x; u < n_units && !s_abort; u += gridDim.x) {
        const Unit un = unit_of(p, u);
        const int passes = (un.n_e + kNP - 1) / kNP;
        const int KB = un.K / kBK;
        for (int ps = 0; ps < passes && !s_abort; ++ps, ++acc) {
          const uint32_t buf = acc & 1u;
          if (acc >= 2 && !wait_or_abort(&acc_empty[buf], ((acc >> 1) - 1) & 1u, p, &s_abort)) break;
          tc_fence_after();
          const int n_rem = min(kNP, un.n_e - ps * kNP);
          const uint32_t idesc = idesc_bf16((n_rem + 15) & ~15);
          const uint32_t d_base = tmem + buf * (kT * kNP);
          for (int kb = 0; kb < KB; ++kb, ++it) {
            const uint32_t stage = it % kFfnStages, round = it / kFfnStages;
            if (!wait_or_abort(&full[stage], round & 1u, p, &s_abort)) break;
            tc_fence_after();
            const uint8_t* st = fsm + stage * kStage;
            const uint64_t bdesc = sw128_desc(st);
#pragma unroll
            for (int t = 0; t < kT; ++t) {
              const uint64_t adesc = sw128_desc(st + kBTile + t * kATile);
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk)  // K = 16 per MMA: 32 bytes along the swizzled row
                tc_mma(d_base + t * kNP, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0);
            }
            tc_commit(&empty[stage]);
          }
          tc_commit(&acc_full[buf]);
        }
      }
    }
  } else {
    // epilogue: warp (w % 4) reads TMEM lanes [32*(w%4), +32), one output feature each
    const int q = warp & 3;
    const int feat = 32 * q + lane;
    uint32_t acc = 0;
    for (int u = blockIdx.x; u < n_units && !s_abort; u += gridDim.x) {
      const Unit un = unit_of(p, u);
      const int passes = (un.n_e + kNP - 1) / kNP;
      for (int ps = 0; ps < passes && !s_abort; ++ps, ++acc) {
        const uint32_t buf = acc & 1u;
        if (!wait_or_abort(&acc_full[buf], (acc >> 1) & 1u, p, &s_abort)) break;
        tc_fence_after();
        const int n_rem = min(kNP, un.n_e - ps * kNP);
        const int chunks = (n_rem + 15) >> 4;
        const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + buf * (kT * kNP);
        const long long row = un.row0 + (long long)ps * kNP;
        for (int c = 0; c < chunks; ++c) {
          if (un.mode == FFN_GATE_UP) {
            uint32_t g[16], v[16];
            tc_ld16(tbase + c * 16, g);
            tc_ld16(tbase + kNP + c * 16, v);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = c * 16 + j;
              if (n < n_rem) {
                const float a = __uint_as_float(g[j]), b = __uint_as_float(v[j]);
                const float h = a / (1.0f + expf(-a)) * b;
                p.h1[(row + n) * p.I + un.tile * 128 + feat] = __float2bfloat16_rn(h);
              }
            }
          } else {
#pragma unroll
            for (int t = 0; t < kT; ++t) {
              uint32_t v[16];
              tc_ld16(tbase + t * kNP + c * 16, v);
              tc_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = c * 16 + j;
                if (n < n_rem)
                  p.y[(row + n) * p.h + un.tile * 256 + t * 128 + feat] =
                      __float2bfloat16_rn(__uint_as_float(v[j]));
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
      }
      if (un.mode == FFN_GATE_UP && passes > 0) {
        // this warp's h1 columns of the unit are stored: make them visible (to
        // the async proxy too: down units read them by TMA), then count them
        // for the expert (four warps a unit; no barrier across the warps)
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        __syncwarp();
        if (lane == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.done + un.e) : "memory");
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D bf16 tensor [rows][cols] (row-major), boxes of 64 columns x box_rows rows,
// 128-byte swizzle; rows past the end read as zeros.
static bool make_map(CUtensorMap* m, const void* base, unsigned long long rows, unsigned long long cols,
                     unsigned box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_ffn(const FfnLaunch& f, cudaStream_t st, int num_sms, void* const* prof_events) {
  const Shape& sh = f.sh;
  const unsigned long long rows = (unsigned long long)sh.W * sh.A;
  CUtensorMap mg, mu, md, mx, mh;
  if (!make_map(&mg, f.w_gate, (unsigned long long)sh.E * f.I, sh.h, 128) ||
      !make_map(&mu, f.w_up, (unsigned long long)sh.E * f.I, sh.h, 128) ||
      !make_map(&md, f.w_down, (unsigned long long)sh.E * sh.h, f.I, 128) ||
      !make_map(&mx, f.expand_x, rows, sh.h, kNP) || !make_map(&mh, f.h1, rows, f.I, kNP))
    return cudaErrorInvalidValue;
  FfnParams p{};
  p.ep = f.ep;
  p.h1 = static_cast<__nv_bfloat16*>(f.h1);
  p.y = static_cast<__nv_bfloat16*>(f.y);
  p.done = f.done;
  p.W = sh.W;
  p.L = sh.L;
  p.E = sh.E;
  p.A = sh.A;
  p.h = sh.h;
  p.I = f.I;
  p.tiles_gu = f.I / 128;
  p.tiles_dn = sh.h / 256;
  p.status = f.status;
  p.timeout_ns = f.timeout_ns;

  int per_sm = 0;  // one CTA per SM by design; the call raises the shared-memory limit once
  cudaError_t e = resident_blocks((const void*)ffn_kernel, kFfnThreads, kFfnSmem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // every CTA must be resident at once (down units wait on other CTAs' gate/up
  // units): one per SM, no more than the SMs
  const int units = p.E * (p.tiles_gu + p.tiles_dn);
  const int grid = units < num_sms ? units : num_sms;
  if (grid <= 0) return cudaSuccess;
  if (prof_events && prof_events[0]) cudaEventRecord(static_cast<cudaEvent_t>(prof_events[0]), st);
  PdlLaunch L(dim3(grid), dim3(kFfnThreads), kFfnSmem, st);
  cudaLaunchAttribute attr[2] = {L.attr[0], {}};
  attr[1].id = cudaLaunchAttributeCooperative;  // co-residency of all CTAs is required
  attr[1].val.cooperative = 1;
  L.cfg.attrs = attr;
  L.cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&L.cfg, ffn_kernel, mg, mu, mx, md, mh, p);
  if (e != cudaSuccess) return e;
  if (prof_events && prof_events[1]) cudaEventRecord(static_cast<cudaEvent_t>(prof_events[1]), st);
  return cudaSuccess;
}

}  // namespace crs
