"""Seeded synthetic inputs for MoE token dispatch / combine.

This module only draws random inputs (tokens, top-K expert ids, active masks,
top-K weights, expert FFN weights). It holds none of the dispatch or combine
arithmetic, so both the CPU oracle and the CUDA path can take their inputs
from it without sharing any of the method.

The shapes follow the workloads the pages run:
  * the SHMEM two-plane combine example (combine_doubleplane README, "运行" and
    "性能测试"): 2 PEs / 8 PEs, bs 8 or 32, h 16 or 7168, topk 2 or 8,
    2 or 8 experts per PE, int32_t data;
  * the aclnnMoeDistributeDispatchV4 parameter blocks: 1D/2D active masks,
    zero / copy expert id ranges, quantMode 0 and 2;
  * the xLLM MegaMoe pull request: a decode MoE layer with intermediate 512.

All draws use numpy's PCG64 generator, so the same seed gives the same bytes
on x86 and Arm hosts. bf16 tensors are held as uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

X_INT32 = "int32"
X_FP16 = "float16"
X_BF16 = "bfloat16"

ES = {X_INT32: 4, X_FP16: 2, X_BF16: 2}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One dispatch/combine problem: W emulated EP ranks, each with bs tokens."""

    name: str
    ep_world_size: int          # W
    bs: int                     # tokens per rank
    h: int                      # hidden size
    topk: int                   # K
    moe_expert_num: int         # E (routed experts; E % W == 0)
    x_dtype: str
    zero_expert_num: int = 0
    copy_expert_num: int = 0
    mask_kind: int = 0          # 0 none, 1 = (bs,), 2 = (bs, K)
    quant_mode: int = 0         # 0 none, 1 static int8, 2 per-token int8, 3 per-group fp8, 4 MX
    y_dtype: str = ""           # quantised element type for modes 3 / 4: fp8_e4m3, fp8_e5m2, fp4_e2m1
    scales_kind: int = 0        # scales input: 0 none, 1 (1,), 2 (h,), 3 (E, h)
    ids: str = "uniform"        # "uniform" distinct ids, or "zipf"
    zipf_s: float = 1.2
    special_p: float = 0.0      # probability that a pick becomes a special expert
    mask_false_p: float = 0.0   # probability that a 2D mask entry is false
    x_range: int = 1000         # int32 x is uniform in [-x_range, x_range]
    scale_lo: int = 1           # int32 weights uniform in [scale_lo, scale_hi]
    scale_hi: int = 4
    ffn_intermediate: int = 0   # > 0: the workload carries SwiGLU expert weights
    seed: int = 0

    @property
    def local_expert_num(self) -> int:
        return self.moe_expert_num // self.ep_world_size

    @property
    def scale_dtype(self) -> str:
        return X_INT32 if self.x_dtype == X_INT32 else "float32"

    @property
    def es(self) -> int:
        return ES[self.x_dtype]

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The workloads, named by what they are.
WORKLOADS = {
    # 2 PEs, bs 8, h 16, topk 2, 2 experts per PE, int32_t (README "运行", 2-card run)
    "w2_bs8_h16_k2_e4_i32": Workload(
        "w2_bs8_h16_k2_e4_i32", 2, 8, 16, 2, 4, X_INT32, x_range=100, seed=0),
    # 8 PEs, 64 experts (README "运行", 8-card run); int32 and fp16 variants
    "w8_bs8_h16_k2_e64_i32": Workload(
        "w8_bs8_h16_k2_e64_i32", 8, 8, 16, 2, 64, X_INT32, x_range=1000, seed=1),
    "w8_bs8_h16_k2_e64_f16": Workload(
        "w8_bs8_h16_k2_e64_f16", 8, 8, 16, 2, 64, X_FP16, seed=1),
    # the perf shape of the README: 8 PEs, bs 32, h 7168, topk 8, 8 experts per PE
    "w8_bs32_h7168_k8_e64_f16": Workload(
        "w8_bs32_h7168_k8_e64_f16", 8, 32, 7168, 8, 64, X_FP16, seed=2),
    "w8_bs32_h7168_k8_e64_f16_q2": Workload(
        "w8_bs32_h7168_k8_e64_f16_q2", 8, 32, 7168, 8, 64, X_FP16, quant_mode=2, seed=2),
    "w8_bs32_h7168_k8_e64_i32": Workload(
        "w8_bs32_h7168_k8_e64_i32", 8, 32, 7168, 8, 64, X_INT32, x_range=1000, seed=2),
    # skewed (Zipf) routing, 2D mask, zero and copy experts, large segments
    "w16_bs256_h7168_k8_e256_bf16_zipf": Workload(
        "w16_bs256_h7168_k8_e256_bf16_zipf", 16, 256, 7168, 8, 256, X_BF16,
        zero_expert_num=4, copy_expert_num=4, mask_kind=2, ids="zipf",
        special_p=0.05, mask_false_p=0.10, seed=3),
    # the same routing law with half the batch (3.75 GB of receive buffers):
    # used for full ncu captures, which must stay small on the device
    "w16_bs128_h7168_k8_e256_bf16_zipf": Workload(
        "w16_bs128_h7168_k8_e256_bf16_zipf", 16, 128, 7168, 8, 256, X_BF16,
        zero_expert_num=4, copy_expert_num=4, mask_kind=2, ids="zipf",
        special_p=0.05, mask_false_p=0.10, seed=3),
    # decode MoE layer with a SwiGLU expert FFN (intermediate 512)
    "w8_bs64_h2048_k8_e128_bf16_ffn": Workload(
        "w8_bs64_h2048_k8_e128_bf16_ffn", 8, 64, 2048, 8, 128, X_BF16,
        ffn_intermediate=512, seed=4),
    # single-shape profiling shape of the README (2 PEs, h 256)
    "w2_bs8_h256_k2_e4_i32": Workload(
        "w2_bs8_h256_k2_e4_i32", 2, 8, 256, 2, 4, X_INT32, x_range=1000, seed=5),
}


def fp32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 samples to the nearest bf16 (ties to even); returns uint16 bits.

    Used only to draw bf16 inputs; the samples are finite.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u >> 16) & np.uint32(1)  # finite values: the sum below stays below 2^32
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_fp32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _distinct_uniform_ids(rng: np.random.Generator, n: int, e: int, k: int) -> np.ndarray:
    # K distinct ids per token, uniform: the first K of a random permutation.
    keys = rng.random((n, e))
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def _zipf_ids(rng: np.random.Generator, n: int, e: int, k: int, s: float) -> np.ndarray:
    # Popularity rank r (1..E) has weight r^-s, over a seeded permutation of the
    # experts. K sequential draws without replacement (weights renormalised after
    # each draw) have the same law as the K largest of log(w) + Gumbel noise,
    # taken in descending key order.
    perm = rng.permutation(e)
    w = np.empty(e, dtype=np.float64)
    w[perm] = np.arange(1, e + 1, dtype=np.float64) ** (-s)
    g = rng.gumbel(size=(n, e))
    keys = np.log(w)[None, :] + g
    order = np.argsort(-keys, axis=1, kind="stable")[:, :k]
    return order.astype(np.int32)


def _softmax_f32(logits: np.ndarray) -> np.ndarray:
    z = logits.astype(np.float32)
    z = z - z.max(axis=-1, keepdims=True)
    ez = np.exp(z, dtype=np.float32)
    return (ez / ez.sum(axis=-1, keepdims=True, dtype=np.float32)).astype(np.float32)


def make_inputs(wl: Workload, seed: Optional[int] = None) -> dict:
    """Draw one batch of inputs for ``wl``.

    Returns numpy arrays with a leading W axis (the W emulated ranks):
      x             [W, bs, h]   int32 / float16 / uint16 (bf16 bits)
      expert_ids    [W, bs, K]   int32
      active_mask   None, [W, bs] or [W, bs, K] uint8
      expert_scales [W, bs, K]   int32 (int32 x) or float32
      w_gate, w_up  [E, I, h]    uint16 bf16 bits   (FFN workloads only; stored
      w_down        [E, h, I]    out-major, like a linear layer's weight)
      quant_scales  float32 (1,), (h,) or (E, h) when scales_kind > 0: static
                    coefficients U[16, 40] (quantMode 1; N(0,1) data then
                    saturates int8 beyond about 3.2 sigma), smoothing weights
                    U[0.5, 2] otherwise
    """
    seed = wl.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    W, bs, h, K, E = wl.ep_world_size, wl.bs, wl.h, wl.topk, wl.moe_expert_num
    n = W * bs
    out = {}

    if wl.x_dtype == X_INT32:
        x = rng.integers(-wl.x_range, wl.x_range + 1, size=(W, bs, h), dtype=np.int32)
    elif wl.x_dtype == X_FP16:
        x = rng.standard_normal(size=(W, bs, h), dtype=np.float32).astype(np.float16)
    else:
        x = fp32_to_bf16_bits(rng.standard_normal(size=(W, bs, h), dtype=np.float32))
    out["x"] = x

    if wl.ids == "zipf":
        ids = _zipf_ids(rng, n, E, K, wl.zipf_s)
    else:
        ids = _distinct_uniform_ids(rng, n, E, K)
    n_special = wl.zero_expert_num + wl.copy_expert_num
    if n_special > 0 and wl.special_p > 0:
        # each pick independently becomes a special expert; the specials of one
        # token are drawn without replacement from the Z + C special ids
        hit = rng.random((n, K)) < wl.special_p
        sperm = np.argsort(rng.random((n, n_special)), axis=1, kind="stable").astype(np.int32)
        slot = np.cumsum(hit, axis=1) - 1
        slot = np.clip(slot, 0, n_special - 1)
        special_ids = E + np.take_along_axis(sperm, slot, axis=1)
        ids = np.where(hit, special_ids, ids).astype(np.int32)
    out["expert_ids"] = ids.reshape(W, bs, K)

    if wl.mask_kind == 2:
        out["active_mask"] = (rng.random((W, bs, K)) >= wl.mask_false_p).astype(np.uint8)
    elif wl.mask_kind == 1:
        # trues first, then falses (the 1D mask must be a prefix)
        n_act = rng.integers(0, bs + 1, size=W)
        out["active_mask"] = (np.arange(bs)[None, :] < n_act[:, None]).astype(np.uint8)
    else:
        out["active_mask"] = None

    if wl.x_dtype == X_INT32:
        out["expert_scales"] = rng.integers(
            wl.scale_lo, wl.scale_hi + 1, size=(W, bs, K), dtype=np.int32)
    else:
        logits = rng.standard_normal(size=(W, bs, K), dtype=np.float32)
        out["expert_scales"] = _softmax_f32(logits)

    if wl.ffn_intermediate > 0:
        I = wl.ffn_intermediate
        for name, shape in (("w_gate", (E, I, h)), ("w_up", (E, I, h)), ("w_down", (E, h, I))):
            w = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(0.02)
            out[name] = fp32_to_bf16_bits(w)

    if wl.scales_kind > 0:
        shape = {1: (1,), 2: (h,), 3: (E, h)}[wl.scales_kind]
        lo, hi = (16.0, 40.0) if wl.quant_mode == 1 else (0.5, 2.0)
        out["quant_scales"] = rng.uniform(lo, hi, size=shape).astype(np.float32)
    return out


def small_random_workload(rng: np.random.Generator, x_dtype: str = X_INT32,
                          max_w: int = 4, max_bs: int = 8) -> Workload:
    """A random small problem for brute-force and parity sweeps."""
    W = int(rng.integers(2, max_w + 1))
    L = int(rng.integers(1, 4))
    K = int(rng.integers(1, min(W * L, 4) + 1))
    bs = int(rng.integers(1, max_bs + 1))
    h = int(rng.choice([8, 16, 24, 40]))
    Z = int(rng.integers(0, 3))
    C = int(rng.integers(0, 3))
    mk = int(rng.integers(0, 3))
    return Workload(
        f"rand_w{W}_l{L}_k{K}_bs{bs}_h{h}", W, bs, h, K, W * L, x_dtype,
        zero_expert_num=Z, copy_expert_num=C, mask_kind=mk,
        special_p=0.25 if Z + C > 0 else 0.0, mask_false_p=0.3, x_range=100,
        seed=int(rng.integers(0, 2**31)))
