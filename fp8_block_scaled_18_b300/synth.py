"""Seeded synthetic inputs shaped like DeepSeek-V3's projections and experts.

This module only draws random numbers and lays them out; it holds none of the
quantisation or GEMM arithmetic.  Both the CUDA path and the CPU oracle are fed
from here, so they see identical bits.  Shapes follow the "DeepSeek-V3"
repository overview (pomoai hub): dim 7168, q_lora_rank 1536,
kv_lora_rank 512 + qk_rope_head_dim 64 (the MLA excerpt's wkv_a output, 576),
256 routed experts with top-8, 8 expert groups of which 4 are kept, sigmoid
scoring, routing weights scaled by 2.5 (config block of "671B 参数如何「激活」37B？").

bf16 tensors are returned as uint16 bit patterns (numpy), rounded from fp32
by torch's round-to-nearest-even cast.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

DIM = 7168
Q_LORA = 1536
KV_OUT = 512 + 64
N_EXPERTS = 256
TOP_K = 8
N_GROUPS = 8
TOPK_GROUPS = 4
ROUTE_SCALE = 2.5
MOE_INTER = 2048
Q_SWEEP_M = (1, 16, 64, 512, 4096, 16384)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 numpy -> bf16 bit patterns (uint16), via torch's RNE cast."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def activations(rng: np.random.Generator, M: int, K: int, n_outlier: int = 0,
                outlier_scale: float = 1.0, student_t: bool = False) -> np.ndarray:
    """X ~ N(0,1) (or Student-t(3)) with `n_outlier` channels scaled up."""
    if student_t:
        x = rng.standard_t(3, size=(M, K)).astype(np.float32)
    else:
        x = rng.standard_normal((M, K), dtype=np.float32)
    if n_outlier:
        ch = rng.choice(K, size=n_outlier, replace=False)
        x[:, ch] *= np.float32(outlier_scale)
    return to_bf16_bits(x)


@dataclass
class DenseCase:
    name: str
    x: np.ndarray  # bf16 bits [M, K]
    w: np.ndarray  # bf16 bits [N, K]

    @property
    def shape(self):
        return self.x.shape[0], self.w.shape[0], self.x.shape[1]


def tiny(seed: int = 0) -> DenseCase:
    """X [128,512] ~N(0,1) with 4 outlier channels x20; W [256,512] ~N(0,0.02)."""
    rng = np.random.default_rng(seed)
    x = activations(rng, 128, 512, n_outlier=4, outlier_scale=20.0)
    w = normal_bf16(rng, (256, 512), 0.02)
    return DenseCase("tiny", x, w)


def kv_down(seed: int = 1, M: int = 4096) -> DenseCase:
    """MLA wkv_a: X [4096,7168] ~N(0,1), 1% of channels x30; W [576,7168]."""
    rng = np.random.default_rng(seed)
    x = activations(rng, M, DIM, n_outlier=round(0.01 * DIM), outlier_scale=30.0)
    w = normal_bf16(rng, (KV_OUT, DIM), 0.02)
    return DenseCase("kv_down", x, w)


def q_down(M: int, seed: int = 2) -> DenseCase:
    """MLA wq_a: W [1536,7168] ~N(0,0.02); X [M,7168] ~N(0,1)."""
    rng = np.random.default_rng(seed)
    w = normal_bf16(rng, (Q_LORA, DIM), 0.02)
    x = activations(np.random.default_rng([seed, M]), M, DIM)
    return DenseCase(f"q_down_m{M}", x, w)


def large_square(seed: int = 3, M: int = 16384) -> DenseCase:
    """X [16384,7168] Student-t(3); W [7168,7168] ~N(0,0.02)."""
    rng = np.random.default_rng(seed)
    x = activations(rng, M, DIM, student_t=True)
    w = normal_bf16(rng, (DIM, DIM), 0.02)
    return DenseCase("large_square", x, w)


@dataclass
class MoECase:
    x_tokens: np.ndarray   # bf16 bits [tokens, K]
    token_of_row: np.ndarray  # int64 [T]: source token of each grouped row
    offsets: np.ndarray    # int32 [G+1]
    n_experts: int
    n: int
    k: int
    expert_seed0: int
    weight_of_row: np.ndarray = None   # fp32 [T]: routing weight of each grouped row
    rows_of_token: np.ndarray = None   # int32 [tokens, top_k]: the grouped rows of each token
    gate_w: np.ndarray = None          # bf16 bits [n_experts, K]: the router's weight
    gate_bias: np.ndarray = None       # fp32 [n_experts]: the router's selection bias

    @property
    def x_rows(self) -> np.ndarray:
        """bf16 bits [T, K]: token rows gathered expert by expert."""
        return self.x_tokens[self.token_of_row]


def route(x_bits: np.ndarray, gate_w_bits: np.ndarray, bias: np.ndarray,
          n_groups: int = N_GROUPS, topk_groups: int = TOPK_GROUPS, top_k: int = TOP_K,
          with_weights: bool = False, route_scale: float = ROUTE_SCALE):
    """Sigmoid-scored, group-limited top-k routing of the synthetic tokens (an
    input generator: it decides which rows each expert receives in the
    workloads that take the routing as given; the library's own router is
    fp8bs_moe_gate).  The bias steers selection only.  The
    group score is the largest biased score in the group; ties go to the lower
    index.  Returns expert ids [tokens, top_k]; with_weights also the routing
    weights: the selected (unbiased) scores normalised to sum 1, times
    route_scale (fp32 [tokens, top_k])."""
    x = torch.from_numpy(bf16_bits_to_f32(x_bits))
    wg = torch.from_numpy(bf16_bits_to_f32(gate_w_bits))
    scores = torch.sigmoid(x @ wg.T).numpy()                  # fp32 [T, E]
    biased = scores + bias[None, :].astype(np.float32)
    T, E = biased.shape
    per = E // n_groups
    gscore = biased.reshape(T, n_groups, per).max(axis=2)
    gorder = np.argsort(-gscore, axis=1, kind="stable")[:, :topk_groups]
    mask = np.full((T, n_groups), -np.inf, dtype=np.float32)
    np.put_along_axis(mask, gorder, 0.0, axis=1)
    masked = biased + np.repeat(mask, per, axis=1)
    experts = np.argsort(-masked, axis=1, kind="stable")[:, :top_k]
    if not with_weights:
        return experts
    w = np.take_along_axis(scores, experts, axis=1).astype(np.float32)
    w = (w / w.sum(axis=1, keepdims=True) * np.float32(route_scale)).astype(np.float32)
    return experts, w


def moe(seed: int = 4, tokens: int = 4096, n_experts: int = N_EXPERTS, n: int = MOE_INTER,
        k: int = DIM, expert_seed0: int = 1000) -> MoECase:
    """4096 tokens X ~N(0,1) routed over 256 experts (8 groups keep 4, top-8);
    gate W ~N(0,0.02), per-expert bias ~U(-0.1,0.1).  Rows are grouped by
    expert, tokens in order within an expert."""
    rng = np.random.default_rng(seed)
    x = activations(rng, tokens, k)
    gw = normal_bf16(rng, (n_experts, k), 0.02)
    bias = rng.uniform(-0.1, 0.1, size=n_experts).astype(np.float32)
    groups = min(N_GROUPS, n_experts)
    experts, weights = route(x, gw, bias, n_groups=groups, topk_groups=max(1, groups // 2),
                             top_k=min(TOP_K, n_experts), with_weights=True)
    flat_e = experts.reshape(-1)
    flat_t = np.repeat(np.arange(tokens, dtype=np.int64), experts.shape[1])
    order = np.argsort(flat_e, kind="stable")
    counts = np.bincount(flat_e, minlength=n_experts)
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    row_of_pair = np.empty_like(order)
    row_of_pair[order] = np.arange(order.size)
    return MoECase(x, flat_t[order], offsets, n_experts, n, k, expert_seed0,
                   weights.reshape(-1)[order].astype(np.float32),
                   row_of_pair.reshape(tokens, experts.shape[1]).astype(np.int32), gw, bias)


def expert_weight(case: MoECase, g: int, device: str = "cpu", which: int = 0) -> torch.Tensor:
    """Expert g's W [N, K] ~N(0,0.02) as a bf16 torch tensor, drawn from a
    torch generator seeded with expert_seed0 + g (+ 100003 * which, so that
    which = 1 gives a second, independent weight per expert, e.g. the up
    projection next to the gate) on `device` (on a GPU this is torch's Philox
    stream, so the same seed gives the same bits every run).  which = 2 is
    the down projection w2, [K, N] (model width by intermediate size); the
    index g = n_experts stands for the shared expert."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(case.expert_seed0) + int(g) + 100003 * int(which))
    shape = (case.k, case.n) if which == 2 else (case.n, case.k)
    w = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return (w * 0.02).to(torch.bfloat16)


def offsets_from_counts(counts) -> np.ndarray:
    counts = np.asarray(counts, dtype=np.int64)
    off = np.zeros(counts.size + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    return off
