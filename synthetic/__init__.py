"""Seeded synthetic inputs for the fine-grained FP8 GEMM path.

This module is shared by the tests, the benchmark and the smoke check.  It
holds no quantisation or GEMM arithmetic: it only draws random BF16 matrices
with the shapes and value distributions of the five workloads below, and the
routing that turns a token batch into per-expert row segments.

Recipe (every workload, seed 0 unless a test says otherwise):
  * one ``torch.Generator`` seeded once; tensors are drawn in the order the
    workload lists them, in fp32, then cast to BF16 (round to nearest even);
  * N(0, 1) activations and N(0, 0.02) weights;
  * outliers: a Bernoulli(p) mask multiplies the chosen fp32 entries by a
    factor before the cast;
  * heavy tails: Student-t with nu = 3, built as Z / sqrt(chi2_3 / 3) from
    generator normals (chi2_3 = sum of three squared normals);
  * routing: logits ~ N(0, 1), score = sigmoid(logit), each token picks the
    top-k experts of score + bias, bias ~ U(-0.1, 0.1) per expert (the bias
    only affects selection); ties go to the lower expert index; rows are then
    sorted by (expert, token).

Shapes (M x K activations, N x K weights unless stated):
  tiny      A 128x512,   W 256x512,   FP32 output
  mla_q     A 4096x1536 with 0.1% outliers x50, W 24576x1536, BF16 output
  mla_kv    A 8192x512,  W 32768x512, BF16 output
  experts   X 4096x7168, 256 experts of W_e 2048x7168, top-8 routing, BF16 out
  dgrad     dY 8192x7168 Student-t(3), W stored [7168, 18432] (K x N), BF16 out
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

FP32_OUT, BF16_OUT = 1, 0


@dataclass
class DenseCase:
    name: str
    a: torch.Tensor            # bf16 [M, K]
    w: torch.Tensor            # bf16 [N, K] (b_major 0) or [K, N] (b_major 1)
    b_major: int
    out_fp32: bool

    @property
    def M(self):
        return self.a.shape[0]

    @property
    def K(self):
        return self.a.shape[1]

    @property
    def N(self):
        return self.w.shape[0] if self.b_major == 0 else self.w.shape[1]


@dataclass
class GroupedCase:
    name: str
    x_sorted: torch.Tensor     # bf16 [M_total, K], rows grouped by expert
    w: torch.Tensor            # bf16 [E, N, K]
    offsets: torch.Tensor      # int32 [E + 1]
    token_of_row: torch.Tensor  # int64 [M_total]
    x: Optional[torch.Tensor] = field(default=None)  # bf16 [tokens, K] before the gather


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std, g, device, outlier_p=0.0, outlier_scale=1.0):
    """fp32 N(0, std^2) draws (optionally with Bernoulli outliers) cast to BF16."""
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if outlier_p > 0.0:
        mask = torch.rand(shape, generator=g, device=device, dtype=torch.float32) < outlier_p
        x = torch.where(mask, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def student_t3_bf16(shape, g, device):
    """Student-t, nu = 3: Z / sqrt(chi2_3 / 3), all from generator normals."""
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(3):
        n = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        chi2.addcmul_(n, n)
    return (z / torch.sqrt(chi2 / 3.0)).to(torch.bfloat16)


def dense_case(name, M, N, K, *, seed=0, device="cpu", w_std=0.02, outlier_p=0.0,
               outlier_scale=50.0, heavy_tail=False, b_major=0, out_fp32=False) -> DenseCase:
    g = generator(seed, device)
    if heavy_tail:
        a = student_t3_bf16((M, K), g, device)
    else:
        a = normal_bf16((M, K), 1.0, g, device, outlier_p, outlier_scale)
    w_shape = (N, K) if b_major == 0 else (K, N)
    w = normal_bf16(w_shape, w_std, g, device)
    return DenseCase(name, a, w, b_major, out_fp32)


@dataclass
class WgradCase:
    """Weight gradient dW = dY^T . X over T tokens: dy [T, M], x [T, N] (BF16)."""
    name: str
    dy: torch.Tensor
    x: torch.Tensor

    @property
    def T(self):
        return self.dy.shape[0]

    @property
    def M(self):
        return self.dy.shape[1]

    @property
    def N(self):
        return self.x.shape[1]


def wgrad_case(name, T, M, N, *, seed=0, device="cpu", heavy_tail=True) -> WgradCase:
    g = generator(seed, device)
    dy = student_t3_bf16((T, M), g, device) if heavy_tail else normal_bf16((T, M), 1.0, g, device)
    x = normal_bf16((T, N), 1.0, g, device)
    return WgradCase(name, dy, x)


def route_topk(logits: torch.Tensor, bias: torch.Tensor, topk: int):
    """Top-k expert choice per token from sigmoid affinities plus a selection
    bias; ties go to the lower expert index (stable descending sort)."""
    score = torch.sigmoid(logits) + bias[None, :]
    order = torch.sort(score, dim=1, descending=True, stable=True).indices
    return order[:, :topk]


def segments_from_choice(choice: torch.Tensor, num_experts: int):
    """Rows sorted by (expert, token): returns (token_of_row, offsets[E+1])."""
    tokens = choice.shape[0]
    expert = choice.reshape(-1)
    token = torch.arange(tokens, device=choice.device).repeat_interleave(choice.shape[1])
    key = expert.to(torch.int64) * tokens + token
    perm = torch.sort(key, stable=True).indices
    token_of_row = token[perm]
    counts = torch.bincount(expert, minlength=num_experts)
    offsets = torch.zeros(num_experts + 1, dtype=torch.int64, device=choice.device)
    offsets[1:] = torch.cumsum(counts, 0)
    return token_of_row, offsets.to(torch.int32)


def grouped_case(name, tokens, E, topk, N, K, *, seed=0, device="cpu", w_std=0.02,
                 keep_x=False) -> GroupedCase:
    g = generator(seed, device)
    x = normal_bf16((tokens, K), 1.0, g, device)
    logits = torch.randn((tokens, E), generator=g, device=device, dtype=torch.float32)
    bias = torch.rand((E,), generator=g, device=device, dtype=torch.float32) * 0.2 - 0.1
    w = torch.empty((E, N, K), dtype=torch.bfloat16, device=device)
    for e in range(E):
        w[e] = normal_bf16((N, K), w_std, g, device)
    choice = route_topk(logits, bias, topk)
    token_of_row, offsets = segments_from_choice(choice, E)
    x_sorted = x.index_select(0, token_of_row)
    return GroupedCase(name, x_sorted, w, offsets, token_of_row, x if keep_x else None)


def grouped_case_with_counts(name, counts, N, K, *, seed=0, device="cpu", w_std=0.02):
    """Grouped case with explicitly chosen per-expert row counts (edge cases:
    empty experts, ragged segments)."""
    g = generator(seed, device)
    counts = [int(c) for c in counts]
    E, M = len(counts), sum(counts)
    x_sorted = normal_bf16((M, K), 1.0, g, device)
    w = torch.empty((E, N, K), dtype=torch.bfloat16, device=device)
    for e in range(E):
        w[e] = normal_bf16((N, K), w_std, g, device)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32,
                           device=device)
    return GroupedCase(name, x_sorted, w, offsets, torch.arange(M, device=device))


# The five workloads at full size.
def tiny(device="cpu", seed=0):
    return dense_case("tiny 128x256x512 fp32-out", 128, 256, 512, seed=seed, device=device,
                      out_fp32=True)


def mla_q(device="cpu", seed=0):
    return dense_case("MLA q up-projection 4096x24576x1536", 4096, 24576, 1536, seed=seed,
                      device=device, outlier_p=0.001, outlier_scale=50.0)


def mla_kv(device="cpu", seed=0):
    return dense_case("MLA kv up-projection 8192x32768x512", 8192, 32768, 512, seed=seed,
                      device=device)


def experts(device="cpu", seed=0, keep_x=False):
    return grouped_case("routed experts 4096 tok top-8 of 256, 2048x7168", 4096, 256, 8,
                        2048, 7168, seed=seed, device=device, keep_x=keep_x)


def experts_small(device="cpu", seed=0, keep_x=False):
    """The routed-expert workload at a quarter of the experts and tokens
    (1024 tokens, top-8 of 64 experts): the same ~128 routed rows per expert
    and the same weight shape, with 0.94 GB of FP8 weights (still far above
    L2).  It is the case the profiler captures of the expert kernels run on."""
    return grouped_case("routed experts 1024 tok top-8 of 64, 2048x7168", 1024, 64, 8,
                        2048, 7168, seed=seed, device=device, keep_x=keep_x)


def dgrad(device="cpu", seed=0):
    return dense_case("dgrad 8192x18432x7168 student-t", 8192, 18432, 7168, seed=seed,
                      device=device, heavy_tail=True, b_major=1)


def wgrad(device="cpu", seed=0):
    """Weight gradient of the data-gradient layer: dY 8192x7168 (Student-t),
    X 8192x18432 ~N(0,1), dW = dY^T . X is 7168x18432 over 8192 tokens."""
    return wgrad_case("wgrad 7168x18432 over 8192 tokens", 8192, 7168, 18432, seed=seed, device=device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a BF16 tensor as its uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
