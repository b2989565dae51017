"""Expert-parallel routed-expert layer with an FP8 all-to-all.

The pages run the routed experts of the MoE layers expert-parallel: each
device holds a subset of the 256 routed experts, the tokens routed to an
expert on another device travel there over an all-to-all, and the activations
are dispatched in FP8 ("DeepSeek-V3 training walkthrough", section 二:
cross-node all-to-all communication and expert parallelism, and section
二(四), last item: activations cached and dispatched in FP8; qqstock.cn
walkthrough, FP8 section, report figure 10).  One step of a rank:

  1. plan (host): every routed copy (token t, slot k) of this rank's tokens
     goes to expert e = choice[t, k], held by rank e // E_local; the copies
     are sent in (expert, token) order, so each destination's rows arrive
     grouped by its local experts;
  2. counts exchange: each rank tells every other how many rows it sends to
     each of that rank's experts;
  3. pack (kernel fp8_ep_dispatch_pack_scatter): 1x128 quantisation of each
     token row once, its codes packed with its FP32 scales into the send row
     of every routed copy;
  4. dispatch (all-to-all of the packed FP8 rows);
  5. unpack (kernel fp8_ep_unpack): received rows into expert-major order and
     the GEMM's scale layout;
  6. the local grouped GEMM (fp8_grouped_gemm_blockscaled) over this rank's
     experts;
  7. return (kernel fp8bs_gather_rows, then an all-to-all of the BF16 expert
     outputs back to their source ranks, then fp8bs_gather_rows into
     (token, slot) order).

The gate-weighted sum of a token's k expert outputs belongs to the model,
not to this layer; ``forward`` returns the per-slot outputs [T * topk, N].

The step is split into three phases around the two exchanges
(``dispatch_send`` -> exchange -> ``expert_compute`` -> exchange ->
``combine_receive``) so that several ranks can also be driven from one
process.  The exchanges go through a ``comm`` object with
``all_to_all_single(out, inp, out_splits, in_splits)`` (torch.distributed in
a real run); host planning uses numpy.  The four data steps (pack, unpack,
grouped GEMM, row gather) go through an ``ops`` object, by default
``KernelOps``: the library's CUDA kernels, the only implementation this
package has.
"""
from dataclasses import dataclass

import numpy as np
import torch

from . import (fp8_ep_dispatch_pack_scatter, fp8_ep_unpack, fp8_grouped_gemm_blockscaled, fp8bs_gather_rows,
               packed_row_bytes)


class KernelOps:
    """The data steps of the layer, as the library's CUDA kernels."""

    @staticmethod
    def pack(x, rows, dest, row_bytes):
        """Send rows: token rows[i] quantised into packed row i; the kernel
        works from the token side (dest[t, j]: the send row of token t's j-th
        copy), encoding each token once."""
        packed = torch.empty((rows.numel(), row_bytes), dtype=torch.uint8, device=x.device)
        return fp8_ep_dispatch_pack_scatter(x, dest, rows.numel(), packed)

    @staticmethod
    def unpack(packed, K, perm):
        return fp8_ep_unpack(packed, K, perm)

    @staticmethod
    def grouped_gemm(q, sA, qw, sw, offsets, out_dtype):
        return fp8_grouped_gemm_blockscaled(q, sA, qw, sw, offsets, out_dtype=out_dtype)

    @staticmethod
    def gather_rows(src, rows):
        return fp8bs_gather_rows(src, rows)


class TorchDistComm:
    """The exchanges over torch.distributed (NCCL for CUDA tensors, gloo for
    CPU tensors)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist, self.group = dist, group

    def all_to_all_single(self, out, inp, out_splits, in_splits):
        self.dist.all_to_all_single(out, inp, list(map(int, out_splits)), list(map(int, in_splits)),
                                    group=self.group)


@dataclass
class SendPlan:
    order: np.ndarray          # [T*topk] flat (t*topk + k) index of each send row
    tokens: np.ndarray         # [T*topk] token of each send row
    send_counts: np.ndarray    # [world] rows to each rank
    expert_counts: np.ndarray  # [E] rows to each global expert


def plan_send(choice: np.ndarray, num_experts: int, world: int) -> SendPlan:
    """Send order of the routed copies: sorted by (expert, token), which
    groups them by destination rank and, within it, by the destination's
    local expert."""
    T, topk = choice.shape
    expert = choice.reshape(-1).astype(np.int64)
    if expert.size and (expert.min() < 0 or expert.max() >= num_experts):
        raise ValueError("expert index out of range")
    token = np.repeat(np.arange(T, dtype=np.int64), topk)
    order = np.lexsort((token, expert))
    e_local = num_experts // world
    counts = np.bincount(expert, minlength=num_experts).astype(np.int64)
    send_counts = counts.reshape(world, e_local).sum(axis=1)
    return SendPlan(order=order, tokens=token[order], send_counts=send_counts, expert_counts=counts)


@dataclass
class RecvPlan:
    perm: np.ndarray           # [M_recv] received-buffer index of each expert-major row
    offsets: np.ndarray        # [E_local + 1] expert segment offsets (expert-major order)
    recv_counts: np.ndarray    # [world] rows received from each rank


def plan_recv(counts_from: np.ndarray) -> RecvPlan:
    """counts_from[src, e]: rows source rank src sends to local expert e.
    The received buffer holds src 0's rows (expert-major), then src 1's, ...;
    the grouped GEMM wants expert-major, and within an expert, by source."""
    world, e_local = counts_from.shape
    recv_counts = counts_from.sum(axis=1)
    src_base = np.concatenate([[0], np.cumsum(recv_counts)[:-1]]).astype(np.int64)
    within = np.concatenate([np.zeros((world, 1), np.int64), np.cumsum(counts_from, axis=1)[:, :-1]], axis=1)
    per_expert = counts_from.sum(axis=0)
    offsets = np.concatenate([[0], np.cumsum(per_expert)]).astype(np.int64)
    perm = np.empty(int(offsets[-1]), np.int64)
    for e in range(e_local):
        pos = offsets[e]
        for s in range(world):
            n = int(counts_from[s, e])
            start = src_base[s] + within[s, e]
            perm[pos:pos + n] = np.arange(start, start + n)
            pos += n
    return RecvPlan(perm=perm, offsets=offsets, recv_counts=recv_counts)


class FP8ExpertParallel:
    """One rank's share of an expert-parallel routed-expert GEMM.

    qw_local [E_local, N, K] / sw_local [E_local, ceil(N/128), K/128]: this
    rank's experts (global ids rank*E_local ... rank*E_local + E_local - 1),
    quantised 128x128 (fp8_quant_w_128x128)."""

    def __init__(self, num_experts, world, rank, qw_local, sw_local, comm=None, ops=KernelOps):
        if num_experts % world != 0:
            raise ValueError("the experts must split evenly over the ranks")
        self.E, self.world, self.rank = num_experts, world, rank
        self.e_local = num_experts // world
        if qw_local.shape[0] != self.e_local:
            raise ValueError("qw_local must hold this rank's experts")
        self.qw, self.sw = qw_local, sw_local
        _, self.N, self.K = qw_local.shape
        self.comm, self.ops = comm, ops
        self.row_bytes = packed_row_bytes(self.K)

    # ---- phase 1: plan and pack ------------------------------------------
    def dispatch_send(self, x: torch.Tensor, choice: torch.Tensor):
        """x [T, K] BF16 and choice [T, topk] expert ids (device).  Returns the
        state of this step, with .packed (send rows), .send_counts and
        .counts_to (rows per destination rank and its local expert)."""
        dev = x.device
        plan = plan_send(choice.detach().cpu().numpy(), self.E, self.world)
        rows = torch.from_numpy(plan.tokens.astype(np.int32)).to(dev)
        n = plan.order.shape[0]
        send_row = np.empty(n, np.int64)
        send_row[plan.order] = np.arange(n)                  # (t, k) -> its row in send order
        dest = torch.from_numpy(send_row.reshape(choice.shape).astype(np.int32)).to(dev)
        packed = self.ops.pack(x, rows, dest, self.row_bytes)
        return _Step(plan=plan, packed=packed, topk=choice.shape[1], T=x.shape[0],
                     counts_to=plan.expert_counts.reshape(self.world, self.e_local))

    # ---- phase 2: expert GEMMs on the received rows -----------------------
    def expert_compute(self, step, packed_recv: torch.Tensor, counts_from: np.ndarray, out_dtype=torch.bfloat16):
        """packed_recv: the rows received from every source rank, in source
        order; counts_from [world, E_local].  Returns this rank's expert
        outputs reordered by source (the rows to send back) and their counts."""
        dev = packed_recv.device
        rp = plan_recv(np.asarray(counts_from, np.int64))
        M = int(rp.offsets[-1])
        step.recv = rp
        perm = torch.from_numpy(rp.perm.astype(np.int32)).to(dev)
        q, sA = self.ops.unpack(packed_recv, self.K, perm)
        offsets = torch.from_numpy(rp.offsets.astype(np.int32)).to(dev)
        y = self.ops.grouped_gemm(q, sA, self.qw, self.sw, offsets, out_dtype)
        # back into received (source-major) order: row perm[i] of the buffer is y[i]
        inv = np.empty(M, np.int64)
        inv[rp.perm] = np.arange(M)
        return self.ops.gather_rows(y, torch.from_numpy(inv.astype(np.int32)).to(dev)), rp.recv_counts

    # ---- phase 3: back into (token, slot) order ----------------------------
    def combine_receive(self, step, y_back: torch.Tensor) -> torch.Tensor:
        """y_back: this rank's rows returned by every expert rank, in send
        order.  Returns [T * topk, N]: row t*topk + k is expert choice[t, k]'s
        output for token t."""
        n = step.T * step.topk
        slot_to_send = np.empty(n, np.int64)
        slot_to_send[step.plan.order] = np.arange(n)
        idx = torch.from_numpy(slot_to_send.astype(np.int32)).to(y_back.device)
        return self.ops.gather_rows(y_back, idx)

    # ---- one whole step over `comm` ----------------------------------------
    def forward(self, x: torch.Tensor, choice: torch.Tensor, out_dtype=torch.bfloat16) -> torch.Tensor:
        if self.comm is None:
            raise ValueError("forward needs a comm (use the phases to drive ranks by hand)")
        dev = x.device
        step = self.dispatch_send(x, choice)
        counts_in = torch.from_numpy(np.ascontiguousarray(step.counts_to).reshape(-1)).to(dev)
        counts_out = torch.empty_like(counts_in)
        self.comm.all_to_all_single(counts_out, counts_in, [self.e_local] * self.world, [self.e_local] * self.world)
        counts_from = counts_out.cpu().numpy().reshape(self.world, self.e_local)
        recv_counts = counts_from.sum(axis=1)
        packed_recv = torch.empty((int(recv_counts.sum()), self.row_bytes), dtype=torch.uint8, device=dev)
        self.comm.all_to_all_single(packed_recv, step.packed, recv_counts, step.plan.send_counts)
        y_src, back_counts = self.expert_compute(step, packed_recv, counts_from, out_dtype)
        y_back = torch.empty((int(step.plan.send_counts.sum()), self.N), dtype=out_dtype, device=dev)
        self.comm.all_to_all_single(y_back, y_src, step.plan.send_counts, back_counts)
        return self.combine_receive(step, y_back)


@dataclass
class _Step:
    plan: SendPlan
    packed: torch.Tensor
    topk: int
    T: int
    counts_to: np.ndarray
    recv: RecvPlan = None
