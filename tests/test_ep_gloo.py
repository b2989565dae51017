"""Expert-parallel dispatch and combine over gloo ranks on the CPU (no GPU).

World sizes 2 and 4 run as spawned processes with a gloo process group and
the layer's real planning and exchange code (``FP8ExpertParallel.forward``
over ``TorchDistComm``).  The four data steps, which on a GPU are the
library's kernels, are supplied here by the test from the CPU oracle: pack =
the oracle's 1x128 quantisation of the routed rows, packed with their scales;
unpack / row gather = numpy indexing; grouped GEMM = the oracle's float64
grouped GEMM.  Every rank's per-slot outputs must then equal, bit for bit,
the oracle's GEMM of each routed token row with its expert's weight computed
directly in one process -- which checks the routing plan, the count and
payload exchanges, the receive permutation, the expert offsets and the
return path.  The GPU test of the same layer (tests/test_gpu_ep.py) runs the
kernels.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

E, K, N, TOPK, T = 8, 256, 136, 2, 48


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(rank):
    """Tokens of one rank, its routing, and every expert's weight (the same
    on every rank)."""
    from synthetic import generator, normal_bf16
    g = generator(100 + rank, "cpu")
    x = normal_bf16((T, K), 1.0, g, "cpu", outlier_p=0.01, outlier_scale=30.0)
    rng = np.random.default_rng(rank)
    # expert 0 is never chosen; rank 1 routes only to the upper half of the
    # experts, so the lower ranks receive nothing from it
    lo = E // 2 if rank == 1 else 1
    choice = np.stack([rng.choice(np.arange(lo, E), size=TOPK, replace=False) for _ in range(T)])
    gw = generator(7, "cpu")
    w = torch.stack([normal_bf16((N, K), 0.02, gw, "cpu") for _ in range(E)])
    return x, torch.from_numpy(choice.astype(np.int64)), w


class OracleOps:
    """CPU stand-ins for the four data steps (test infrastructure)."""

    @staticmethod
    def pack(x, rows, dest, row_bytes):
        import oracle
        from synthetic import bf16_bits
        xr = x[rows.long()]
        q, s = oracle.quant_act_1x128(bf16_bits(xr))
        M, Kx = q.shape
        out = np.zeros((M, row_bytes), np.uint8)
        out[:, :Kx] = q
        out[:, Kx:Kx + 4 * (Kx // 128)] = np.ascontiguousarray(s.T).view(np.uint8).reshape(M, -1)
        return torch.from_numpy(out)

    @staticmethod
    def unpack(packed, Kx, perm):
        p = packed.numpy()[perm.numpy()]
        q = np.ascontiguousarray(p[:, :Kx])
        s = np.ascontiguousarray(p[:, Kx:Kx + 4 * (Kx // 128)]).view(np.float32).T
        return torch.from_numpy(q), torch.from_numpy(np.ascontiguousarray(s))

    @staticmethod
    def grouped_gemm(q, sA, qw, sw, offsets, out_dtype):
        import oracle
        c = oracle.grouped_gemm_f64(q.numpy(), sA.numpy(), qw.numpy(), sw.numpy(), offsets.numpy())
        return torch.from_numpy(c)

    @staticmethod
    def gather_rows(src, rows):
        return src[rows.long()].contiguous()


def _rank_main(rank, world, port, result_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from synthetic import bf16_bits
        from fp8_fine_grained_26_b300.ep import FP8ExpertParallel, TorchDistComm
        x, choice, w = _inputs(rank)
        e_local = E // world
        mine = range(rank * e_local, (rank + 1) * e_local)
        qw, sw = zip(*[oracle.quant_w_128x128(bf16_bits(w[e])) for e in mine])
        layer = FP8ExpertParallel(E, world, rank, torch.from_numpy(np.stack(qw)), torch.from_numpy(np.stack(sw)),
                                  comm=TorchDistComm(), ops=OracleOps)
        y = layer.forward(x, choice, out_dtype=torch.float64).numpy()
        # the same outputs computed directly: token row quantised alone, times its expert
        ref = np.empty_like(y)
        qx, sx = oracle.quant_act_1x128(bf16_bits(x))
        qws = {}
        for t in range(T):
            for k in range(TOPK):
                e = int(choice[t, k])
                if e not in qws:
                    qws[e] = oracle.quant_w_128x128(bf16_bits(w[e]))
                ref[t * TOPK + k] = oracle.gemm_f64(qx[t:t + 1], np.ascontiguousarray(sx[:, t:t + 1]),
                                                   *qws[e])[0]
        result_q.put((rank, bool(np.array_equal(y, ref)), float(np.max(np.abs(y - ref)))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_ep_forward_over_gloo_matches_direct_oracle(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, equal, diff in sorted(results):
        assert equal, f"rank {rank}: largest difference {diff}"


def test_plans_conserve_and_order_rows():
    from fp8_fine_grained_26_b300.ep import plan_recv, plan_send
    rng = np.random.default_rng(3)
    choice = np.stack([rng.choice(16, size=3, replace=False) for _ in range(40)])   # distinct top-3
    sp = plan_send(choice, 16, 4)
    assert sp.send_counts.sum() == 120 and np.array_equal(np.sort(sp.order), np.arange(120))
    experts = choice.reshape(-1)[sp.order]
    assert np.all(np.diff(experts) >= 0)                          # grouped by expert (so by rank)
    toks = sp.tokens
    for e in np.unique(experts):
        assert np.all(np.diff(toks[experts == e]) > 0)            # then by token
    counts_from = rng.integers(0, 5, size=(4, 4))
    counts_from[2, 1] = 0
    rp = plan_recv(counts_from)
    assert np.array_equal(np.sort(rp.perm), np.arange(counts_from.sum()))
    assert np.array_equal(np.diff(rp.offsets), counts_from.sum(axis=0))
    # the rows of expert e, in source order, are the e-blocks of each source's chunk
    base = np.concatenate([[0], np.cumsum(counts_from.sum(axis=1))])
    within = np.concatenate([np.zeros((4, 1), int), np.cumsum(counts_from, axis=1)], axis=1)
    for e in range(4):
        want = np.concatenate([np.arange(base[s] + within[s, e], base[s] + within[s, e + 1]) for s in range(4)])
        assert np.array_equal(rp.perm[rp.offsets[e]:rp.offsets[e + 1]], want)
