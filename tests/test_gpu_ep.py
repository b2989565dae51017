"""Expert-parallel dispatch/combine on the GPU: the kernels and the layer.

* fp8_ep_dispatch_pack: codes and scales bit-equal to the gather quantiser
  (and so to the oracle's quantisation of the gathered rows), scales packed
  after the codes of each row; fp8_ep_dispatch_pack_scatter (the form the
  layer uses: each token encoded once) bit-equal to it.
* fp8_ep_unpack and fp8bs_gather_rows: pure data movement, bit-equal to
  numpy indexing; an out-of-range index gives a zero row and FP8BS_ERR_INDEX.
* The layer at world size 1 (the exchanges are copies) on the routed-expert
  workload: every row of 16 experts against the oracle's GEMM.
* 2, 4 and 8 ranks emulated in one process on one GPU, each phase of every
  rank run in turn with the exchanges done by slicing (no rank waits on
  another on the device): every rank's outputs are bit-identical to the
  world-1 run over all tokens, since each output row depends only on its own
  token row and its expert.  Multi-GPU runs are not measured here (one GPU).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import ErrorStats, host_u8
from synthetic import bf16_bits, generator, normal_bf16

pytestmark = pytest.mark.gpu
import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
from fp8_fine_grained_26_b300.ep import FP8ExpertParallel

DEV = "cuda"


def test_dispatch_pack_equals_gather_quantiser():
    g = generator(3, DEV)
    T, K = 300, 1024
    x = normal_bf16((T, K), 1.0, g, DEV, outlier_p=0.01, outlier_scale=60.0)
    x[17] = 0
    rows = torch.randint(0, T, (777,), generator=g, device=DEV, dtype=torch.int64).to(torch.int32)
    rows[5] = 17
    packed = fp8.fp8_ep_dispatch_pack(x, rows)
    q, s = fp8.fp8_quant_act_1x128_gather(x, rows)
    assert fp8.fp8bs_last_error() == 0
    KB = K // 128
    assert packed.shape[1] == fp8.packed_row_bytes(K)
    assert torch.equal(packed[:, :K], q)
    ps = packed[:, K:K + 4 * KB].contiguous().view(torch.float32)          # [M, KB]
    assert torch.equal(ps.t().contiguous().view(torch.int32), s.view(torch.int32))
    oq, os_ = oracle.quant_act_1x128(bf16_bits(x[rows.long()]))
    assert np.array_equal(host_u8(packed[:, :K]), oq)
    assert np.array_equal(ps.cpu().numpy().T.copy().view(np.uint32), os_.view(np.uint32))


def test_dispatch_pack_scatter_equals_gather_form():
    g = generator(5, DEV)
    T, K, topk = 200, 1024, 3
    x = normal_bf16((T, K), 1.0, g, DEV, outlier_p=0.01, outlier_scale=60.0)
    M = T * topk
    send_row = torch.randperm(M, generator=torch.Generator().manual_seed(1)).to(torch.int32)
    dest = send_row.view(T, topk).to(DEV)
    rows = torch.empty(M, dtype=torch.int32)
    rows[send_row.long()] = torch.arange(T, dtype=torch.int32).repeat_interleave(topk)
    a = fp8.fp8_ep_dispatch_pack_scatter(x, dest, M)
    b = fp8.fp8_ep_dispatch_pack(x, rows.to(DEV))
    assert fp8.fp8bs_last_error() == 0
    KB = K // 128
    assert torch.equal(a[:, :K + 4 * KB], b[:, :K + 4 * KB])


def test_unpack_and_gather_rows_are_exact_data_movement():
    g = generator(4, DEV)
    K, n_src, M = 768, 500, 640
    ld = fp8.packed_row_bytes(K)
    packed = torch.randint(0, 256, (n_src, ld), generator=g, device=DEV, dtype=torch.int64).to(torch.uint8)
    perm = torch.randint(0, n_src, (M,), generator=g, device=DEV, dtype=torch.int64).to(torch.int32)
    q, sA = fp8.fp8_ep_unpack(packed, K, perm)
    assert fp8.fp8bs_last_error() == 0
    p = packed.cpu().numpy()[perm.cpu().numpy()]
    assert np.array_equal(host_u8(q), p[:, :K])
    assert np.array_equal(sA.cpu().numpy().view(np.uint8).reshape(K // 128, M, 4).transpose(1, 0, 2).reshape(M, -1),
                          p[:, K:K + 4 * (K // 128)])
    y = torch.randn((n_src, 2048), generator=g, device=DEV).to(torch.bfloat16)
    z = fp8.fp8bs_gather_rows(y, perm)
    assert torch.equal(z, y[perm.long()])
    # out-of-range indices: zero rows and an index error
    bad = perm.clone()
    bad[7] = n_src
    bad[9] = -1
    z = fp8.fp8bs_gather_rows(y, bad)
    assert fp8.fp8bs_last_error() == fp8.FP8BS_ERR_INDEX
    assert torch.all(z[7] == 0) and torch.all(z[9] == 0) and torch.equal(z[8], y[bad[8].long()])
    q, sA = fp8.fp8_ep_unpack(packed, K, bad)
    assert fp8.fp8bs_last_error() == fp8.FP8BS_ERR_INDEX
    assert torch.all(q[7] == 0) and torch.all(sA[:, 9] == 0)


class LoopbackComm:
    """World size 1: every exchange is a copy."""

    def all_to_all_single(self, out, inp, out_splits, in_splits):
        out.copy_(inp)


def _experts_layer_inputs(device):
    case = synthetic.experts(device=device, keep_x=True)
    E, N, K = case.w.shape
    qw, sw = fp8.fp8_quant_w_128x128(case.w.view(E * N, K))
    qw, sw = qw.view(E, N, K), sw.view(E, -1, K // 128)
    tokens = case.x.shape[0]
    # the routing the workload drew: slot k of token t is the k-th expert it chose
    topk = 8
    tok = case.token_of_row.cpu().numpy()
    off = case.offsets.cpu().numpy()
    expert_of_row = np.repeat(np.arange(E), np.diff(off))
    choice = np.empty((tokens, topk), np.int64)
    fill = np.zeros(tokens, np.int64)
    for r in range(tok.shape[0]):                      # rows are (expert, token) sorted: experts ascend per token
        t = tok[r]
        choice[t, fill[t]] = expert_of_row[r]
        fill[t] += 1
    assert np.all(fill == topk)
    return case, qw, sw, torch.from_numpy(choice).to(device)


@pytest.fixture(scope="module")
def experts_world1():
    case, qw, sw, choice = _experts_layer_inputs(DEV)
    E = qw.shape[0]
    layer = FP8ExpertParallel(E, 1, 0, qw, sw, comm=LoopbackComm())
    y = layer.forward(case.x, choice)
    assert fp8.fp8bs_last_error() == 0
    return case, qw, sw, choice, y


def test_ep_world1_matches_oracle(experts_world1):
    case, qw, sw, choice, y = experts_world1
    E, N, K = qw.shape
    T, topk = choice.shape
    ch = choice.cpu().numpy()
    qx, sx = oracle.quant_act_1x128(bf16_bits(case.x))
    an_all = oracle.act_row_norms(qx, sx)
    rng = np.random.default_rng(1)
    st = ErrorStats("EP world 1, experts workload, 16 experts' rows")
    for e in sorted(set(rng.integers(0, E, 14).tolist()) | {0, E - 1}):
        t_idx, k_idx = np.nonzero(ch == e)
        if t_idx.size == 0:
            continue
        oqb, osb = oracle.quant_w_128x128(bf16_bits(case.w[e]))
        ref = oracle.gemm_f64(qx[t_idx], np.ascontiguousarray(sx[:, t_idx]), oqb, osb)
        got = y[torch.from_numpy(t_idx * topk + k_idx).to(DEV)].double().cpu().numpy()
        st.add(got, ref, an_all[t_idx], oracle.b_row_norms(oqb, osb))
    st.check()


def test_ep_world1_over_nccl_equals_loopback(experts_world1, tmp_path):
    # The layer's exchanges through torch.distributed with the NCCL backend (a
    # one-rank group on this GPU): the FP8 payload rows, the per-expert counts
    # and the BF16 return rows go through NCCL's all-to-all, and the result is
    # bit-equal to the in-process loopback.  Larger worlds are covered by the
    # gloo tests on the CPU and the emulated ranks below.
    import datetime
    import os
    import torch.distributed as dist
    from fp8_fine_grained_26_b300.ep import TorchDistComm
    case, qw, sw, choice, y = experts_world1
    E = qw.shape[0]
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    store = dist.FileStore(str(tmp_path / "nccl_store"), 1)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120), device_id=torch.device(DEV, 0))
    try:
        layer = FP8ExpertParallel(E, 1, 0, qw, sw, comm=TorchDistComm())
        y2 = layer.forward(case.x, choice)
        torch.cuda.synchronize()
        assert fp8.fp8bs_last_error() == 0
        assert torch.equal(y, y2)
    finally:
        dist.destroy_process_group()


def _emulate(world, x, choice, qw, sw):
    """Every rank's three phases run in turn; the exchanges are slices."""
    E = qw.shape[0]
    el = E // world
    T = x.shape[0] // world
    layers = [FP8ExpertParallel(E, world, r, qw[r * el:(r + 1) * el], sw[r * el:(r + 1) * el]) for r in range(world)]
    steps = [layers[r].dispatch_send(x[r * T:(r + 1) * T], choice[r * T:(r + 1) * T]) for r in range(world)]
    send_off = [np.concatenate([[0], np.cumsum(s.plan.send_counts)]) for s in steps]
    y_src, back_off = [], []
    for d in range(world):
        recv = torch.cat([steps[s].packed[send_off[s][d]:send_off[s][d + 1]] for s in range(world)])
        counts_from = np.stack([steps[s].counts_to[d] for s in range(world)])
        ys, back_counts = layers[d].expert_compute(steps[d], recv, counts_from)
        y_src.append(ys)
        back_off.append(np.concatenate([[0], np.cumsum(back_counts)]))
    outs = []
    for s in range(world):
        y_back = torch.cat([y_src[d][back_off[d][s]:back_off[d][s + 1]] for d in range(world)])
        outs.append(layers[s].combine_receive(steps[s], y_back))
    return torch.cat(outs)


@pytest.mark.parametrize("world", [2, 4, 8])
def test_ep_emulated_ranks_equal_world1(experts_world1, world):
    case, qw, sw, choice, y1 = experts_world1
    y = _emulate(world, case.x, choice, qw, sw)
    assert fp8.fp8bs_last_error() == 0
    assert torch.equal(y.view(torch.int16), y1.view(torch.int16)), f"world {world}"


def test_bench_ep_step_equals_experts_step():
    """The benchmark's expert-parallel step (world size 1) gives, for routed
    copy (t, k), the same row as the dispatch + grouped GEMM step gives for
    that copy's row in (expert, token) order."""
    import bench
    s1 = bench.ExpertsStep(synthetic.experts_small(device=DEV, keep_x=True), fp8, torch)
    s2 = bench.ExpertsEPStep(synthetic.experts_small(device=DEV, keep_x=True), fp8, torch)
    s1.run(0)
    s2.run(0)
    assert fp8.fp8bs_last_error() == 0
    assert torch.equal(s2.c.view(torch.int16), s1.c[s2.slot.long()].view(torch.int16))
