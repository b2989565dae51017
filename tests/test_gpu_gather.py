"""Fused gather + 1x128 quantisation (expert dispatch) on the GPU: bit-exact
against the oracle quantising the gathered BF16 rows, equal to the GPU
quantiser on the gathered matrix, and an out-of-range index reported as
FP8BS_ERR_INDEX by the kernel's own bounds check (no out-of-bounds access)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import host_u8
from synthetic import bf16_bits, generator, normal_bf16

pytestmark = pytest.mark.gpu
import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
DEV = "cuda"


# K in tiles: 1, 3, 9 (= 8 + 1), 56 (= 7 x 8), 33 (= 4 x 8 + 1), 64 (= 8 x 8):
# a warp task is eight tiles, four lanes each, so partial last tasks of 1 and
# 3 tiles and whole ones are all covered
@pytest.mark.parametrize("T,K,M", [(64, 128, 100), (300, 384, 777), (50, 1152, 64), (4096, 7168, 256),
                                   (100, 4224, 50), (20, 8192, 40)])
def test_gather_quantiser_matches_oracle(T, K, M):
    g = generator(T + K + M, DEV)
    x = normal_bf16((T, K), 1.0, g, DEV, outlier_p=0.003, outlier_scale=50.0)
    x[3 % T] = 0
    rows = torch.randint(0, T, (M,), generator=g, device=DEV, dtype=torch.int64).to(torch.int32)
    rows[0] = 3 % T
    q, s = fp8.fp8_quant_act_1x128_gather(x, rows)
    assert fp8.fp8bs_last_error() == 0
    xg = bf16_bits(x)[rows.cpu().numpy()]
    oq, os_ = oracle.quant_act_1x128(xg)
    assert np.array_equal(host_u8(q), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    q2, s2 = fp8.fp8_quant_act_1x128(x.index_select(0, rows.long()))
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s.view(torch.int32), s2.view(torch.int32))


def test_gather_quantiser_adversarial_rows():
    # ties at every E4M3 midpoint, signed zeros, subnormals and extremes,
    # gathered in a scrambled order with repeats
    from test_gpu_quant import _adversarial_rows
    base = _adversarial_rows()
    x = torch.cat([base, base.flip(0)], dim=1).repeat(1, 17).to(DEV)    # K = 34 tiles
    T = x.shape[0]
    g = generator(123, DEV)
    rows = torch.randint(0, T, (3 * T,), generator=g, device=DEV, dtype=torch.int64).to(torch.int32)
    q, s = fp8.fp8_quant_act_1x128_gather(x, rows)
    assert fp8.fp8bs_last_error() == 0
    oq, os_ = oracle.quant_act_1x128(bf16_bits(x)[rows.cpu().numpy()])
    assert np.array_equal(host_u8(q), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))


def test_gather_quantiser_experts_dispatch():
    case = synthetic.experts(device=DEV, keep_x=True)
    rows = case.token_of_row.to(torch.int32)
    q, s = fp8.fp8_quant_act_1x128_gather(case.x, rows)
    q2, s2 = fp8.fp8_quant_act_1x128(case.x_sorted)
    assert fp8.fp8bs_last_error() == 0
    assert torch.equal(q, q2) and torch.equal(s.view(torch.int32), s2.view(torch.int32))


def test_gather_quantiser_bad_index_is_reported():
    g = generator(9, DEV)
    x = normal_bf16((32, 256), 1.0, g, DEV)
    rows = torch.tensor([0, 5, 32, -1, 7], dtype=torch.int32, device=DEV)   # 32 and -1 are out of range
    q = torch.full((5, 256), 0x33, dtype=torch.uint8, device=DEV)
    s = torch.full((2, 5), 9.0, dtype=torch.float32, device=DEV)
    fp8.fp8_quant_act_1x128_gather(x, rows, q=q, sA=s)
    assert fp8.fp8bs_last_error() == fp8.FP8BS_ERR_INDEX
    assert fp8.fp8bs_last_error() == fp8.FP8BS_OK
    assert torch.all(q[2] == 0) and torch.all(q[3] == 0) and torch.all(s[:, 2:4] == 0)
    q2, s2 = fp8.fp8_quant_act_1x128(x.index_select(0, torch.tensor([0, 5, 7], device=DEV)))
    torch.cuda.synchronize()
    assert torch.equal(q[[0, 1, 4]], q2) and torch.equal(s[:, [0, 1, 4]], s2)


# ------------------------------------------------------------ scatter form
def _dest_from_rows(token_of_row, T, topk):
    """dest[t, j]: the j-th output row that holds token t (rows ascending)."""
    order = np.argsort(token_of_row, kind="stable")
    return order.reshape(T, topk).astype(np.int32)


def test_scatter_quantiser_equals_gather_on_the_experts_dispatch():
    case = synthetic.experts(device=DEV, keep_x=True)
    T = case.x.shape[0]
    rows = case.token_of_row.to(torch.int32)
    M = rows.numel()
    dest = torch.from_numpy(_dest_from_rows(case.token_of_row.cpu().numpy(), T, 8)).to(DEV)
    q, s = fp8.fp8_quant_act_1x128_scatter(case.x, dest, M)
    q2, s2 = fp8.fp8_quant_act_1x128_gather(case.x, rows)
    assert fp8.fp8bs_last_error() == 0
    assert torch.equal(q, q2) and torch.equal(s.view(torch.int32), s2.view(torch.int32))


@pytest.mark.parametrize("T,K,topk", [(64, 128, 1), (300, 384, 3), (50, 1152, 8), (100, 4224, 2)])
def test_scatter_quantiser_matches_oracle(T, K, topk):
    g = generator(T * K + topk, DEV)
    x = normal_bf16((T, K), 1.0, g, DEV, outlier_p=0.003, outlier_scale=50.0)
    x[1] = 0
    M = T * topk + 5                                          # 5 rows nobody writes
    perm = torch.randperm(T * topk, generator=torch.Generator().manual_seed(T)).to(torch.int32)
    dest = perm.view(T, topk).to(DEV)
    q = torch.full((M, K), 0x66, dtype=torch.uint8, device=DEV)
    s = torch.full((K // 128, M), 3.5, dtype=torch.float32, device=DEV)
    fp8.fp8_quant_act_1x128_scatter(x, dest, M, q=q, sA=s)
    assert fp8.fp8bs_last_error() == 0
    oq, os_ = oracle.quant_act_1x128(bf16_bits(x))
    d = dest.cpu().numpy()
    qh, sh = host_u8(q), s.cpu().numpy()
    for j in range(topk):
        assert np.array_equal(qh[d[:, j]], oq)
        assert np.array_equal(sh[:, d[:, j]].view(np.uint32), os_.view(np.uint32))
    assert np.all(qh[T * topk:] == 0x66) and np.all(sh[:, T * topk:] == 3.5)       # untouched


def test_scatter_quantiser_bad_destination_is_reported():
    g = generator(10, DEV)
    x = normal_bf16((4, 256), 1.0, g, DEV)
    dest = torch.tensor([[0, 1], [2, 9], [-1, 3], [4, 5]], dtype=torch.int32, device=DEV)   # 9 and -1: out of range
    q = torch.full((6, 256), 0x33, dtype=torch.uint8, device=DEV)
    s = torch.full((2, 6), 9.0, dtype=torch.float32, device=DEV)
    fp8.fp8_quant_act_1x128_scatter(x, dest, 6, q=q, sA=s)
    assert fp8.fp8bs_last_error() == fp8.FP8BS_ERR_INDEX
    q2, s2 = fp8.fp8_quant_act_1x128(x)
    torch.cuda.synchronize()
    for (t, j), row in {(0, 0): 0, (0, 1): 1, (1, 0): 2, (2, 1): 3, (3, 0): 4, (3, 1): 5}.items():
        assert torch.equal(q[row], q2[t]) and torch.equal(s[:, row], s2[:, t])
