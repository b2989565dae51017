"""GPU parity of fp8_quant_act_w (both operands of one GEMM quantised in one
launch) against the CPU oracle: the activation's 1x128 codes and scales and
the weight's 128x128 codes and scales must be bit-identical to the oracle's,
and to the two single-operand calls."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import bf16_bits, generator, normal_bf16
from parity import host_u8

pytestmark = pytest.mark.gpu

import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
DEV = "cuda"


def _bits_f32(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def check_pair(x, w, what):
    qa, sA, qw, sW = fp8.fp8_quant_act_w(x, w)
    torch.cuda.synchronize()
    assert fp8.fp8bs_last_error() == 0
    if x.numel():
        qo, so = oracle.quant_act_1x128(bf16_bits(x))
        qg = host_u8(qa)
        nbad = int(np.count_nonzero(qg != qo))
        assert nbad == 0, f"{what} activation: {nbad} E4M3 codes differ, first at {np.argwhere(qg != qo)[:5].tolist()}"
        np.testing.assert_array_equal(_bits_f32(sA.cpu().numpy()), _bits_f32(so), err_msg=what)
    if w.numel():
        qo, so = oracle.quant_w_128x128(bf16_bits(w))
        qg = host_u8(qw)
        nbad = int(np.count_nonzero(qg != qo))
        assert nbad == 0, f"{what} weight: {nbad} E4M3 codes differ"
        np.testing.assert_array_equal(_bits_f32(sW.cpu().numpy()), _bits_f32(so), err_msg=what)
    return qa, sA, qw, sW


@pytest.mark.parametrize("M,K,R,C", [(1, 128, 1, 128), (17, 256, 200, 384), (300, 640, 513, 640),
                                     (1025, 1536, 128, 128), (4, 384, 1300, 256)])
def test_pair_random_ragged(M, K, R, C):
    g = generator(M * 7 + R, DEV)
    x = normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.01, outlier_scale=50.0)
    w = normal_bf16((R, C), 0.02, g, DEV)
    check_pair(x, w, f"act {M}x{K} + weight {R}x{C}")


@pytest.mark.parametrize("which", ["act", "weight"])
def test_pair_with_one_empty_operand(which):
    g = generator(31, DEV)
    if which == "act":
        x = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
        w = normal_bf16((300, 256), 0.02, g, DEV)
    else:
        x = normal_bf16((300, 256), 1.0, g, DEV)
        w = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    check_pair(x, w, f"empty {which}")


def test_pair_strided_rows_and_outputs():
    g = generator(5, DEV)
    big_x = normal_bf16((64, 1024), 2.0, g, DEV)
    big_w = normal_bf16((300, 1024), 0.02, g, DEV)
    x, w = big_x[:, 256:768], big_w[:, 128:640]            # row strides 1024 > 512
    qa_big = torch.zeros((64, 640), dtype=torch.uint8, device=DEV)
    qw_big = torch.zeros((300, 640), dtype=torch.uint8, device=DEV)
    qa, sA, qw, sW = fp8.fp8_quant_act_w(x, w, qa=qa_big[:, :512], qw=qw_big[:, :512])
    torch.cuda.synchronize()
    qo, so = oracle.quant_act_1x128(bf16_bits(x))
    np.testing.assert_array_equal(host_u8(qa), qo)
    np.testing.assert_array_equal(_bits_f32(sA.cpu().numpy()), _bits_f32(so))
    qo, so = oracle.quant_w_128x128(bf16_bits(w))
    np.testing.assert_array_equal(host_u8(qw), qo)
    np.testing.assert_array_equal(_bits_f32(sW.cpu().numpy()), _bits_f32(so))
    # the bytes past each output row's K columns are not written
    assert int(qa_big[:, 512:].count_nonzero()) == 0 and int(qw_big[:, 512:].count_nonzero()) == 0


def test_pair_equals_single_operand_calls_on_adversarial_blocks():
    # constant, all-zero and single-outlier tiles, plus values at the
    # E4M3 rounding midpoints, in both operands
    g = generator(11, DEV)
    x = normal_bf16((256, 512), 1.0, g, DEV)
    x[0:8, :] = 0
    x[8:16, :] = 3.0
    x[16, 5] = 1.0e4
    w = normal_bf16((384, 512), 0.02, g, DEV)
    w[:128, :128] = 0
    w[128:256, 128:256] = -0.5
    w[300, 400] = -7.0e3
    qa, sA, qw, sW = check_pair(x, w, "adversarial")
    qa1, sA1 = fp8.fp8_quant_act_1x128(x)
    qw1, sW1 = fp8.fp8_quant_w_128x128(w)
    assert torch.equal(qa, qa1) and torch.equal(sA.view(torch.int32), sA1.view(torch.int32))
    assert torch.equal(qw, qw1) and torch.equal(sW.view(torch.int32), sW1.view(torch.int32))


def test_pair_full_mla_q():
    # the forward step's launch: A 4096x1536 (outliers) and W 24576x1536 together
    c = synthetic.mla_q(device=DEV)
    check_pair(c.a, c.w, "mla_q A 4096x1536 + W 24576x1536")


def test_pair_full_mla_kv():
    c = synthetic.mla_kv(device=DEV)
    check_pair(c.a, c.w, "mla_kv A 8192x512 + W 32768x512")


def test_pair_full_dgrad():
    c = synthetic.dgrad(device=DEV)
    check_pair(c.a, c.w, "dgrad dY 8192x7168 + W stored 7168x18432")
