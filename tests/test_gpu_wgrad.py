"""Weight-gradient path on the GPU against the oracle: the token-dimension
quantiser (bit-exact) and the GEMM whose operands both carry 1x128 scales
along the tokens (within the GEMM tolerance, normalised by the dequantised
row norms of both operands)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import assert_gemm_ok, gemm_errors, host_f64, host_u8, output_rounding_errors
from synthetic import bf16_bits, generator, normal_bf16

pytestmark = pytest.mark.gpu
import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
DEV = "cuda"


# F is a multiple of 8: BF16 rows must start on 16-byte boundaries (TMA)
@pytest.mark.parametrize("T,F", [(128, 128), (256, 296), (512, 64), (384, 8), (1024, 264)])
def test_token_quantiser_bit_exact(T, F):
    g = generator(T + F, DEV)
    x = normal_bf16((T, F), 1.0, g, DEV, outlier_p=0.005, outlier_scale=60.0)
    x[:, 0] = 0                                                   # an all-zero column
    if F > 3:
        x[128:256 if T > 128 else 128, 3] = -0.0                  # a run of negative zeros
    q, s = fp8.fp8_quant_tokens_1x128(x)
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_tokens_1x128(bf16_bits(x))
    assert np.array_equal(host_u8(q), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))


def test_token_quantiser_equals_row_quantiser_of_transpose():
    g = generator(77, DEV)
    x = synthetic.student_t3_bf16((640, 384), g, DEV)
    q, s = fp8.fp8_quant_tokens_1x128(x)
    q2, s2 = fp8.fp8_quant_act_1x128(x.t().contiguous())
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s.view(torch.int32), s2.view(torch.int32))


def _check(T, M, N, seed, out_dtype=torch.bfloat16):
    case = synthetic.wgrad_case("t", T, M, N, seed=seed, device=DEV)
    qa, sa = fp8.fp8_quant_tokens_1x128(case.dy)
    qb, sb = fp8.fp8_quant_tokens_1x128(case.x)
    c = fp8.fp8_gemm_wgrad(qa, sa, qb, sb, out_dtype=out_dtype)
    assert fp8.fp8bs_last_error() == 0
    oqa, osa = oracle.quant_tokens_1x128(bf16_bits(case.dy))
    oqb, osb = oracle.quant_tokens_1x128(bf16_bits(case.x))
    assert np.array_equal(host_u8(qa), oqa) and np.array_equal(host_u8(qb), oqb)
    ref = oracle.gemm_f64_tokens(oqa, osa, oqb, osb)
    an, bn = oracle.act_row_norms(oqa, osa), oracle.act_row_norms(oqb, osb)
    e, bad = gemm_errors(host_f64(c), ref, an, bn)
    assert_gemm_ok(e, bad, f"wgrad {M}x{N} over {T} tokens", e_out=output_rounding_errors(ref, an, bn, out_dtype))


@pytest.mark.parametrize("T,M,N", [(128, 128, 256), (256, 296, 520), (512, 136, 264), (384, 64, 1000),
                                   (1024, 512, 768)])
def test_wgrad_gemm_matches_oracle(T, M, N):
    _check(T, M, N, seed=T + M + N)


def test_wgrad_gemm_fp32_out():
    _check(256, 200, 384, seed=3, out_dtype=torch.float32)


def test_wgrad_promotion_exact():
    # codes in {0, +-2^j} and power-of-two per-row scales per slice: every
    # partial and sum is exact in FP32, so the GPU must equal the oracle exactly
    rng = np.random.default_rng(17)
    T, M, N = 512, 256, 384
    dy = (448.0 * 2.0 ** (-rng.integers(0, 4, size=(T, M)))) * rng.choice([-1.0, 0.0, 1.0], size=(T, M))
    x = (448.0 * 2.0 ** (-rng.integers(0, 4, size=(T, N)))) * rng.choice([-1.0, 0.0, 1.0], size=(T, N))
    for tb in range(T // 128):                          # one exact 448 * 2^-j amax per run
        dy[tb * 128, :] = 448.0 * 2.0 ** -(tb % 3)
        x[tb * 128, :] = 448.0 * 2.0 ** -(tb % 2)
    dy_t = torch.tensor(dy, dtype=torch.float32).to(torch.bfloat16).to(DEV)
    x_t = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(DEV)
    qa, sa = fp8.fp8_quant_tokens_1x128(dy_t)
    qb, sb = fp8.fp8_quant_tokens_1x128(x_t)
    c = fp8.fp8_gemm_wgrad(qa, sa, qb, sb, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle.gemm_f64_tokens(host_u8(qa), sa.cpu().numpy(), host_u8(qb), sb.cpu().numpy())
    assert np.array_equal(c.cpu().numpy().astype(np.float64), ref)
