"""Parity of the GEMM with an E4M3 output (the output quantised per 1x128 row
tile in the epilogue, `fp8_gemm_blockscaled_e4m3_out`).

Two checks:
1. Bit for bit, it equals the BF16-output GEMM followed by the activation
   quantiser on that BF16 matrix (same arithmetic, same encoder rule).
2. Against the float64 oracle, its dequantised output stays within a bound
   derived from the arithmetic. With x the BF16 output value, s = amax_tile(|x|)/448
   and v = x/s, the E4M3 code is within half a step of v: 2^-4 |v| in the normal range
   and 2^-10 below 2^-6. So |dec(q)*s - x| <= 2^-4 |x| + 2^-10 s, and the GEMM's
   own acceptance bound E = 2e-3 ||a_m|| ||b_n|| covers |x - ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import MAX_E, host_u8
from synthetic import bf16_bits, generator, normal_bf16

pytestmark = pytest.mark.gpu
import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
DEV = "cuda"


def operands(M, N, K, b_major, seed, zero_rows=()):
    g = generator(seed, DEV)
    a = normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.002, outlier_scale=40.0)
    for r in zero_rows:
        a[r] = 0
    w = normal_bf16((N, K) if b_major == 0 else (K, N), 0.02, g, DEV)
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    return a, w, qa, sa, qb, sb


@pytest.mark.parametrize("M,N,K,b_major", [
    (128, 256, 512, 0), (300, 384, 640, 0), (129, 128, 256, 0), (512, 1024, 1024, 0),
    (1, 128, 128, 0), (200, 384, 512, 1), (333, 640, 896, 1), (64, 256, 384, 1)])
def test_e4m3_out_equals_gemm_then_quantiser(M, N, K, b_major):
    _, _, qa, sa, qb, sb = operands(M, N, K, b_major, seed=M + N + K + b_major)
    qc, sc = fp8.fp8_gemm_blockscaled_e4m3_out(qa, sa, qb, sb, b_major=b_major)
    c = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, b_major=b_major)
    q2, s2 = fp8.fp8_quant_act_1x128(c)
    assert fp8.fp8bs_last_error() == 0
    assert torch.equal(qc, q2), f"{M}x{N}x{K}: codes differ"
    assert torch.equal(sc.view(torch.int32), s2.view(torch.int32)), f"{M}x{N}x{K}: scales differ"


@pytest.mark.parametrize("b_major", [0, 1])
def test_e4m3_out_within_derived_bound_of_oracle(b_major):
    M, N, K = 300, 512, 768
    a, w, qa, sa, qb, sb = operands(M, N, K, b_major, seed=41 + b_major, zero_rows=(7, 260))
    qc, sc = fp8.fp8_gemm_blockscaled_e4m3_out(qa, sa, qb, sb, b_major=b_major)
    torch.cuda.synchronize()
    oqa, osa = oracle.quant_act_1x128(bf16_bits(a))
    oqb, osb = oracle.quant_w_128x128(bf16_bits(w))
    assert np.array_equal(host_u8(qa), oqa) and np.array_equal(host_u8(qb), oqb)
    ref = oracle.gemm_f64(oqa, osa, oqb, osb, b_major=b_major)
    e_bound = MAX_E * np.outer(oracle.act_row_norms(oqa, osa), oracle.b_row_norms(oqb, osb, b_major=b_major))
    codes = host_u8(qc)
    scales = sc.cpu().numpy().astype(np.float64)                    # [N/128, M]
    deq = oracle.e4m3_decode_table()[codes] * np.repeat(scales.T, 128, axis=1)
    tiles = np.abs(ref).reshape(M, N // 128, 128)
    amax_ref = np.repeat(tiles.max(axis=2), 128, axis=1)
    e_tile = np.repeat(e_bound.reshape(M, N // 128, 128).max(axis=2), 128, axis=1)
    bound = (2.0 ** -4) * (np.abs(ref) + e_bound) + (amax_ref + e_tile) / (448.0 * 1024.0) * 1.001 \
        + e_bound * 1.001 + 1e-7 * np.abs(ref)
    err = np.abs(deq - ref)
    assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e}"
    # scales: fp32(amax/448) of the BF16 output tile, within the GEMM bound of the oracle's
    sc_ref = tiles.max(axis=2).T / 448.0
    et = e_bound.reshape(M, N // 128, 128).max(axis=2).T / 448.0
    assert np.all(np.abs(scales - sc_ref) <= et + 2e-7 * sc_ref)
    # rows of zeros: scale 0 and +0 codes
    for r in (7, 260):
        assert np.all(scales[:, r] == 0) and np.all(codes[r] == 0)


def test_e4m3_out_row_stride_and_k0():
    _, _, qa, sa, qb, sb = operands(130, 256, 256, 0, seed=5)
    big = torch.full((130, 288), 0xAB, dtype=torch.uint8, device=DEV)
    qc, sc = fp8.fp8_gemm_blockscaled_e4m3_out(qa, sa, qb, sb, qC=big[:, :256])
    q_ref, s_ref = fp8.fp8_gemm_blockscaled_e4m3_out(qa, sa, qb, sb)
    torch.cuda.synchronize()
    assert torch.equal(big[:, :256], q_ref) and torch.equal(sc, s_ref)
    assert torch.all(big[:, 256:] == 0xAB)
    # K == 0: C is the empty sum, so zero codes and zero scales
    qa0 = torch.empty((10, 0), dtype=torch.uint8, device=DEV)
    sa0 = torch.empty((0, 10), dtype=torch.float32, device=DEV)
    qb0 = torch.empty((128, 0), dtype=torch.uint8, device=DEV)
    sb0 = torch.empty((1, 0), dtype=torch.float32, device=DEV)
    q0 = torch.full((10, 128), 0x55, dtype=torch.uint8, device=DEV)
    s0 = torch.full((1, 10), 3.0, dtype=torch.float32, device=DEV)
    fp8.fp8_gemm_blockscaled_e4m3_out(qa0, sa0, qb0, sb0, qC=q0, sC=s0)
    torch.cuda.synchronize()
    assert torch.all(q0 == 0) and torch.all(s0 == 0)


@pytest.mark.parametrize("wl", ["mla_q", "mla_kv"])
def test_e4m3_out_full_size_equals_gemm_then_quantiser(wl):
    import synthetic
    case = getattr(synthetic, wl)(device=DEV)
    qa, sa = fp8.fp8_quant_act_1x128(case.a)
    qb, sb = fp8.fp8_quant_w_128x128(case.w)
    qc, sc = fp8.fp8_gemm_blockscaled_e4m3_out(qa, sa, qb, sb)
    c = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb)
    q2, s2 = fp8.fp8_quant_act_1x128(c)
    assert fp8.fp8bs_last_error() == 0
    assert torch.equal(qc, q2) and torch.equal(sc.view(torch.int32), s2.view(torch.int32))
