"""GPU parity of the block-scaled FP8 GEMMs against the float64 CPU oracle.

The GPU side runs the whole path (quantise A and B on the device, GEMM); the
oracle quantises the same BF16 inputs itself and computes the float64 GEMM
over its own dequantised operands, so no oracle input comes from the CUDA
path.  Acceptance is the normalised-error rule in ``parity.py``; the
exact-arithmetic cases require bit equality.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import bf16_bits, generator, normal_bf16
from parity import assert_gemm_ok, gemm_errors, host_f64, host_u8, output_rounding_errors

pytestmark = pytest.mark.gpu

import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
DEV = "cuda"


def gpu_path(a, w, b_major, out_dtype):
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    c = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, b_major=b_major, out_dtype=out_dtype)
    assert fp8.fp8bs_last_error() == 0
    return qa, sa, qb, sb, c


def oracle_operands(a, w):
    qa, sa = oracle.quant_act_1x128(bf16_bits(a))
    qb, sb = oracle.quant_w_128x128(bf16_bits(w))
    return qa, sa, qb, sb


def full_check(a, w, b_major, out_dtype, what):
    qa, sa, qb, sb, c = gpu_path(a, w, b_major, out_dtype)
    oqa, osa, oqb, osb = oracle_operands(a, w)
    assert np.array_equal(host_u8(qa), oqa) and np.array_equal(host_u8(qb), oqb), \
        f"{what}: quantised operands differ"
    ref = oracle.gemm_f64(oqa, osa, oqb, osb, b_major=b_major)
    an = oracle.act_row_norms(oqa, osa)
    bn = oracle.b_row_norms(oqb, osb, b_major=b_major)
    e, bad = gemm_errors(host_f64(c), ref, an, bn)
    assert_gemm_ok(e, bad, what, e_out=output_rounding_errors(ref, an, bn, out_dtype))
    return c, ref


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 520, 640), (1, 1, 128),
                                   (129, 257, 256), (512, 768, 1024)])
def test_gemm_kmajor_ragged(M, N, K, out_dtype):
    g = generator(M * 7 + N + K, DEV)
    a = normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.002, outlier_scale=50.0)
    w = normal_bf16((N, K), 0.02, g, DEV)
    full_check(a, w, 0, out_dtype, f"K-major {M}x{N}x{K} {out_dtype}")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(200, 384, 512), (128, 128, 128), (333, 640, 896)])
def test_gemm_mnmajor(M, N, K, out_dtype):
    g = generator(M + N * 3 + K, DEV)
    a = synthetic.student_t3_bf16((M, K), g, DEV)
    w = normal_bf16((K, N), 0.02, g, DEV)             # stored [K][N]
    full_check(a, w, 1, out_dtype, f"MN-major {M}x{N}x{K} {out_dtype}")


def _pow2_case(M, N, K, seed, b_major):
    """BF16 inputs whose quantisation is exact: every 1x128 tile / 128x128 block
    holds +-448 * 2^(a - t), t in 0..3, or 0, with its amax 448 * 2^a, a in
    {-1, 0, 1}: the scale is 2^a and the codes are +-448 * 2^-t.  Every FP8
    product, 128-term partial and promoted sum is then exact in FP32."""
    rng = np.random.default_rng(seed)

    def make(rows, cols, block_rows):
        v = np.zeros((rows, cols), np.float32)
        for r0 in range(0, rows, block_rows):
            for c0 in range(0, cols, 128):
                a = rng.integers(-1, 2)
                blk = (448.0 * 2.0 ** (a - rng.integers(0, 4, size=(min(block_rows, rows - r0), 128)))
                       * rng.choice([-1.0, 0.0, 1.0], size=(min(block_rows, rows - r0), 128)))
                blk[0, 0] = 448.0 * 2.0 ** a
                v[r0:r0 + blk.shape[0], c0:c0 + 128] = blk
        return v

    a = make(M, K, 1)
    if b_major == 0:
        w = make(N, K, 128)
    else:
        w = make(K, N, 128)
    return (torch.from_numpy(a).to(torch.bfloat16).to(DEV),
            torch.from_numpy(w).to(torch.bfloat16).to(DEV))


@pytest.mark.parametrize("b_major", [0, 1])
def test_gemm_promotion_exact(b_major):
    """Exact-arithmetic pin: FP32 output must equal the float64 oracle bit for bit."""
    M, N, K = 256, 512, 1024
    a, w = _pow2_case(M, N, K, seed=11 + b_major, b_major=b_major)
    qa, sa, qb, sb, c = gpu_path(a, w, b_major, torch.float32)
    oqa, osa, oqb, osb = oracle_operands(a, w)
    assert np.all(np.log2(osa[osa > 0]) % 1 == 0) and np.all(np.log2(osb[osb > 0]) % 1 == 0)
    ref = oracle.gemm_f64(oqa, osa, oqb, osb, b_major=b_major)
    assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref)
    got = c.cpu().numpy().astype(np.float64)
    nbad = int(np.count_nonzero(got != ref))
    assert nbad == 0, f"{nbad} outputs differ; first {np.argwhere(got != ref)[:4].tolist()}"


def test_gemm_single_k_block_is_scaled_dot_product():
    g = generator(3, DEV)
    a = normal_bf16((64, 128), 1.0, g, DEV)
    w = normal_bf16((96, 128), 0.02, g, DEV)
    full_check(a, w, 0, torch.float32, "K=128")


def test_gemm_zero_rows_and_k0():
    g = generator(4, DEV)
    a = normal_bf16((200, 256), 1.0, g, DEV)
    a[5] = 0
    a[150] = -0.0
    w = normal_bf16((300, 256), 0.02, g, DEV)
    w[7] = 0
    c, _ = full_check(a, w, 0, torch.bfloat16, "zero rows")
    assert torch.all(c[5] == 0) and torch.all(c[150] == 0) and torch.all(c[:, 7] == 0)
    # K == 0: the sum is empty, C is written with zeros
    qa = torch.empty((10, 0), dtype=torch.uint8, device=DEV)
    sa = torch.empty((0, 10), dtype=torch.float32, device=DEV)
    qb = torch.empty((20, 0), dtype=torch.uint8, device=DEV)
    sb = torch.empty((1, 0), dtype=torch.float32, device=DEV)
    c0 = torch.full((10, 24), 7.0, dtype=torch.float32, device=DEV)[:, :20]
    out = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, C=c0)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_gemm_output_row_stride():
    g = generator(6, DEV)
    a = normal_bf16((130, 256), 1.0, g, DEV)
    w = normal_bf16((200, 256), 0.02, g, DEV)
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    big = torch.full((130, 264), 5.0, dtype=torch.bfloat16, device=DEV)
    fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, C=big[:, :200])
    ref = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb)
    torch.cuda.synchronize()
    assert torch.equal(big[:, :200], ref)
    assert torch.all(big[:, 200:] == 5.0)


@pytest.mark.parametrize("b_major", [0, 1])
def test_gemm_pair_tail_rows_untouched(b_major):
    # 3 M-blocks: the CTA-pair kernel runs a second pair whose second CTA has
    # no rows; nothing may be written below row M or right of column N.
    g = generator(8 + b_major, DEV)
    M, N, K = 300, 512 if b_major else 520, 384
    a = normal_bf16((M, K), 1.0, g, DEV)
    w = normal_bf16((N, K) if b_major == 0 else (K, N), 0.02, g, DEV)
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    big = torch.full((M + 12, N + 24), 3.0, dtype=torch.bfloat16, device=DEV)
    fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, b_major=b_major, C=big[:M, :N])
    ref = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, b_major=b_major)
    torch.cuda.synchronize()
    assert torch.equal(big[:M, :N], ref)
    assert torch.all(big[M:] == 3.0) and torch.all(big[:, N:] == 3.0)


@pytest.mark.parametrize("b_major", [0, 1])
def test_gemm_pair_matches_single_cta(b_major):
    # M > 128 runs on CTA pairs, M <= 128 on single CTAs: the same rows must
    # come out bit-identical (same slices, same promotion order).
    g = generator(12 + b_major, DEV)
    M, N, K = 384, 768, 1024
    a = normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.01, outlier_scale=30.0)
    w = normal_bf16((N, K) if b_major == 0 else (K, N), 0.02, g, DEV)
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    for dt in (torch.bfloat16, torch.float32):
        c_pair = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, b_major=b_major, out_dtype=dt)
        for r0 in (0, 128, 256):
            c_one = fp8.fp8_gemm_blockscaled(qa[r0:r0 + 128], sa[:, r0:r0 + 128].contiguous(), qb, sb,
                                             b_major=b_major, out_dtype=dt)
            torch.cuda.synchronize()
            assert torch.equal(c_pair[r0:r0 + 128].view(torch.int16 if dt == torch.bfloat16 else torch.int32),
                               c_one.view(torch.int16 if dt == torch.bfloat16 else torch.int32)), (dt, r0)


def test_gemm_tiny_workload_full():
    c = synthetic.tiny(device=DEV)
    full_check(c.a, c.w, 0, torch.float32, "tiny 128x256x512 fp32")


# ------------------------------------------------------------------ grouped
def grouped_gpu(case, out_dtype=torch.bfloat16):
    E, N, K = case.w.shape
    qa, sa = fp8.fp8_quant_act_1x128(case.x_sorted)
    qb, sb = fp8.fp8_quant_w_128x128(case.w.view(E * N, K))
    c = fp8.fp8_grouped_gemm_blockscaled(qa, sa, qb.view(E, N, K), sb.view(E, -1, K // 128),
                                         case.offsets, out_dtype=out_dtype)
    assert fp8.fp8bs_last_error() == 0
    return c


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_grouped_small_with_empty_and_ragged_segments(out_dtype):
    counts = [0, 130, 5, 0, 256, 1, 300, 0]
    case = synthetic.grouped_case_with_counts("grouped small", counts, 384, 512, seed=3, device=DEV)
    c = grouped_gpu(case, out_dtype)
    E, N, K = case.w.shape
    qa, sa = oracle.quant_act_1x128(bf16_bits(case.x_sorted))
    qbs, sbs = zip(*[oracle.quant_w_128x128(bf16_bits(case.w[e])) for e in range(E)])
    qb, sb = np.stack(qbs), np.stack(sbs)
    off = case.offsets.cpu().numpy()
    ref = oracle.grouped_gemm_f64(qa, sa, qb, sb, off)
    got = host_f64(c)
    an = oracle.act_row_norms(qa, sa)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        bn = oracle.b_row_norms(qb[e], sb[e])
        e_, bad = gemm_errors(got[r0:r1], ref[r0:r1], an[r0:r1], bn)
        assert_gemm_ok(e_, bad, f"expert {e}")


def test_grouped_all_rows_in_one_expert_equals_dense():
    counts = [0, 0, 700, 0]
    case = synthetic.grouped_case_with_counts("one expert", counts, 512, 256, seed=9, device=DEV)
    c = grouped_gpu(case, torch.float32)
    qa, sa = fp8.fp8_quant_act_1x128(case.x_sorted)
    qb, sb = fp8.fp8_quant_w_128x128(case.w[2])
    d = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(c, d)
