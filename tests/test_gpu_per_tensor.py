"""GPU parity of the per-tensor FP8 contrast variant, and the accuracy
comparison the fine-grained scheme exists for.

* Quantisers (current and delayed scaling): codes and scale bit-exact
  against the oracle, recorded amax exact.
* GEMM over per-tensor operands: against the oracle's float64 GEMM of the
  same quantised operands, under the normalised-error rule of ``parity.py``.
  This GEMM accumulates the whole K on the tensor cores (no promotion), so
  its FP32-output error is the tensor cores' own accumulation error.
* Accuracy: on the MLA-q activations (0.1% outliers x50) and the dgrad
  operands (Student-t, nu = 3), both schemes' outputs against the float64
  product of the UNQUANTISED BF16 inputs, normalised by the BF16 row norms.
  The pages motivate the 1x128 / 128x128 groups by exactly this comparison
  ("qqstock.cn walkthrough", FP8 section: fine-grained rather than
  per-tensor quantisation, report figure 7a; "DeepSeek-V3 Technical Report
  digest", section 3, fine-grained quantisation bullet).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import ErrorStats, host_u8, record_stats
from synthetic import bf16_bits, generator, normal_bf16

pytestmark = pytest.mark.gpu
import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
DEV = "cuda"


def _scale_bits(t):
    return t.cpu().numpy().view(np.uint32)[0]


@pytest.mark.parametrize("R,C", [(1, 128), (300, 384), (128, 128), (129, 256), (4096, 1536), (24576, 1536)])
def test_per_tensor_quantiser_bit_exact(R, C):
    g = generator(R + C, DEV)
    x = normal_bf16((R, C), 1.0, g, DEV, outlier_p=0.001, outlier_scale=50.0)
    q, s = fp8.fp8_quant_per_tensor(x)
    assert fp8.fp8bs_last_error() == 0
    oq, os_ = oracle.quant_per_tensor(bf16_bits(x))
    assert _scale_bits(s) == np.float32(os_).view(np.uint32)
    assert np.array_equal(host_u8(q), oq)


def test_per_tensor_quantiser_zero_tensor_strided_rows_and_workspace_rules():
    x = torch.zeros((200, 512), dtype=torch.bfloat16, device=DEV)
    x[3, 7] = -0.0
    q, s = fp8.fp8_quant_per_tensor(x)
    torch.cuda.synchronize()
    assert s.item() == 0.0 and q[3, 7].item() == 0x80 and int(torch.count_nonzero(q)) == 1
    # strided input and output rows, a workspace reused across calls
    g = generator(5, DEV)
    big = synthetic.student_t3_bf16((130, 640), g, DEV)
    qbig = torch.full((130, 528), 0x33, dtype=torch.uint8, device=DEV)
    ws = torch.full((fp8.fp8_quant_per_tensor_workspace_size(130, 512),), 0xFF, dtype=torch.uint8, device=DEV)
    for _ in range(2):
        q2, s2 = fp8.fp8_quant_per_tensor(big[:, :512], q=qbig[:, :512], workspace=ws)
        torch.cuda.synchronize()
        oq, os_ = oracle.quant_per_tensor(bf16_bits(big[:, :512]))
        assert np.array_equal(host_u8(qbig[:, :512]), oq) and _scale_bits(s2) == np.float32(os_).view(np.uint32)
        assert torch.all(qbig[:, 512:] == 0x33)
    with pytest.raises(fp8.Fp8bsError):
        fp8.fp8_quant_per_tensor(big[:, :512], workspace=ws[:-4])


@pytest.mark.parametrize("factor", [1.0, 0.25, 8.0, 1.37, 0.0])
def test_delayed_scaling_bit_exact(factor):
    """amax_in = factor x the tensor's amax: 1 equals current scaling, 0.25
    saturates the largest values, 8 leaves headroom, 1.37 is not a BF16 value
    (the IEEE-division path), 0 is a zero scale (codes of x itself)."""
    g = generator(int(factor * 100) + 7, DEV)
    x = synthetic.student_t3_bf16((640, 768), g, DEV)
    amax = float(torch.max(torch.abs(x.float())))
    amax_in = torch.tensor([np.float32(amax * factor)], dtype=torch.float32, device=DEV)
    q, s, amax_out = fp8.fp8_quant_per_tensor_delayed(x, amax_in)
    assert fp8.fp8bs_last_error() == 0
    oq, os_, oa = oracle.quant_per_tensor_delayed(bf16_bits(x), np.float32(amax * factor))
    assert _scale_bits(s) == np.float32(os_).view(np.uint32)
    assert np.array_equal(host_u8(q), oq)
    assert _scale_bits(amax_out) == np.float32(oa).view(np.uint32) == np.float32(amax).view(np.uint32)
    if factor == 0.25:
        assert int(torch.count_nonzero((q & 0x7F) == 0x7E)) > 0


def _pt_gemm_check(M, N, K, b_major, out_dtype, seed, heavy=False):
    g = generator(seed, DEV)
    a = (synthetic.student_t3_bf16((M, K), g, DEV) if heavy
         else normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.001, outlier_scale=50.0))
    w = normal_bf16((N, K) if b_major == 0 else (K, N), 0.02, g, DEV)
    qa, sa = fp8.fp8_quant_per_tensor(a)
    qb, sb = fp8.fp8_quant_per_tensor(w)
    c = fp8.fp8_gemm_per_tensor(qa, sa, qb, sb, b_major=b_major, out_dtype=out_dtype)
    assert fp8.fp8bs_last_error() == 0
    oqa, osa = oracle.quant_per_tensor(bf16_bits(a))
    oqb, osb = oracle.quant_per_tensor(bf16_bits(w))
    assert np.array_equal(host_u8(qa), oqa) and np.array_equal(host_u8(qb), oqb)
    if b_major == 1:
        oqb = np.ascontiguousarray(oqb.T)                   # the same elements, K-major
    ref = oracle.gemm_f64_per_tensor(oqa, osa, oqb, osb)
    # normalised by the dequantised row norms (per-tensor scales: norm * scale)
    an = np.sqrt(np.sum(oracle.e4m3_decode_table()[oqa] ** 2, axis=1)) * float(osa)
    bn = np.sqrt(np.sum(oracle.e4m3_decode_table()[oqb] ** 2, axis=1)) * float(osb)
    st = ErrorStats(f"per-tensor GEMM {M}x{N}x{K} b_major={b_major} {out_dtype}")
    st.add(c.double().cpu().numpy(), ref, an, bn)
    return st


@pytest.mark.parametrize("M,N,K,b_major", [(128, 256, 512, 0), (300, 520, 640, 0), (1000, 15000, 512, 0),
                                           (100, 3000, 1024, 0), (333, 640, 896, 1), (1000, 15232, 384, 1)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_per_tensor_gemm_matches_oracle(M, N, K, b_major, out_dtype):
    _pt_gemm_check(M, N, K, b_major, out_dtype, seed=M + N + K).check()


def test_per_tensor_gemm_long_k_accumulation():
    """K = 7168 (the dgrad contraction) accumulated entirely on the tensor
    cores, FP32 output: the recorded error is the tensor cores' own
    accumulation error over 7168 products."""
    st = _pt_gemm_check(512, 2048, 7168, 0, torch.float32, seed=99, heavy=True)
    st.check()


def _fine_grained(a, w, b_major):
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    return fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, b_major=b_major, out_dtype=torch.float32)


def _per_tensor(a, w, b_major):
    qa, sa = fp8.fp8_quant_per_tensor(a)
    qb, sb = fp8.fp8_quant_per_tensor(w)
    return fp8.fp8_gemm_per_tensor(qa, sa, qb, sb, b_major=b_major, out_dtype=torch.float32)


@pytest.mark.parametrize("workload", ["mla_q", "dgrad"])
def test_fine_grained_is_more_accurate_than_per_tensor(workload):
    """Both schemes, FP32 outputs, on the full operands of the workload (the
    quantisers see the whole tensors), compared on 256 rows x every column
    with the float64 product of the unquantised BF16 inputs."""
    case = getattr(synthetic, workload)(device=DEV)
    fg = _fine_grained(case.a, case.w, case.b_major)
    pt = _per_tensor(case.a, case.w, case.b_major)
    assert fp8.fp8bs_last_error() == 0
    rows = np.r_[0:128, case.M - 128:case.M]
    a_bits = bf16_bits(case.a[torch.from_numpy(rows).to(DEV)])
    w_bits = bf16_bits(case.w)
    if case.b_major == 1:
        w_bits = np.ascontiguousarray(w_bits.T)             # [N][K]: the same elements, K contiguous
    exact = oracle.gemm_bf16_f64(a_bits, w_bits, b_major=0)
    af = (a_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wf = (w_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    an = np.sqrt(np.sum(af ** 2, axis=1))
    bn = np.sqrt(np.sum(wf ** 2, axis=1))
    res = {}
    for name, c in (("fine-grained 1x128/128x128", fg), ("per-tensor", pt)):
        st = ErrorStats(f"{workload}: {name} vs unquantised BF16 product")
        st.add(c[torch.from_numpy(rows).to(DEV)].double().cpu().numpy(), exact, an, bn)
        record_stats(st.what, st.max, st.mean, st.n)
        res[name] = st
    fgs, pts = res["fine-grained 1x128/128x128"], res["per-tensor"]
    assert fgs.mean < pts.mean, (fgs.mean, pts.mean)
