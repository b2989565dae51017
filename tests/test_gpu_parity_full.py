"""Element-by-element GPU parity on the persistent multi-tile paths and at the
workloads' full sizes.

Every output element of every case below is compared with the float64 CPU
oracle under the acceptance rule of ``parity.py`` (max normalised error
<= 2e-3, mean <= 1e-4, zero-norm outputs exactly 0).  The multi-tile cases
are sized so that every persistent CTA (or CTA pair) of the kernel runs at
least three output tiles, which exercises what a one-wave shape cannot: the
TMEM buffer parity and the scale-ring slots carried from tile to tile, the
reuse of the epilogue staging boxes, the rasterisation groups of the pair
schedule (including a ragged last group), and long grouped schedules with
empty and ragged expert segments.  The full-size cases compare the whole
output of the MLA-q and MLA-kv GEMMs, full-width row slabs from the first and
last rasterisation groups of the data-gradient GEMM, every row of a set of
experts of the routed-expert GEMM, and a full-width slab of the
weight-gradient GEMM.

As everywhere, the GPU side quantises the BF16 inputs itself and the oracle
quantises the same BF16 inputs itself; no oracle input comes from the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity import (ErrorStats, assert_e4m3_out_within_bound, compare_by_slabs, host_u8, record_stats,
                    slabs)
from synthetic import bf16_bits, generator, normal_bf16

pytestmark = pytest.mark.gpu
import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
DEV = "cuda"
BM, BN = 128, 256


def num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def cdiv(a, b):
    return -(-a // b)


def quantise_both(a, w):
    """GPU quantisation of both operands and the oracle's own quantisation of
    the same BF16 inputs; the codes and scales must agree bit for bit."""
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    oqa, osa = oracle.quant_act_1x128(bf16_bits(a))
    oqb, osb = oracle.quant_w_128x128(bf16_bits(w))
    assert np.array_equal(host_u8(qa), oqa) and np.array_equal(host_u8(qb), oqb), "codes differ"
    assert np.array_equal(sa.cpu().numpy().view(np.uint32), osa.view(np.uint32)), "activation scales differ"
    assert np.array_equal(sb.cpu().numpy().view(np.uint32), osb.view(np.uint32)), "weight scales differ"
    return (qa, sa, qb, sb), (oqa, osa, oqb, osb)


def k_major_view(oqb, osb, b_major):
    """The oracle's B operand in the K-major layout: a stored [K][N] weight
    (MN-major) is the transpose of the [N][K] one, with its scale grid
    transposed (a relabelling of the same elements; the oracle's own pins show
    the two layouts give identical results)."""
    if b_major == 0:
        return oqb, osb
    return np.ascontiguousarray(oqb.T), np.ascontiguousarray(osb.T)


def dense_full_compare(what, a, w, b_major, out_dtype, row_ranges=None, slab_rows=512):
    (qa, sa, qb, sb), (oqa, osa, oqb, osb) = quantise_both(a, w)
    c = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, b_major=b_major, out_dtype=out_dtype)
    assert fp8.fp8bs_last_error() == 0
    M, N = c.shape
    kqb, ksb = k_major_view(oqb, osb, b_major)
    an = oracle.act_row_norms(oqa, osa)
    bn = oracle.b_row_norms(kqb, ksb)

    def ref_rows(r0, r1):
        return oracle.gemm_f64(oqa[r0:r1], np.ascontiguousarray(osa[:, r0:r1]), kqb, ksb)

    ranges = row_ranges if row_ranges is not None else slabs(0, M, slab_rows)
    return compare_by_slabs(what, c, ref_rows, an, bn, [s for r in ranges for s in slabs(*r, slab_rows)])


# ------------------------------------------------------------ multi-tile shapes
@pytest.mark.parametrize("M,N,K,out_dtype", [
    (1000, 15000, 512, torch.bfloat16),      # 4 M-pairs x 59 N-blocks, ragged in M and N
    (4252, 3400, 256, torch.bfloat16),       # 17 M-pairs: two rasterisation groups, the last ragged
    (1000, 15000, 384, torch.float32),       # FP32 output (direct stores) across many tiles
])
def test_pair_kmajor_every_cta_runs_several_tiles(M, N, K, out_dtype):
    tiles = cdiv(cdiv(M, BM), 2) * cdiv(N, BN)
    assert tiles >= 3 * (num_sms() // 2), "shape must give every CTA pair 3+ tiles"
    g = generator(M + N + K, DEV)
    a = normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.002, outlier_scale=50.0)
    w = normal_bf16((N, K), 0.02, g, DEV)
    dense_full_compare(f"pair K-major {M}x{N}x{K} {out_dtype}", a, w, 0, out_dtype)


@pytest.mark.parametrize("M,N,K", [(1000, 15232, 384), (4352, 3456, 256)])
def test_pair_mnmajor_every_cta_runs_several_tiles(M, N, K):
    tiles = cdiv(cdiv(M, BM), 2) * cdiv(N, BN)
    assert tiles >= 3 * (num_sms() // 2)
    g = generator(M * 3 + N + K, DEV)
    a = synthetic.student_t3_bf16((M, K), g, DEV)
    w = normal_bf16((K, N), 0.02, g, DEV)                       # stored [K][N]
    dense_full_compare(f"pair MN-major {M}x{N}x{K}", a, w, 1, torch.bfloat16)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_single_cta_every_cta_runs_several_tiles(out_dtype):
    M, N, K = 100, 114000, 256                                  # M <= 128: single-CTA kernel
    assert cdiv(N, BN) >= 3 * num_sms()
    g = generator(5 + (out_dtype == torch.float32), DEV)
    a = normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.01, outlier_scale=30.0)
    w = normal_bf16((N, K), 0.02, g, DEV)
    dense_full_compare(f"single-CTA {M}x{N}x{K} {out_dtype}", a, w, 0, out_dtype)


def test_single_cta_mnmajor_every_cta_runs_several_tiles():
    M, N, K = 128, 113920, 256
    assert cdiv(N, BN) >= 3 * num_sms()
    g = generator(8, DEV)
    a = normal_bf16((M, K), 1.0, g, DEV)
    w = normal_bf16((K, N), 0.02, g, DEV)
    dense_full_compare(f"single-CTA MN-major {M}x{N}x{K}", a, w, 1, torch.bfloat16)


def grouped_compare(what, case, out_dtype=torch.bfloat16, experts=None):
    """Grouped GEMM of `case` on the GPU; every row of the chosen experts (all
    by default) against the oracle's grouped GEMM.  The oracle quantises each
    expert's weight from its BF16 input."""
    E, N, K = case.w.shape
    qa, sa = fp8.fp8_quant_act_1x128(case.x_sorted)
    qb, sb = fp8.fp8_quant_w_128x128(case.w.view(E * N, K))
    c = fp8.fp8_grouped_gemm_blockscaled(qa, sa, qb.view(E, N, K), sb.view(E, -1, K // 128), case.offsets,
                                         out_dtype=out_dtype)
    assert fp8.fp8bs_last_error() == 0
    off = case.offsets.cpu().numpy().astype(np.int64)
    oqa, osa = oracle.quant_act_1x128(bf16_bits(case.x_sorted))
    assert np.array_equal(host_u8(qa), oqa)
    an = oracle.act_row_norms(oqa, osa)
    st = ErrorStats(what)
    for e in (range(E) if experts is None else experts):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        oqb, osb = oracle.quant_w_128x128(bf16_bits(case.w[e]))
        assert np.array_equal(host_u8(qb.view(E, N, K)[e]), oqb)
        bn = oracle.b_row_norms(oqb, osb)
        ref = oracle.gemm_f64(oqa[r0:r1], np.ascontiguousarray(osa[:, r0:r1]), oqb, osb)
        st.add(c[r0:r1].double().cpu().numpy(), ref, an[r0:r1], bn)
    st.check()
    return c


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_grouped_hundreds_of_tiles_with_empty_and_ragged_segments(out_dtype):
    rng = np.random.default_rng(31)
    counts = rng.integers(0, 400, size=48)
    counts[[0, 5, 17, 47]] = 0                                   # empty experts, first and last included
    counts[[3, 9]] = [1, 129]                                    # a one-row and a just-over-one-block segment
    N, K = 2304, 384
    tiles = int(sum(cdiv(int(c), BM) for c in counts)) * cdiv(N, BN)
    assert tiles >= 3 * num_sms()
    case = synthetic.grouped_case_with_counts("grouped multi-tile", counts, N, K, seed=7, device=DEV)
    grouped_compare(f"grouped {len(counts)} experts, {tiles} tiles, {out_dtype}", case, out_dtype)


def test_grouped_max_experts_accepted():
    """E = FP8BS_MAX_EXPERTS (2048) experts, most of them empty: accepted, and
    the routed rows match the oracle (first and last expert included)."""
    E, N, K = 2048, 256, 128
    counts = np.zeros(E, np.int64)
    counts[[0, 1, 700, 1500, 2047]] = [130, 3, 256, 77, 200]
    case = synthetic.grouped_case_with_counts("2048 experts", counts, N, K, seed=13, device=DEV)
    grouped_compare("grouped E=2048", case, torch.float32, experts=[0, 1, 700, 1500, 2047])


def test_wgrad_every_cta_runs_several_tiles():
    T, M, N = 512, 1000, 14336
    tiles = cdiv(cdiv(M, BM), 2) * cdiv(N, BN)
    assert tiles >= 3 * (num_sms() // 2)
    case = synthetic.wgrad_case("wgrad multi-tile", T, M, N, seed=19, device=DEV)
    qa, sa = fp8.fp8_quant_tokens_1x128(case.dy)
    qb, sb = fp8.fp8_quant_tokens_1x128(case.x)
    c = fp8.fp8_gemm_wgrad(qa, sa, qb, sb)
    assert fp8.fp8bs_last_error() == 0
    oqa, osa = oracle.quant_tokens_1x128(bf16_bits(case.dy))
    oqb, osb = oracle.quant_tokens_1x128(bf16_bits(case.x))
    assert np.array_equal(host_u8(qa), oqa) and np.array_equal(host_u8(qb), oqb)
    an, bn = oracle.act_row_norms(oqa, osa), oracle.act_row_norms(oqb, osb)
    compare_by_slabs(f"wgrad {M}x{N} over {T} tokens", c,
                     lambda r0, r1: oracle.gemm_f64_tokens(oqa[r0:r1], np.ascontiguousarray(osa[:, r0:r1]),
                                                           oqb, osb),
                     an, bn, slabs(0, M, 256))


@pytest.mark.parametrize("b_major", [0, 1])
def test_e4m3_out_against_oracle_every_cta_runs_several_tiles(b_major):
    M, N, K = 1000, 15104, 384
    tiles = cdiv(cdiv(M, BM), 2) * cdiv(N, BN)
    assert tiles >= 3 * (num_sms() // 2)
    g = generator(61 + b_major, DEV)
    a = normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.002, outlier_scale=40.0)
    a[17] = 0
    w = normal_bf16((N, K) if b_major == 0 else (K, N), 0.02, g, DEV)
    (qa, sa, qb, sb), (oqa, osa, oqb, osb) = quantise_both(a, w)
    qc, sc = fp8.fp8_gemm_blockscaled_e4m3_out(qa, sa, qb, sb, b_major=b_major)
    assert fp8.fp8bs_last_error() == 0
    kqb, ksb = k_major_view(oqb, osb, b_major)
    ref = oracle.gemm_f64(oqa, osa, kqb, ksb)
    ratio = assert_e4m3_out_within_bound(host_u8(qc), sc.cpu().numpy(), ref, oracle.act_row_norms(oqa, osa),
                                         oracle.b_row_norms(kqb, ksb), oracle.e4m3_decode_table())
    record_stats(f"e4m3-out {M}x{N}x{K} b_major={b_major} (error / derived bound)", ratio, float("nan"), M * N)
    assert torch.all(qc[17] == 0) and torch.all(sc[:, 17] == 0)


# ------------------------------------------------------------ full sizes
def test_mla_q_full_output():
    case = synthetic.mla_q(device=DEV)
    dense_full_compare("mla_q 4096x24576x1536, every output", case.a, case.w, 0, torch.bfloat16)


def test_mla_kv_full_output():
    case = synthetic.mla_kv(device=DEV)
    dense_full_compare("mla_kv 8192x32768x512, every output", case.a, case.w, 0, torch.bfloat16)


def test_dgrad_full_width_slabs():
    """Rows [0, 512) (first rasterisation group) and [7680, 8192) (last), all
    18432 columns."""
    case = synthetic.dgrad(device=DEV)
    dense_full_compare("dgrad 8192x18432x7168, rows 0-511 and 7680-8191", case.a, case.w, 1, torch.bfloat16,
                       row_ranges=[(0, 512), (7680, 8192)])


def test_experts_full_rows_of_many_experts():
    """Every row and column of 24 of the 256 experts: the largest and smallest
    segments, the first and last expert and 20 more chosen at random."""
    case = synthetic.experts(device=DEV, keep_x=True)
    counts = np.diff(case.offsets.cpu().numpy())
    assert counts.sum() == 4096 * 8
    rng = np.random.default_rng(0)
    picks = {int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 10 ** 9))), 0, 255}
    while len(picks) < 24:
        picks.add(int(rng.integers(0, 256)))
    grouped_compare("experts 256x(2048x7168), every row of 24 experts", case, experts=sorted(picks))


def test_wgrad_full_width_slab():
    case = synthetic.wgrad(device=DEV)
    qa, sa = fp8.fp8_quant_tokens_1x128(case.dy)
    qb, sb = fp8.fp8_quant_tokens_1x128(case.x)
    c = fp8.fp8_gemm_wgrad(qa, sa, qb, sb)
    assert fp8.fp8bs_last_error() == 0
    rows = (6912, 7168)                                         # the last 256 output rows, full width
    oqa, osa = oracle.quant_tokens_1x128(bf16_bits(case.dy[:, rows[0]:rows[1]]))
    oqb, osb = oracle.quant_tokens_1x128(bf16_bits(case.x))
    assert np.array_equal(host_u8(qa)[rows[0]:rows[1]], oqa) and np.array_equal(host_u8(qb), oqb)
    an, bn = oracle.act_row_norms(oqa, osa), oracle.act_row_norms(oqb, osb)
    st = ErrorStats("wgrad 7168x18432 over 8192 tokens, rows 6912-7167")
    for r0, r1 in slabs(0, rows[1] - rows[0], 64):
        ref = oracle.gemm_f64_tokens(oqa[r0:r1], np.ascontiguousarray(osa[:, r0:r1]), oqb, osb)
        st.add(c[rows[0] + r0:rows[0] + r1].double().cpu().numpy(), ref, an[r0:r1], bn)
    st.check()
