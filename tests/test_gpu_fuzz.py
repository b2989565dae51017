"""Seeded random shapes for the GEMMs (every output element against the float64
oracle) and the quantisers (bit-exact against the oracle).

The fixed-shape tests pin particular tile counts, tails and layouts; these
draw M, N, K, the B layout, the output type and (grouped) the segment lengths
at random from a fixed seed, so that shapes nobody chose by hand (odd tails in
M and N, a single row or column, K of one slice, runs of empty experts) pass
the same acceptance rule.  Each case is small enough for the oracle to finish
in well under a second.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import bf16_bits, generator, normal_bf16
from parity import assert_gemm_ok, gemm_errors, host_f64, host_u8, output_rounding_errors

from test_gpu_gemm import full_check, grouped_gpu

pytestmark = pytest.mark.gpu

import fp8_fine_grained_26_b300 as fp8  # noqa: F401  (a missing or broken build fails loudly)
DEV = "cuda"


def _dense_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        b_major = int(rng.integers(0, 2))
        M = int(rng.choice([1, 2, 127, 128, 129]) if rng.random() < 0.25 else rng.integers(1, 900))
        if b_major == 0:
            N = int(rng.choice([1, 17, 255, 256, 257]) if rng.random() < 0.25 else rng.integers(1, 1300))
        else:
            N = 128 * int(rng.integers(1, 10))                  # [K][N] storage: N a multiple of 128
        K = 128 * int(rng.integers(1, 13))
        out = torch.bfloat16 if rng.random() < 0.6 else torch.float32
        cases.append((i, M, N, K, b_major, out))
    return cases


@pytest.mark.parametrize("i,M,N,K,b_major,out_dtype", _dense_cases(20, 20261203))
def test_dense_random_shapes(i, M, N, K, b_major, out_dtype):
    g = generator(1000 + i, DEV)
    a = normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.002, outlier_scale=50.0)
    w = normal_bf16((N, K) if b_major == 0 else (K, N), 0.02, g, DEV)
    full_check(a, w, b_major, out_dtype, f"case {i}: {M}x{N}x{K} b_major={b_major} {out_dtype}")


def _grouped_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        E = int(rng.integers(1, 13))
        counts = [int(c) for c in rng.integers(0, 400, size=E)]
        zero = rng.random(E) < 0.3                              # runs of empty experts
        counts = [0 if z else c for c, z in zip(counts, zero)]
        if sum(counts) == 0:
            counts[-1] = 1
        N = 128 * int(rng.integers(1, 6))
        K = 128 * int(rng.integers(1, 9))
        out = torch.bfloat16 if rng.random() < 0.6 else torch.float32
        cases.append((i, counts, N, K, out))
    return cases


@pytest.mark.parametrize("i,counts,N,K,out_dtype", _grouped_cases(10, 77))
def test_grouped_random_segments(i, counts, N, K, out_dtype):
    case = synthetic.grouped_case_with_counts(f"fuzz {i}", counts, N, K, seed=500 + i, device=DEV)
    c = grouped_gpu(case, out_dtype)
    E = len(counts)
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
        err, bad = gemm_errors(got[r0:r1], ref[r0:r1], an[r0:r1], bn)
        assert_gemm_ok(err, bad, f"case {i} expert {e} ({counts}, N={N}, K={K})",
                       e_out=output_rounding_errors(ref[r0:r1], an[r0:r1], bn, out_dtype))


# ---------------------------------------------------------------- quantisers (bit-exact)
from test_gpu_quant import check_act, check_w          # noqa: E402
from test_gpu_quant_pair import check_pair              # noqa: E402


def _random_bf16(shape, rng, g):
    """N(0, s^2) with s drawn over six decades, some outliers and zeroed runs,
    or Student-t: the value mixes the quantisers see."""
    kind = rng.integers(0, 3)
    if kind == 2:
        x = synthetic.student_t3_bf16(shape, g, DEV)
    else:
        x = normal_bf16(shape, float(10.0 ** rng.uniform(-3, 3)), g, DEV,
                        outlier_p=float(rng.choice([0.0, 0.001, 0.02])), outlier_scale=float(rng.choice([10, 100])))
    if rng.random() < 0.5 and shape[0] > 1:
        r = int(rng.integers(0, shape[0]))
        x[r] = 0                                            # an all-zero row
    return x


def _quant_cases(n, seed):
    rng = np.random.default_rng(seed)
    return [(i, int(rng.integers(1, 1500)), 128 * int(rng.integers(1, 17)), int(rng.integers(1, 1500)),
             128 * int(rng.integers(1, 17))) for i in range(n)]


@pytest.mark.parametrize("i,M,K,R,C", _quant_cases(12, 4242))
def test_quantisers_random_shapes(i, M, K, R, C):
    rng = np.random.default_rng(9000 + i)
    g = generator(9000 + i, DEV)
    x = _random_bf16((M, K), rng, g)
    w = _random_bf16((R, C), rng, g)
    check_act(x, f"case {i} act {M}x{K}")
    check_w(w, f"case {i} weight {R}x{C}")
    check_pair(x, w, f"case {i} pair")


@pytest.mark.parametrize("i", range(6))
def test_token_quantiser_random_shapes(i):
    rng = np.random.default_rng(7000 + i)
    g = generator(7000 + i, DEV)
    T, F = 128 * int(rng.integers(1, 9)), 8 * int(rng.integers(1, 160))   # F: 16-byte BF16 rows
    x = _random_bf16((T, F), rng, g)
    q, s = fp8.fp8_quant_tokens_1x128(x)
    torch.cuda.synchronize()
    assert fp8.fp8bs_last_error() == 0
    oq, os_ = oracle.quant_tokens_1x128(bf16_bits(x))
    assert np.array_equal(host_u8(q), oq), f"case {i} {T}x{F}"
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32)), f"case {i} {T}x{F}"


@pytest.mark.parametrize("i", range(6))
def test_dispatch_quantisers_random_routing(i):
    # gather (a row list with repeats) and scatter (every token to topk
    # distinct rows of a larger buffer) against the oracle's quantiser of the
    # gathered rows
    rng = np.random.default_rng(8000 + i)
    g = generator(8000 + i, DEV)
    T, K, topk = int(rng.integers(1, 400)), 128 * int(rng.integers(1, 40)), int(rng.integers(1, 9))
    x = _random_bf16((T, K), rng, g)
    oq, os_ = oracle.quant_act_1x128(bf16_bits(x))
    rows = torch.from_numpy(rng.integers(0, T, size=int(rng.integers(1, 3 * T + 2))).astype(np.int32)).to(DEV)
    q, s = fp8.fp8_quant_act_1x128_gather(x, rows)
    assert fp8.fp8bs_last_error() == 0
    r = rows.cpu().numpy()
    assert np.array_equal(host_u8(q), oq[r]), f"case {i} gather"
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_[:, r].view(np.uint32)), f"case {i} gather scales"
    M = T * topk + int(rng.integers(0, 7))
    dest = torch.from_numpy(rng.permutation(M)[: T * topk].astype(np.int32).reshape(T, topk)).to(DEV)
    q = torch.full((M, K), 0x5A, dtype=torch.uint8, device=DEV)
    s = torch.full((K // 128, M), -1.25, dtype=torch.float32, device=DEV)
    fp8.fp8_quant_act_1x128_scatter(x, dest, M, q=q, sA=s)
    assert fp8.fp8bs_last_error() == 0
    d = dest.cpu().numpy()
    qh, sh = host_u8(q), s.cpu().numpy()
    written = np.zeros(M, bool)
    for j in range(topk):
        assert np.array_equal(qh[d[:, j]], oq), f"case {i} scatter copy {j}"
        assert np.array_equal(sh[:, d[:, j]].view(np.uint32), os_.view(np.uint32)), f"case {i} scatter scales {j}"
        written[d[:, j]] = True
    assert np.all(qh[~written] == 0x5A) and np.all(sh[:, ~written] == -1.25)     # untouched rows


# ---------------------------------------------------------------- weight gradient and E4M3 output
from test_gpu_wgrad import _check as wgrad_check               # noqa: E402


@pytest.mark.parametrize("i", range(6))
def test_wgrad_random_shapes(i):
    rng = np.random.default_rng(6000 + i)
    T = 128 * int(rng.integers(1, 9))
    M, N = 8 * int(rng.integers(1, 90)), 8 * int(rng.integers(1, 140))     # 16-byte BF16 rows
    wgrad_check(T, M, N, seed=6000 + i, out_dtype=torch.bfloat16 if rng.random() < 0.6 else torch.float32)


@pytest.mark.parametrize("i", range(6))
def test_e4m3_output_random_shapes(i):
    # the fused epilogue is bit-equal to the BF16 GEMM followed by the
    # activation quantiser, whose own parity with the oracle is bit-exact
    rng = np.random.default_rng(5000 + i)
    M, N, K = int(rng.integers(1, 700)), 128 * int(rng.integers(1, 9)), 128 * int(rng.integers(1, 12))
    b_major = int(rng.integers(0, 2))
    g = generator(5000 + i, DEV)
    a = normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.002, outlier_scale=40.0)
    w = normal_bf16((N, K) if b_major == 0 else (K, N), 0.02, g, DEV)
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    qc, sc = fp8.fp8_gemm_blockscaled_e4m3_out(qa, sa, qb, sb, b_major=b_major)
    c = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, b_major=b_major)
    q2, s2 = fp8.fp8_quant_act_1x128(c)
    assert fp8.fp8bs_last_error() == 0
    assert torch.equal(qc, q2), f"case {i} {M}x{N}x{K}: codes differ"
    assert torch.equal(sc.view(torch.int32), s2.view(torch.int32)), f"case {i} {M}x{N}x{K}: scales differ"
    full_check(a, w, b_major, torch.bfloat16, f"case {i} BF16 GEMM under the E4M3 output")
