"""Seeded random shapes for the dense and grouped GEMMs, every output element
compared with the float64 oracle.

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
from parity import assert_gemm_ok, gemm_errors, host_f64, output_rounding_errors

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
