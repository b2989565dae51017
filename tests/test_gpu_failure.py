"""Failure detection on the GPU without a GPU fault: a device wait that
nothing ends runs out after a short limit, the kernel records the time-out in
the error word and returns, the host reads FP8BS_ERR_TIMEOUT, and the
context keeps working (the next GEMM matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import oracle
from parity import assert_gemm_ok, gemm_errors, host_f64, host_u8
from synthetic import bf16_bits, generator, normal_bf16

pytestmark = pytest.mark.gpu
import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
DEV = "cuda"


def test_wait_timeout_is_reported_and_cleared():
    assert fp8.fp8bs_last_error() == fp8.FP8BS_OK
    t0 = time.perf_counter()
    fp8.fp8bs_selftest_wait_timeout(20000)            # 20 ms
    st = fp8.fp8bs_last_error()
    dt = time.perf_counter() - t0
    assert st == fp8.FP8BS_ERR_TIMEOUT
    assert 0.015 < dt < 5.0, dt                       # the wait really ran to its limit
    assert fp8.fp8bs_last_error() == fp8.FP8BS_OK     # reading clears it


def test_context_usable_after_timeout():
    fp8.fp8bs_selftest_wait_timeout(5000)
    assert fp8.fp8bs_last_error() == fp8.FP8BS_ERR_TIMEOUT
    g = generator(21, DEV)
    a = normal_bf16((256, 384), 1.0, g, DEV)
    w = normal_bf16((320, 384), 0.02, g, DEV)
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    c = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32)
    assert fp8.fp8bs_last_error() == fp8.FP8BS_OK
    oqa, osa = oracle.quant_act_1x128(bf16_bits(a))
    oqb, osb = oracle.quant_w_128x128(bf16_bits(w))
    assert np.array_equal(host_u8(qa), oqa) and np.array_equal(host_u8(qb), oqb)
    ref = oracle.gemm_f64(oqa, osa, oqb, osb, b_major=0)
    e, bad = gemm_errors(host_f64(c), ref, oracle.act_row_norms(oqa, osa), oracle.b_row_norms(oqb, osb))
    assert_gemm_ok(e, bad, "GEMM after a time-out")


def test_timeout_on_a_side_stream_is_seen_on_that_stream():
    s = torch.cuda.Stream()
    fp8.fp8bs_selftest_wait_timeout(2000, stream=s)
    assert fp8.fp8bs_last_error(stream=s) == fp8.FP8BS_ERR_TIMEOUT


def test_timeout_and_index_errors_are_reported_one_per_call():
    """Both conditions set: the time-out is reported first, then the index
    error, then nothing; each call clears only the bit it reports."""
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device=DEV)
    rows = torch.tensor([0, 9, 1], dtype=torch.int32, device=DEV)       # 9 is out of range
    fp8.fp8_quant_act_1x128_gather(x, rows)
    fp8.fp8bs_selftest_wait_timeout(2000)
    assert fp8.fp8bs_last_error() == fp8.FP8BS_ERR_TIMEOUT
    assert fp8.fp8bs_last_error() == fp8.FP8BS_ERR_INDEX
    assert fp8.fp8bs_last_error() == fp8.FP8BS_OK


# ---------------------------------------------------------------- abort paths
# With a wait limit of a few microseconds, a real kernel's wait that has to
# wait for memory or for the tensor core runs out: the kernel must record the
# time-out, drain its own copies and MMAs, free its tensor memory and return,
# writing nothing outside its outputs; the next call (default limit) must be
# correct.  Only single-CTA kernels take the short limit (CTA-pair GEMMs keep
# the default), so these are the paths exercised here.
SHORT_NS = 1000


def _with_short_limit(fn, attempts=5):
    """Runs fn() with the short wait limit until a call reports a time-out;
    returns the list of statuses.  The default limit is always restored."""
    seen = []
    try:
        fp8.fp8bs_selftest_set_wait_limit(SHORT_NS)
        for _ in range(attempts):
            fn()
            seen.append(fp8.fp8bs_last_error())
            if seen[-1] == fp8.FP8BS_ERR_TIMEOUT:
                break
    finally:
        fp8.fp8bs_selftest_set_wait_limit(0)
    assert all(s in (fp8.FP8BS_OK, fp8.FP8BS_ERR_TIMEOUT) for s in seen), seen
    return seen


def test_single_cta_gemm_abort_path():
    # one 128 x 256 tile over K = 65536 (512 slices): the store issuer waits
    # for the whole K loop and the promote warps wait on every slice
    g = generator(71, DEV)
    M, N, K = 100, 256, 65536
    a = normal_bf16((M, K), 1.0, g, DEV)
    w = normal_bf16((N, K), 0.02, g, DEV)
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    big = torch.full((M + 8, N + 64), 7.0, dtype=torch.bfloat16, device=DEV)
    seen = _with_short_limit(lambda: fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, C=big[:M, :N]))
    assert fp8.FP8BS_ERR_TIMEOUT in seen, seen
    assert torch.all(big[M:] == 7.0) and torch.all(big[:, N:] == 7.0), "written outside C"
    c = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32)
    assert fp8.fp8bs_last_error() == fp8.FP8BS_OK
    oqa, osa = oracle.quant_act_1x128(bf16_bits(a))
    oqb, osb = oracle.quant_w_128x128(bf16_bits(w))
    assert np.array_equal(host_u8(qa), oqa) and np.array_equal(host_u8(qb), oqb)
    ref = oracle.gemm_f64(oqa, osa, oqb, osb)
    e, bad = gemm_errors(host_f64(c), ref, oracle.act_row_norms(oqa, osa), oracle.b_row_norms(oqb, osb))
    assert_gemm_ok(e, bad, "GEMM after an aborted GEMM")


def test_grouped_gemm_abort_path():
    import synthetic
    counts = [300, 0, 17, 129]
    case = synthetic.grouped_case_with_counts("abort", counts, 512, 16384, seed=3, device=DEV)
    E, N, K = case.w.shape
    qa, sa = fp8.fp8_quant_act_1x128(case.x_sorted)
    qb, sb = fp8.fp8_quant_w_128x128(case.w.view(E * N, K))
    qb, sb = qb.view(E, N, K), sb.view(E, -1, K // 128)
    M = case.x_sorted.shape[0]
    big = torch.full((M + 8, N + 64), 5.0, dtype=torch.bfloat16, device=DEV)
    seen = _with_short_limit(lambda: fp8.fp8_grouped_gemm_blockscaled(qa, sa, qb, sb, case.offsets,
                                                                      C=big[:M, :N]))
    assert torch.all(big[M:] == 5.0) and torch.all(big[:, N:] == 5.0), "written outside C"
    ref_after = fp8.fp8_grouped_gemm_blockscaled(qa, sa, qb, sb, case.offsets)
    again = fp8.fp8_grouped_gemm_blockscaled(qa, sa, qb, sb, case.offsets)
    assert fp8.fp8bs_last_error() == fp8.FP8BS_OK
    assert torch.equal(ref_after, again)                # the context and the kernel are intact
    print("grouped abort statuses", seen)


def test_quantiser_abort_path():
    g = generator(73, DEV)
    M, K = 8192, 8192                                   # 128 MB of BF16: many units per CTA
    x = normal_bf16((M, K), 1.0, g, DEV)
    q = torch.full((M + 4, K), 0x5A, dtype=torch.uint8, device=DEV)
    s = torch.full((K // 128 + 1, M), -1.0, dtype=torch.float32, device=DEV)
    seen = _with_short_limit(lambda: fp8.fp8_quant_act_1x128(x, q[:M], s[:K // 128]))
    assert torch.all(q[M:] == 0x5A) and torch.all(s[K // 128:] == -1.0), "written outside the outputs"
    q2, s2 = fp8.fp8_quant_act_1x128(x)
    assert fp8.fp8bs_last_error() == fp8.FP8BS_OK
    oq, os_ = oracle.quant_act_1x128(bf16_bits(x[:256]))
    assert np.array_equal(host_u8(q2[:256]), oq)
    assert np.array_equal(s2[:, :256].cpu().numpy().view(np.uint32), os_.view(np.uint32))
    print("quantiser abort statuses", seen)


def test_pair_gemm_keeps_the_default_limit():
    """While a short limit is set, a CTA-pair GEMM (M > 128) still runs with
    the default one and completes normally."""
    g = generator(79, DEV)
    a = normal_bf16((512, 4096), 1.0, g, DEV)
    w = normal_bf16((1024, 4096), 0.02, g, DEV)
    qa, sa = fp8.fp8_quant_act_1x128(a)
    qb, sb = fp8.fp8_quant_w_128x128(w)
    ref = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb)
    try:
        fp8.fp8bs_selftest_set_wait_limit(SHORT_NS)
        c = fp8.fp8_gemm_blockscaled(qa, sa, qb, sb)
        st = fp8.fp8bs_last_error()
    finally:
        fp8.fp8bs_selftest_set_wait_limit(0)
    assert st == fp8.FP8BS_OK and torch.equal(c, ref)
