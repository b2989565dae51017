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
fp8 = pytest.importorskip("fp8_fine_grained_26_b300")
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
