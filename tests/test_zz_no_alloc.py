"""The allocation-free per-tensor quantiser, called through the C ABI.

fp8_quant_per_tensor_noalloc serves callers that cannot allocate device
memory around a call (a host application that owns every device buffer and
grants none for scratch, a serving loop that allows no allocation after
start-up): it keeps its scratch in a fixed array inside the library instead
of taking a workspace.  Its result must equal the workspace call's, bit for
bit, on consecutive calls that share that array -- the second call on a
smaller tensor than the first, so stale words from the first call are still
in the array when it runs -- and a tensor too large for the array must be
refused before anything is enqueued.

This file is collected after every other test file, and passes both alone in
a fresh process (where it makes the library's first call on the device, the
one that looks up the array's address) and after the rest of the suite.
"""
import ctypes

import pytest
import torch

import synthetic
from synthetic import generator, normal_bf16

pytestmark = pytest.mark.gpu
import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
DEV = "cuda"


def _noalloc(x, q, scale, stream):
    """The C entry point, called directly with ctypes (no binding logic)."""
    R, C = x.shape
    return fp8.lib.fp8_quant_per_tensor_noalloc(
        ctypes.c_void_p(x.data_ptr()), R, C, x.stride(0), ctypes.c_void_p(q.data_ptr()), q.stride(0),
        ctypes.c_void_p(scale.data_ptr()), ctypes.c_void_p(stream.cuda_stream))


def test_noalloc_equals_workspace_call_on_two_calls_in_a_row():
    stream = torch.cuda.current_stream()
    g = generator(2024, DEV)
    inputs = [normal_bf16((3000, 2048), 1.0, g, DEV, outlier_p=0.001, outlier_scale=50.0),   # 24 x 16 units
              synthetic.student_t3_bf16((300, 640), g, DEV)]                                   # 3 x 5 units
    for i, x in enumerate(inputs):
        R, C = x.shape
        q = torch.empty((R, C), dtype=torch.uint8, device=DEV)
        s = torch.empty((1,), dtype=torch.float32, device=DEV)
        assert _noalloc(x, q, s, stream) == fp8.FP8BS_OK, f"call {i}"
        assert fp8.fp8bs_last_error(stream) == fp8.FP8BS_OK
        q_ref, s_ref = fp8.fp8_quant_per_tensor(x)          # the workspace entry point
        torch.cuda.synchronize()
        assert torch.equal(q, q_ref), f"call {i}: codes differ"
        assert s.view(torch.int32).item() == s_ref.view(torch.int32).item(), f"call {i}: scales differ"


def test_noalloc_refuses_a_tensor_too_large_for_its_scratch():
    stream = torch.cuda.current_stream()
    x = torch.zeros((128, 256), dtype=torch.bfloat16, device=DEV)
    q = torch.zeros((128, 256), dtype=torch.uint8, device=DEV)
    s = torch.full((1,), 7.0, dtype=torch.float32, device=DEV)
    units_max = 16384                                       # FP8BS_NOALLOC_MAX_UNITS
    R, C = 128 * (units_max // 2 + 1), 256                  # one 128x128 unit over the limit
    rc = fp8.lib.fp8_quant_per_tensor_noalloc(
        ctypes.c_void_p(x.data_ptr()), R, C, C, ctypes.c_void_p(q.data_ptr()), C, ctypes.c_void_p(s.data_ptr()),
        ctypes.c_void_p(stream.cuda_stream))
    assert rc == fp8.FP8BS_ERR_SCRATCH
    torch.cuda.synchronize()
    assert s.item() == 7.0 and int(torch.count_nonzero(q)) == 0      # nothing was enqueued
    # exactly at the limit is accepted (shape check only: 128 x 2^21 elements would be 512 MB)
    R_ok = 128 * (units_max // 2)
    xb = torch.empty((R_ok, C), dtype=torch.bfloat16, device=DEV).normal_()
    qb = torch.empty((R_ok, C), dtype=torch.uint8, device=DEV)
    assert _noalloc(xb, qb, s, stream) == fp8.FP8BS_OK
    q_ref, s_ref = fp8.fp8_quant_per_tensor(xb)
    torch.cuda.synchronize()
    assert torch.equal(qb, q_ref) and s.view(torch.int32).item() == s_ref.view(torch.int32).item()
    assert fp8.fp8bs_last_error(stream) == fp8.FP8BS_OK
