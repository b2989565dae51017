"""C-ABI boundary checks that need no GPU: the library loads, exports every
entry point the public header declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*int\s+(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted([
        "fp8_quant_act_1x128", "fp8_quant_w_128x128", "fp8_quant_act_w", "fp8_gemm_blockscaled",
        "fp8_gemm_blockscaled_e4m3_out", "fp8_quant_tokens_1x128", "fp8_gemm_wgrad",
        "fp8_quant_act_1x128_gather", "fp8_grouped_gemm_blockscaled", "fp8bs_last_error",
        "fp8bs_selftest_wait_timeout", "fp8bs_selftest_set_wait_limit",
        "fp8_quant_per_tensor_workspace_size", "fp8_quant_per_tensor", "fp8_quant_per_tensor_delayed",
        "fp8_gemm_per_tensor", "fp8_quant_per_tensor_noalloc", "fp8_ep_dispatch_pack", "fp8_ep_unpack",
        "fp8bs_gather_rows", "fp8_quant_act_1x128_scatter", "fp8_ep_dispatch_pack_scatter",
        "fp8bs_selftest_encode_e4m3"])


def test_library_loads_and_exports_every_declared_symbol():
    import fp8_fine_grained_26_b300 as fp8
    assert os.path.exists(fp8.LIB_PATH)
    for name in declared_functions():
        assert hasattr(fp8.lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", fp8.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(declared_functions()) <= exported


def test_oracle_is_not_linked_into_the_library():
    import fp8_fine_grained_26_b300 as fp8
    out = subprocess.run(["nm", "-D", fp8.LIB_PATH], capture_output=True, text=True).stdout
    assert "oracle_" not in out
    out = subprocess.run(["ldd", fp8.LIB_PATH], capture_output=True, text=True).stdout
    assert "liboracle" not in out


def test_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "fp8_fine_grained_26_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "liboracle" not in src and "fp8_oracle" not in src, f


# Host-side validation: these calls return before any CUDA call.
def _raw():
    import fp8_fine_grained_26_b300 as fp8
    return fp8.lib


P = ctypes.c_void_p


def test_quant_act_rejects_bad_shapes_and_pointers():
    lib = _raw()
    assert lib.fp8_quant_act_1x128(P(0), 4, 100, 100, P(0), 100, P(0), P(0)) == -2   # K % 128
    assert lib.fp8_quant_act_1x128(P(0), -1, 128, 128, P(0), 128, P(0), P(0)) == -2  # M < 0
    assert lib.fp8_quant_act_1x128(P(0), 0, 128, 128, P(0), 128, P(0), P(0)) == 0    # empty
    assert lib.fp8_quant_act_1x128(P(0), 4, 128, 128, P(0), 128, P(0), P(0)) == -1   # NULL
    assert lib.fp8_quant_act_1x128(P(16), 4, 128, 64, P(16), 128, P(16), P(0)) == -2  # ldx < K
    assert lib.fp8_quant_act_1x128(P(8), 4, 128, 128, P(16), 128, P(16), P(0)) == -3  # align
    assert lib.fp8_quant_act_1x128(P(16), 4, 128, 132, P(16), 128, P(16), P(0)) == -3  # ldx*2 % 16


def test_quant_w_rejects_bad_shapes():
    lib = _raw()
    assert lib.fp8_quant_w_128x128(P(0), 4, 130, 130, P(0), 130, P(0), P(0)) == -2
    assert lib.fp8_quant_w_128x128(P(0), 0, 128, 128, P(0), 128, P(0), P(0)) == 0
    assert lib.fp8_quant_w_128x128(P(16), 4, 128, 128, P(16), 136, P(16), P(0)) == -3


def test_quant_act_w_rejects_either_bad_operand():
    lib = _raw()
    q = lib.fp8_quant_act_w
    good_a = (P(16), 4, 128, 128, P(16), 128, P(16))
    good_w = (P(16), 4, 128, 128, P(16), 128, P(16))
    empty_a = (P(0), 0, 128, 128, P(0), 128, P(0))
    empty_w = (P(0), 0, 128, 128, P(0), 128, P(0))
    assert q(*empty_a, *empty_w, P(0)) == 0                                          # both empty
    assert q(P(16), 4, 100, 128, P(16), 128, P(16), *good_w, P(0)) == -2             # K % 128
    assert q(*good_a, P(16), 4, 130, 130, P(16), 130, P(16), P(0)) == -2             # C % 128
    assert q(P(0), 4, 128, 128, P(16), 128, P(16), *good_w, P(0)) == -1              # NULL x
    assert q(*good_a, P(16), 4, 128, 128, P(0), 128, P(16), P(0)) == -1              # NULL qw
    assert q(*good_a, P(16), 4, 128, 64, P(16), 128, P(16), P(0)) == -2              # ldw < C
    assert q(P(8), 4, 128, 128, P(16), 128, P(16), *empty_w, P(0)) == -3             # x align
    assert q(*empty_a, P(16), 4, 128, 128, P(16), 136, P(16), P(0)) == -3            # ldqw % 16
    assert q(P(16), -1, 128, 128, P(16), 128, P(16), *good_w, P(0)) == -2     # M < 0


def test_gemm_rejects_bad_arguments():
    lib = _raw()
    g = lib.fp8_gemm_blockscaled
    assert g(P(16), P(16), P(16), P(16), 4, 4, 128, 2, P(16), 0, 8, P(0)) == -4       # b_major
    assert g(P(16), P(16), P(16), P(16), 4, 4, 128, 0, P(16), 7, 8, P(0)) == -4       # c_dtype
    assert g(P(16), P(16), P(16), P(16), 4, 4, 100, 0, P(16), 0, 8, P(0)) == -2       # K % 128
    assert g(P(16), P(16), P(16), P(16), 0, 4, 128, 0, P(16), 0, 8, P(0)) == 0        # M == 0
    assert g(P(0), P(16), P(16), P(16), 4, 4, 128, 0, P(16), 0, 8, P(0)) == -1        # NULL qA
    assert g(P(16), P(16), P(16), P(16), 4, 8, 128, 0, P(16), 0, 4, P(0)) == -2       # ldc < N
    assert g(P(16), P(16), P(16), P(16), 4, 4, 128, 0, P(17), 0, 4, P(0)) == -3       # C align
    assert g(P(8), P(16), P(16), P(16), 4, 4, 128, 0, P(16), 0, 8, P(0)) == -3        # qA align
    gg = lib.fp8_grouped_gemm_blockscaled
    assert gg(P(16), P(16), P(16), P(16), P(16), 0, 4, 4, 128, P(16), 0, 8, P(0)) == -4   # E < 1
    assert gg(P(16), P(16), P(16), P(16), P(0), 2, 4, 4, 128, P(16), 0, 8, P(0)) == -1    # offsets


def test_grouped_gemm_expert_count_limit():
    """The header's FP8BS_MAX_EXPERTS (2048) is the largest accepted E: one
    more is FP8BS_ERR_ARG before any device call; E == 2048 passes the host
    checks (and, with no GPU, stops at the device check).  256 routed experts
    per MoE layer is the pages' configuration ("DeepSeek-V3 training
    walkthrough", section 一, DeepSeekMoE item)."""
    text = open(HEADER).read()
    assert "FP8BS_MAX_EXPERTS = 2048" in text
    gg = _raw().fp8_grouped_gemm_blockscaled
    assert gg(P(16), P(16), P(16), P(16), P(16), 2049, 4, 4, 128, P(16), 0, 8, P(0)) == -4
    assert gg(P(16), P(16), P(16), P(16), P(16), 4096, 4, 4, 128, P(16), 0, 8, P(0)) == -4
    if not os.path.exists("/dev/nvidia0"):
        assert gg(P(16), P(16), P(16), P(16), P(16), 2048, 4, 4, 128, P(16), 0, 8, P(0)) == -6


def test_e4m3_out_gemm_rejects_bad_arguments():
    lib = _raw()
    g = lib.fp8_gemm_blockscaled_e4m3_out
    assert g(P(16), P(16), P(16), P(16), 4, 200, 128, 0, P(16), 208, P(16), P(0)) == -2   # N % 128
    assert g(P(16), P(16), P(16), P(16), 4, 256, 100, 0, P(16), 256, P(16), P(0)) == -2   # K % 128
    assert g(P(16), P(16), P(16), P(16), 4, 256, 128, 3, P(16), 256, P(16), P(0)) == -4   # b_major
    assert g(P(16), P(16), P(16), P(16), 0, 256, 128, 0, P(0), 256, P(0), P(0)) == 0      # M == 0
    assert g(P(16), P(16), P(16), P(16), 4, 256, 128, 0, P(0), 256, P(16), P(0)) == -1   # NULL qC
    assert g(P(16), P(16), P(16), P(16), 4, 256, 128, 0, P(16), 256, P(0), P(0)) == -1   # NULL sC
    assert g(P(16), P(16), P(16), P(16), 4, 256, 128, 0, P(16), 128, P(16), P(0)) == -2  # ldqc < N
    assert g(P(16), P(16), P(16), P(16), 4, 256, 128, 0, P(16), 264, P(16), P(0)) == -3  # ldqc % 16
    assert g(P(16), P(16), P(16), P(16), 4, 256, 128, 0, P(8), 256, P(16), P(0)) == -3   # qC align


def test_token_quantiser_and_wgrad_reject_bad_arguments():
    lib = _raw()
    q = lib.fp8_quant_tokens_1x128
    assert q(P(16), 100, 8, 8, P(16), 112, P(16), P(0)) == -2      # T % 128
    assert q(P(16), 0, 8, 8, P(16), 128, P(16), P(0)) == 0         # empty
    assert q(P(0), 128, 8, 8, P(16), 128, P(16), P(0)) == -1       # NULL
    assert q(P(16), 128, 8, 4, P(16), 128, P(16), P(0)) == -2      # ldx < F
    assert q(P(16), 128, 8, 8, P(16), 120, P(16), P(0)) == -2      # ldq < T
    assert q(P(16), 128, 8, 12, P(16), 128, P(16), P(0)) == -3     # ldx * 2 % 16
    w = lib.fp8_gemm_wgrad
    assert w(P(16), P(16), P(16), P(16), 4, 4, 100, P(16), 0, 8, P(0)) == -2     # K % 128
    assert w(P(16), P(16), P(16), P(16), 4, 4, 128, P(16), 5, 8, P(0)) == -4     # c_dtype
    assert w(P(0), P(16), P(16), P(16), 4, 4, 128, P(16), 0, 8, P(0)) == -1      # NULL
    assert w(P(16), P(16), P(16), P(16), 0, 4, 128, P(16), 0, 8, P(0)) == 0      # M == 0


def test_gather_quantiser_rejects_bad_arguments():
    lib = _raw()
    g = lib.fp8_quant_act_1x128_gather
    assert g(P(16), 8, 100, 128, P(16), 4, P(16), 128, P(16), P(0)) == -2    # K % 128
    assert g(P(16), 8, 128, 128, P(16), 0, P(16), 128, P(16), P(0)) == 0     # M == 0
    assert g(P(16), 8, 128, 128, P(0), 4, P(16), 128, P(16), P(0)) == -1     # NULL rows
    assert g(P(16), 8, 128, 64, P(16), 4, P(16), 128, P(16), P(0)) == -2     # ldx < K
    assert g(P(16), 8, 128, 128, P(18), 4, P(16), 128, P(16), P(0)) == -3    # rows align
    assert g(P(16), 8, 128, 132, P(16), 4, P(16), 128, P(16), P(0)) == -3    # ldx * 2 % 16


def test_per_tensor_calls_reject_bad_arguments():
    lib = _raw()
    n = ctypes.c_int64(0)
    assert lib.fp8_quant_per_tensor_workspace_size(300, 384, ctypes.byref(n)) == 0
    assert n.value == 4 * (3 * 3 + 1)                                   # one word per 128x128 unit, plus one
    assert lib.fp8_quant_per_tensor_workspace_size(300, 100, ctypes.byref(n)) == -2
    assert lib.fp8_quant_per_tensor_workspace_size(300, 128, None) == -1
    q = lib.fp8_quant_per_tensor
    assert q(P(16), 4, 100, 128, P(16), 128, P(16), P(16), 64, P(0)) == -2         # C % 128
    assert q(P(16), 0, 128, 128, P(16), 128, P(16), P(16), 0, P(0)) == 0           # empty: no-op
    assert q(P(16), 4, 128, 128, P(16), 128, P(16), P(0), 64, P(0)) == -1          # no workspace
    assert q(P(16), 4, 128, 128, P(16), 128, P(16), P(18), 64, P(0)) == -3         # workspace align
    assert q(P(16), 300, 384, 384, P(16), 384, P(16), P(16), 39, P(0)) == -4      # workspace too small
    d = lib.fp8_quant_per_tensor_delayed
    assert d(P(16), 4, 128, 128, P(0), P(16), 128, P(16), P(32), P(0)) == -1       # no amax_in
    assert d(P(16), 4, 128, 128, P(32), P(16), 128, P(16), P(32), P(0)) == -4      # amax_in == amax_out
    assert d(P(16), 4, 128, 128, P(34), P(16), 128, P(16), P(32), P(0)) == -3      # amax_in align
    g = lib.fp8_gemm_per_tensor
    assert g(P(16), P(16), P(16), P(16), 4, 4, 128, 2, P(16), 0, 8, P(0)) == -4      # b_major
    assert g(P(16), P(16), P(16), P(16), 4, 4, 100, 0, P(16), 0, 8, P(0)) == -2      # K % 128
    assert g(P(16), P(16), P(16), P(16), 4, 20, 128, 1, P(16), 0, 20, P(0)) == -2    # MN-major N % 16
    assert g(P(16), P(0), P(16), P(16), 4, 4, 128, 0, P(16), 0, 8, P(0)) == -1       # NULL sA


def test_selftest_rejects_out_of_range_limits():
    lib = _raw()
    assert lib.fp8bs_selftest_wait_timeout(0, P(0)) == -4
    assert lib.fp8bs_selftest_wait_timeout(-5, P(0)) == -4
    assert lib.fp8bs_selftest_wait_timeout(1000001, P(0)) == -4
    s = lib.fp8bs_selftest_set_wait_limit
    assert s(-1) == -4 and s(2000000001) == -4
    assert s(0) == 0                                  # the default; host-only
    e = lib.fp8bs_selftest_encode_e4m3
    e.argtypes = [ctypes.c_uint32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    assert e(0, -1, P(16), P(0)) == -4
    assert e(0xFFFFFFF0, 17, P(16), P(0)) == -4       # past the last pattern
    assert e(5, 0, P(0), P(0)) == 0                   # nothing to do; host-only


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="checks the no-GPU answer")
def test_no_gpu_is_reported_as_device_error():
    lib = _raw()
    st = lib.fp8_quant_act_1x128(P(16), 4, 128, 128, P(16), 128, P(16), P(0))
    assert st == -6


def test_build_entry_does_not_need_the_library_to_exist():
    # a fresh checkout has no libfp8bs.so, and the package refuses to import
    # without it: build() must reach the build script without importing the
    # package first
    import subprocess
    code = ("import sys, __graft_entry__ as g, os; "
            "m = g._module_from_file('fp8bs_lib_build', os.path.join(g.ROOT, 'fp8_fine_grained_26_b300', 'build.py')); "
            "assert 'fp8_fine_grained_26_b300' not in sys.modules; "
            "assert callable(m.build) and m.LIB.endswith('libfp8bs.so'); print('ok')")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stderr[-2000:]
