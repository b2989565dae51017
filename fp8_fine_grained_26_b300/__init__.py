"""Python binding of the fine-grained FP8 block-scaled GEMM library.

Argument marshalling only: every function here checks tensor dtypes, shapes
and devices, allocates outputs with torch when the caller did not pass them,
and calls the same-named C entry point of ``libfp8bs.so`` (declared in
``include/fp8bs.h``) on the current torch CUDA stream.  All arithmetic runs
in the library's CUDA kernels; there is no fallback of any kind.  Importing
this package fails if the library has not been built.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8bs.so")

FP8BS_OK = 0
FP8BS_ERR_NULL = -1
FP8BS_ERR_SHAPE = -2
FP8BS_ERR_ALIGN = -3
FP8BS_ERR_ARG = -4
FP8BS_ERR_LAUNCH = -5
FP8BS_ERR_DEVICE = -6
FP8BS_ERR_TIMEOUT = -7
FP8BS_ERR_INDEX = -8
FP8BS_ERR_SCRATCH = -9
OUT_BF16, OUT_FP32 = 0, 1
B_KMAJOR, B_MNMAJOR = 0, 1

_STATUS_NAMES = {
    FP8BS_ERR_NULL: "FP8BS_ERR_NULL", FP8BS_ERR_SHAPE: "FP8BS_ERR_SHAPE",
    FP8BS_ERR_ALIGN: "FP8BS_ERR_ALIGN", FP8BS_ERR_ARG: "FP8BS_ERR_ARG",
    FP8BS_ERR_LAUNCH: "FP8BS_ERR_LAUNCH", FP8BS_ERR_DEVICE: "FP8BS_ERR_DEVICE",
    FP8BS_ERR_TIMEOUT: "FP8BS_ERR_TIMEOUT", FP8BS_ERR_INDEX: "FP8BS_ERR_INDEX",
    FP8BS_ERR_SCRATCH: "FP8BS_ERR_SCRATCH",
}

EXPORTED = ("fp8_quant_act_1x128", "fp8_quant_w_128x128", "fp8_quant_act_w", "fp8_gemm_blockscaled",
            "fp8_gemm_blockscaled_e4m3_out", "fp8_quant_tokens_1x128", "fp8_gemm_wgrad",
            "fp8_quant_act_1x128_gather", "fp8_grouped_gemm_blockscaled", "fp8bs_last_error",
            "fp8bs_selftest_wait_timeout", "fp8bs_selftest_set_wait_limit",
            "fp8_quant_per_tensor_workspace_size", "fp8_quant_per_tensor", "fp8_quant_per_tensor_delayed",
            "fp8_gemm_per_tensor", "fp8_quant_per_tensor_noalloc", "fp8_ep_dispatch_pack", "fp8_ep_unpack",
            "fp8bs_gather_rows", "fp8_quant_act_1x128_scatter", "fp8_ep_dispatch_pack_scatter",
            "fp8bs_selftest_encode_e4m3")


class Fp8bsError(RuntimeError):
    def __init__(self, status, call):
        self.status = status
        super().__init__(f"{call} returned {_STATUS_NAMES.get(status, status)}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                          "(python fp8_fine_grained_26_b300/build.py, or __graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    i64, p, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    sigs = {
        "fp8_quant_act_1x128": [p, i64, i64, i64, p, i64, p, p],
        "fp8_quant_w_128x128": [p, i64, i64, i64, p, i64, p, p],
        "fp8_quant_act_w": [p, i64, i64, i64, p, i64, p, p, i64, i64, i64, p, i64, p, p],
        "fp8_gemm_blockscaled": [p, p, p, p, i64, i64, i64, i32, p, i32, i64, p],
        "fp8_gemm_blockscaled_e4m3_out": [p, p, p, p, i64, i64, i64, i32, p, i64, p, p],
        "fp8_quant_tokens_1x128": [p, i64, i64, i64, p, i64, p, p],
        "fp8_quant_act_1x128_gather": [p, i64, i64, i64, p, i64, p, i64, p, p],
        "fp8_gemm_wgrad": [p, p, p, p, i64, i64, i64, p, i32, i64, p],
        "fp8_grouped_gemm_blockscaled": [p, p, p, p, p, i32, i64, i64, i64, p, i32, i64, p],
        "fp8bs_last_error": [p],
        "fp8bs_selftest_wait_timeout": [i64, p],
        "fp8bs_selftest_set_wait_limit": [i64],
        "fp8bs_selftest_encode_e4m3": [ctypes.c_uint32, i64, p, p],
        "fp8_quant_per_tensor_workspace_size": [i64, i64, p],
        "fp8_quant_per_tensor": [p, i64, i64, i64, p, i64, p, p, i64, p],
        "fp8_quant_per_tensor_delayed": [p, i64, i64, i64, p, p, i64, p, p, p],
        "fp8_gemm_per_tensor": [p, p, p, p, i64, i64, i64, i32, p, i32, i64, p],
        "fp8_quant_per_tensor_noalloc": [p, i64, i64, i64, p, i64, p, p],
        "fp8_ep_dispatch_pack": [p, i64, i64, i64, p, i64, p, i64, p],
        "fp8_ep_unpack": [p, i64, i64, i64, p, i64, p, i64, p, p],
        "fp8bs_gather_rows": [p, i64, i64, p, i64, i64, p, i64, p],
        "fp8_quant_act_1x128_scatter": [p, i64, i64, i64, p, i32, i64, p, i64, p, p],
        "fp8_ep_dispatch_pack_scatter": [p, i64, i64, i64, p, i32, i64, p, i64, p],
    }
    for name, args in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    return lib


lib = _load()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _check(status, call):
    if status != FP8BS_OK:
        raise Fp8bsError(status, call)


def _need(t, dtype, name, ndim):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.dim() != ndim or not t.is_cuda:
        raise TypeError(f"{name}: expected a {ndim}-D CUDA tensor of {dtype}")


def _row_major(t, name):
    if t.dim() >= 1 and t.numel() > 0 and t.stride(-1) != 1:
        raise ValueError(f"{name}: innermost dimension must be contiguous")


def fp8_quant_act_1x128(x, q=None, sA=None, stream=None):
    """1x128 tile quantisation of BF16 ``x [M, K]`` (row stride may exceed K).

    Returns ``(q uint8 [M, K], sA float32 [K/128, M])``; E4M3 codes are
    returned as their bytes (view them as ``torch.float8_e4m3fn`` if wanted)."""
    _need(x, torch.bfloat16, "x", 2)
    _row_major(x, "x")
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sA is None:
        sA = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    _need(q, torch.uint8, "q", 2)
    _row_major(q, "q")
    if tuple(q.shape) != (M, K) or not sA.is_contiguous() or sA.numel() != (K // 128) * M:
        raise ValueError("output shapes do not match x")
    ldx = x.stride(0) if M > 0 else K
    ldq = q.stride(0) if M > 0 else K
    _check(lib.fp8_quant_act_1x128(_ptr(x), M, K, ldx, _ptr(q), ldq, _ptr(sA), _stream(stream)),
           "fp8_quant_act_1x128")
    return q, sA


def fp8_quant_w_128x128(w, q=None, sW=None, stream=None):
    """128x128 block quantisation of BF16 ``w [R, C]``.

    Returns ``(q uint8 [R, C], sW float32 [ceil(R/128), C/128])``."""
    _need(w, torch.bfloat16, "w", 2)
    _row_major(w, "w")
    R, C = w.shape
    if q is None:
        q = torch.empty((R, C), dtype=torch.uint8, device=w.device)
    if sW is None:
        sW = torch.empty(((R + 127) // 128, C // 128), dtype=torch.float32, device=w.device)
    _need(q, torch.uint8, "q", 2)
    _row_major(q, "q")
    if tuple(q.shape) != (R, C) or not sW.is_contiguous() or \
            sW.numel() != ((R + 127) // 128) * (C // 128):
        raise ValueError("output shapes do not match w")
    ldw = w.stride(0) if R > 0 else C
    ldq = q.stride(0) if R > 0 else C
    _check(lib.fp8_quant_w_128x128(_ptr(w), R, C, ldw, _ptr(q), ldq, _ptr(sW), _stream(stream)),
           "fp8_quant_w_128x128")
    return q, sW


def fp8_quant_act_w(x, w, qa=None, sA=None, qw=None, sW=None, stream=None):
    """Both operands of one GEMM in one launch: 1x128 quantisation of BF16
    ``x [M, K]`` and 128x128 quantisation of BF16 ``w [R, C]``, bit-equal to
    fp8_quant_act_1x128(x) and fp8_quant_w_128x128(w).

    Returns ``(qa, sA, qw, sW)`` with the shapes of those two calls."""
    _need(x, torch.bfloat16, "x", 2)
    _need(w, torch.bfloat16, "w", 2)
    _row_major(x, "x")
    _row_major(w, "w")
    M, K = x.shape
    R, C = w.shape
    if qa is None:
        qa = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sA is None:
        sA = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    if qw is None:
        qw = torch.empty((R, C), dtype=torch.uint8, device=w.device)
    if sW is None:
        sW = torch.empty(((R + 127) // 128, C // 128), dtype=torch.float32, device=w.device)
    _need(qa, torch.uint8, "qa", 2)
    _need(qw, torch.uint8, "qw", 2)
    _row_major(qa, "qa")
    _row_major(qw, "qw")
    if tuple(qa.shape) != (M, K) or not sA.is_contiguous() or sA.numel() != (K // 128) * M:
        raise ValueError("activation output shapes do not match x")
    if tuple(qw.shape) != (R, C) or not sW.is_contiguous() or sW.numel() != ((R + 127) // 128) * (C // 128):
        raise ValueError("weight output shapes do not match w")
    ldx = x.stride(0) if M > 0 else K
    ldqa = qa.stride(0) if M > 0 else K
    ldw = w.stride(0) if R > 0 else C
    ldqw = qw.stride(0) if R > 0 else C
    _check(lib.fp8_quant_act_w(_ptr(x), M, K, ldx, _ptr(qa), ldqa, _ptr(sA),
                               _ptr(w), R, C, ldw, _ptr(qw), ldqw, _ptr(sW), _stream(stream)),
           "fp8_quant_act_w")
    return qa, sA, qw, sW


def _out(C, M, N, out_dtype, device):
    if C is None:
        C = torch.empty((M, N), dtype=out_dtype, device=device)
    if C.dtype not in (torch.bfloat16, torch.float32) or C.dim() != 2 or \
            tuple(C.shape) != (M, N) or not C.is_cuda:
        raise ValueError("C must be a [M, N] CUDA tensor of bfloat16 or float32")
    _row_major(C, "C")
    ldc = C.stride(0) if M > 0 else N
    return C, (OUT_FP32 if C.dtype == torch.float32 else OUT_BF16), ldc


def fp8_gemm_blockscaled(qA, sA, qB, sB, b_major=B_KMAJOR, out_dtype=torch.bfloat16, C=None,
                         stream=None):
    """``C = A . B^T`` from 1x128-quantised ``qA [M, K]`` / ``sA [K/128, M]`` and
    128x128-quantised B: ``qB [N, K]`` / ``sB [ceil(N/128), K/128]`` (K-major),
    or ``qB [K, N]`` / ``sB [K/128, N/128]`` (``b_major=B_MNMAJOR``)."""
    _need(qA, torch.uint8, "qA", 2)
    _need(qB, torch.uint8, "qB", 2)
    _need(sA, torch.float32, "sA", 2)
    _need(sB, torch.float32, "sB", 2)
    for t, n in ((qA, "qA"), (qB, "qB"), (sA, "sA"), (sB, "sB")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    M, K = qA.shape
    if b_major == B_KMAJOR:
        N, Kb = qB.shape
    else:
        Kb, N = qB.shape
    if Kb != K:
        raise ValueError("qA and qB disagree on K")
    C, cd, ldc = _out(C, M, N, out_dtype, qA.device)
    _check(lib.fp8_gemm_blockscaled(_ptr(qA), _ptr(sA), _ptr(qB), _ptr(sB), M, N, K, b_major,
                                    _ptr(C), cd, ldc, _stream(stream)), "fp8_gemm_blockscaled")
    return C


def fp8_gemm_blockscaled_e4m3_out(qA, sA, qB, sB, b_major=B_KMAJOR, qC=None, sC=None, stream=None):
    """``C = A . B^T`` as :func:`fp8_gemm_blockscaled`, returned quantised per
    1x128 row tile: ``qC uint8 [M, N]`` (E4M3 codes) and ``sC float32
    [N/128, M]``.  N must be a multiple of 128."""
    _need(qA, torch.uint8, "qA", 2)
    _need(qB, torch.uint8, "qB", 2)
    _need(sA, torch.float32, "sA", 2)
    _need(sB, torch.float32, "sB", 2)
    for t, n in ((qA, "qA"), (qB, "qB"), (sA, "sA"), (sB, "sB")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    M, K = qA.shape
    if b_major == B_KMAJOR:
        N, Kb = qB.shape
    else:
        Kb, N = qB.shape
    if Kb != K:
        raise ValueError("qA and qB disagree on K")
    if qC is None:
        qC = torch.empty((M, N), dtype=torch.uint8, device=qA.device)
    if sC is None:
        sC = torch.empty((N // 128, M), dtype=torch.float32, device=qA.device)
    _need(qC, torch.uint8, "qC", 2)
    _need(sC, torch.float32, "sC", 2)
    if tuple(qC.shape) != (M, N) or tuple(sC.shape) != (N // 128, M) or not sC.is_contiguous():
        raise ValueError("qC must be [M, N] and sC a contiguous [N/128, M]")
    _row_major(qC, "qC")
    ldq = qC.stride(0) if M > 0 else N
    _check(lib.fp8_gemm_blockscaled_e4m3_out(_ptr(qA), _ptr(sA), _ptr(qB), _ptr(sB), M, N, K, b_major,
                                             _ptr(qC), ldq, _ptr(sC), _stream(stream)),
           "fp8_gemm_blockscaled_e4m3_out")
    return qC, sC


def fp8_quant_act_1x128_gather(x, rows, q=None, sA=None, stream=None):
    """1x128 quantisation of the gathered rows ``x[rows]`` of a BF16 ``[T, K]``
    matrix (``rows``: int32 CUDA tensor), without materialising them; returns
    ``(q uint8 [M, K], sA float32 [K/128, M])`` with ``M = len(rows)``."""
    _need(x, torch.bfloat16, "x", 2)
    _need(rows, torch.int32, "rows", 1)
    _row_major(x, "x")
    if not rows.is_contiguous():
        raise ValueError("rows must be contiguous")
    T, K = x.shape
    M = rows.numel()
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sA is None:
        sA = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    _row_major(q, "q")
    ldx = x.stride(0) if T > 0 else K
    ldq = q.stride(0) if M > 0 else K
    _check(lib.fp8_quant_act_1x128_gather(_ptr(x), T, K, ldx, _ptr(rows), M, _ptr(q), ldq, _ptr(sA),
                                          _stream(stream)), "fp8_quant_act_1x128_gather")
    return q, sA


def fp8_quant_tokens_1x128(x, qT=None, s=None, stream=None):
    """Quantise a BF16 ``[T, F]`` matrix per 1x128 run of tokens in each
    feature column; returns ``(qT uint8 [F, T], s float32 [T/128, F])``."""
    _need(x, torch.bfloat16, "x", 2)
    _row_major(x, "x")
    T, F = x.shape
    if qT is None:
        qT = torch.empty((F, T), dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty((T // 128, F), dtype=torch.float32, device=x.device)
    _row_major(qT, "qT")
    ldx = x.stride(0) if T > 0 else F
    ldq = qT.stride(0) if F > 0 else T
    _check(lib.fp8_quant_tokens_1x128(_ptr(x), T, F, ldx, _ptr(qT), ldq, _ptr(s), _stream(stream)),
           "fp8_quant_tokens_1x128")
    return qT, s


def fp8_gemm_wgrad(qA, sA, qB, sB, out_dtype=torch.bfloat16, C=None, stream=None):
    """Weight-gradient GEMM ``C = A . B^T`` with both operands scaled per row
    and 128-wide K-slice: ``qA [M, K]`` / ``sA [K/128, M]``, ``qB [N, K]`` /
    ``sB [K/128, N]`` (outputs of :func:`fp8_quant_tokens_1x128`)."""
    for t, n, d in ((qA, "qA", torch.uint8), (qB, "qB", torch.uint8), (sA, "sA", torch.float32),
                    (sB, "sB", torch.float32)):
        _need(t, d, n, 2)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    M, K = qA.shape
    N, Kb = qB.shape
    if Kb != K:
        raise ValueError("qA and qB disagree on K")
    C, cd, ldc = _out(C, M, N, out_dtype, qA.device)
    _check(lib.fp8_gemm_wgrad(_ptr(qA), _ptr(sA), _ptr(qB), _ptr(sB), M, N, K, _ptr(C), cd, ldc,
                              _stream(stream)), "fp8_gemm_wgrad")
    return C


def fp8_grouped_gemm_blockscaled(qA, sA, qB, sB, seg_offsets, out_dtype=torch.bfloat16, C=None,
                                 stream=None):
    """Per-expert ``C[rows of e] = A[rows of e] . B_e^T`` with ``qB [E, N, K]``,
    ``sB [E, ceil(N/128), K/128]`` and device ``seg_offsets int32 [E+1]``."""
    _need(qA, torch.uint8, "qA", 2)
    _need(qB, torch.uint8, "qB", 3)
    _need(sA, torch.float32, "sA", 2)
    _need(sB, torch.float32, "sB", 3)
    _need(seg_offsets, torch.int32, "seg_offsets", 1)
    for t, n in ((qA, "qA"), (qB, "qB"), (sA, "sA"), (sB, "sB"), (seg_offsets, "seg_offsets")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    M, K = qA.shape
    E, N, Kb = qB.shape
    if Kb != K or seg_offsets.numel() != E + 1:
        raise ValueError("grouped GEMM shapes disagree")
    C, cd, ldc = _out(C, M, N, out_dtype, qA.device)
    _check(lib.fp8_grouped_gemm_blockscaled(_ptr(qA), _ptr(sA), _ptr(qB), _ptr(sB),
                                            _ptr(seg_offsets), E, M, N, K, _ptr(C), cd, ldc,
                                            _stream(stream)), "fp8_grouped_gemm_blockscaled")
    return C


def fp8_quant_per_tensor_workspace_size(R, C):
    """Bytes of device workspace fp8_quant_per_tensor needs for an [R, C] tensor."""
    n = ctypes.c_int64(0)
    _check(lib.fp8_quant_per_tensor_workspace_size(int(R), int(C), ctypes.byref(n)),
           "fp8_quant_per_tensor_workspace_size")
    return n.value


def _per_tensor_outputs(x, q, scale):
    R, C = x.shape
    if q is None:
        q = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((1,), dtype=torch.float32, device=x.device)
    _need(q, torch.uint8, "q", 2)
    _row_major(q, "q")
    if tuple(q.shape) != (R, C) or scale.dtype != torch.float32 or scale.numel() < 1 or not scale.is_cuda:
        raise ValueError("output shapes do not match x")
    return q, scale


def fp8_quant_per_tensor(x, q=None, scale=None, workspace=None, stream=None):
    """Per-tensor quantisation of BF16 ``x [R, C]`` with its own amax (one
    scale fp32(amax/448) for every element).  ``workspace``: a device uint8
    tensor of at least fp8_quant_per_tensor_workspace_size(R, C) bytes
    (allocated here when not given).  Returns ``(q uint8 [R, C], scale float32 [1])``."""
    _need(x, torch.bfloat16, "x", 2)
    _row_major(x, "x")
    R, C = x.shape
    q, scale = _per_tensor_outputs(x, q, scale)
    need = fp8_quant_per_tensor_workspace_size(R, C)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=x.device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    ldx = x.stride(0) if R > 0 else C
    ldq = q.stride(0) if R > 0 else C
    _check(lib.fp8_quant_per_tensor(_ptr(x), R, C, ldx, _ptr(q), ldq, _ptr(scale), _ptr(workspace), nbytes,
                                    _stream(stream)), "fp8_quant_per_tensor")
    return q, scale


def fp8_quant_per_tensor_delayed(x, amax_in, q=None, scale=None, amax_out=None, stream=None):
    """Per-tensor quantisation of BF16 ``x [R, C]`` with delayed scaling: the
    scale is fp32(amax_in/448) for a given device float ``amax_in`` (e.g. the
    largest amax of earlier steps); this tensor's own amax goes to
    ``amax_out``.  Returns ``(q, scale, amax_out)``."""
    _need(x, torch.bfloat16, "x", 2)
    _row_major(x, "x")
    R, C = x.shape
    q, scale = _per_tensor_outputs(x, q, scale)
    if amax_out is None:
        amax_out = torch.empty((1,), dtype=torch.float32, device=x.device)
    for t, n in ((amax_in, "amax_in"), (amax_out, "amax_out")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.numel() < 1 or not t.is_cuda:
            raise TypeError(f"{n}: expected a CUDA float32 tensor")
    ldx = x.stride(0) if R > 0 else C
    ldq = q.stride(0) if R > 0 else C
    _check(lib.fp8_quant_per_tensor_delayed(_ptr(x), R, C, ldx, _ptr(amax_in), _ptr(q), ldq, _ptr(scale),
                                            _ptr(amax_out), _stream(stream)), "fp8_quant_per_tensor_delayed")
    return q, scale, amax_out


def fp8_gemm_per_tensor(qA, sA, qB, sB, b_major=B_KMAJOR, out_dtype=torch.bfloat16, C=None, stream=None):
    """``C = sA sB (qA . qB^T)`` for per-tensor scaled operands (``sA``, ``sB``
    one-element device float32 tensors), the whole K accumulated on the
    tensor cores.  ``qB`` is ``[N, K]`` or (b_major=1) stored ``[K, N]``."""
    _need(qA, torch.uint8, "qA", 2)
    _need(qB, torch.uint8, "qB", 2)
    M, K = qA.shape
    N = qB.shape[0] if b_major == B_KMAJOR else qB.shape[1]
    Kb = qB.shape[1] if b_major == B_KMAJOR else qB.shape[0]
    if Kb != K:
        raise ValueError("qA and qB disagree on K")
    for t, n in ((sA, "sA"), (sB, "sB")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.numel() < 1 or not t.is_cuda:
            raise TypeError(f"{n}: expected a CUDA float32 tensor")
    C, cd, ldc = _out(C, M, N, out_dtype, qA.device)
    _check(lib.fp8_gemm_per_tensor(_ptr(qA), _ptr(sA), _ptr(qB), _ptr(sB), M, N, K, int(b_major), _ptr(C), cd,
                                   ldc, _stream(stream)), "fp8_gemm_per_tensor")
    return C


def fp8_quant_act_1x128_scatter(x, dest, M, q=None, sA=None, stream=None):
    """Token row t of BF16 ``x [T, K]`` quantised once per 1x128 tile and
    written to rows ``dest[t, j]`` of ``q [M, K]`` / columns of ``sA [K/128, M]``
    (``dest``: CUDA int32 ``[T, topk]``)."""
    _need(x, torch.bfloat16, "x", 2)
    _row_major(x, "x")
    if dest.dtype != torch.int32 or dest.dim() != 2 or not dest.is_cuda or dest.shape[0] != x.shape[0]:
        raise TypeError("dest: expected a CUDA int32 tensor [T, topk]")
    T, K = x.shape
    topk = dest.shape[1]
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sA is None:
        sA = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    _need(q, torch.uint8, "q", 2)
    _row_major(q, "q")
    if tuple(q.shape) != (M, K) or not sA.is_contiguous() or sA.numel() != (K // 128) * M:
        raise ValueError("output shapes do not match")
    ldx = x.stride(0) if T > 0 else K
    ldq = q.stride(0) if M > 0 else K
    _check(lib.fp8_quant_act_1x128_scatter(_ptr(x), T, K, ldx, _ptr(dest.contiguous()), topk, M, _ptr(q), ldq,
                                           _ptr(sA), _stream(stream)), "fp8_quant_act_1x128_scatter")
    return q, sA


def packed_row_bytes(K):
    """Row stride (bytes) of a packed dispatch row: K codes + K/128 FP32
    scales, rounded up to 16."""
    return (K + 4 * (K // 128) + 15) // 16 * 16


def fp8_ep_dispatch_pack(x, rows, packed=None, stream=None):
    """Gather + 1x128 quantisation of the routed rows ``x[rows]`` into packed
    rows ``[M, packed_row_bytes(K)]`` (codes, then the row's scales)."""
    _need(x, torch.bfloat16, "x", 2)
    _row_major(x, "x")
    if rows.dtype != torch.int32 or rows.dim() != 1 or not rows.is_cuda:
        raise TypeError("rows: expected a 1-D CUDA int32 tensor")
    T, K = x.shape
    M = rows.numel()
    if packed is None:
        packed = torch.empty((M, packed_row_bytes(K)), dtype=torch.uint8, device=x.device)
    _need(packed, torch.uint8, "packed", 2)
    _row_major(packed, "packed")
    if packed.shape[0] != M:
        raise ValueError("packed must have one row per routed copy")
    ldx = x.stride(0) if T > 0 else K
    ld = packed.stride(0) if M > 0 else packed.shape[1]
    _check(lib.fp8_ep_dispatch_pack(_ptr(x), T, K, ldx, _ptr(rows.contiguous()), M, _ptr(packed), ld,
                                    _stream(stream)), "fp8_ep_dispatch_pack")
    return packed


def fp8_ep_dispatch_pack_scatter(x, dest, M, packed=None, stream=None):
    """Token row t of BF16 ``x [T, K]`` quantised once and packed (codes, then
    its scales) into send rows ``dest[t, j]`` of ``packed [M, packed_row_bytes(K)]``."""
    _need(x, torch.bfloat16, "x", 2)
    _row_major(x, "x")
    if dest.dtype != torch.int32 or dest.dim() != 2 or not dest.is_cuda or dest.shape[0] != x.shape[0]:
        raise TypeError("dest: expected a CUDA int32 tensor [T, topk]")
    T, K = x.shape
    if packed is None:
        packed = torch.empty((M, packed_row_bytes(K)), dtype=torch.uint8, device=x.device)
    _need(packed, torch.uint8, "packed", 2)
    _row_major(packed, "packed")
    if packed.shape[0] != M:
        raise ValueError("packed must have M rows")
    ldx = x.stride(0) if T > 0 else K
    ld = packed.stride(0) if M > 0 else packed.shape[1]
    _check(lib.fp8_ep_dispatch_pack_scatter(_ptr(x), T, K, ldx, _ptr(dest.contiguous()), dest.shape[1], M,
                                            _ptr(packed), ld, _stream(stream)), "fp8_ep_dispatch_pack_scatter")
    return packed


def fp8_ep_unpack(packed, K, perm, q=None, sA=None, stream=None):
    """Packed rows, reordered by ``perm``: ``q[i], sA[:, i]`` = codes and
    scales of ``packed[perm[i]]``.  Returns ``(q uint8 [M, K], sA [K/128, M])``."""
    _need(packed, torch.uint8, "packed", 2)
    _row_major(packed, "packed")
    if perm.dtype != torch.int32 or perm.dim() != 1 or not perm.is_cuda:
        raise TypeError("perm: expected a 1-D CUDA int32 tensor")
    M = perm.numel()
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=packed.device)
    if sA is None:
        sA = torch.empty((K // 128, M), dtype=torch.float32, device=packed.device)
    _need(q, torch.uint8, "q", 2)
    if not sA.is_contiguous() or sA.numel() != (K // 128) * M:
        raise ValueError("sA must be a contiguous [K/128, M] tensor")
    ld = packed.stride(0) if packed.shape[0] > 0 else packed.shape[1]
    ldq = q.stride(0) if M > 0 else K
    _check(lib.fp8_ep_unpack(_ptr(packed), packed.shape[0], ld, K, _ptr(perm.contiguous()), M, _ptr(q), ldq,
                             _ptr(sA), _stream(stream)), "fp8_ep_unpack")
    return q, sA


def fp8bs_gather_rows(src, rows, dst=None, stream=None):
    """``dst[i] = src[rows[i]]`` for the rows of a 2-D CUDA tensor (any dtype;
    a row must be a multiple of 16 bytes)."""
    if src.dim() != 2 or not src.is_cuda:
        raise TypeError("src: expected a 2-D CUDA tensor")
    _row_major(src, "src")
    if rows.dtype != torch.int32 or rows.dim() != 1 or not rows.is_cuda:
        raise TypeError("rows: expected a 1-D CUDA int32 tensor")
    M = rows.numel()
    if dst is None:
        dst = torch.empty((M, src.shape[1]), dtype=src.dtype, device=src.device)
    if dst.dtype != src.dtype or dst.dim() != 2 or dst.shape[1] != src.shape[1] or dst.shape[0] != M:
        raise ValueError("dst must be [len(rows), src.shape[1]] of src's dtype")
    _row_major(dst, "dst")
    es = src.element_size()
    row_bytes = src.shape[1] * es
    ld_src = (src.stride(0) if src.shape[0] > 0 else src.shape[1]) * es
    ld_dst = (dst.stride(0) if M > 0 else dst.shape[1]) * es
    _check(lib.fp8bs_gather_rows(_ptr(src), src.shape[0], ld_src, _ptr(rows.contiguous()), M, row_bytes, _ptr(dst),
                                 ld_dst, _stream(stream)), "fp8bs_gather_rows")
    return dst


def fp8bs_last_error(stream=None):
    """Synchronise the stream and return (and clear) the device error status."""
    return lib.fp8bs_last_error(_stream(stream))


def fp8bs_selftest_wait_timeout(limit_us=20000, stream=None):
    """Enqueue the failure-detection self-test: a device wait that nothing
    ends runs out after ``limit_us`` and is recorded in the error word (read
    it with fp8bs_last_error)."""
    _check(lib.fp8bs_selftest_wait_timeout(int(limit_us), _stream(stream)), "fp8bs_selftest_wait_timeout")


def fp8bs_selftest_set_wait_limit(limit_ns):
    """Test hook: time limit (ns) of the pipeline waits of quantisers and
    single-CTA GEMMs launched from now on; 0 restores the default (2 s)."""
    _check(lib.fp8bs_selftest_set_wait_limit(int(limit_ns)), "fp8bs_selftest_set_wait_limit")


def fp8bs_selftest_encode_e4m3(first_bits, n, q=None, stream=None):
    """Test hook: ``q[i]`` = the E4M3 code the quantisers' conversion gives
    the fp32 value with bit pattern ``first_bits + i`` (uint8 CUDA tensor of
    ``n`` codes)."""
    if q is None:
        q = torch.empty(int(n), dtype=torch.uint8, device="cuda")
    if q.dtype != torch.uint8 or not q.is_cuda or not q.is_contiguous() or q.numel() < n:
        raise TypeError("q: expected a contiguous uint8 CUDA tensor of at least n elements")
    _check(lib.fp8bs_selftest_encode_e4m3(int(first_bits), int(n), _ptr(q), _stream(stream)),
           "fp8bs_selftest_encode_e4m3")
    return q


__all__ = ["fp8_quant_act_1x128", "fp8_quant_w_128x128", "fp8_quant_act_w", "fp8_gemm_blockscaled",
           "fp8_gemm_blockscaled_e4m3_out", "fp8_quant_tokens_1x128", "fp8_gemm_wgrad",
           "fp8_quant_act_1x128_gather", "FP8BS_ERR_INDEX",
           "fp8_grouped_gemm_blockscaled", "fp8bs_last_error", "fp8bs_selftest_wait_timeout",
           "fp8bs_selftest_set_wait_limit", "fp8_quant_per_tensor_workspace_size", "fp8_quant_per_tensor",
           "fp8_quant_per_tensor_delayed", "fp8_gemm_per_tensor", "fp8_quant_act_1x128_scatter", "packed_row_bytes", "fp8_ep_dispatch_pack", "fp8_ep_dispatch_pack_scatter",
           "fp8_ep_unpack", "fp8bs_gather_rows", "fp8bs_selftest_encode_e4m3", "Fp8bsError", "lib",
           "LIB_PATH", "EXPORTED", "B_KMAJOR", "B_MNMAJOR", "OUT_BF16", "OUT_FP32"]
