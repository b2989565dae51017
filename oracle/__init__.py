"""CPU oracle for the fine-grained FP8 block-scaled GEMM path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library (``fp8_fine_grained_26_b300``) never imports, links or loads it, and
the two share no code: this is a ctypes wrapper over ``fp8_oracle.c``, a plain
C restatement of the method (see that file's header for the passages it
follows).

All arrays are numpy arrays on the host:
  * bf16 inputs are passed as ``uint16`` bit patterns,
  * E4M3 codes are ``uint8``,
  * scales are ``float32``, GEMM results ``float64``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode_n.argtypes = [p, i64, p]
        lib.oracle_e4m3_encode_n.restype = None
        lib.oracle_quant_act_1x128.argtypes = [p, i64, i64, i64, p, i64, p]
        lib.oracle_quant_w_128x128.argtypes = [p, i64, i64, i64, p, i64, p]
        lib.oracle_gemm_f64.argtypes = [p, p, i64, p, p, i64, ctypes.c_int, i64, i64, i64, p, i64]
        lib.oracle_gemm_f64_at.argtypes = [p, p, i64, p, p, i64, ctypes.c_int, i64, i64, i64,
                                           p, p, i64, p]
        lib.oracle_grouped_gemm_f64.argtypes = [p, p, i64, p, p, p, ctypes.c_int, i64, i64, i64,
                                                p, i64]
        lib.oracle_gemm_f64_tokens.argtypes = [p, p, i64, p, p, i64, i64, i64, i64, p, i64]
        lib.oracle_act_row_norms.argtypes = [p, p, i64, i64, i64, p]
        lib.oracle_act_row_norms.restype = None
        lib.oracle_b_row_norms.argtypes = [p, p, i64, ctypes.c_int, i64, i64, p]
        lib.oracle_b_row_norms.restype = None
        lib.oracle_quant_per_tensor.argtypes = [p, i64, i64, i64, p, i64, p]
        lib.oracle_quant_per_tensor.restype = ctypes.c_int
        lib.oracle_quant_per_tensor_delayed.argtypes = [p, i64, i64, i64, ctypes.c_float, p, i64, p, p]
        lib.oracle_quant_per_tensor_delayed.restype = ctypes.c_int
        lib.oracle_gemm_f64_per_tensor.argtypes = [p, ctypes.c_float, i64, p, ctypes.c_float, i64, ctypes.c_int,
                                                   i64, i64, i64, p, i64]
        lib.oracle_gemm_f64_per_tensor.restype = ctypes.c_int
        lib.oracle_gemm_bf16_f64.argtypes = [p, i64, p, i64, ctypes.c_int, i64, i64, i64, p, i64]
        lib.oracle_gemm_bf16_f64.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_threads.restype = None
        lib.oracle_get_threads.argtypes = []
        lib.oracle_get_threads.restype = ctypes.c_int
        for f in ("oracle_quant_act_1x128", "oracle_quant_w_128x128", "oracle_gemm_f64",
                  "oracle_gemm_f64_at", "oracle_grouped_gemm_f64", "oracle_gemm_f64_tokens"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (status {rc})")


def _as_c(a, dtype):
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def set_threads(n: int) -> None:
    """Number of OpenMP threads the GEMMs and row norms use (0 = all the
    process may use).  Threads take whole output rows; each output element is
    the same in-order sum over k on one thread, so results do not depend on it."""
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    """Threads the GEMMs currently use."""
    return int(_load().oracle_get_threads())


def e4m3_encode(v: float) -> int:
    """E4M3 code of one finite fp32 value (RNE, saturating to +-448)."""
    return int(_load().oracle_e4m3_encode(ctypes.c_float(v)))


def e4m3_decode(c: int) -> float:
    """Exact value of one E4M3 code (NaN for S.1111.111)."""
    return float(_load().oracle_e4m3_decode(ctypes.c_uint8(c)))


def e4m3_encode_array(v) -> np.ndarray:
    """Element-wise ``e4m3_encode`` of a float32 array."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32).ravel())
    out = np.empty(v.shape[0], np.uint8)
    _load().oracle_e4m3_encode_n(_ptr(v), v.shape[0], _ptr(out))
    return out


def e4m3_decode_table() -> np.ndarray:
    """float64 value of every code 0..255."""
    lib = _load()
    return np.array([lib.oracle_e4m3_decode(ctypes.c_uint8(c)) for c in range(256)])


def quant_act_1x128(x_bf16_bits):
    """1x128 tile quantisation of a bf16 ``[M, K]`` matrix (given as uint16 bits).

    Returns ``(q uint8 [M, K], sA float32 [K/128, M])``."""
    x = _as_c(x_bf16_bits, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    _check(_load().oracle_quant_act_1x128(_ptr(x), M, K, K, _ptr(q), K, _ptr(s)), "quant_act")
    return q, s


def quant_tokens_1x128(x_bf16_bits):
    """1x128 tiles along the token (row) dimension of a bf16 ``[T, F]`` matrix:
    each feature column is cut into runs of 128 tokens, each with its own scale
    -- the operands of the weight-gradient GEMM, whose contraction runs over
    tokens.  By definition this is the 1x128 row quantisation of the
    transposed matrix.

    Returns ``(q uint8 [F, T], s float32 [T/128, F])``."""
    x = _as_c(x_bf16_bits, np.uint16)
    return quant_act_1x128(np.ascontiguousarray(x.T))


def quant_w_128x128(w_bf16_bits):
    """128x128 block quantisation of a bf16 ``[R, C]`` matrix (uint16 bits).

    Returns ``(q uint8 [R, C], sW float32 [ceil(R/128), C/128])``."""
    w = _as_c(w_bf16_bits, np.uint16)
    R, C = w.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty(((R + 127) // 128, C // 128), np.float32)
    _check(_load().oracle_quant_w_128x128(_ptr(w), R, C, C, _ptr(q), C, _ptr(s)), "quant_w")
    return q, s


def _gemm_shapes(qA, qB, b_major):
    M, K = qA.shape
    if b_major == 0:
        N, Kb = qB.shape
    else:
        Kb, N = qB.shape
    if Kb != K:
        raise ValueError("K mismatch")
    return M, N, K


def gemm_f64(qA, sA, qB, sB, b_major: int = 0) -> np.ndarray:
    """float64 ``C = A^ . B^T`` over the dequantised operands.

    ``b_major`` 0: ``qB`` is ``[N, K]`` with ``sB [ceil(N/128), K/128]``;
    ``b_major`` 1: ``qB`` is ``[K, N]`` with ``sB [K/128, ceil(N/128)]``."""
    qA, sA = _as_c(qA, np.uint8), _as_c(sA, np.float32)
    qB, sB = _as_c(qB, np.uint8), _as_c(sB, np.float32)
    M, N, K = _gemm_shapes(qA, qB, b_major)
    C = np.empty((M, N), np.float64)
    ldb = qB.shape[1]
    _check(_load().oracle_gemm_f64(_ptr(qA), _ptr(sA), K, _ptr(qB), _ptr(sB), ldb, b_major,
                                   M, N, K, _ptr(C), N), "gemm")
    return C


def gemm_f64_at(qA, sA, qB, sB, rows, cols, b_major: int = 0) -> np.ndarray:
    """The float64 GEMM evaluated only at positions ``(rows[i], cols[i])``."""
    qA, sA = _as_c(qA, np.uint8), _as_c(sA, np.float32)
    qB, sB = _as_c(qB, np.uint8), _as_c(sB, np.float32)
    rows = _as_c(np.asarray(rows, np.int64), np.int64)
    cols = _as_c(np.asarray(cols, np.int64), np.int64)
    M, N, K = _gemm_shapes(qA, qB, b_major)
    out = np.empty(rows.shape[0], np.float64)
    ldb = qB.shape[1]
    _check(_load().oracle_gemm_f64_at(_ptr(qA), _ptr(sA), K, _ptr(qB), _ptr(sB), ldb, b_major,
                                      M, N, K, _ptr(rows), _ptr(cols), rows.shape[0], _ptr(out)),
           "gemm_at")
    return out


def grouped_gemm_f64(qA, sA, qB, sB, offsets) -> np.ndarray:
    """Per-expert float64 GEMM: rows ``[off[e], off[e+1])`` of ``A`` times
    expert ``e``'s ``qB[e] [N, K]`` (scales ``sB[e] [ceil(N/128), K/128]``)."""
    qA, sA = _as_c(qA, np.uint8), _as_c(sA, np.float32)
    qB, sB = _as_c(qB, np.uint8), _as_c(sB, np.float32)
    off = _as_c(np.asarray(offsets, np.int32), np.int32)
    M, K = qA.shape
    E, N, Kb = qB.shape
    if Kb != K or off.shape[0] != E + 1 or off[0] != 0 or off[-1] != M:
        raise ValueError("bad grouped shapes/offsets")
    C = np.zeros((M, N), np.float64)
    _check(_load().oracle_grouped_gemm_f64(_ptr(qA), _ptr(sA), K, _ptr(qB), _ptr(sB), _ptr(off),
                                           E, M, N, K, _ptr(C), N), "grouped_gemm")
    return C


def gemm_f64_tokens(qA, sA, qB, sB) -> np.ndarray:
    """float64 ``C = A^ . B^T`` where both operands carry 1x128 scales along K:
    ``qA [M, K]`` with ``sA [K/128, M]`` and ``qB [N, K]`` with ``sB [K/128, N]``
    (the weight-gradient GEMM dW = dY^T . X over tokens)."""
    qA, sA = _as_c(qA, np.uint8), _as_c(sA, np.float32)
    qB, sB = _as_c(qB, np.uint8), _as_c(sB, np.float32)
    M, K = qA.shape
    N, Kb = qB.shape
    if Kb != K or sA.shape != (K // 128, M) or sB.shape != (K // 128, N):
        raise ValueError("shape mismatch")
    C = np.empty((M, N), np.float64)
    _check(_load().oracle_gemm_f64_tokens(_ptr(qA), _ptr(sA), K, _ptr(qB), _ptr(sB), K, M, N, K,
                                          _ptr(C), N), "gemm_tokens")
    return C


def quant_per_tensor(x_bf16_bits):
    """Per-tensor quantisation with the tensor's own amax (current scaling):
    one scale fp32(amax/448) for every element.  Returns ``(q uint8 [R, C],
    scale float32)``."""
    x = _as_c(x_bf16_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty(1, np.float32)
    _check(_load().oracle_quant_per_tensor(_ptr(x), R, C, C, _ptr(q), C, _ptr(s)), "quant_per_tensor")
    return q, np.float32(s[0])


def quant_per_tensor_delayed(x_bf16_bits, amax_in):
    """Per-tensor quantisation with a given amax (delayed scaling): scale =
    fp32(amax_in/448), larger values saturate.  Returns ``(q, scale, amax of
    this tensor)``."""
    x = _as_c(x_bf16_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty(1, np.float32)
    a = np.empty(1, np.float32)
    _check(_load().oracle_quant_per_tensor_delayed(_ptr(x), R, C, C, ctypes.c_float(float(amax_in)), _ptr(q), C,
                                                   _ptr(s), _ptr(a)), "quant_per_tensor_delayed")
    return q, np.float32(s[0]), np.float32(a[0])


def gemm_f64_per_tensor(qA, sA, qB, sB, b_major: int = 0) -> np.ndarray:
    """float64 ``C = (sA qA^) . (sB qB^)^T`` for per-tensor scales sA, sB
    (scalars); ``qB`` is ``[N, K]`` (b_major 0) or ``[K, N]`` (b_major 1)."""
    qA, qB = _as_c(qA, np.uint8), _as_c(qB, np.uint8)
    M, N, K = _gemm_shapes(qA, qB, b_major)
    C = np.empty((M, N), np.float64)
    _check(_load().oracle_gemm_f64_per_tensor(_ptr(qA), ctypes.c_float(float(sA)), K, _ptr(qB),
                                              ctypes.c_float(float(sB)), qB.shape[1], b_major, M, N, K,
                                              _ptr(C), N), "gemm_per_tensor")
    return C


def gemm_bf16_f64(a_bits, b_bits, b_major: int = 0) -> np.ndarray:
    """float64 product of the UNQUANTISED BF16 inputs (uint16 bits): ``a [M,
    K]`` times ``b [N, K]`` (b_major 0) or stored ``[K, N]`` (b_major 1)."""
    a, b = _as_c(a_bits, np.uint16), _as_c(b_bits, np.uint16)
    M, K = a.shape
    N = b.shape[0] if b_major == 0 else b.shape[1]
    if (b.shape[1] if b_major == 0 else b.shape[0]) != K:
        raise ValueError("K mismatch")
    C = np.empty((M, N), np.float64)
    _check(_load().oracle_gemm_bf16_f64(_ptr(a), K, _ptr(b), b.shape[1], b_major, M, N, K, _ptr(C), N),
           "gemm_bf16")
    return C


def act_row_norms(qA, sA) -> np.ndarray:
    """||A^[m, :]||_2 of the dequantised activation rows."""
    qA, sA = _as_c(qA, np.uint8), _as_c(sA, np.float32)
    M, K = qA.shape
    out = np.empty(M, np.float64)
    _load().oracle_act_row_norms(_ptr(qA), _ptr(sA), K, M, K, _ptr(out))
    return out


def b_row_norms(qB, sB, b_major: int = 0) -> np.ndarray:
    """||B^[n, :]||_2 of the dequantised weight rows (rows of B^T's transpose)."""
    qB, sB = _as_c(qB, np.uint8), _as_c(sB, np.float32)
    if b_major == 0:
        N, K = qB.shape
    else:
        K, N = qB.shape
    out = np.empty(N, np.float64)
    _load().oracle_b_row_norms(_ptr(qB), _ptr(sB), qB.shape[1], b_major, N, K, _ptr(out))
    return out


__all__ = ["set_threads", "get_threads", "e4m3_encode", "e4m3_decode", "e4m3_encode_array", "e4m3_decode_table",
           "quant_act_1x128", "quant_w_128x128", "gemm_f64", "gemm_f64_at",
           "grouped_gemm_f64", "act_row_norms", "b_row_norms", "quant_per_tensor",
           "quant_per_tensor_delayed", "gemm_f64_per_tensor", "gemm_bf16_f64"]
