"""Helpers shared by the parity tests: host copies and the GEMM acceptance rule.

GEMM acceptance (normalised error against the float64 oracle):
    e[m, n] = |C_gpu[m, n] - C_ref[m, n]| / (||A^[m, :]||_2 * ||B^[n, :]||_2)
over the dequantised operands; pass if max e <= 2e-3 and mean e <= 1e-4, and
rows or columns whose dequantised norm is 0 must be exactly 0 on the GPU.
The bound on max e covers the BF16 output rounding (|C| <= ||a|| ||w||, so
rounding adds at most 2^-9 ~ 1.95e-3 in e); the mean bound leaves about half
of its budget to accumulation error after the BF16 rounding's mean share.
"""
import numpy as np
import torch

MAX_E = 2e-3
MEAN_E = 1e-4


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint8)


def host_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.float32, copy=False)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def gemm_errors(c_gpu: np.ndarray, c_ref: np.ndarray, a_norms: np.ndarray, b_norms: np.ndarray):
    """Normalised errors of full matrices; returns (e array, zero-norm violations)."""
    denom = np.outer(a_norms, b_norms)
    zero = denom == 0
    bad_zero = int(np.count_nonzero(c_gpu[zero] != 0))
    e = np.abs(c_gpu - c_ref)[~zero] / denom[~zero]
    return e, bad_zero


def sampled_errors(c_gpu_vals, c_ref_vals, a_norm_vals, b_norm_vals):
    denom = a_norm_vals * b_norm_vals
    zero = denom == 0
    bad_zero = int(np.count_nonzero(np.asarray(c_gpu_vals)[zero] != 0))
    e = np.abs(np.asarray(c_gpu_vals) - np.asarray(c_ref_vals))[~zero] / denom[~zero]
    return e, bad_zero


def assert_gemm_ok(e: np.ndarray, bad_zero: int, what: str, max_e=MAX_E, mean_e=MEAN_E):
    assert bad_zero == 0, f"{what}: {bad_zero} zero-norm outputs are not exactly 0"
    if e.size == 0:
        return
    mx, mn = float(e.max()), float(e.mean())
    assert mx <= max_e and mn <= mean_e, f"{what}: max e {mx:.3e} (<= {max_e}), mean e {mn:.3e} (<= {mean_e})"


def b_norms_at(oracle, qb: np.ndarray, sb: np.ndarray, cols, b_major: int = 0) -> np.ndarray:
    """||B^[n, :]||_2 for each n in ``cols`` (one oracle call per distinct n, so
    each call sees a one-row operand with its own scale row)."""
    cols = np.asarray(cols)
    uc, inv = np.unique(cols, return_inverse=True)
    out = np.empty(len(uc))
    for i, n in enumerate(uc):
        nb = n // 128
        if b_major == 0:
            out[i] = oracle.b_row_norms(np.ascontiguousarray(qb[n:n + 1]),
                                        np.ascontiguousarray(sb[nb:nb + 1]))[0]
        else:
            out[i] = oracle.b_row_norms(np.ascontiguousarray(qb[:, n:n + 1]),
                                        np.ascontiguousarray(sb[:, nb:nb + 1]), b_major=1)[0]
    return out[inv]
