"""Helpers shared by the parity tests: host copies and the GEMM acceptance rule.

GEMM acceptance (normalised error against the float64 oracle):
    e[m, n] = |C_gpu[m, n] - C_ref[m, n]| / (||A^[m, :]||_2 * ||B^[n, :]||_2)
over the dequantised operands; pass if max e <= 2e-3 and mean e <= 1e-4, and
rows or columns whose dequantised norm is 0 must be exactly 0 on the GPU.
The bound on max e covers the BF16 output rounding (|C| <= ||a|| ||w||, so
rounding adds at most 2^-9 ~ 1.95e-3 in e).  The mean bound is for the error
beyond what the output format itself imposes: when a check passes the
normalised error of rounding the float64 reference to the output type
(``output_rounding_errors``), the mean bound is 1e-4 above that error's mean.
For BF16 output that share is about 2^-9 * 0.72 * E|cos(a, w)|: rounding to an
8-bit significand errs by a quarter ulp on average, significands spread
log-uniformly over [1, 2) (mean of 1/m = 0.72), and E|cos| = sqrt(2 / (pi K))
for independent rows.  That is 1.0e-4 at K = 128 and 2.5e-5 at K = 2048.
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


def output_rounding_errors(c_ref: np.ndarray, a_norms: np.ndarray, b_norms: np.ndarray, out_dtype):
    """Normalised error of rounding the float64 reference itself to the output
    type (None for FP32 output, whose rounding is far below the bounds)."""
    if out_dtype != torch.bfloat16:
        return None
    denom = np.outer(a_norms, b_norms)
    nz = denom != 0
    r = torch.from_numpy(np.ascontiguousarray(c_ref, dtype=np.float64)).to(torch.bfloat16).double().numpy()
    return np.abs(r - c_ref)[nz] / denom[nz]


def sampled_errors(c_gpu_vals, c_ref_vals, a_norm_vals, b_norm_vals):
    denom = a_norm_vals * b_norm_vals
    zero = denom == 0
    bad_zero = int(np.count_nonzero(np.asarray(c_gpu_vals)[zero] != 0))
    e = np.abs(np.asarray(c_gpu_vals) - np.asarray(c_ref_vals))[~zero] / denom[~zero]
    return e, bad_zero


def assert_gemm_ok(e: np.ndarray, bad_zero: int, what: str, max_e=MAX_E, mean_e=MEAN_E, e_out=None):
    assert bad_zero == 0, f"{what}: {bad_zero} zero-norm outputs are not exactly 0"
    if e.size == 0:
        return
    if e_out is not None and e_out.size:
        mean_e = mean_e + float(e_out.mean())
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


class ErrorStats:
    """Running max / mean of the normalised error over many slabs of one output,
    plus the count of zero-norm outputs that are not exactly 0."""

    def __init__(self, what):
        self.what, self.max, self.sum, self.n, self.bad_zero = what, 0.0, 0.0, 0, 0

    def add(self, c_gpu: np.ndarray, c_ref: np.ndarray, a_norms: np.ndarray, b_norms: np.ndarray):
        e, bad = gemm_errors(c_gpu, c_ref, a_norms, b_norms)
        self.bad_zero += bad
        if e.size:
            self.max = max(self.max, float(e.max()))
            self.sum += float(e.sum())
            self.n += int(e.size)

    @property
    def mean(self):
        return self.sum / self.n if self.n else 0.0

    def check(self, max_e=MAX_E, mean_e=MEAN_E):
        record_stats(self.what, self.max, self.mean, self.n)
        assert self.bad_zero == 0, f"{self.what}: {self.bad_zero} zero-norm outputs are not exactly 0"
        assert self.max <= max_e and self.mean <= mean_e, \
            f"{self.what}: max e {self.max:.3e} (<= {max_e}), mean e {self.mean:.3e} (<= {mean_e})"


def record_stats(what, max_e, mean_e, count):
    """Appends one JSON line per checked output to the file named by the
    PARITY_STATS environment variable, if set (a record of the errors seen)."""
    import json
    import os
    path = os.environ.get("PARITY_STATS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": what, "max_e": max_e, "mean_e": mean_e, "outputs": count}) + "\n")


def compare_by_slabs(what, c_gpu, ref_rows, a_norms, b_norms, row_ranges):
    """Every output element of the rows in `row_ranges` (a list of (r0, r1)),
    one slab at a time: ``ref_rows(r0, r1)`` returns the float64 oracle rows
    and ``c_gpu`` is the device output.  Returns the ErrorStats (checked)."""
    st = ErrorStats(what)
    for r0, r1 in row_ranges:
        got = c_gpu[r0:r1].double().cpu().numpy()
        st.add(got, ref_rows(r0, r1), a_norms[r0:r1], b_norms)
    st.check()
    return st


def slabs(r0, r1, rows):
    return [(a, min(a + rows, r1)) for a in range(r0, r1, rows)]


def assert_e4m3_out_within_bound(codes, scales, ref, a_norms, b_norms, dec_table):
    """Quantised-output check against the float64 oracle.  With x the BF16
    output value, s = amax_tile(|x|)/448 and v = x/s, the E4M3 code is within
    half a step of v: 2^-4 |v| in the normal range and 2^-10 below 2^-6.  So
    |dec(q)*s - x| <= 2^-4 |x| + 2^-10 s, and the GEMM acceptance bound
    E = 2e-3 ||a_m|| ||b_n|| covers |x - ref|.  codes [M][N] uint8, scales
    [N/128][M] float; returns the largest error / bound ratio."""
    M, N = ref.shape
    e_bound = MAX_E * np.outer(a_norms, b_norms)
    sc = np.asarray(scales, np.float64)
    deq = dec_table[codes] * np.repeat(sc.T, 128, axis=1)
    tiles = np.abs(ref).reshape(M, N // 128, 128)
    amax_ref = np.repeat(tiles.max(axis=2), 128, axis=1)
    e_tile = np.repeat(e_bound.reshape(M, N // 128, 128).max(axis=2), 128, axis=1)
    bound = (2.0 ** -4) * (np.abs(ref) + e_bound) + (amax_ref + e_tile) / (448.0 * 1024.0) * 1.001 \
        + e_bound * 1.001 + 1e-7 * np.abs(ref)
    err = np.abs(deq - ref)
    assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e}"
    sc_ref = tiles.max(axis=2).T / 448.0
    et = e_bound.reshape(M, N // 128, 128).max(axis=2).T / 448.0
    assert np.all(np.abs(sc - sc_ref) <= et + 2e-7 * sc_ref)
    return float(np.max(err / np.maximum(bound, 1e-300)))
