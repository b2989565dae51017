"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself:
  * torch's own float8_e4m3fn conversion (an independent E4M3 implementation)
    for decoding every code and for encoding values below the rounding
    boundary to 480;
  * closed forms: saturation, ties-to-even midpoints, exact power-of-two
    scales, constant and all-zero tiles, the E4M3 rounding-error bound;
  * invariants the method fixes: the amax element maps to +-448, locality of
    each 1x128 tile / 128x128 block (tile sizes read from the golden fixture
    that cites the pages), quantise-then-gather == gather-then-quantise,
    transposing a weight transposes its block grid;
  * numpy float64 matmul on dequantised operands decoded by torch (brute force
    on tiny shapes), and exact-arithmetic cases.
Each group is chosen so that a plausible slip in the oracle (wrong exponent
bias, rounding direction, subnormal formula, scale index, transposed operand,
dropped block) fails at least one test here.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from synthetic import bf16_bits, dense_case, normal_bf16, generator

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fine_grained_tiling.txt")


def golden_tiling():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def torch_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_encode(v: np.ndarray) -> np.ndarray:
    """torch float32 -> float8_e4m3fn (round to nearest even; NaN above 464)."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def f32_bits_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 values that are exactly representable in bf16 -> bf16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not representable in bf16"
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- E4M3 codec
def test_decode_matches_torch_for_all_codes():
    ours = oracle.e4m3_decode_table()
    ref = torch_decode(np.arange(256, dtype=np.uint8))
    nan_codes = {0x7F, 0xFF}
    for c in range(256):
        if c in nan_codes:
            assert np.isnan(ours[c]) and np.isnan(ref[c])
        else:
            assert ours[c] == ref[c], hex(c)
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0
    assert ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_roundtrip_every_finite_code():
    table = oracle.e4m3_decode_table()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = np.float32(table[c])
        if c == 0x80:
            v = np.float32(-0.0)
        assert oracle.e4m3_encode(float(v)) == c, hex(c)


def _structured_values():
    """Every finite E4M3 value, every midpoint between neighbours, and the
    fp32 values one and two ulps either side of each midpoint."""
    table = oracle.e4m3_decode_table()
    pos = np.array(sorted({table[c] for c in range(0x7F)}))      # 0 .. 448
    mids = (pos[:-1] + pos[1:]) / 2.0                             # exact in fp32
    vals = [pos.astype(np.float32), mids.astype(np.float32)]
    m32 = mids.astype(np.float32)
    for k in (1, 2):
        up, dn = m32.copy(), m32.copy()
        for _ in range(k):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(0))
        vals += [up, dn]
    # below the smallest subnormal's half, around it, and the 448..464 band
    vals.append(np.array([2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11, 1e-30, 1e-45,
                          448.0, 449.0, 456.0, 463.9], np.float32))
    v = np.concatenate(vals)
    return np.concatenate([v, -v])


def test_encode_matches_torch_structured():
    v = _structured_values()
    assert np.all(np.abs(v) < 464)
    np.testing.assert_array_equal(oracle.e4m3_encode_array(v), torch_encode(v))


def test_encode_matches_torch_random_fp32():
    rng = np.random.default_rng(1234)
    # random bit patterns over the whole finite range below 464, incl. fp32 subnormals
    bits = rng.integers(0, 0x43E80000, size=2_000_000, dtype=np.uint32)
    v = bits.view(np.float32)
    v = np.concatenate([v, -v, rng.uniform(-464, 464, 500_000).astype(np.float32)])
    v = v[np.abs(v) < 464]
    np.testing.assert_array_equal(oracle.e4m3_encode_array(v), torch_encode(v))


def test_encode_saturates_finite():
    big = np.array([448.0, 450.0, 463.99, 464.0, 470.0, 480.0, 1e6, 3.4e38], np.float32)
    assert np.all(oracle.e4m3_encode_array(big) == 0x7E)
    assert np.all(oracle.e4m3_encode_array(-big) == 0xFE)


def test_ties_go_to_even_code():
    table = oracle.e4m3_decode_table()
    for c in range(0, 0x7E):
        lo, hi = table[c], table[c + 1]
        mid = np.float32((lo + hi) / 2)
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(mid)) == want, hex(c)
        assert oracle.e4m3_encode(float(-mid)) == (want | 0x80)


def test_signed_zero_and_underflow_keep_sign():
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-30) == 0x80
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00          # tie between 0 and 2^-9 -> even
    assert oracle.e4m3_encode(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 0x01


# ---------------------------------------------------------------- quantisers
def _random_act(M, K, seed=0, std=1.0):
    g = generator(seed, "cpu")
    return bf16_bits(normal_bf16((M, K), std, g, "cpu", outlier_p=0.01, outlier_scale=50.0))


def test_scale_is_ieee_fp32_division_of_amax():
    x = _random_act(64, 512)
    q, s = oracle.quant_act_1x128(x)
    xf = bf16_bits_to_f32(x).reshape(64, 4, 128)
    amax = np.abs(xf).max(axis=2).T                       # [KB, M]
    np.testing.assert_array_equal(s, amax / np.float32(448.0))
    # binary64 then one rounding to binary32 is the same correctly-rounded
    # quotient for binary32 operands (53 >= 2*24 + 2)
    np.testing.assert_array_equal(s, (amax.astype(np.float64) / 448.0).astype(np.float32))


def test_quant_act_matches_numpy_division_and_torch_encoder():
    x = _random_act(96, 384, seed=3)
    q, s = oracle.quant_act_1x128(x)
    xf = bf16_bits_to_f32(x).reshape(96, 3, 128)
    y = xf / s.T[:, :, None]                                # numpy IEEE fp32 division
    assert np.all(np.abs(y) < 464)
    np.testing.assert_array_equal(q.reshape(96, 3, 128), torch_encode(y).reshape(96, 3, 128))


def test_amax_element_maps_to_448():
    x = _random_act(128, 1024, seed=5)
    q, s = oracle.quant_act_1x128(x)
    xf = bf16_bits_to_f32(x).reshape(128, 8, 128)
    idx = np.abs(xf).argmax(axis=2)
    qm = np.take_along_axis(q.reshape(128, 8, 128), idx[:, :, None], axis=2)[:, :, 0]
    sign = np.take_along_axis(xf, idx[:, :, None], axis=2)[:, :, 0] < 0
    assert np.all(qm == np.where(sign, 0xFE, 0x7E))


def test_constant_and_zero_tiles():
    M, K = 4, 256
    x = np.zeros((M, K), np.float32)
    x[0, :128] = 3.0
    x[1, :128] = -0.15625
    x[2, 128:] = -0.0                                      # all-zero tile with -0
    x[3, :] = 0.0
    h = f32_bits_to_bf16_bits(x)
    q, s = oracle.quant_act_1x128(h)
    assert s[0, 0] == np.float32(3.0) / np.float32(448.0) and np.all(q[0, :128] == 0x7E)
    assert s[0, 1] == np.float32(0.15625) / np.float32(448.0) and np.all(q[1, :128] == 0xFE)
    assert s[1, 2] == 0.0 and np.all(q[2, 128:] == 0x80)
    assert s[0, 3] == 0.0 and s[1, 3] == 0.0 and np.all(q[3] == 0x00)
    assert np.all(q[0, 128:] == 0x00) and s[1, 0] == 0.0


@pytest.mark.parametrize("k", [-20, -7, -1, 0, 3, 12])
def test_power_of_two_amax_gives_exact_scale(k):
    g = generator(7 + k + 20, "cpu")
    xf = bf16_bits_to_f32(bf16_bits(normal_bf16((8, 128), 2.0 ** k * 100.0, g, "cpu")))
    xf = np.clip(xf, -(448.0 * 2.0 ** k) * 0.999, 448.0 * 2.0 ** k * 0.999).astype(np.float32)
    xf = bf16_bits_to_f32(f32_bits_to_bf16_bits(
        (np.ascontiguousarray(xf).view(np.uint32) & 0xFFFF0000).view(np.float32)))
    xf[:, 17] = np.float32(448.0 * 2.0 ** k)
    xf[3, 17] = np.float32(-448.0 * 2.0 ** k)
    q, s = oracle.quant_act_1x128(f32_bits_to_bf16_bits(xf))
    assert np.all(s == np.float32(2.0 ** k))
    np.testing.assert_array_equal(q, torch_encode(xf * np.float32(2.0 ** -k)).reshape(q.shape))


def test_dequantised_error_within_e4m3_bound():
    x = _random_act(64, 512, seed=11, std=3.0)
    q, s = oracle.quant_act_1x128(x)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    deq = torch_decode(q) * np.repeat(s.T, 128, axis=1).astype(np.float64)
    sc = np.repeat(s.T, 128, axis=1).astype(np.float64)
    bound = (2.0 ** -4 * np.abs(xf) + 2.0 ** -10 * sc) * (1 + 2.0 ** -20)
    assert np.all(np.abs(deq - xf) <= bound)


def test_subnormal_scales_are_kept():
    x = np.zeros((2, 128), np.float32)
    x[0, 5] = np.float32(2.0 ** -130)                      # bf16 subnormal
    x[1, 9] = np.float32(-1.5 * 2.0 ** -120)
    q, s = oracle.quant_act_1x128(f32_bits_to_bf16_bits(x))
    assert s[0, 0] > 0 and s[0, 1] > 0
    assert s[0, 0] == np.float32(2.0 ** -130) / np.float32(448.0)
    assert s[0, 1] == np.float32(1.5 * 2.0 ** -120) / np.float32(448.0)
    assert q[0, 5] == 0x7E and q[1, 9] == 0xFE


def test_act_tile_locality_matches_golden_geometry():
    geo = golden_tiling()
    tc = geo["act_tile_cols"]
    assert geo["act_tile_rows"] == 1
    x = _random_act(8, 4 * tc, seed=21)
    q0, s0 = oracle.quant_act_1x128(x)
    assert s0.shape == (4, 8)
    for col in (tc - 1, tc, 3 * tc - 1):
        x1 = x.copy()
        x1[5, col] = f32_bits_to_bf16_bits(np.array([1000.0], np.float32))[0]
        q1, s1 = oracle.quant_act_1x128(x1)
        kb = col // tc
        changed_s = np.argwhere(s1 != s0)
        assert changed_s.tolist() == [[kb, 5]]
        rows, cols = np.nonzero(q1 != q0)
        assert set(rows.tolist()) == {5}
        assert cols.min() >= kb * tc and cols.max() < (kb + 1) * tc


def test_quantise_then_gather_equals_gather_then_quantise():
    x = _random_act(50, 256, seed=31)
    rows = np.array([7, 7, 0, 49, 13, 2, 13, 30])
    q, s = oracle.quant_act_1x128(x)
    qg, sg = oracle.quant_act_1x128(x[rows])
    np.testing.assert_array_equal(qg, q[rows])
    np.testing.assert_array_equal(sg, s[:, rows])


def _random_w(R, C, seed=0):
    g = generator(seed, "cpu")
    return bf16_bits(normal_bf16((R, C), 0.02, g, "cpu", outlier_p=0.001, outlier_scale=30.0))


def test_weight_block_geometry_scale_and_locality():
    geo = golden_tiling()
    br, bc = geo["weight_block_rows"], geo["weight_block_cols"]
    w = _random_w(3 * br, 2 * bc, seed=41)
    q, s = oracle.quant_w_128x128(w)
    wf = bf16_bits_to_f32(w).reshape(3, br, 2, bc)
    amax = np.abs(wf).max(axis=(1, 3))
    np.testing.assert_array_equal(s, amax / np.float32(448.0))
    y = wf / s[:, None, :, None]
    np.testing.assert_array_equal(q.reshape(3, br, 2, bc), torch_encode(y).reshape(3, br, 2, bc))
    w1 = w.copy()
    w1[br, bc - 1] = f32_bits_to_bf16_bits(np.array([5.0], np.float32))[0]
    q1, s1 = oracle.quant_w_128x128(w1)
    assert np.argwhere(s1 != s).tolist() == [[1, 0]]
    r, c = np.nonzero(q1 != q)
    assert r.min() >= br and r.max() < 2 * br and c.max() < bc


def test_weight_partial_row_block_uses_existing_rows_only():
    w = _random_w(200, 256, seed=43)
    q, s = oracle.quant_w_128x128(w)
    assert s.shape == (2, 2)
    pad = np.zeros((256, 256), np.uint16)                   # +0 padding leaves amax unchanged
    pad[:200] = w
    qp, sp = oracle.quant_w_128x128(pad)
    np.testing.assert_array_equal(s, sp)
    np.testing.assert_array_equal(q, qp[:200])
    tail = np.abs(bf16_bits_to_f32(w[128:])).reshape(72, 2, 128).max(axis=(0, 2))
    np.testing.assert_array_equal(s[1], tail / np.float32(448.0))


def test_weight_transpose_invariance():
    w = _random_w(256, 384, seed=47)
    q, s = oracle.quant_w_128x128(w)
    qt, st = oracle.quant_w_128x128(np.ascontiguousarray(w.T))
    np.testing.assert_array_equal(qt, q.T)
    np.testing.assert_array_equal(st, s.T)


# ---------------------------------------------------------------- GEMM
def _deq_np(q, s_rows_by_k):
    return torch_decode(q) * s_rows_by_k


def _tiny_operands(M, N, K, seed):
    c = dense_case("pin", M, N, K, seed=seed)
    qa, sa = oracle.quant_act_1x128(bf16_bits(c.a))
    qb, sb = oracle.quant_w_128x128(bf16_bits(c.w))
    return qa, sa, qb, sb


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (3, 5, 128), (8, 8, 256), (5, 130, 256)])
def test_gemm_matches_numpy_matmul_of_torch_dequantised(M, N, K):
    qa, sa, qb, sb = _tiny_operands(M, N, K, seed=M * 100 + N)
    A = torch_decode(qa) * np.repeat(sa.T, 128, axis=1).astype(np.float64)
    sb_full = np.repeat(np.repeat(sb, 128, axis=0)[:N], 128, axis=1).astype(np.float64)
    B = torch_decode(qb) * sb_full
    ref = A @ B.T
    got = oracle.gemm_f64(qa, sa, qb, sb)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-300)
    # brute-force triple loop over the torch-decoded values
    for m in range(min(M, 3)):
        for n in range(min(N, 3)):
            acc = 0.0
            for k in range(K):
                acc += A[m, k] * B[n, k]
            assert abs(got[m, n] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_gemm_constant_blocks_closed_form():
    # every 1x128 tile of A constant and every 128x128 block of B constant in
    # magnitude: all codes are +-448, so C = sum_kb 128 * 448^2 * sA*sB*sign
    M, N, K = 3, 4, 384
    a = np.zeros((M, K), np.float32)
    b = np.zeros((N, K), np.float32)
    av = [0.5, -2.0, 3.0]
    bv = [0.25, -1.0, 0.75]
    for kb in range(3):
        for m in range(M):
            a[m, kb * 128:(kb + 1) * 128] = av[(m + kb) % 3] * (m + 1)
        for n in range(N):
            b[n, kb * 128:(kb + 1) * 128] = bv[kb] * (-1.0 if n % 2 else 1.0)
    qa, sa = oracle.quant_act_1x128(f32_bits_to_bf16_bits(a))
    qb, sb = oracle.quant_w_128x128(f32_bits_to_bf16_bits(b))
    got = oracle.gemm_f64(qa, sa, qb, sb)
    for m in range(M):
        for n in range(N):
            want = 0.0
            for kb in range(3):
                sgn = float(np.sign(a[m, kb * 128]) * np.sign(b[n, kb * 128]))
                want += 128 * 448.0 * 448.0 * float(sa[kb, m]) * float(sb[0, kb]) * sgn
            assert got[m, n] == pytest.approx(want, rel=1e-14)


def test_gemm_exact_powers_of_two():
    # codes in {0, +-2^j}, power-of-two data: the result is an exact small integer
    rng = np.random.default_rng(5)
    M, N, K = 6, 7, 256
    a = rng.choice([0.0, 1.0, -1.0, 2.0, -0.5, 448.0], size=(M, K)).astype(np.float32)
    b = rng.choice([0.0, 1.0, -1.0, 4.0, -0.25, 448.0], size=(N, K)).astype(np.float32)
    a[:, 0] = 448.0
    a[:, 128] = 448.0
    b[:, 0] = 448.0
    b[:, 128] = 448.0
    qa, sa = oracle.quant_act_1x128(f32_bits_to_bf16_bits(a))
    qb, sb = oracle.quant_w_128x128(f32_bits_to_bf16_bits(b))
    assert np.all(sa == 1.0) and np.all(sb == 1.0)
    got = oracle.gemm_f64(qa, sa, qb, sb)
    want = a.astype(np.float64) @ b.astype(np.float64).T
    np.testing.assert_array_equal(got, want)


def test_gemm_mn_major_b_equals_k_major():
    qa, sa, qb, sb = _tiny_operands(4, 256, 256, seed=77)
    c_k = oracle.gemm_f64(qa, sa, qb, sb, b_major=0)
    qbt, sbt = np.ascontiguousarray(qb.T), np.ascontiguousarray(sb.T)
    c_mn = oracle.gemm_f64(qa, sa, qbt, sbt, b_major=1)
    np.testing.assert_array_equal(c_k, c_mn)


def test_gemm_at_matches_full():
    qa, sa, qb, sb = _tiny_operands(9, 140, 256, seed=13)
    full = oracle.gemm_f64(qa, sa, qb, sb)
    rows = np.array([0, 8, 3, 4])
    cols = np.array([139, 0, 128, 77])
    np.testing.assert_array_equal(oracle.gemm_f64_at(qa, sa, qb, sb, rows, cols), full[rows, cols])


def test_grouped_equals_per_expert_dense():
    rng = np.random.default_rng(9)
    counts = [3, 0, 5, 1, 0]
    E, N, K = len(counts), 136, 256
    M = sum(counts)
    qa, sa = oracle.quant_act_1x128(_random_act(M, K, seed=2))
    qbs, sbs = [], []
    for e in range(E):
        qb, sb = oracle.quant_w_128x128(_random_w(N, K, seed=100 + e))
        qbs.append(qb)
        sbs.append(sb)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    got = oracle.grouped_gemm_f64(qa, sa, np.stack(qbs), np.stack(sbs), off)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        A = torch_decode(qa[r0:r1]) * np.repeat(sa[:, r0:r1].T, 128, axis=1)
        sbf = np.repeat(np.repeat(sbs[e], 128, axis=0)[:N], 128, axis=1)
        B = torch_decode(qbs[e]) * sbf
        np.testing.assert_allclose(got[r0:r1], A @ B.T, rtol=1e-12, atol=1e-300)
    del rng


def test_row_norms_match_numpy():
    qa, sa, qb, sb = _tiny_operands(5, 200, 256, seed=17)
    A = torch_decode(qa) * np.repeat(sa.T, 128, axis=1)
    B = torch_decode(qb) * np.repeat(np.repeat(sb, 128, axis=0)[:200], 128, axis=1)
    np.testing.assert_allclose(oracle.act_row_norms(qa, sa), np.linalg.norm(A, axis=1), rtol=1e-13)
    np.testing.assert_allclose(oracle.b_row_norms(qb, sb), np.linalg.norm(B, axis=1), rtol=1e-13)
    np.testing.assert_allclose(oracle.b_row_norms(np.ascontiguousarray(qb.T),
                                                  np.ascontiguousarray(sb.T), b_major=1),
                               np.linalg.norm(B, axis=1), rtol=1e-13)


def test_oracle_rejects_k_not_multiple_of_128():
    with pytest.raises(ValueError):
        oracle.quant_act_1x128(np.zeros((2, 100), np.uint16))


# ---- weight-gradient GEMM: both operands with 1x128 scales along the tokens
def _token_operands(T, M, N, seed):
    g = generator(seed, "cpu")
    dy = normal_bf16((T, M), 1.0, g, "cpu")
    x = normal_bf16((T, N), 1.0, g, "cpu", outlier_p=0.01, outlier_scale=20.0)
    qa, sa = oracle.quant_tokens_1x128(bf16_bits(dy))
    qb, sb = oracle.quant_tokens_1x128(bf16_bits(x))
    return dy, x, qa, sa, qb, sb


def test_token_quantiser_brute_force():
    # per feature column, per run of 128 tokens: amax, fp32 IEEE division, the
    # torch E4M3 encoder -- written as a plain loop over columns of the input
    g = generator(31, "cpu")
    x = normal_bf16((256, 5), 1.0, g, "cpu", outlier_p=0.02, outlier_scale=30.0)
    q, s = oracle.quant_tokens_1x128(bf16_bits(x))
    assert q.shape == (5, 256) and s.shape == (2, 5)
    xf = x.float().numpy()
    for f in range(5):
        for tb in range(2):
            col = xf[tb * 128:(tb + 1) * 128, f]
            amax = np.float32(np.max(np.abs(col)))
            sc = np.float32(amax / np.float32(448.0))
            assert s[tb, f] == sc
            want = torch.from_numpy((col / sc).astype(np.float32)).to(torch.float8_e4m3fn)
            np.testing.assert_array_equal(q[f, tb * 128:(tb + 1) * 128], want.view(torch.uint8).numpy())
            assert np.max(q[f, tb * 128:(tb + 1) * 128] & 0x7F) == 0x7E     # amax -> 448


@pytest.mark.parametrize("T,M,N", [(128, 3, 5), (256, 8, 6), (384, 2, 130)])
def test_gemm_tokens_matches_numpy_matmul_of_torch_dequantised(T, M, N):
    _, _, qa, sa, qb, sb = _token_operands(T, M, N, seed=T + M + N)
    A = torch_decode(qa) * np.repeat(sa.T, 128, axis=1).astype(np.float64)
    B = torch_decode(qb) * np.repeat(sb.T, 128, axis=1).astype(np.float64)
    got = oracle.gemm_f64_tokens(qa, sa, qb, sb)
    np.testing.assert_allclose(got, A @ B.T, rtol=1e-12, atol=1e-300)


def test_gemm_tokens_reduces_to_block_scaled_gemm():
    # if every 128-row block of B shares one scale per slice, the per-row B
    # scales are a 128x128 block grid and the two GEMM definitions coincide
    _, _, qa, sa, qb, _ = _token_operands(256, 4, 256, seed=3)
    rng = np.random.default_rng(4)
    s_block = rng.uniform(0.01, 2.0, size=(2, 2)).astype(np.float32)      # [N/128][K/128]
    s_rows = np.repeat(s_block.T, 128, axis=1)                             # [K/128][N]
    np.testing.assert_array_equal(oracle.gemm_f64_tokens(qa, sa, qb, s_rows),
                                  oracle.gemm_f64(qa, sa, qb, s_block))


def test_gemm_tokens_constant_closed_form():
    # constant magnitude per (row, 128-token run): codes +-448, so
    # C[m][n] = sum_kb 128 * 448^2 * sA[kb][m] * sB[kb][n] * sign
    T, M, N = 256, 2, 3
    dy = np.zeros((T, M), np.float32)
    x = np.zeros((T, N), np.float32)
    for tb in range(2):
        for m in range(M):
            dy[tb * 128:(tb + 1) * 128, m] = (m + 1) * (0.5 if tb else -1.5)
        for n in range(N):
            x[tb * 128:(tb + 1) * 128, n] = (n + 2) * (0.25 if tb else 3.0)
    qa, sa = oracle.quant_tokens_1x128(f32_bits_to_bf16_bits(dy))
    qb, sb = oracle.quant_tokens_1x128(f32_bits_to_bf16_bits(x))
    got = oracle.gemm_f64_tokens(qa, sa, qb, sb)
    for m in range(M):
        for n in range(N):
            want = sum(128 * 448.0 * 448.0 * float(sa[tb, m]) * float(sb[tb, n]) *
                       float(np.sign(dy[tb * 128, m]) * np.sign(x[tb * 128, n])) for tb in range(2))
            assert got[m, n] == pytest.approx(want, rel=1e-14)


def test_weight_gradient_close_to_unquantised_product():
    # dW = dY^T . X through the quantised operands stays within the E4M3
    # rounding of the operands of the float64 product of the BF16 inputs
    dy, x, qa, sa, qb, sb = _token_operands(512, 16, 24, seed=9)
    got = oracle.gemm_f64_tokens(qa, sa, qb, sb)
    dyf, xf = dy.double().numpy(), x.double().numpy()
    ref = dyf.T @ xf
    # per element: half an E4M3 step, 2^-4 relative (normal) or 2^-10 * scale (subnormal)
    ea = 2.0 ** -4 * np.abs(dyf) + 2.0 ** -10 * np.repeat(sa.astype(np.float64), 128, axis=0)
    eb = 2.0 ** -4 * np.abs(xf) + 2.0 ** -10 * np.repeat(sb.astype(np.float64), 128, axis=0)
    bound = np.abs(dyf).T @ eb + ea.T @ np.abs(xf) + ea.T @ eb
    assert np.all(np.abs(got - ref) <= bound * (1 + 1e-9))


# ---------------------------------------------------------------- threads
def _with_threads(n, fn):
    old = oracle.get_threads()
    try:
        oracle.set_threads(n)
        return fn()
    finally:
        oracle.set_threads(0 if old == oracle.get_threads() else old)


@pytest.mark.parametrize("b_major", [0, 1])
def test_gemm_result_does_not_depend_on_thread_count(b_major):
    """The GEMMs split whole output rows over threads; each element is the
    same in-order sum, so 1 thread and many give identical bits (the
    single-threaded result is the plain loop)."""
    qa, sa, qb, sb = _tiny_operands(37, 300, 512, seed=5)
    if b_major == 1:
        qb, sb = np.ascontiguousarray(qb.T), np.ascontiguousarray(sb.T)
    one = _with_threads(1, lambda: oracle.gemm_f64(qa, sa, qb, sb, b_major=b_major))
    many = _with_threads(max(2, os.cpu_count() or 2), lambda: oracle.gemm_f64(qa, sa, qb, sb, b_major=b_major))
    np.testing.assert_array_equal(one, many)
    rows, cols = np.arange(37) % 37, (np.arange(37) * 7) % 300
    np.testing.assert_array_equal(_with_threads(3, lambda: oracle.gemm_f64_at(qa, sa, qb, sb, rows, cols,
                                                                               b_major=b_major)),
                                  one[rows, cols])


def test_grouped_tokens_and_norms_do_not_depend_on_thread_count():
    counts = [9, 0, 14, 3]
    E, N, K = len(counts), 260, 256
    M = sum(counts)
    qa, sa = oracle.quant_act_1x128(_random_act(M, K, seed=3))
    qbs, sbs = zip(*[oracle.quant_w_128x128(_random_w(N, K, seed=200 + e)) for e in range(E)])
    qb, sb = np.stack(qbs), np.stack(sbs)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    runs = [_with_threads(n, lambda: oracle.grouped_gemm_f64(qa, sa, qb, sb, off)) for n in (1, 4)]
    np.testing.assert_array_equal(runs[0], runs[1])
    ta, tsa = oracle.quant_tokens_1x128(_random_act(256, 40, seed=4))
    tb, tsb = oracle.quant_tokens_1x128(_random_act(256, 70, seed=6))
    runs = [_with_threads(n, lambda: oracle.gemm_f64_tokens(ta, tsa, tb, tsb)) for n in (1, 5)]
    np.testing.assert_array_equal(runs[0], runs[1])
    norms = [_with_threads(n, lambda: oracle.act_row_norms(qa, sa)) for n in (1, 6)]
    np.testing.assert_array_equal(norms[0], norms[1])


def test_k_major_view_of_a_stored_kxn_weight_gives_the_same_gemm():
    """The GPU parity tests compare the MN-major GEMM with the oracle's K-major
    GEMM of the transposed weight (codes transposed, scale grid transposed):
    both layouts of the oracle give the same bits."""
    g = generator(23, "cpu")
    a = bf16_bits(normal_bf16((20, 384), 1.0, g, "cpu"))
    w_kn = bf16_bits(normal_bf16((384, 256), 0.02, g, "cpu"))            # stored [K][N]
    qa, sa = oracle.quant_act_1x128(a)
    qb, sb = oracle.quant_w_128x128(w_kn)
    c_mn = oracle.gemm_f64(qa, sa, qb, sb, b_major=1)
    c_k = oracle.gemm_f64(qa, sa, np.ascontiguousarray(qb.T), np.ascontiguousarray(sb.T), b_major=0)
    np.testing.assert_array_equal(c_mn, c_k)


# ---------------------------------------------------------------- per-tensor scaling
def _numpy_torch_per_tensor(x_bits, amax):
    """Independent restatement: scale by numpy fp32 IEEE division, codes by
    torch's float8_e4m3fn conversion (saturated first: torch maps > 464 to
    NaN), zero scale -> codes of x itself."""
    xf = bf16_bits_to_f32(x_bits)
    s = np.float32(amax) / np.float32(448.0)
    y = xf / s if s != 0 else xf
    y = np.clip(y, -448.0, 448.0).astype(np.float32)
    return torch_encode(y), s


def test_per_tensor_matches_numpy_division_and_torch_encoder():
    x = _random_act(300, 384, seed=91)
    q, s = oracle.quant_per_tensor(x)
    want_q, want_s = _numpy_torch_per_tensor(x, np.abs(bf16_bits_to_f32(x)).max())
    assert np.float32(s).view(np.uint32) == np.float32(want_s).view(np.uint32)
    np.testing.assert_array_equal(q, want_q)


def test_per_tensor_amax_element_maps_to_448():
    x = _random_act(64, 256, seed=92)
    q, _ = oracle.quant_per_tensor(x)
    xf = bf16_bits_to_f32(x)
    i = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
    assert q[i] in (0x7E, 0xFE)
    # 448's rounding interval starts at the midpoint 432 to the next code
    # down (416); the tie at 432 goes to 448 (even mantissa)
    s = np.float32(np.abs(xf[i])) / np.float32(448.0)
    assert np.count_nonzero((q & 0x7F) == 0x7E) == np.count_nonzero(np.abs(xf / s) >= 432.0)


def test_per_tensor_of_one_group_equals_the_group_quantisers():
    """A 128x128 tensor is one weight block and a 1x128 tensor is one
    activation tile: per-tensor scaling must give the same codes and scale."""
    w = _random_w(128, 128, seed=93)
    q, s = oracle.quant_per_tensor(w)
    qb, sb = oracle.quant_w_128x128(w)
    np.testing.assert_array_equal(q, qb)
    assert np.float32(s).view(np.uint32) == sb[0, 0].view(np.uint32)
    a = _random_act(1, 128, seed=94)
    q, s = oracle.quant_per_tensor(a)
    qa, sa = oracle.quant_act_1x128(a)
    np.testing.assert_array_equal(q, qa)
    assert np.float32(s).view(np.uint32) == sa[0, 0].view(np.uint32)


def test_per_tensor_zero_tensor():
    x = np.zeros((3, 128), np.uint16)
    x[1, 5] = 0x8000                                                  # -0
    q, s = oracle.quant_per_tensor(x)
    assert s == 0.0 and q[1, 5] == 0x80 and np.count_nonzero(q) == 1


def test_delayed_scaling_rules():
    x = _random_act(200, 256, seed=95)
    amax = np.abs(bf16_bits_to_f32(x)).max()
    # the tensor's own amax: identical to current scaling
    q0, s0 = oracle.quant_per_tensor(x)
    q1, s1, a1 = oracle.quant_per_tensor_delayed(x, amax)
    np.testing.assert_array_equal(q0, q1)
    assert s0 == s1 and a1 == amax
    # a quarter of it (a history that missed a growth): the largest values
    # saturate; every code follows numpy division + torch encoding
    q2, s2, a2 = oracle.quant_per_tensor_delayed(x, amax / 4)
    want, want_s = _numpy_torch_per_tensor(x, np.float32(amax / 4))
    np.testing.assert_array_equal(q2, want)
    assert s2 == want_s and a2 == amax
    assert np.any((q2 & 0x7F) == 0x7E)
    # a larger history amax: nothing saturates except exactly-448 codes
    q3, _, _ = oracle.quant_per_tensor_delayed(x, amax * 8)
    want, _ = _numpy_torch_per_tensor(x, np.float32(amax * 8))
    np.testing.assert_array_equal(q3, want)
    assert not np.any((q3 & 0x7F) == 0x7E)


@pytest.mark.parametrize("b_major", [0, 1])
def test_per_tensor_gemm_matches_numpy_and_block_gemm_with_constant_scales(b_major):
    g = generator(96, "cpu")
    a = bf16_bits(normal_bf16((9, 384), 1.0, g, "cpu", outlier_p=0.02, outlier_scale=50.0))
    w = bf16_bits(normal_bf16((140, 384) if b_major == 0 else (384, 256), 0.02, g, "cpu"))
    qa, sa = oracle.quant_per_tensor(a)
    qb, sb = oracle.quant_per_tensor(w)
    got = oracle.gemm_f64_per_tensor(qa, sa, qb, sb, b_major=b_major)
    A = torch_decode(qa) * np.float64(sa)
    B = torch_decode(qb) * np.float64(sb)
    np.testing.assert_allclose(got, A @ (B.T if b_major == 0 else B), rtol=1e-12, atol=1e-300)
    # the block oracle with every group scale equal to the tensor's scale
    KB = 384 // 128
    if b_major == 0:
        sb_grid = np.full(((140 + 127) // 128, KB), sb, np.float32)
    else:
        sb_grid = np.full((KB, 256 // 128), sb, np.float32)
    blk = oracle.gemm_f64(qa, np.full((KB, 9), sa, np.float32), qb, sb_grid, b_major=b_major)
    np.testing.assert_array_equal(got, blk)


@pytest.mark.parametrize("b_major", [0, 1])
def test_unquantised_bf16_product_matches_numpy(b_major):
    g = generator(97, "cpu")
    a = normal_bf16((7, 256), 1.0, g, "cpu", outlier_p=0.02, outlier_scale=50.0)
    w = normal_bf16((130, 256) if b_major == 0 else (256, 130), 0.02, g, "cpu")
    got = oracle.gemm_bf16_f64(bf16_bits(a), bf16_bits(w), b_major=b_major)
    A, W = a.double().numpy(), w.double().numpy()
    np.testing.assert_allclose(got, A @ (W.T if b_major == 0 else W), rtol=1e-12, atol=1e-300)


def test_array_encoder_does_not_depend_on_thread_count():
    """The array encoder spreads independent elements over threads: 1 thread
    and many give the same codes, equal to the one-value encoder."""
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    one = _with_threads(1, lambda: oracle.e4m3_encode_array(v))
    many = _with_threads(0, lambda: oracle.e4m3_encode_array(v))
    assert np.array_equal(one, many)
    idx = rng.integers(0, v.shape[0], size=2000)
    assert all(int(one[i]) == oracle.e4m3_encode(float(v[i])) for i in idx)


def test_output_rounding_share_of_the_gemm_error_rule():
    # The GEMM acceptance rule lets the mean error rise by the normalised error
    # of rounding the float64 reference itself to BF16.  That share is bounded
    # by 2^-9 element-wise (|C| <= ||a|| ||w||, half an ulp of an 8-bit
    # significand) and, for independent random rows, averages about
    # 2^-9 * 0.72 * E|cos| with E|cos| = sqrt(2 / (pi K)): ~1e-4 at K = 128.
    import torch
    from parity import output_rounding_errors
    rng = np.random.default_rng(5)
    for K in (128, 2048):
        a = rng.standard_normal((300, K))
        w = rng.standard_normal((200, K))
        ref = a @ w.T
        an, wn = np.linalg.norm(a, axis=1), np.linalg.norm(w, axis=1)
        assert output_rounding_errors(ref, an, wn, torch.float32) is None
        e = output_rounding_errors(ref, an, wn, torch.bfloat16)
        assert e.max() <= 2.0 ** -9
        predicted = 2.0 ** -9 * (1.0 - 0.5) / np.log(2.0) * np.sqrt(2.0 / (np.pi * K))
        assert 0.85 * predicted < e.mean() < 1.15 * predicted, (K, e.mean(), predicted)
