"""GPU parity of the two quantisers against the CPU oracle: E4M3 bytes and FP32
scales must be bit-identical (scales compared as uint32 bit patterns)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import bf16_bits, generator, normal_bf16
from parity import host_u8

pytestmark = pytest.mark.gpu

import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly
DEV = "cuda"


def _bits_f32(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def check_act(x_dev: torch.Tensor, what: str):
    q, s = fp8.fp8_quant_act_1x128(x_dev)
    assert fp8.fp8bs_last_error() == 0
    qo, so = oracle.quant_act_1x128(bf16_bits(x_dev))
    qg, sg = host_u8(q), s.cpu().numpy()
    nbad = int(np.count_nonzero(qg != qo))
    assert nbad == 0, f"{what}: {nbad} E4M3 codes differ, first at {np.argwhere(qg != qo)[:5].tolist()}"
    np.testing.assert_array_equal(_bits_f32(sg), _bits_f32(so), err_msg=what)
    return q, s


def check_w(w_dev: torch.Tensor, what: str):
    q, s = fp8.fp8_quant_w_128x128(w_dev)
    assert fp8.fp8bs_last_error() == 0
    qo, so = oracle.quant_w_128x128(bf16_bits(w_dev))
    qg, sg = host_u8(q), s.cpu().numpy()
    nbad = int(np.count_nonzero(qg != qo))
    assert nbad == 0, f"{what}: {nbad} E4M3 codes differ"
    np.testing.assert_array_equal(_bits_f32(sg), _bits_f32(so), err_msg=what)
    return q, s


@pytest.mark.parametrize("M,K", [(1, 128), (17, 256), (300, 640), (1025, 1536)])
def test_quant_act_random_ragged(M, K):
    g = generator(M + K, DEV)
    x = normal_bf16((M, K), 1.0, g, DEV, outlier_p=0.01, outlier_scale=50.0)
    check_act(x, f"act {M}x{K}")


def test_quant_act_strided_rows():
    g = generator(5, DEV)
    big = normal_bf16((64, 1024), 2.0, g, DEV)
    x = big[:, 256:768]                      # row stride 1024 > K = 512
    q, s = fp8.fp8_quant_act_1x128(x)
    qo, so = oracle.quant_act_1x128(bf16_bits(x))
    np.testing.assert_array_equal(host_u8(q), qo)
    np.testing.assert_array_equal(_bits_f32(s.cpu().numpy()), _bits_f32(so))


def _adversarial_rows():
    """Rows exercising ties, saturation, signed zeros, subnormals and extremes."""
    rows = []
    table = oracle.e4m3_decode_table()
    pos = np.array(sorted({table[c] for c in range(0x7F)}), np.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)       # exact E4M3 midpoints
    # amax = 448 -> scale 1, so x / s = x exactly: every midpoint is a tie
    for i in range(0, len(mids), 127):
        r = np.zeros(128, np.float32)
        chunk = mids[i:i + 127]
        r[:len(chunk)] = chunk
        r[127] = 448.0
        rows.append(r)
        rows.append(-r)
    rows.append(np.zeros(128, np.float32))                      # all +0
    rows.append(-np.zeros(128, np.float32))                     # all -0
    z = np.zeros(128, np.float32)
    z[::2] = -0.0
    rows.append(z)                                              # mixed signed zeros
    rows.append(np.full(128, 3.0, np.float32))                  # constant
    rows.append(np.full(128, -1e-38, np.float32))               # tiny constant
    sub = np.zeros(128, np.float32)
    sub[3] = 2.0 ** -130                                        # bf16 subnormal amax
    sub[4] = -2.0 ** -133
    rows.append(sub)
    big = np.linspace(-3e38, 3e38, 128).astype(np.float32)      # near the bf16 maximum
    rows.append(big)
    wide = (np.float32(2.0) ** np.arange(-64, 64, dtype=np.float32))  # 128 binades
    rows.append(wide)
    rows.append(-wide[::-1])
    m = np.stack(rows)
    # round to bf16 (values chosen are representable or rounded here once)
    t = torch.from_numpy(m).to(torch.bfloat16)
    return t


def test_quant_act_adversarial():
    x = _adversarial_rows().to(DEV)
    x = torch.cat([x, x], dim=1)                                # K = 256, two tiles per row
    check_act(x, "act adversarial")


def test_quant_act_scaled_midpoints_all_scales():
    # the same tie pattern under power-of-two and non-power-of-two amax
    base = _adversarial_rows()[:4].float()
    outs = []
    for k in (-60, -9, -1, 1, 7, 60):
        outs.append(base * (2.0 ** k))
    for f in (0.3, 1.7, 3.0, 5.0 / 7.0):
        outs.append(base * f)
    x = torch.cat(outs).to(torch.bfloat16).to(DEV)
    check_act(x, "act scaled midpoints")


@pytest.mark.parametrize("R,C", [(1, 128), (128, 128), (200, 384), (513, 640)])
def test_quant_w_random_ragged(R, C):
    g = generator(R * 3 + C, DEV)
    w = normal_bf16((R, C), 0.02, g, DEV, outlier_p=0.001, outlier_scale=30.0)
    check_w(w, f"w {R}x{C}")


def test_quant_w_adversarial_blocks():
    a = _adversarial_rows()
    w = torch.cat([a, a.flip(0)], dim=0)[:256]
    w = torch.cat([w, torch.zeros_like(w)], dim=1).to(DEV)       # includes all-zero blocks
    check_w(w, "w adversarial")


def test_quant_w_transpose_invariance_on_gpu():
    g = generator(77, DEV)
    w = normal_bf16((256, 384), 0.02, g, DEV)
    q1, s1 = fp8.fp8_quant_w_128x128(w)
    q2, s2 = fp8.fp8_quant_w_128x128(w.t().contiguous())
    assert torch.equal(q1.t(), q2) and torch.equal(s1.t(), s2)


# ------------------------------------------------- full workload sizes
def test_quant_full_mla_q():
    c = synthetic.mla_q(device=DEV)
    check_act(c.a, "mla_q A 4096x1536 (outliers)")
    check_w(c.w, "mla_q W 24576x1536")


def test_quant_full_mla_kv():
    c = synthetic.mla_kv(device=DEV)
    check_act(c.a, "mla_kv A 8192x512")
    check_w(c.w, "mla_kv W 32768x512")


def test_quant_full_dgrad():
    c = synthetic.dgrad(device=DEV)
    check_act(c.a, "dgrad dY 8192x7168 student-t")
    check_w(c.w, "dgrad W stored 7168x18432")


def test_quant_experts_sampled():
    c = synthetic.experts(device=DEV, keep_x=True)
    q, s = check_act(c.x, "experts X 4096x7168")
    # quantise-then-gather equals gather-then-quantise (on the device)
    qs, ss = fp8.fp8_quant_act_1x128(c.x_sorted)
    assert torch.equal(qs, q.index_select(0, c.token_of_row))
    assert torch.equal(ss, s.index_select(1, c.token_of_row))
    # weights: the whole [E*N, K] matrix at once on the GPU, a sample of
    # experts (first, last, two interior) checked against the oracle
    E, N, K = c.w.shape
    qw, sw = fp8.fp8_quant_w_128x128(c.w.view(E * N, K))
    for e in (0, 1, 137, E - 1):
        qo, so = oracle.quant_w_128x128(bf16_bits(c.w[e]))
        np.testing.assert_array_equal(host_u8(qw[e * N:(e + 1) * N]), qo)
        np.testing.assert_array_equal(_bits_f32(sw[e * N // 128:(e + 1) * N // 128].cpu().numpy()),
                                      _bits_f32(so))
