"""The quantisers' E4M3 conversion (cvt.rn.satfinite.e4m3x2.f32, through the
fp8bs_selftest_encode_e4m3 hook) against the oracle's encoder, written from
the format definition, on EVERY finite fp32 bit pattern: the encoder is the
one step every quantiser and the E4M3-output epilogue share, and the oracle's
reading of it (round to nearest even, saturation to +-448, the input's sign
kept on zero) is thereby checked on all 2^32 - 2^24 finite inputs, not a
sample."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
import fp8_fine_grained_26_b300 as fp8  # a missing or broken build fails loudly

CHUNK = 1 << 28


def test_device_encoder_equals_oracle_on_every_finite_fp32():
    q = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    idx = np.arange(CHUNK, dtype=np.uint32)
    checked = 0
    for c in range((1 << 32) // CHUNK):
        first = c * CHUNK
        fp8.fp8bs_selftest_encode_e4m3(first, CHUNK, q)
        got = q.cpu().numpy()
        bits = idx + np.uint32(first)
        finite = (bits & np.uint32(0x7F800000)) != np.uint32(0x7F800000)
        ref = oracle.e4m3_encode_array(bits[finite].view(np.float32))
        dev = got[finite]
        bad = np.nonzero(dev != ref)[0]
        if bad.size:
            b = bits[finite][bad[:8]]
            pytest.fail(f"{bad.size} codes differ in chunk {c}; e.g. bits {[hex(int(x)) for x in b]}: "
                        f"device {[hex(int(x)) for x in dev[bad[:8]]]}, oracle {[hex(int(x)) for x in ref[bad[:8]]]}")
        checked += int(finite.sum())
    assert checked == (1 << 32) - (1 << 24)          # every pattern but the 2^24 with exponent 255
