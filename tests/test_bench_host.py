"""Host-side logic of bench.py that needs no GPU: the DRAM-traffic record
lookup and its source hash, the quantisers' algorithmic byte count, and the
reporting helpers."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _record():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


def test_traffic_lookup_returns_the_record_for_its_sources(monkeypatch):
    # a capture is reported only while the kernel sources hash to the value
    # stored with it; otherwise the bench reports null
    rec = _record()
    keys = [k for k in rec if not k.startswith("_")]
    assert keys
    for k in keys:
        kernel, workload = k.split(":")
        assert rec[k]["bytes"] == rec[k]["read"] + rec[k]["write"]
        assert len(rec[k]["src_sha"]) == 16
        assert bench.gemm_traffic(kernel, workload) in (rec[k]["bytes"], None), k
        with monkeypatch.context() as m:
            m.setattr(bench, "kernel_src_sha", lambda e4m3_out=False, s=rec[k]["src_sha"]: s)
            assert bench.gemm_traffic(kernel, workload) == rec[k]["bytes"], k


def test_traffic_lookup_is_null_for_unknown_workloads_and_stale_sources(monkeypatch):
    assert bench.gemm_traffic("gemm", "no_such_workload") is None
    monkeypatch.setattr(bench, "kernel_src_sha", lambda e4m3_out=False: "0" * 16)
    assert bench.gemm_traffic("gemm", "mla_q") is None
    assert bench.gemm_traffic("gemm_e4m3", "mla_kv") is None


def test_source_hash_covers_the_encoder_only_for_the_e4m3_epilogue():
    plain, e4m3 = bench.kernel_src_sha(), bench.kernel_src_sha(True)
    assert len(plain) == 16 and len(e4m3) == 16 and plain != e4m3
    assert bench.kernel_src_sha() == plain            # deterministic


def test_quantiser_algorithmic_bytes():
    # 3 bytes per element plus 4 per scale
    assert bench.quant_alg_bytes((4096, 1536), "act") == 4096 * 1536 * 3 + 12 * 4096 * 4
    assert bench.quant_alg_bytes((24576, 1536), "w") == 24576 * 1536 * 3 + 192 * 12 * 4
    # a partial last row block still has its own weight scale
    assert bench.quant_alg_bytes((200, 384), "w") == 200 * 384 * 3 + 2 * 3 * 4
    # the operands timed alone are the configurations' own shapes
    shapes = {label: shape for label, _, shape in bench.QUANT_ALONE_CASES}
    assert shapes["mla_q A 4096x1536"] == (4096, 1536)
    assert shapes["dgrad W stored 7168x18432"] == (7168, 18432)
    assert all(c % 128 == 0 for _, kind, shape in bench.QUANT_ALONE_CASES
               for (_, c) in (shape if kind == "act+w" else (shape,)))


def test_cpu_model_is_a_name_or_none():
    m = bench.cpu_model()
    assert m is None or (isinstance(m, str) and m)


def test_peak_rule_burst_unless_long_and_power_capped():
    import bench
    peaks = {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "hbm_gbs": 6400.0}
    p, kind, _ = bench.choose_peaks(peaks, 0.004, {"reasons": []})
    assert (p, kind) == (3600.0, "burst")
    p, kind, _ = bench.choose_peaks(peaks, 0.2, {"reasons": ["sw_power_cap"]})      # short: burst
    assert kind == "burst"
    p, kind, _ = bench.choose_peaks(peaks, 3.0, {"reasons": []})                     # long, no cap
    assert kind == "burst"
    p, kind, why = bench.choose_peaks(peaks, 3.0, {"reasons": ["sw_power_cap"]})
    assert (p, kind) == (2800.0, "sustained") and "power_cap" in why


def test_default_headline_is_the_largest_configuration():
    import bench
    sizes = {"mla_q": (4096, 24576, 1536), "mla_kv": (8192, 32768, 512), "dgrad": (8192, 18432, 7168),
             "tiny": (128, 256, 512), "experts": (32768, 2048, 7168)}
    flops = {k: 2.0 * m * n * k_ for k, (m, n, k_) in sizes.items()}
    # the expert GEMM has the most FLOPs but is HBM-bound on weights; of the
    # dense GEMMs dgrad is the largest
    assert max((v, k) for k, v in flops.items() if k != "experts")[1] == bench.HEADLINE


def test_ep_world1_plan_maps_every_routed_copy_to_its_row():
    """The expert-parallel bench step's routing plan, on a small synthetic
    routing: copy (t, k) goes to a row of token t under expert choice[t, k],
    every row is used once, and at world size 1 the receive permutation is
    the identity and the expert offsets are the routing's own."""
    import numpy as np
    import torch
    import synthetic
    g = synthetic.generator(2, "cpu")
    T, E, topk = 64, 16, 4
    logits = torch.randn((T, E), generator=g)
    bias = torch.rand((E,), generator=g) * 0.2 - 0.1
    choice = synthetic.route_topk(logits, bias, topk)
    token_of_row, offsets = synthetic.segments_from_choice(choice, E)
    tok, off = token_of_row.numpy(), offsets.numpy()
    plan = bench.ep_world1_plan(tok, off, T)
    M = T * topk
    slot = plan["slot"]
    assert plan["topk"] == topk
    assert np.array_equal(np.sort(slot), np.arange(M))
    assert np.array_equal(plan["dest"].reshape(-1), slot)
    assert np.array_equal(plan["perm"], np.arange(M)) and np.array_equal(plan["inv"], np.arange(M))
    assert np.array_equal(plan["offsets"], off)
    expert_of_row = np.repeat(np.arange(E), np.diff(off))
    assert np.array_equal(tok[slot], np.repeat(np.arange(T), topk))
    assert np.array_equal(expert_of_row[slot].reshape(T, topk), plan["choice"])
    assert np.array_equal(np.sort(choice.numpy(), axis=1), plan["choice"])


class _FakeNvml:
    """Stands in for the NVML reader: a scripted SM clock and reason list."""

    def __init__(self, script):
        self.script, self.i, self.shut = script, 0, False

    def handle(self, uuid, index):
        return (uuid, index)

    def max_clock_sm(self, h):
        return 2032.0

    def clock_sm(self, h):
        return self.script[min(self.i, len(self.script) - 1)][0]

    def reasons(self, h):
        why = self.script[min(self.i, len(self.script) - 1)][1]
        self.i += 1
        return why

    def shutdown(self):
        self.shut = True


def test_clock_record_keeps_only_samples_inside_the_timed_region():
    # before the region: idle at full clock; inside: 1800 MHz under the power
    # cap; after it: a slowdown that must not be counted
    import time
    fake = _FakeNvml([(2032.0, [])])
    s = bench.ClockSampler(0, "GPU-fake", nvml_factory=lambda: fake)
    s.start()
    time.sleep(0.02)
    fake.script, fake.i = [(1800.0, ["sw_power_cap"])], 0
    time.sleep(0.005)                        # let the poller see the change
    s.mark_start()
    time.sleep(0.03)
    s.mark_end()
    fake.script, fake.i = [(2032.0, ["hw_slowdown"])], 0
    time.sleep(0.01)
    rec = s.stop()
    assert fake.shut
    assert rec["sm_mhz"] == 1800 and rec["sm_max_mhz"] == 2032
    assert rec["reasons"] == ["sw_power_cap"] and rec["samples"] >= 5
    assert rec["source"].startswith("NVML")


def test_clock_record_of_a_region_shorter_than_the_poll_uses_the_samples_around_it():
    import time
    fake = _FakeNvml([(1900.0, ["sw_power_cap"])])
    s = bench.ClockSampler(0, None, nvml_factory=lambda: fake)
    s.NVML_POLL_S = 0.02
    s.start()
    time.sleep(0.05)
    s.mark_start()
    s.mark_end()                             # no poll lands inside
    time.sleep(0.05)
    rec = s.stop()
    assert rec["samples"] == 2 and rec["sm_mhz"] == 1900 and rec["reasons"] == ["sw_power_cap"]
