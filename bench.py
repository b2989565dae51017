"""Benchmark of the fine-grained FP8 GEMM path on one node.

One step = one pass of the whole path over one batch of synthetic input:
    quantise A per 1x128 tile, quantise W per 128x128 block, block-scaled
    FP8 GEMM with per-128-K promotion -> C (BF16)
on the data-gradient shape by default -- dY 8192x7168 (Student-t, nu = 3),
W stored 7168x18432, dX = dY . W 8192x18432 BF16 -- the largest of the
configurations that fit one GPU; A and W are quantised in one launch
(``--quant split`` runs the two single-operand quantisers concurrently
instead).  The default run adds, in the same JSON line, one sub-record per
other configuration (MLA q, MLA kv, routed experts, weight gradient, tiny),
each timed in its own region, the expert-parallel layer's device steps on the
routed-expert workload, the per-tensor contrast scheme on the dgrad and MLA q
shapes, and the quantisers-alone table.
``--workload`` selects another headline shape (mla_q, mla_kv, wgrad,
experts, experts_ep, tiny, and the 64-expert experts_small and
experts_ep_small that profiler captures run on) and then measures only that one.  For ``experts`` a step is the dispatch
quantisation (each token row encoded once and its codes written to each of
its routed rows) plus the grouped GEMM (expert weights
are quantised once, before timing, as they are once per weight update); for
``wgrad`` it is the token-dimension quantisation of dY and X plus the
weight-gradient GEMM; ``experts_ep`` runs the device steps of the
expert-parallel layer at world size 1 on the experts workload (pack, unpack
into expert order, grouped GEMM, the two row gathers of the return path; the
all-to-alls move nothing at world size 1).

Printed (rank 0, one JSON line): whole-job GEMM TFLOP/s over the step time,
per-kernel times from CUDA events on the launching stream, the GEMM's
roofline fraction against the measured peaks (the burst peak unless the timed
region lasts a second or more under the power cap), quantiser GB/s against HBM,
an end-to-end number through the same C-ABI calls with pinned host buffers
(host<->device copies inside the timed region), the oracle timed on a
bounded sample on the host cores, and SM clocks sampled during the timed
region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

``--quant-alone`` instead times the quantisers alone on every operand of the
configurations (back-to-back calls, inputs rotating over more than 2x L2) and
prints their GB/s against HBM as its own JSON line.

Multi-GPU: launched by torch.distributed.run, each rank runs an independent
replica (the path has no exchange step); the time is the max over ranks.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 block-scaled GEMM TFLOP/s & % dense-FP8 peak; quantiser GB/s & % HBM"
L2_BYTES = 126 * 1024 * 1024
FP8_OVER_BF16 = 2.0          # nominal dense FP8 : BF16 tensor ratio (4.5 : 2.25 PFLOP/s)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks
class NvmlReader:
    """The few NVML calls the clock record needs, through ctypes on the
    driver's libnvidia-ml (reads only; no GPU setting is touched)."""
    CLOCK_SM = 1
    REASON_BITS = {"gpu_idle": 0x1, "applications_clocks_setting": 0x2, "sw_power_cap": 0x4,
                   "hw_slowdown": 0x8, "sync_boost": 0x10, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80,
                   "display_clock_setting": 0x100}

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        try:
            self._reasons = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def handle(self, uuid, index):
        h = self.c.c_void_p()
        if uuid and self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), self.c.byref(h)) == 0:
            return h
        if self.lib.nvmlDeviceGetHandleByIndex_v2(self.c.c_uint(index), self.c.byref(h)) != 0:
            raise OSError("no NVML handle")
        return h

    def _clock(self, fn, h):
        v = self.c.c_uint()
        if fn(h, self.c.c_int(self.CLOCK_SM), self.c.byref(v)) != 0:
            raise OSError("NVML clock read failed")
        return float(v.value)

    def clock_sm(self, h):
        return self._clock(self.lib.nvmlDeviceGetClockInfo, h)

    def max_clock_sm(self, h):
        return self._clock(self.lib.nvmlDeviceGetMaxClockInfo, h)

    def reasons(self, h):
        v = self.c.c_ulonglong()
        if self._reasons(h, self.c.byref(v)) != 0:
            raise OSError("NVML reason read failed")
        names = [n for n, b in self.REASON_BITS.items() if v.value & b]
        rest = v.value & ~sum(self.REASON_BITS.values())
        return names + ([f"other_0x{rest:x}"] if rest else [])

    def shutdown(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock and clock-event reasons during a timed region.

    A host thread polls NVML every half millisecond; only the samples taken
    between mark_start() and mark_end() count, so the record covers the timed
    region itself even when it lasts a few milliseconds.  Without NVML the
    fallback is nvidia-smi's 200 ms loop: it is given time for a first sample,
    and when none lands inside a short region all its samples count."""
    NVML_POLL_S = 0.0005
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")
    REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int, uuid=None, nvml_factory=None):
        self.index, self.uuid = index, uuid
        self.nvml_factory = nvml_factory or NvmlReader
        self.proc = self.nvml = self.handle = self.max_mhz = None
        self.samples = []                   # (host time, sm MHz, reason names)
        self.window = [None, None]
        self.stop_flag = threading.Event()

    def start(self):
        try:
            self.nvml = self.nvml_factory()
            self.handle = self.nvml.handle(self.uuid, self.index)
            self.max_mhz = self.nvml.max_clock_sm(self.handle)
            self.thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self.thread.start()
            return
        except Exception:                   # no NVML: nvidia-smi loop
            self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.SMI_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()
            t0 = time.perf_counter()
            while not self.samples and time.perf_counter() - t0 < 1.0:
                time.sleep(0.01)            # the first sample, before the region starts
        except (OSError, ValueError):
            self.proc = None

    def mark_start(self):
        self.window[0] = time.perf_counter()

    def mark_end(self):
        self.window[1] = time.perf_counter()

    def _poll_nvml(self):
        nv, h = self.nvml, self.handle
        while not self.stop_flag.is_set():
            try:
                mhz = nv.clock_sm(h)
                why = nv.reasons(h)
            except Exception:
                break
            self.samples.append((time.perf_counter(), mhz, why))
            time.sleep(self.NVML_POLL_S)

    def _read_smi(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) < 7:
                continue
            try:
                mhz, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            self.max_mhz = mx
            self.samples.append((time.perf_counter(), mhz,
                                 [n for n, v in zip(self.REASON_NAMES, parts[3:7]) if v.lower().startswith("active")]))

    def stop(self):
        if self.nvml is None and self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.thread.join(timeout=5)
        t0, t1 = self.window
        inside = [x for x in self.samples if (t0 is None or x[0] >= t0) and (t1 is None or x[0] <= t1)]
        if not inside and self.samples:
            if self.nvml is None:
                inside = self.samples        # 200 ms samples can miss a short region: keep them all
            else:                            # a region shorter than the poll: the samples around it
                before = [x for x in self.samples if t0 is not None and x[0] < t0][-1:]
                after = [x for x in self.samples if t1 is not None and x[0] > t1][:1]
                inside = before + after
        if self.nvml is not None:
            try:
                self.nvml.shutdown()
            except Exception:
                pass
        reasons = sorted({n for x in inside for n in x[2]})
        return {"sm_mhz": statistics.median(x[1] for x in inside) if inside else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(inside),
                "source": ("NVML, polled every 0.5 ms inside the timed region" if self.nvml is not None
                           else "nvidia-smi -lms 200")}


def clock_sampler(local):
    """The sampler for this rank's GPU, found by UUID so that it is the right
    device whatever CUDA_VISIBLE_DEVICES holds."""
    import torch
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        uuid = None
    return ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local, uuid)


# ---------------------------------------------------------------- workloads
def make_workload(name, device):
    import synthetic
    name = name.replace("_per_tensor", "")
    if name == "mla_q":
        return synthetic.mla_q(device=device)
    if name == "mla_kv":
        return synthetic.mla_kv(device=device)
    if name == "dgrad":
        return synthetic.dgrad(device=device)
    if name == "tiny":
        return synthetic.tiny(device=device)
    if name in ("experts", "experts_ep"):
        return synthetic.experts(device=device, keep_x=True)
    if name in ("experts_small", "experts_ep_small"):
        return synthetic.experts_small(device=device, keep_x=True)
    if name == "wgrad":
        return synthetic.wgrad(device=device)
    raise ValueError(name)


class DenseStep:
    """quantise A and W -> GEMM, over rotating input sets (> 2x L2).

    quant "pair": both operands in one launch (fp8_quant_act_w).  quant
    "split": the two single-operand quantisers, the activation's on a side
    stream forked from the step's stream, concurrently with the weight's; the
    GEMM waits for both."""

    def __init__(self, case, fp8, torch, e4m3_out=None, quant="pair"):
        self.fp8, self.torch, self.case = fp8, torch, case
        self.quant = quant
        M, K, N = case.M, case.K, case.N
        self.M, self.N, self.K, self.b_major = M, N, K, case.b_major
        self.out_dtype = torch.float32 if case.out_fp32 else torch.bfloat16
        # e4m3_out "fused": the GEMM writes C quantised per 1x128 row tile
        # (codes + scales) instead of BF16; "unfused": the same result from the
        # BF16 GEMM followed by the activation quantiser on C
        self.e4m3_out = e4m3_out
        in_bytes = (case.a.numel() + case.w.numel()) * 2
        self.nsets = max(1, min(8, -(-2 * L2_BYTES // in_bytes) + 1))
        self.sets = [(case.a, case.w)] + [(case.a.clone(), case.w.clone())
                                          for _ in range(self.nsets - 1)]
        dev = case.a.device
        self.qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        self.sa = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
        self.qb = torch.empty(tuple(case.w.shape), dtype=torch.uint8, device=dev)
        R, C = case.w.shape
        self.sb = torch.empty(((R + 127) // 128, C // 128), dtype=torch.float32, device=dev)
        if e4m3_out:
            self.c = torch.empty((M, N), dtype=torch.uint8, device=dev)
            self.sc = torch.empty((N // 128, M), dtype=torch.float32, device=dev)
            out_bytes = M * N + self.sc.numel() * 4
            if e4m3_out == "unfused":
                self.c16 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        else:
            self.c = torch.empty((M, N), dtype=self.out_dtype, device=dev)
            self.sc = None
            out_bytes = M * N * self.c.element_size()
        self.flops = 2.0 * M * N * K
        qa_bytes = M * K * 3 + (K // 128) * M * 4
        qw_bytes = R * C * 3 + self.sb.numel() * 4
        if quant == "pair":
            self.kernels = ["quant_act_w", "gemm"]
            self.kernel_bytes = {"quant_act_w": qa_bytes + qw_bytes}
        else:
            self.kernels = ["quant_act", "quant_w", "gemm"]
            self.kernel_bytes = {"quant_act": qa_bytes, "quant_w": qw_bytes}
        self.kernel_bytes["gemm"] = M * K + R * C + (self.sa.numel() + self.sb.numel()) * 4 + out_bytes
        if e4m3_out == "unfused":
            self.kernels.append("quant_out")
            self.kernel_bytes["gemm"] += M * N * 2 - out_bytes
            self.kernel_bytes["quant_out"] = M * N * 3 + self.sc.numel() * 4
        self.h2d_bytes = in_bytes
        self.d2h_bytes = out_bytes
        self.launches_per_step = len(self.kernels)
        self.side = torch.cuda.Stream(device=dev)
        self.schedule = ("quant_act_w" if quant == "pair" else "quant_act || quant_w") + " -> gemm" + \
            (" -> quant_out" if e4m3_out == "unfused" else "")

    def _quantise(self, a, w, events=None):
        """Both operands into qa / sa and qb / sb; records the quantiser
        kernels' (start, end) events, if given, and returns how many it used."""
        f, torch = self.fp8, self.torch
        main = torch.cuda.current_stream()
        if self.quant == "pair":
            if events: events[0].record(main)
            f.fp8_quant_act_w(a, w, self.qa, self.sa, self.qb, self.sb)
            if events: events[1].record(main)
            return 2
        self.side.wait_stream(main)            # the previous step's GEMM has read qa / sa
        with torch.cuda.stream(self.side):
            if events: events[0].record(self.side)
            f.fp8_quant_act_1x128(a, self.qa, self.sa, stream=self.side)
            if events: events[1].record(self.side)
        if events: events[2].record(main)
        f.fp8_quant_w_128x128(w, self.qb, self.sb)
        if events: events[3].record(main)
        main.wait_stream(self.side)
        return 4

    def run(self, i, events=None):
        """events: (start, end) per kernel in `kernels` order, or None."""
        a, w = self.sets[i % self.nsets]
        main = self.torch.cuda.current_stream()
        e = self._quantise(a, w, events)
        if events: events[e].record(main)
        self._gemm()
        if events: events[e + 1].record(main)
        if self.e4m3_out == "unfused":
            if events: events[e + 2].record(main)
            self.fp8.fp8_quant_act_1x128(self.c16, self.c, self.sc)
            if events: events[e + 3].record(main)

    def _gemm(self):
        if self.e4m3_out == "unfused":
            self.fp8.fp8_gemm_blockscaled(self.qa, self.sa, self.qb, self.sb, b_major=self.b_major,
                                          C=self.c16)
        elif self.e4m3_out:
            self.fp8.fp8_gemm_blockscaled_e4m3_out(self.qa, self.sa, self.qb, self.sb, b_major=self.b_major,
                                                   qC=self.c, sC=self.sc)
        else:
            self.fp8.fp8_gemm_blockscaled(self.qa, self.sa, self.qb, self.sb, b_major=self.b_major,
                                          C=self.c)

    # ---- end-to-end interface (see run_e2e): inputs on the host, outputs back
    def host_inputs(self):
        return [self.case.a.cpu().pin_memory(), self.case.w.cpu().pin_memory()]

    def out_buffers(self):
        outs = [torch_empty_like(self.torch, self.c)]
        if self.sc is not None:
            outs.append(torch_empty_like(self.torch, self.sc))
        return outs

    def compute(self, dev_in, outs):
        """The whole path on device inputs [a, w] into outs [c (, sc)]."""
        a, w = dev_in
        f = self.fp8
        self._quantise(a, w)
        if self.e4m3_out == "unfused":
            f.fp8_gemm_blockscaled(self.qa, self.sa, self.qb, self.sb, b_major=self.b_major, C=self.c16)
            f.fp8_quant_act_1x128(self.c16, outs[0], outs[1])
        elif self.e4m3_out:
            f.fp8_gemm_blockscaled_e4m3_out(self.qa, self.sa, self.qb, self.sb, b_major=self.b_major,
                                            qC=outs[0], sC=outs[1])
        else:
            f.fp8_gemm_blockscaled(self.qa, self.sa, self.qb, self.sb, b_major=self.b_major, C=outs[0])


class PerTensorStep:
    """The per-tensor contrast scheme on a dense workload: quantise A and W
    with one scale each (fp8_quant_per_tensor: unit amaxes, reduction,
    encoding -- it reads each operand twice) -> GEMM accumulating the whole K
    on the tensor cores (fp8_gemm_per_tensor), over rotating input sets."""

    def __init__(self, case, fp8, torch):
        self.fp8, self.torch, self.case = fp8, torch, case
        M, K, N = case.M, case.K, case.N
        self.M, self.N, self.K, self.b_major = M, N, K, case.b_major
        in_bytes = (case.a.numel() + case.w.numel()) * 2
        self.nsets = max(1, min(8, -(-2 * L2_BYTES // in_bytes) + 1))
        self.sets = [(case.a, case.w)] + [(case.a.clone(), case.w.clone()) for _ in range(self.nsets - 1)]
        dev = case.a.device
        R, C = case.w.shape
        self.qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        self.qb = torch.empty((R, C), dtype=torch.uint8, device=dev)
        self.sa = torch.empty((1,), dtype=torch.float32, device=dev)
        self.sb = torch.empty((1,), dtype=torch.float32, device=dev)
        self.wsa = torch.empty((fp8.fp8_quant_per_tensor_workspace_size(M, K),), dtype=torch.uint8, device=dev)
        self.wsb = torch.empty((fp8.fp8_quant_per_tensor_workspace_size(R, C),), dtype=torch.uint8, device=dev)
        self.c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.flops = 2.0 * M * N * K
        self.kernels = ["quant_a_per_tensor", "quant_w_per_tensor", "gemm"]
        # two reads (the amax pass, then the encoding pass) and one write per element
        self.kernel_bytes = {"quant_a_per_tensor": M * K * 5, "quant_w_per_tensor": R * C * 5,
                             "gemm": M * K + R * C + 8 + M * N * 2}
        self.h2d_bytes = in_bytes
        self.d2h_bytes = M * N * 2
        self.launches_per_step = 7
        self.schedule = "quant_per_tensor(A) -> quant_per_tensor(W) -> gemm_per_tensor (whole K on the tensor cores)"

    def run(self, i, events=None):
        a, w = self.sets[i % self.nsets]
        self.compute([a, w], [self.c], events)

    def host_inputs(self):
        return [self.case.a.cpu().pin_memory(), self.case.w.cpu().pin_memory()]

    def out_buffers(self):
        return [torch_empty_like(self.torch, self.c)]

    def compute(self, dev_in, outs, events=None):
        a, w = dev_in
        f = self.fp8
        if events: events[0].record()
        f.fp8_quant_per_tensor(a, self.qa, self.sa, self.wsa)
        if events: events[1].record()
        if events: events[2].record()
        f.fp8_quant_per_tensor(w, self.qb, self.sb, self.wsb)
        if events: events[3].record()
        if events: events[4].record()
        f.fp8_gemm_per_tensor(self.qa, self.sa, self.qb, self.sb, b_major=self.b_major, C=outs[0])
        if events: events[5].record()


class WgradStep:
    """quant_tokens(dY) || quant_tokens(X) -> weight-gradient GEMM, over
    rotating input sets (> 2x L2): dW = dY^T . X with both operands quantised
    per 1x128 run of tokens."""

    def __init__(self, case, fp8, torch):
        self.fp8, self.torch, self.case = fp8, torch, case
        T, M, N = case.T, case.M, case.N
        self.M, self.N, self.K = M, N, T
        in_bytes = (case.dy.numel() + case.x.numel()) * 2
        self.nsets = max(1, min(8, -(-2 * L2_BYTES // in_bytes) + 1))
        self.sets = [(case.dy, case.x)] + [(case.dy.clone(), case.x.clone()) for _ in range(self.nsets - 1)]
        dev = case.dy.device
        self.qa = torch.empty((M, T), dtype=torch.uint8, device=dev)
        self.sa = torch.empty((T // 128, M), dtype=torch.float32, device=dev)
        self.qb = torch.empty((N, T), dtype=torch.uint8, device=dev)
        self.sb = torch.empty((T // 128, N), dtype=torch.float32, device=dev)
        self.c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.flops = 2.0 * M * N * T
        self.kernels = ["quant_dy", "quant_x", "gemm"]
        self.kernel_bytes = {
            "quant_dy": T * M * 3 + self.sa.numel() * 4,
            "quant_x": T * N * 3 + self.sb.numel() * 4,
            "gemm": M * T + N * T + (self.sa.numel() + self.sb.numel()) * 4 + M * N * 2,
        }
        self.h2d_bytes = in_bytes
        self.d2h_bytes = M * N * 2
        self.launches_per_step = 3
        self.side = torch.cuda.Stream(device=dev)
        self.schedule = "quant_tokens(dY) || quant_tokens(X) -> wgrad gemm"

    def run(self, i, events=None):
        """events: (start, end) per kernel in `kernels` order, or None."""
        dy, x = self.sets[i % self.nsets]
        f, torch = self.fp8, self.torch
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            if events: events[0].record(self.side)
            f.fp8_quant_tokens_1x128(dy, self.qa, self.sa, stream=self.side)
            if events: events[1].record(self.side)
        if events: events[2].record(main)
        f.fp8_quant_tokens_1x128(x, self.qb, self.sb)
        if events: events[3].record(main)
        main.wait_stream(self.side)
        if events: events[4].record(main)
        f.fp8_gemm_wgrad(self.qa, self.sa, self.qb, self.sb, C=self.c)
        if events: events[5].record(main)

    def host_inputs(self):
        return [self.case.dy.cpu().pin_memory(), self.case.x.cpu().pin_memory()]

    def out_buffers(self):
        return [torch_empty_like(self.torch, self.c)]

    def compute(self, dev_in, outs):
        dy, x = dev_in
        f, torch = self.fp8, self.torch
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            f.fp8_quant_tokens_1x128(dy, self.qa, self.sa, stream=self.side)
        f.fp8_quant_tokens_1x128(x, self.qb, self.sb)
        main.wait_stream(self.side)
        f.fp8_gemm_wgrad(self.qa, self.sa, self.qb, self.sb, C=outs[0])


class ExpertsStep:
    """Dispatch + grouped GEMM: the routed copies of the token rows are
    gathered and quantised in one pass (fp8_quant_act_1x128_gather, bit-equal
    to quantising the gathered BF16 rows), then the grouped GEMM.  The expert
    weights are quantised once, untimed, as they are once per weight update."""

    def __init__(self, case, fp8, torch):
        self.fp8, self.torch, self.case = fp8, torch, case
        E, N, K = case.w.shape
        M = case.x_sorted.shape[0]
        self.M, self.N, self.K, self.E = M, N, K, E
        dev = case.x_sorted.device
        qb, sb = fp8.fp8_quant_w_128x128(case.w.view(E * N, K))
        self.qb, self.sb = qb.view(E, N, K), sb.view(E, -1, K // 128)
        case.w = None                       # the BF16 weights are not needed any more
        torch.cuda.empty_cache()
        self.x = case.x                      # [tokens, K] BF16, before the dispatch
        T = self.x.shape[0]
        # dest[t, j]: the j-th routed row that holds token t (the scatter form of the dispatch)
        import numpy as np
        tok = case.token_of_row.cpu().numpy()
        self.topk = tok.shape[0] // T
        self.dest = torch.from_numpy(np.argsort(tok, kind="stable").reshape(T, self.topk).astype(np.int32)).to(dev)
        case.x_sorted = None
        self.qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        self.sa = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
        self.c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.nsets = 1                      # 3.76 GB of expert weights stream per step (> L2)
        self.flops = 2.0 * M * N * K
        self.kernels = ["quant_scatter", "grouped_gemm"]
        self.kernel_bytes = {
            # each token row read once, every routed copy written once
            "quant_scatter": T * K * 2 + M * 4 + M * K + (K // 128) * M * 4,
            "grouped_gemm": M * K + E * N * K + (self.sa.numel() + self.sb.numel()) * 4 + M * N * 2,
        }
        self.h2d_bytes = T * K * 2 + M * 4
        self.d2h_bytes = M * N * 2
        self.launches_per_step = 2
        self.schedule = "quant_scatter(X -> its routed rows) -> grouped_gemm"

    def run(self, i, events=None):
        """events: (start, end) per kernel in `kernels` order, or None."""
        f = self.fp8
        if events: events[0].record()
        f.fp8_quant_act_1x128_scatter(self.x, self.dest, self.M, self.qa, self.sa)
        if events: events[1].record()
        if events: events[2].record()
        f.fp8_grouped_gemm_blockscaled(self.qa, self.sa, self.qb, self.sb, self.case.offsets,
                                       C=self.c)
        if events: events[3].record()

    def host_inputs(self):
        # the token rows and their routed destinations come from the host every step
        return [self.x.cpu().pin_memory(), self.dest.cpu().pin_memory()]

    def out_buffers(self):
        return [torch_empty_like(self.torch, self.c)]

    def compute(self, dev_in, outs):
        x, dest = dev_in
        f = self.fp8
        f.fp8_quant_act_1x128_scatter(x, dest, self.M, self.qa, self.sa)
        f.fp8_grouped_gemm_blockscaled(self.qa, self.sa, self.qb, self.sb, self.case.offsets, C=outs[0])


def ep_world1_plan(token_of_row, offsets, tokens):
    """The expert-parallel layer's routing plan at world size 1 for a routing
    given as rows sorted by (expert, token) (token_of_row, expert offsets):
    dest[t, k] = send row of token t's k-th copy, perm = received row of each
    expert-major row, inv = its inverse, slot[t*topk + k] = send row of copy
    (t, k), and the expert offsets.  Host numpy, through the layer's own
    planning functions."""
    import numpy as np
    from fp8_fine_grained_26_b300.ep import plan_recv, plan_send
    tok = np.asarray(token_of_row, np.int64)
    off = np.asarray(offsets, np.int64)
    E = off.shape[0] - 1
    topk = tok.shape[0] // tokens
    expert_of_row = np.repeat(np.arange(E), np.diff(off))
    choice = np.empty((tokens, topk), np.int64)
    fill = np.zeros(tokens, np.int64)
    for r in range(tok.shape[0]):                        # experts ascend within each token's copies
        choice[tok[r], fill[tok[r]]] = expert_of_row[r]
        fill[tok[r]] += 1
    plan = plan_send(choice, E, 1)
    M = plan.order.shape[0]
    send_row = np.empty(M, np.int64)
    send_row[plan.order] = np.arange(M)
    rp = plan_recv(plan.expert_counts.reshape(1, E))
    inv = np.empty(M, np.int64)
    inv[rp.perm] = np.arange(M)
    return {"topk": topk, "dest": send_row.reshape(tokens, topk), "perm": rp.perm, "inv": inv, "slot": send_row,
            "offsets": rp.offsets, "choice": choice}


class ExpertsEPStep:
    """The device steps of the expert-parallel layer (fp8_fine_grained_26_b300.ep)
    at world size 1, on the routed-expert workload: pack (each token row
    quantised once, its codes and scales packed into the send row of every
    routed copy) -> [all-to-all: at world size 1 the send buffer is the
    receive buffer] -> unpack into expert order -> grouped GEMM -> row gather
    back into source order -> [all-to-all] -> row gather into (token, slot)
    order.  The routing plan (host numpy, once per routing) is made before
    timing; the weights are quantised once, untimed."""

    def __init__(self, case, fp8, torch):
        import numpy as np
        self.fp8, self.torch, self.case = fp8, torch, case
        E, N, K = case.w.shape
        dev = case.x.device
        qb, sb = fp8.fp8_quant_w_128x128(case.w.view(E * N, K))
        self.qb, self.sb = qb.view(E, N, K), sb.view(E, -1, K // 128)
        case.w = None
        case.x_sorted = None
        torch.cuda.empty_cache()
        self.x = case.x
        T = self.x.shape[0]
        plan = ep_world1_plan(case.token_of_row.cpu().numpy(), case.offsets.cpu().numpy(), T)
        self.topk = plan["topk"]
        M = plan["slot"].shape[0]
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a).astype(np.int32)).to(dev)
        self.dest, self.perm, self.inv, self.slot = (i32(plan["dest"]), i32(plan["perm"]), i32(plan["inv"]),
                                                     i32(plan["slot"]))
        self.offsets = i32(plan["offsets"])
        self.M, self.N, self.K, self.E = M, N, K, E
        rb = fp8.packed_row_bytes(K)
        self.packed = torch.empty((M, rb), dtype=torch.uint8, device=dev)
        self.qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        self.sa = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.y_src = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.nsets = 1
        self.flops = 2.0 * M * N * K
        self.kernels = ["ep_pack", "ep_unpack", "grouped_gemm", "gather_src", "gather_slot"]
        kb = K // 128
        self.kernel_bytes = {
            "ep_pack": T * K * 2 + M * 4 + M * (K + 4 * kb),
            "ep_unpack": M * 4 + 2 * M * (K + 4 * kb),
            "grouped_gemm": M * K + E * N * K + (self.sa.numel() + self.sb.numel()) * 4 + M * N * 2,
            "gather_src": M * 4 + 2 * M * N * 2,
            "gather_slot": M * 4 + 2 * M * N * 2,
        }
        self.h2d_bytes = T * K * 2 + 4 * M * 4
        self.d2h_bytes = M * N * 2
        self.launches_per_step = 5
        self.schedule = ("ep_pack -> [exchange] -> ep_unpack -> grouped_gemm -> gather_src -> [exchange] -> "
                         "gather_slot (world size 1: the exchanges move nothing)")

    def _steps(self, x, dest, perm, inv, slot, out, events=None):
        f = self.fp8
        calls = [
            lambda: f.fp8_ep_dispatch_pack_scatter(x, dest, self.M, self.packed),
            lambda: f.fp8_ep_unpack(self.packed, self.K, perm, self.qa, self.sa),
            lambda: f.fp8_grouped_gemm_blockscaled(self.qa, self.sa, self.qb, self.sb, self.offsets, C=self.y),
            lambda: f.fp8bs_gather_rows(self.y, inv, self.y_src),
            lambda: f.fp8bs_gather_rows(self.y_src, slot, out),
        ]
        for j, call in enumerate(calls):
            if events: events[2 * j].record()
            call()
            if events: events[2 * j + 1].record()

    def run(self, i, events=None):
        self._steps(self.x, self.dest, self.perm, self.inv, self.slot, self.c, events)

    def host_inputs(self):
        return [t.cpu().pin_memory() for t in (self.x, self.dest, self.perm, self.inv, self.slot)]

    def out_buffers(self):
        return [torch_empty_like(self.torch, self.c)]

    def compute(self, dev_in, outs):
        self._steps(*dev_in, outs[0])


def torch_empty_like(torch, t):
    return torch.empty(tuple(t.shape), dtype=t.dtype, device=t.device)


def run_e2e(step, n, torch):
    """End to end through the C-ABI calls, inputs from pinned host memory and
    the result back to pinned host memory, every step.  Consecutive steps are
    pipelined on three streams with double-buffered device inputs and outputs:
    step i+1's host->device copy and step i-1's device->host copy overlap
    step i's kernels (the PCIe link carries both directions at once).
    Returns the time per step in ms (first copy in to last copy out)."""
    host_in = step.host_inputs()
    dev_in = [[torch.empty(tuple(h.shape), dtype=h.dtype, device="cuda") for h in host_in] for _ in range(2)]
    outs = [step.out_buffers() for _ in range(2)]
    host_out = [[torch.empty(tuple(o.shape), dtype=o.dtype).pin_memory() for o in outs[b]] for b in range(2)]
    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def loop(count):
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        ev_in = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):
            ev_comp[b].record(main)
            ev_out[b].record(main)
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        for i in range(count):
            b = i % 2
            s_in.wait_event(ev_comp[b])            # step i-2's kernels have read dev_in[b]
            with torch.cuda.stream(s_in):
                for d, h in zip(dev_in[b], host_in):
                    d.copy_(h, non_blocking=True)
            ev_in[b].record(s_in)
            main.wait_event(ev_in[b])
            main.wait_event(ev_out[b])             # step i-2's result has left outs[b]
            step.compute(dev_in[b], outs[b])
            ev_comp[b].record(main)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                for h, d in zip(host_out[b], outs[b]):
                    h.copy_(d, non_blocking=True)
            ev_out[b].record(s_out)
        main.wait_stream(s_out)
        main.wait_stream(s_in)

    loop(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    loop(n)
    e1.record(main)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


# ---------------------------------------------------------------- CPU oracle
def cpu_model():
    """The host CPU's model name (from /proc/cpuinfo), for the baseline line."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def oracle_sample(workload_name, case_cpu_fn, rows=32):
    """The oracle, as it stands, on a bounded sample of the workload: quantise
    `rows` rows of A and the whole weight (single-threaded C), then the
    float64 GEMM of those rows against every column (its OpenMP threads over
    the host cores).  Returns (flops, seconds, description)."""
    import numpy as np
    import oracle
    import synthetic
    a_bits, w_bits, b_major = case_cpu_fn()
    t0 = time.perf_counter()
    qa, sa = oracle.quant_act_1x128(a_bits[:rows])
    qb, sb = oracle.quant_w_128x128(w_bits)
    c = oracle.gemm_f64(qa, sa, qb, sb, b_major=b_major)
    dt = time.perf_counter() - t0
    K = a_bits.shape[1]
    N = c.shape[1]
    del np, synthetic
    return 2.0 * rows * N * K, dt, (f"{rows} rows of A x all {N} columns (quantise those rows and "
                                    f"the whole {w_bits.shape[0]}x{w_bits.shape[1]} weight, single-threaded; "
                                    f"float64 GEMM on {oracle.get_threads()} threads)")


def oracle_sample_wgrad(case, cols=2):
    """The oracle on a bounded sample of the weight-gradient workload: quantise
    the whole dY along tokens and `cols` input-feature columns of X, then the
    float64 GEMM of every dY feature against those columns."""
    import oracle
    import synthetic
    dy_bits = synthetic.bf16_bits(case.dy)
    x_bits = synthetic.bf16_bits(case.x[:, :cols])
    t0 = time.perf_counter()
    qa, sa = oracle.quant_tokens_1x128(dy_bits)
    qb, sb = oracle.quant_tokens_1x128(x_bits)
    c = oracle.gemm_f64_tokens(qa, sa, qb, sb)
    dt = time.perf_counter() - t0
    return 2.0 * c.shape[0] * c.shape[1] * case.T, dt, (
        f"all {case.M} dY features x {cols} X features over {case.T} tokens (quantise dY and those "
        f"columns along tokens, single-threaded; float64 GEMM on {oracle.get_threads()} threads)")


def dense_host_inputs(case):
    import synthetic
    return synthetic.bf16_bits(case.a), synthetic.bf16_bits(case.w), case.b_major


def kernel_src_sha(e4m3_out=False):
    """First 16 hex digits of sha256 over the sources a GEMM kernel is built
    from: gemm.cuh, ptx.cuh and common.cuh, plus quant.cuh (the encoder) for
    the E4M3-output epilogue, the only GEMM variant that uses it."""
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm.cuh", "ptx.cuh", "common.cuh") + (("quant.cuh",) if e4m3_out else ()):
        with open(os.path.join(ROOT, "fp8_fine_grained_26_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def gemm_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu record, or None when there
    is none for this workload or the kernel source changed since it was taken."""
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(prof):
        return None
    with open(prof) as f:
        rec = json.load(f).get(f"{kernel}:{workload}")
    if rec is None or rec.get("src_sha") != kernel_src_sha(kernel.endswith("_e4m3")):
        return None
    return rec["bytes"]


# ---------------------------------------------------------------- main arms
# Peak rule: the measured burst peaks apply to a kernel in a short timed
# region; the sustained ones only when the timed region is long (>= 1 s) AND
# the clocks sampled during it show the power cap.
SUSTAINED_MIN_S = 1.0

HEADLINE = "dgrad"                                  # the largest configuration that fits one GPU
SUBRECORD_WORKLOADS = ("mla_q", "mla_kv", "experts", "experts_ep", "wgrad", "tiny", "dgrad_per_tensor",
                       "mla_q_per_tensor")


def choose_peaks(peaks, region_s, clk):
    """(fp8 tensor peak TFLOP/s, which one, why) for a timed region of
    region_s seconds with clock record clk."""
    burst = peaks["bf16_tflops"] * FP8_OVER_BF16
    sust = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * FP8_OVER_BF16
    capped = "sw_power_cap" in (clk.get("reasons") or [])
    if region_s >= SUSTAINED_MIN_S and capped:
        return sust, "sustained", f"timed region {region_s:.2f} s under sw_power_cap"
    why = (f"timed region {region_s:.3f} s" + (" (< 1 s)" if region_s < SUSTAINED_MIN_S else "") +
           ("" if capped else ", no power cap seen"))
    return burst, "burst", why


def build_step(name, case, fp8, torch, args):
    if name.endswith("_per_tensor"):
        return PerTensorStep(case, fp8, torch)
    if name in ("experts_ep", "experts_ep_small"):
        return ExpertsEPStep(case, fp8, torch)
    if name in ("experts", "experts_small"):
        return ExpertsStep(case, fp8, torch)
    if name == "wgrad":
        return WgradStep(case, fp8, torch)
    return DenseStep(case, fp8, torch, e4m3_out=args.e4m3_out, quant=args.quant)


def measure(args, name, fp8, torch, peaks, peak_src, world, rank, local, device, with_cpu, with_e2e):
    """One workload: warm-up, K timed steps (one CUDA graph, events around
    every kernel), end to end from host buffers, rooflines.  Returns the
    record (the JSON line's body for the headline, a sub-record otherwise)."""
    case = make_workload(name, device)
    if args.e4m3_out and (name in ("experts", "experts_small", "experts_ep", "experts_ep_small", "wgrad")
                          or name.endswith("_per_tensor")):
        raise SystemExit("--e4m3-out applies to the dense forward workloads")
    step = build_step(name, case, fp8, torch, args)
    stream = torch.cuda.current_stream()

    for i in range(args.warmup):
        step.run(i)
    if fp8.fp8bs_last_error() != 0:
        raise RuntimeError(f"{name}: device error during warm-up")

    # The K timed steps are captured once into a CUDA graph (no host launch
    # gaps between kernels, and nothing between consecutive kernels, so a
    # kernel's on-chip set-up may overlap the end of the one before it).  A
    # second graph of the same K steps records a timing event before and
    # after every kernel, on the stream that kernel runs on: it gives the
    # per-kernel times (each kernel then runs alone between its events).  One
    # untimed replay of each uploads it.
    nk = len(step.kernels)
    evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2 * nk)]
           for _ in range(args.steps)]
    graph = graph_evt = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                step.run(i)
        graph_evt = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_evt):
            for i in range(args.steps):
                step.run(i, evs[i])
        graph.replay()
        graph_evt.replay()
        torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = clock_sampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.05)                        # the sampler is running before the region starts
    clocks.mark_start()
    t_start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step.run(i, evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    clk = clocks.stop()
    if graph_evt is not None:
        graph_evt.replay()                  # per-kernel times
        torch.cuda.synchronize()
    barrier(world)
    if fp8.fp8bs_last_error() != 0:
        raise RuntimeError(f"{name}: device error in the timed region")

    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, world, device)
    per_kernel = {}
    for j, kname in enumerate(step.kernels):
        per_kernel[kname] = sum(e[2 * j].elapsed_time(e[2 * j + 1]) for e in evs) / args.steps
    ms_per_step = elapsed_ms / args.steps
    value = world * step.flops / (ms_per_step * 1e-3) / 1e12
    del graph, graph_evt

    # ---- end-to-end through the same C-ABI calls from pinned host buffers
    e2e = None
    if with_e2e:
        n_e2e = max(3, min(args.steps, 20))
        barrier(world)
        e2e_ms = max_over_ranks(run_e2e(step, n_e2e, torch), world, device)
        e2e = {"value": round(world * step.flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
               "ms_per_step": round(e2e_ms, 4), "steps": n_e2e,
               "h2d_bytes_per_step": int(step.h2d_bytes), "d2h_bytes_per_step": int(step.d2h_bytes),
               "pipelining": "copy in / kernels / copy out of consecutive steps overlap (3 streams)"}

    # ---- roofline of the dominant kernel (the GEMM) and the quantisers.  The
    # bound is whichever of the tensor and HBM times of the kernel's
    # algorithmic work is longer (the expert GEMM streams weights).
    region_s = elapsed_ms * 1e-3
    fp8_peak, peak_kind, peak_why = choose_peaks(peaks, region_s, clk)
    fp8_burst = peaks["bf16_tflops"] * FP8_OVER_BF16
    fp8_sust = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * FP8_OVER_BF16
    gemm_name = "grouped_gemm" if "grouped_gemm" in step.kernels else "gemm"
    gemm_ms = per_kernel[gemm_name]
    achieved = step.flops / (gemm_ms * 1e-3) / 1e12
    gemm_bytes = step.kernel_bytes[gemm_name]
    achieved_gbs = gemm_bytes / (gemm_ms * 1e-3) / 1e9
    traffic = gemm_traffic(gemm_name + ("_e4m3" if getattr(step, "e4m3_out", None) == "fused" else ""), name)
    hbm_bound = gemm_bytes / (peaks["hbm_gbs"] * 1e9) > step.flops / (fp8_peak * 1e12)
    if hbm_bound:
        roofline = {"kernel": gemm_name, "bound": "hbm", "achieved": round(achieved_gbs, 1),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
                    "traffic": traffic, "peak_source": f"{peak_src} hbm_gbs",
                    "tensor_tflops": round(achieved, 1),
                    "tensor_frac_of_burst": round(achieved / fp8_burst, 4)}
    else:
        roofline = {"kernel": gemm_name, "bound": "tensor", "achieved": round(achieved, 1),
                    "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                    "frac": round(achieved / fp8_peak, 4), "traffic": traffic,
                    "peak_source": f"{peak_src} bf16 {peak_kind} x {FP8_OVER_BF16} (nominal FP8:BF16)",
                    "peak_rule": f"{peak_kind}: {peak_why}",
                    "frac_of_burst": round(achieved / fp8_burst, 4),
                    "frac_of_sustained": round(achieved / fp8_sust, 4)}
    hbm = peaks["hbm_gbs"]
    kernels = {}
    for kname in step.kernels:
        ms = per_kernel[kname]
        gbs = step.kernel_bytes[kname] / (ms * 1e-3) / 1e9
        entry = {"ms": round(ms, 5), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4)}
        if kname in ("gemm", "grouped_gemm"):
            entry["TFLOP/s"] = round(achieved, 1)
            entry["frac_fp8_burst"] = round(achieved / fp8_burst, 4)
            entry["frac_fp8_sustained"] = round(achieved / fp8_sust, 4)
        kernels[kname] = entry

    # ---- CPU baseline (oracle) on a bounded sample, rank 0 at N=1 only
    cpu = None
    if with_cpu and rank == 0 and world == 1:
        import oracle
        if name == "wgrad":
            flops, secs, desc = oracle_sample_wgrad(case)
        elif name not in ("experts", "experts_small", "experts_ep", "experts_ep_small") and not name.endswith("_per_tensor"):
            flops, secs, desc = oracle_sample(name, lambda: dense_host_inputs(case))
        else:
            flops = None
        if flops is not None:
            cpu = {"value": round(flops / secs / 1e12, 9), "unit": "TFLOP/s", "cores": oracle.get_threads(),
                   "kind": "oracle", "sample": desc, "seconds": round(secs, 2), "cpu_model": cpu_model()}

    rec = {
        "value": round(value, 2), "unit": "TFLOP/s", "ms_per_step": round(ms_per_step, 5),
        "config": {"workload": case.name if hasattr(case, "name") else name,
                   "M": step.M, "N": step.N, "K": step.K,
                   "step": step.schedule,
                   "out": (f"e4m3 + fp32 scale per 1x128 row tile ({step.e4m3_out})"
                           if getattr(step, "e4m3_out", None)
                           else "bf16" if step.c.dtype == torch.bfloat16 else "fp32"),
                   "l2": (f"inputs rotate over {step.nsets} sets (> 2x the 126 MB L2)"
                          if step.nsets > 1 else "inputs larger than L2"),
                   "parallelism": f"replicas x{world}",
                   "launch": "eager" if args.eager else
                   "CUDA graph of the timed steps; per-kernel times from a second replay with events around each kernel"},
        "kernels": kernels, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": step.launches_per_step * args.steps * world,
        "clocks": clk,
    }
    del step, case, evs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    import fp8_fine_grained_26_b300 as fp8
    device = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    common = (fp8, torch, peaks, peak_src, world, rank, local, device)

    head = measure(args, args.workload, *common, with_cpu=not args.no_cpu, with_e2e=not args.no_e2e)
    out = {"metric": METRIC, "value": head.pop("value"), "unit": head.pop("unit"), "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": head.pop("ms_per_step"),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "e4m3 (fp32 accumulate)", "data": "synthetic"}
    out.update(head)
    if args.subrecords:
        # the other configurations, each its own timed region in this run
        subs = {}
        for wl in SUBRECORD_WORKLOADS:
            if wl == args.workload:
                continue
            r = measure(args, wl, *common, with_cpu=False, with_e2e=not args.no_e2e)
            subs[wl] = {k: r[k] for k in ("value", "unit", "ms_per_step", "config", "kernels", "roofline",
                                          "e2e", "gpu_launches", "clocks")}
        out["workloads"] = subs
        out["quantisers_alone"] = run_quant_alone(args, emit=False)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The oracle as the reference arm, on the host's cores: each step a
    bounded sample -- as many rows of A as the oracle has threads and one
    128-column block of the weight, quantised, and their float64 GEMM block
    (the GEMM spreads the rows over the threads)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    if args.workload in ("experts", "experts_small", "experts_ep", "experts_ep_small", "wgrad"):
        print(json.dumps({"impl": "reference", "unavailable":
                          "the oracle arm samples the dense forward workloads only"}), flush=True)
        return
    import numpy as np
    import oracle
    import synthetic
    case = make_workload(args.workload, "cpu")
    a_bits, w_bits = synthetic.bf16_bits(case.a), synthetic.bf16_bits(case.w)
    b_major, K, N = case.b_major, case.K, case.N
    NB = (N + 127) // 128
    cores = oracle.get_threads()
    rows = min(cores, a_bits.shape[0])

    def one(i):
        m = (i * rows) % (a_bits.shape[0] - rows + 1)
        nb = i % NB
        qa, sa = oracle.quant_act_1x128(a_bits[m:m + rows])
        if b_major == 0:
            blk = np.ascontiguousarray(w_bits[nb * 128:(nb + 1) * 128])
        else:
            blk = np.ascontiguousarray(w_bits[:, nb * 128:(nb + 1) * 128])
        qb, sb = oracle.quant_w_128x128(blk)
        c = oracle.gemm_f64(qa, sa, qb, sb, b_major)
        return 2.0 * K * c.shape[0] * c.shape[1]

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    flops = 0.0
    for i in range(args.steps):
        flops += one(i)
    dt = time.perf_counter() - t0
    v = flops / dt / 1e12
    out = {"metric": METRIC, "impl": "reference", "value": round(v, 9), "unit": "TFLOP/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
           "config": {"workload": case.name, "M": case.M, "N": case.N, "K": case.K},
           "cpu_baseline": {"value": round(v, 9), "unit": "TFLOP/s", "kind": "oracle", "cores": cores,
                            "cpu_model": cpu_model(),
                            "sample": f"per step: {rows} rows of A (one per oracle thread) and one 128-column "
                                      f"block of the weight quantised, and their {rows}x128 float64 GEMM block"},
           "e2e": {"value": round(v, 9), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ------------------------------------------------- quantisers alone
# Each operand of the five configurations that the quantisers see, as
# (label, kind, rows, cols): "act" takes the 1x128 rule, "w" the 128x128 rule,
# "act+w" both operands of one GEMM in one fp8_quant_act_w launch.
QUANT_ALONE_CASES = [
    ("mla_q A 4096x1536", "act", (4096, 1536)),
    ("mla_q W 24576x1536", "w", (24576, 1536)),
    ("mla_q A+W (one launch)", "act+w", ((4096, 1536), (24576, 1536))),
    ("mla_kv A 8192x512", "act", (8192, 512)),
    ("mla_kv W 32768x512", "w", (32768, 512)),
    ("mla_kv A+W (one launch)", "act+w", ((8192, 512), (32768, 512))),
    ("experts X 4096x7168", "act", (4096, 7168)),
    ("dgrad dY 8192x7168", "act", (8192, 7168)),
    ("dgrad W stored 7168x18432", "w", (7168, 18432)),
]


def quant_alg_bytes(shape, kind):
    """Algorithmic bytes of one quantisation of a BF16 [R][C] operand: 2 B
    read and 1 B written per element, plus 4 B per scale (one per 1x128 tile
    for "act", one per 128x128 block for "w")."""
    R, C = shape
    nscale = (C // 128) * R if kind == "act" else ((R + 127) // 128) * (C // 128)
    return R * C * 3 + nscale * 4


def run_quant_alone(args, emit=True):
    """The quantisers timed alone: for each operand, `steps` back-to-back
    calls captured in one CUDA graph, cycling over copies of the input whose
    total size is at least twice L2 (so every call reads from HBM), timed with
    CUDA events around the replay; the steady-state time per call and the
    algorithmic GB/s (2 B read + 1 B written per element + 4 B per scale)
    against the measured HBM peak.  One JSON line (or, with emit=False, the
    same record returned); `value` is the aggregate GB/s over all the listed
    operands."""
    import torch
    import fp8_fine_grained_26_b300 as fp8
    import synthetic
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    dev = torch.device("cuda", local)
    g = synthetic.generator(0, dev)

    results, tot_bytes, tot_ms = {}, 0.0, 0.0
    clocks = clock_sampler(local)
    clocks.start()
    clocks.mark_start()
    for label, kind, shape in QUANT_ALONE_CASES:
        shapes = list(shape) if kind == "act+w" else [shape]
        in_bytes = sum(r * c * 2 for r, c in shapes)
        nsets = max(1, min(32, -(-2 * L2_BYTES // in_bytes)))
        sets = [[synthetic.normal_bf16(sh, 1.0, g, dev) for sh in shapes] for _ in range(nsets)]
        outs = [(torch.empty(sh, dtype=torch.uint8, device=dev),) for sh in shapes]
        if kind == "act+w":
            (M, K), (R, C) = shapes
            sa = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
            sw = torch.empty(((R + 127) // 128, C // 128), dtype=torch.float32, device=dev)
            call = lambda xs: fp8.fp8_quant_act_w(xs[0], xs[1], outs[0][0], sa, outs[1][0], sw)
            nbytes = quant_alg_bytes(shapes[0], "act") + quant_alg_bytes(shapes[1], "w")
        elif kind == "act":
            (M, K), = shapes
            sa = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
            call = lambda xs: fp8.fp8_quant_act_1x128(xs[0], outs[0][0], sa)
            nbytes = quant_alg_bytes(shapes[0], "act")
        else:
            (R, C), = shapes
            sw = torch.empty(((R + 127) // 128, C // 128), dtype=torch.float32, device=dev)
            call = lambda xs: fp8.fp8_quant_w_128x128(xs[0], outs[0][0], sw)
            nbytes = quant_alg_bytes(shapes[0], "w")
        calls = args.steps if emit else max(args.steps, 200)
        for i in range(max(3, args.warmup)):
            call(sets[i % nsets])
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(calls):
                call(sets[i % nsets])
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        if fp8.fp8bs_last_error() != 0:
            raise RuntimeError(f"device error while timing {label}")
        ms = e0.elapsed_time(e1) / calls
        gbs = nbytes / (ms * 1e-3) / 1e9
        results[label] = {"us": round(ms * 1e3, 3), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
                          "bytes": int(nbytes), "input_copies": nsets}
        tot_bytes += nbytes
        tot_ms += ms
        del sets, graph
        torch.cuda.empty_cache()
    clocks.mark_end()
    clk = clocks.stop()
    value = tot_bytes / (tot_ms * 1e-3) / 1e9
    rec = {
        "metric": "quantiser GB/s alone (back-to-back calls, inputs rotating over > 2x L2)",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "frac_hbm": round(value / hbm, 4),
        "peak": {"hbm_gbs": hbm, "source": peak_src},
        "dtype": "bf16 -> e4m3", "data": "synthetic N(0,1)", "quantisers": results, "clocks": clk,
        "gpu_launches": calls * len(QUANT_ALONE_CASES)}
    if emit and rank == 0:
        print(json.dumps(rec), flush=True)
    return rec


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=HEADLINE,
                    choices=["mla_q", "mla_kv", "dgrad", "experts", "experts_ep", "tiny", "wgrad", "experts_small",
                             "experts_ep_small",
                             "dgrad_per_tensor", "mla_q_per_tensor", "mla_kv_per_tensor"],
                    help="the headline workload (default: dgrad, the largest configuration)")
    ap.add_argument("--no-subrecords", action="store_true",
                    help="with the default workload, skip the other configurations' sub-records and the "
                         "quantisers-alone table")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end run")
    ap.add_argument("--quant", choices=["pair", "split"], default="pair",
                    help="dense workloads: quantise A and W in one launch (pair) or as two "
                         "concurrent kernels (split)")
    ap.add_argument("--e4m3-out", choices=["fused", "unfused"], default=None,
                    help="dense workloads: the step's output is C quantised per 1x128 row tile (E4M3 codes "
                         "+ scales), by the GEMM's epilogue (fused) or by the activation quantiser on the "
                         "BF16 C (unfused)")
    ap.add_argument("--quant-alone", action="store_true",
                    help="time the quantisers alone on every operand of the configurations "
                         "(back-to-back calls in a CUDA graph, inputs rotating over > 2x L2)")
    ap.add_argument("--eager", action="store_true",
                    help="launch the timed steps one by one instead of replaying a CUDA graph")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    args.subrecords = args.workload == HEADLINE and not args.no_subrecords and not args.e4m3_out
    if args.impl == "reference":
        run_reference(args)
    elif args.quant_alone:
        run_quant_alone(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
