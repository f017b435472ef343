"""Benchmark of the fine-grained FP8 path on B300.

One step = one pass of the whole path over one batch of synthetic input:
online quantization of the activations (1x128 tiles) and of the weights
(128x128 blocks), then the block-scaled FP8 GEMM.  Default workload: the
grouped MoE problem (32 experts, 16384 tokens routed with Zipf 1.1, each
expert's rows rounded up to 128, K = 7168, N = 2048, BF16 in and out), the
largest configuration that fits one GPU.  The same JSON line also carries the
weight-gradient GEMM dW[7168][2048] = dY^T X over T = 8192 (the largest dense
shape) under "dense_headline".  Other workloads (--workload forward | wgrad |
accum | backward | mlp_down | forward_norm) use the same step structure with
their own quantizers and GEMM form.

Prints ONE JSON line (rank 0).  `value` is whole-step throughput in TFLOPS
(2*M*N*K of the GEMM per step, over the step's device time with inputs
resident in HBM), summed over ranks (each rank runs its own replica: weak
scaling, no collective on the data path).  Each step is one replay of a CUDA
graph holding the step's three kernels, timed with CUDA events on the
launching stream; L2 is flushed between timed steps, outside the timed events
(a 256 MB write, then a 256 MB read, so the step starts on a clean L2).

--impl reference times the CPU oracle (test infrastructure, plain C) on a
bounded sample of the same workload on this host's cores.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import fp8q_inputs as fi  # noqa: E402

METRIC = "block-scaled FP8 GEMM TFLOPS (% of FP8 peak); quantize GB/s (% of HBM)"
FLUSH_BYTES = 256 << 20
RMS_EPS = 1e-6                  # RMSNorm epsilon of the forward_norm workload


# ------------------------------------------------------------------ helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def kernel_source_hash():
    """Hash of the GEMM kernel sources the committed DRAM-traffic figures were taken on."""
    h = hashlib.sha256()
    for f in ("gemm.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "fp8_fine_grained_21_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "k_gemm_dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
            sel = ["-i", uuid]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", *sel, "--query-gpu=" + self.FIELDS,
                    "--format=csv,noheader,nounits", "-lms", "20"]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            time.sleep(0.2)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def describe(name):
    return {
        "forward": "forward: A[4096][7168] bf16 1x128-quantized x W[2048][7168] bf16 "
                   "128x128-quantized -> C[4096][2048] bf16",
        "wgrad": "wgrad: dW[7168][2048] = dY^T X over T=8192, dY and X bf16 128x1-quantized -> f32",
        "accum": "accum: A[1024][16384] x B[1024][16384] bf16 U(-1,1), 1x128 / 128x128 -> f32",
        "grouped": "grouped: 32 experts (Multinomial(16384, Zipf 1.1), M_e rounded up to 128), "
                   "N=2048, K=7168, bf16 -> bf16",
        "forward_norm": "forward with fused RMSNorm: X[4096][7168] bf16 -> fused RMSNorm (g[7168], "
                        "eps 1e-6) + 1x128 FP8 cast, x W[2048][7168] bf16 128x128-quantized -> "
                        "C[4096][2048] bf16",
        "mlp_down": "SwiGLU MLP down projection: gate_up[4096][2*2048] bf16 -> fused "
                    "silu(gate)*up + 1x128 FP8 cast, W2[7168][2048] bf16 128x128-quantized, "
                    "C[4096][7168] = h W2^T -> bf16",
        "backward": "backward data path of forward: dY[4096][2048] bf16 1x128-quantized, stored "
                    "W8[2048][7168] transposed, stored A8 tiles regrouped 1x128 -> 128x1, "
                    "dX[4096][7168] = dY W -> bf16",
    }[name]


# ------------------------------------------------------- replicas on N ranks
def max_over_ranks(x, dist, device):
    """The slowest rank's time (every rank runs its own replica; the job ends
    when the last one does)."""
    if dist is None:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_replica, ms):
    """Whole-job throughput: the work of all replicas over the slowest rank's time."""
    return world * flops_per_replica / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------- workloads
class Workload:
    """Device buffers and the step of one workload (all kernels are fp8q's)."""

    def __init__(self, name, seed, device):
        import fp8_fine_grained_21_b300 as fq

        self.fq = fq
        self.name = name
        d = fi.make(name, seed=seed)
        self.host = d
        self.launches_per_step = 3
        if name in ("forward", "accum"):
            Ah, Bh = (d["A"], d["W"]) if name == "forward" else (d["A"], d["B"])
            self.M, self.K = Ah.shape
            self.N = Bh.shape[0]
            self.inputs_host = [Ah, Bh]
            self.out_dtype = torch.bfloat16 if name == "forward" else torch.float32
            if name == "accum":
                # 32 tiles of 128 K blocks: the stream-K schedule cuts every tile,
                # so the GEMM call adds the kernel that sums the pieces
                self.launches_per_step = 4
        elif name == "wgrad":
            dY, X = d["dY"], d["X"]
            T, self.M = dY.shape
            self.N = X.shape[1]
            self.K = T
            self.inputs_host = [dY, X]
            self.out_dtype = torch.float32
        elif name == "backward":
            self.M, self.N = d["dY"].shape[0], d["W"].shape[1]
            self.K = d["dY"].shape[1]
            self.inputs_host = [d["dY"], d["A"], d["W"]]
            self.out_dtype = torch.bfloat16
            self.launches_per_step = 4
        elif name == "forward_norm":
            self.M, self.K = d["X"].shape
            self.N = d["W"].shape[0]
            self.inputs_host = [d["X"], d["W"], d["g"]]
            self.out_dtype = torch.bfloat16
        elif name == "mlp_down":
            gu, W2 = d["gate_up"], d["W2"]
            self.M, self.K = gu.shape[0], gu.shape[1] // 2
            self.N = W2.shape[0]
            self.inputs_host = [gu, W2]
            self.out_dtype = torch.bfloat16
        elif name == "grouped":
            A, W, offs = d["A"], d["W"], d["m_offsets"]
            self.G, self.N, self.K = W.shape
            self.M = A.shape[0]
            self.inputs_host = [A, W.reshape(self.G * self.N, self.K)]
            self.offs = torch.from_numpy(offs.astype(np.int32)).to(device)
            self.out_dtype = torch.bfloat16
        else:
            raise ValueError(name)
        self.desc = describe(name)
        self.inputs = [torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(device)
                       for h in self.inputs_host]
        x0, x1 = self.inputs[:2]
        if name == "backward":
            # the forward pass's stored FP8 tiles (set-up, not part of the step)
            self.af8, self.saf = fq.quant_act_1x128(self.inputs[1])
            self.wf8, self.swf = fq.quant_w_128x128(self.inputs[2])
            self.inputs = self.inputs[:1]                 # the step's only new input is dY
            self.inputs_host = self.inputs_host[:1]
            self.a8, self.sa = fq.quant_act_1x128(x0)      # dY 1x128 (inner dim N = 2048)
            self.b8, self.sb = fq.transpose_w_128x128(self.wf8, self.swf)
            self.at8, self.sat = fq.retile_1x128_to_128x1(self.af8, self.saf)
        elif name == "wgrad":
            self.a8, self.sa = fq.quant_act_128x1(x0)
            self.b8, self.sb = fq.quant_act_128x1(x1)
        elif name == "forward_norm":
            self.a8, self.sa = fq.rmsnorm_quant_1x128(x0, self.inputs[2], RMS_EPS)
            self.b8, self.sb = fq.quant_w_128x128(x1)
        elif name == "mlp_down":
            self.a8, self.sa = fq.swiglu_quant_1x128(x0[:, :self.K], x0[:, self.K:])
            self.b8, self.sb = fq.quant_w_128x128(x1)
        else:
            self.a8, self.sa = fq.quant_act_1x128(x0)
            self.b8, self.sb = fq.quant_w_128x128(x1)
        self.C = torch.empty((self.M, self.N), dtype=self.out_dtype, device=device)
        self.side = torch.cuda.Stream(device)
        # stream-K workspace (counters start at zero; every call leaves them zero)
        self.ws = torch.zeros(fq.fp8q_gemm_workspace_size(), dtype=torch.uint8, device=device)
        self.flops = 2.0 * self.M * self.N * self.K
        e0, e1 = x0.numel(), x1.numel()
        # algorithmic bytes: BF16 in + FP8 out + FP32 scales
        if name == "backward":
            ew, ea = self.wf8.numel(), self.af8.numel()
            # dY quantization; weight transpose + activation regrouping (side stream)
            self.quant_bytes = [e0 * 3 + e0 * 4 // 128,
                                (2 * ew + 8 * ew // 16384) + (2 * ea + 2 * (ea * 4 // 128))]
        elif name == "wgrad":
            self.quant_bytes = [e0 * 3 + e0 * 4 // 128, e1 * 3 + e1 * 4 // 128]
        elif name == "mlp_down":
            h = e0 // 2                     # gate and up in (BF16), h out (FP8 + scales)
            self.quant_bytes = [e0 * 2 + h + h * 4 // 128, e1 * 3 + e1 * 4 // 16384]
        else:
            self.quant_bytes = [e0 * 3 + e0 * 4 // 128, e1 * 3 + e1 * 4 // 16384]
        self.gemm_bytes = (self.a8.numel() + self.b8.numel() + 4 * (self.sa.numel() + self.sb.numel())
                           + self.C.numel() * self.C.element_size())

    def quant0(self, stream=None):
        fq = self.fq
        if self.name == "backward":
            fq.fp8q_quant_act_1x128(self.inputs[0], self.a8, self.sa, stream)
        elif self.name == "wgrad":
            fq.fp8q_quant_act_128x1(self.inputs[0], self.a8, self.sa, stream)
        elif self.name == "mlp_down":
            self._swiglu(self.inputs[0], self.a8, self.sa, stream)
        elif self.name == "forward_norm":
            self._rmsnorm(self.inputs[0], self.a8, self.sa, stream)
        else:
            fq.fp8q_quant_act_1x128(self.inputs[0], self.a8, self.sa, stream)

    def _rmsnorm(self, x, q, s, stream):
        self.fq.fp8q_rmsnorm_quant_1x128(x, self.inputs[2], q, s, RMS_EPS, stream)

    def _swiglu(self, gu, q, s, stream):
        self.fq.fp8q_swiglu_quant_1x128(gu[:, :self.K], gu[:, self.K:], q, s, stream)

    def quant1(self, stream=None):
        fq = self.fq
        if self.name == "backward":
            fq.fp8q_transpose_w_128x128(self.wf8, self.swf, self.b8, self.sb, stream)
            fq.fp8q_retile_1x128_to_128x1(self.af8, self.saf, self.at8, self.sat, stream)
        elif self.name == "wgrad":
            fq.fp8q_quant_act_128x1(self.inputs[1], self.b8, self.sb, stream)
        else:
            fq.fp8q_quant_w_128x128(self.inputs[1], self.b8, self.sb, stream)

    def gemm(self, stream=None):
        fq = self.fq
        if self.name == "grouped":
            fq.fp8q_gemm_grouped_ws(self.a8, self.sa, self.b8.view(self.G, self.N, self.K),
                                    self.sb.view(self.G, self.N // 128, self.K // 128), self.C,
                                    self.offs, self.ws, stream)
        elif self.name == "wgrad":
            fq.fp8q_gemm_ws(self.a8, self.sa, self.b8, self.sb, self.C, fq.BSCALE_ROW1x128,
                            self.ws, stream)
        else:
            fq.fp8q_gemm_ws(self.a8, self.sa, self.b8, self.sb, self.C, fq.BSCALE_BLOCK128,
                            self.ws, stream)

    def quant_kernels(self):
        """(input, launch(x, q, s, stream), q, s) of each standalone quantizer of the step."""
        fq = self.fq
        if self.name == "wgrad":
            return [(self.inputs[0], fq.fp8q_quant_act_128x1, self.a8, self.sa),
                    (self.inputs[1], fq.fp8q_quant_act_128x1, self.b8, self.sb)]
        if self.name == "backward":
            return [(self.inputs[0], fq.fp8q_quant_act_1x128, self.a8, self.sa)]
        if self.name == "forward_norm":
            return [(self.inputs[0], self._rmsnorm, self.a8, self.sa),
                    (self.inputs[1], fq.fp8q_quant_w_128x128, self.b8, self.sb)]
        if self.name == "mlp_down":
            return [(self.inputs[0], self._swiglu, self.a8, self.sa),
                    (self.inputs[1], fq.fp8q_quant_w_128x128, self.b8, self.sb)]
        return [(self.inputs[0], fq.fp8q_quant_act_1x128, self.a8, self.sa),
                (self.inputs[1], fq.fp8q_quant_w_128x128, self.b8, self.sb)]

    def fused_step(self, stream=None):
        """Forward workload with the activations quantized inside the GEMM:
        the weight quantization, then fp8q_gemm_quant_a on the BF16
        activations, which also writes the stored 1x128 tiles (A8, sA)."""
        self.quant1(stream)
        self.fused_gemm(stream)

    def fused_gemm(self, stream=None):
        self.fq.fp8q_gemm_quant_a(self.inputs[0], self.b8, self.sb, self.C, self.a8, self.sa,
                                  self.ws, stream)

    def step(self, stream=None):
        """Quantize both operands, then the GEMM.  The two quantizations are
        independent, so B's runs on a side stream (a fork and join inside the
        captured graph) while A's runs on the main one."""
        main = torch.cuda.current_stream() if stream is None else stream
        self.side.wait_stream(main)
        self.quant0(main)
        with torch.cuda.stream(self.side):
            self.quant1(self.side)
        main.wait_stream(self.side)
        self.gemm(main)


def capture(fn):
    """CUDA graph of fn() (the library launches on torch's capture stream)."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                                   # warm-up outside capture (attributes, caches)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


class L2Flush:
    """Evicts the step's data from L2 between timed steps: a write of a buffer
    twice the size of L2, then a read of another one.  The read makes the
    flush's own dirty lines drain to HBM here, outside the timed events, so
    the next step starts with a clean L2 holding none of its inputs instead
    of paying for the flush's write-backs."""

    def __init__(self, device):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def time_graph(g, n, stream, flush, median=False):
    """Device time of n replays, each preceded by an L2 flush that is outside
    the events (and long enough to hide the host's enqueue time): (mean, min,
    mean), or (median, min, mean) with median=True.  Per-kernel figures use the median: a
    replay whose launch reached the GPU late (a stall of the host thread
    between the start event and the launch) is counted whole in its event
    pair and would pull the mean of a ~20 us kernel far up."""
    evs = []
    for _ in range(n):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    t = np.array([a.elapsed_time(b) for a, b in evs])
    return float(np.median(t) if median else t.mean()), float(t.min()), float(t.mean())


KERNEL_REPLAYS = 200             # per-kernel timing: replays, whatever --steps is


def mma_peak(fq, stream, launches=40, blocks=8192):
    """Dense FP8 tensor-pipe rate measured on this GPU: the library's
    MMA-only probe (128 x 256 x 32 E4M3 MMAs back to back on every SM),
    `launches` launches of `blocks` 128-K blocks per SM each, timed with CUDA
    events; the SM clock is sampled meanwhile."""
    sms = fq.fp8q_num_sms()
    flops = sms * blocks * 2.0 * 128 * 256 * 128
    fq.fp8q_bench_mma_peak(blocks, stream)          # warm-up
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    evs = []
    for _ in range(launches):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fq.fp8q_bench_mma_peak(blocks, stream)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    clocks = sampler.stop()
    status = fq.fp8q_get_device_status()
    if status != 0:
        raise RuntimeError("MMA probe: %s" % fq.fp8q_status_string(status))
    ms = float(np.median([a.elapsed_time(b) for a, b in evs]))
    return {"tflops": flops / (ms * 1e-3) / 1e12, "ms_per_launch": ms, "sms": sms,
            "probe": "tcgen05.mma.cta_group::1.kind::f8f6f4 128x256x32, %d per SM per launch, "
                     "median of %d launches" % (4 * blocks, launches),
            "clocks": clocks}


def time_quant_back_to_back(wl, stream, flush, reps=20):
    """Per-launch time of each quantizer when launched back to back (one CUDA
    graph) over R distinct copies of its input, R chosen so that the copies
    together exceed 384 MB (three times L2): every launch still reads from
    HBM, but launch ramp and tail overlap between neighbours.  Inputs of
    256 MB or more are left out (a single launch already is that long)."""
    out = []
    for x, fn, q, s in wl.quant_kernels():
        if x.numel() * x.element_size() >= FLUSH_BYTES:
            out.append(None)
            continue
        R = max(2, -(-(384 << 20) // (x.numel() * x.element_size())))
        bufs = [(x.clone(), torch.empty_like(q), torch.empty_like(s)) for _ in range(R)]

        def run(bufs=bufs, fn=fn):
            st = torch.cuda.current_stream()
            for xi, qi, si in bufs:
                fn(xi, qi, si, st)

        g = capture(run)
        ms, _, _ = time_graph(g, reps, stream, flush, median=True)
        out.append({"launches": R, "ms_per_launch": ms / R})
        del g, bufs
    return out


def time_e2e(wl, steps, stream):
    """Host buffers in, host result out: pinned H2D of the step's inputs, the
    three library calls, D2H of C -- all inside the timed region."""
    hin = [torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).pin_memory()
           for h in wl.inputs_host]
    hout = torch.empty(wl.C.shape, dtype=wl.C.dtype).pin_memory()

    def one():
        for d, h in zip(wl.inputs, hin):
            d.copy_(h, non_blocking=True)
        wl.step()
        hout.copy_(wl.C, non_blocking=True)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    a.record(stream)
    for _ in range(steps):
        one()
    b.record(stream)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) * 1e3 / steps
    dev = a.elapsed_time(b) / steps
    h2d = sum(h.numel() * h.element_size() for h in hin)
    d2h = hout.numel() * hout.element_size()
    return {"ms": max(wall, dev), "h2d": h2d, "d2h": d2h}


def dense_headline(fq, device, stream, flush):
    """The weight-gradient workload (the largest dense shape) timed beside the
    default grouped one: its step, its GEMM and its two quantizers, each
    kernel over KERNEL_REPLAYS replays with the same flush discipline."""
    wl = Workload("wgrad", seed=0, device=device)
    g_step = capture(wl.step)
    g_parts = [capture(wl.quant0), capture(wl.quant1), capture(wl.gemm)]
    for _ in range(3):
        flush()
        g_step.replay()
    torch.cuda.synchronize()
    step_ms, _, _ = time_graph(g_step, 50, stream, flush)
    kt = [time_graph(g, KERNEL_REPLAYS, stream, flush, median=True) for g in g_parts]
    status = fq.fp8q_get_device_status()
    if status != 0:
        raise RuntimeError("device status after the dense headline: %s" % fq.fp8q_status_string(status))
    gemm_tflops = wl.flops / (kt[2][0] * 1e-3) / 1e12
    out = {"workload": wl.desc, "M": wl.M, "N": wl.N, "K": wl.K, "step_ms": step_ms,
           "step_tflops": wl.flops / (step_ms * 1e-3) / 1e12, "gemm_tflops": gemm_tflops,
           "gemm_ms": kt[2][0], "quant_ms": [kt[0][0], kt[1][0]],
           "quant_gbs": [wl.quant_bytes[i] / (kt[i][0] * 1e-3) / 1e9 for i in range(2)],
           "gemm_traffic": profiled_traffic("gemm_wgrad")}
    del g_step, g_parts, wl
    torch.cuda.synchronize()
    return out


# --------------------------------------------------------------- CPU oracle
def oracle_sample(name, rows, kcols=None, seed=0, threads=0, data=None):
    """Time the oracle on a sub-problem of the workload -- `rows` x `rows`
    outputs over the first `kcols` of K (quantize both operands' slices, then
    the FP64 GEMM) -- and extrapolate linearly to one full step: the cost per
    quantized element and per multiply-add are measured separately and scaled
    by the full step's counts."""
    import oracle

    d = data if data is not None else fi.make(name, seed=seed)
    if name == "wgrad":
        dY, X = d["dY"], d["X"]
        T, M = dY.shape
        N = X.shape[1]
        K = T
        kc = K if kcols is None else min(kcols, K)
        full_elems = dY.size + X.size
        t0 = time.perf_counter()
        a8, sa = oracle.quant_128x1(np.ascontiguousarray(dY[:kc, :rows]))
        b8, sb = oracle.quant_128x1(np.ascontiguousarray(X[:kc, :rows]))
        tq = time.perf_counter() - t0
        bmode = 1
    else:
        if name == "grouped":
            A, B = d["A"], d["W"][0]
            M, K = A.shape
            N = d["W"].shape[1]
            full_elems = A.size + d["W"].size
        elif name == "backward":
            A, B = d["dY"], np.ascontiguousarray(d["W"].T)   # dX = dY (W^T)^T
            M, K = A.shape
            N = B.shape[0]
            full_elems = A.size + d["A"].size + d["W"].size
        elif name == "mlp_down":
            A, B = d["gate_up"], d["W2"]
            M, K = A.shape[0], A.shape[1] // 2
            N = B.shape[0]
            full_elems = M * K + B.size
        elif name == "forward_norm":
            A, B = d["X"], d["W"]
            M, K = A.shape
            N = B.shape[0]
            full_elems = A.size + B.size
        else:
            A, B = (d["A"], d["W"]) if name == "forward" else (d["A"], d["B"])
            M, K = A.shape
            N = B.shape[0]
            full_elems = A.size + B.size
        kc = K if kcols is None else min(kcols, K)
        t0 = time.perf_counter()
        if name == "forward_norm":
            a8, sa, _ = oracle.rmsnorm_quant_1x128(np.ascontiguousarray(A[:rows, :kc]),
                                                   np.ascontiguousarray(d["g"][:kc]), RMS_EPS)
        elif name == "mlp_down":
            a8, sa, _ = oracle.swiglu_quant_1x128(np.ascontiguousarray(A[:rows, :kc]),
                                                  np.ascontiguousarray(A[:rows, K:K + kc]))
        else:
            a8, sa = oracle.quant_1x128(np.ascontiguousarray(A[:rows, :kc]))
        b8, sb = oracle.quant_128x128(np.ascontiguousarray(B[:rows, :kc]))
        tq = time.perf_counter() - t0
        bmode = 0
    t0 = time.perf_counter()
    oracle.gemm(a8, sa, b8, sb, bmode=bmode, threads=threads)
    tg = time.perf_counter() - t0
    q_elems = 2 * rows * kc
    macs = rows * rows * kc
    full_macs = M * N * K
    est_s = tq / q_elems * full_elems + tg / macs * full_macs
    return {"tflops": 2.0 * full_macs / est_s / 1e12, "sample_s": tq + tg,
            "sample": "%dx%d outputs over the first %d of K=%d (quantize %d elements, %d MACs), "
                      "extrapolated per element and per MAC to the full step" % (
                          rows, rows, kc, K, q_elems, macs),
            "cores": threads or oracle.max_threads()}


# ------------------------------------------------------------------- arms
def run_reference(args):
    """The CPU oracle as the reference arm, on this host's cores.  Each step is
    a bounded sample whose K extent is sized so that warm-up + timed steps fit
    in about two minutes.  Under torchrun only rank 0 works."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    d = fi.make(args.workload, seed=0)
    budget_s = 120.0
    nsteps = max(1, args.steps + args.warmup)
    probe = oracle_sample(args.workload, 128, kcols=128, data=d)   # one 128 x 128 x 128 block
    per_block = max(probe["sample_s"], 1e-3)
    kblocks = int(max(1, min(56, (budget_s / nsteps) / per_block)))
    vals, secs, last = [], [], probe
    for i in range(nsteps):
        last = oracle_sample(args.workload, 128, kcols=128 * kblocks, data=d)
        if i >= args.warmup:
            vals.append(last["tflops"])
            secs.append(last["sample_s"])
    v = float(np.mean(vals)) if vals else float(last["tflops"])
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOPS", "n_gpus": args.gpus,
           "steps": len(vals), "warmup": args.warmup,
           "ms_per_step": float(np.mean(secs)) * 1e3 if secs else None,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded PCG64; distributions of the named workload)",
           "config": {"workload": describe(args.workload)},
           "cpu_baseline": {"value": v, "unit": "TFLOPS", "cores": last["cores"], "kind": "oracle",
                            "sample": last["sample"]},
           "e2e": {"value": v, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def run_fp8q(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    import fp8_fine_grained_21_b300 as fq

    fq.load()
    wl = Workload(args.workload, seed=rank, device=device)
    stream = torch.cuda.current_stream(device)
    flush = L2Flush(device)

    g_step = capture(wl.step)
    g_parts = [capture(wl.quant0), capture(wl.quant1), capture(wl.gemm)]
    for _ in range(args.warmup):
        flush()
        g_step.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(device)
    sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    step_ms, step_min, _ = time_graph(g_step, args.steps, stream, flush)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall_ms = (time.perf_counter() - t_wall0) * 1e3
    # per-kernel device times (same flush discipline), for the roofline line
    kt = [time_graph(g, KERNEL_REPLAYS, stream, flush, median=True) for g in g_parts]
    q_b2b = time_quant_back_to_back(wl, stream, flush)
    clocks = sampler.stop()
    status = fq.fp8q_get_device_status()
    if status != 0:
        raise RuntimeError("device status after timing: %s" % fq.fp8q_status_string(status))
    fused = None
    if args.workload == "forward":
        # the same forward step with the activations quantized inside the GEMM
        g_fs, g_fg = capture(wl.fused_step), capture(wl.fused_gemm)
        fs_ms, _, _ = time_graph(g_fs, KERNEL_REPLAYS, stream, flush)
        fg_ms, _, _ = time_graph(g_fg, KERNEL_REPLAYS, stream, flush, median=True)
        fused = {"step_ms": fs_ms, "gemm_ms": fg_ms,
                 "step_tflops": wl.flops / (fs_ms * 1e-3) / 1e12,
                 "gemm_tflops": wl.flops / (fg_ms * 1e-3) / 1e12,
                 "two_step": {"step_ms": step_ms, "quant_a_ms": kt[0][0], "gemm_ms": kt[2][0],
                              "quant_a_plus_gemm_ms": kt[0][0] + kt[2][0]},
                 "what": "weight quantization, then fp8q_gemm_quant_a on the BF16 activations "
                         "(1x128 quantization inside the GEMM, stored A8/sA written)"}
        status = fq.fp8q_get_device_status()
        if status != 0:
            raise RuntimeError("device status after the fused step: %s" % fq.fp8q_status_string(status))
        del g_fs, g_fg
    dense = None
    if args.workload == "grouped" and not args.no_dense_headline:
        dense = dense_headline(fq, device, stream, flush)
    peak_probe = mma_peak(fq, stream) if not args.no_mma_peak else None

    step_ms = max_over_ranks(step_ms, dist, device)
    e2e = time_e2e(wl, max(3, min(args.steps, 20)), stream) if not args.no_e2e else None
    e2e_ms = max_over_ranks(e2e["ms"], dist, device) if e2e else None
    if rank != 0:
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return

    peaks = measured_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]          # FP8 dense = 2 x BF16 dense (nominal ratio)
    mma_meas = peak_probe["tflops"] if peak_probe else None
    gemm_ms = kt[2][0]
    gemm_tflops = wl.flops / (gemm_ms * 1e-3) / 1e12
    value = job_tflops(world, wl.flops, step_ms)
    q_gbs = [wl.quant_bytes[i] / (kt[i][0] * 1e-3) / 1e9 for i in range(2)]
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate)",
        "data": "synthetic (seeded PCG64; N(0,1) activations with 0.1% x100 outliers, "
                "N(0,0.02) weights)",
        "config": {"workload": wl.desc, "M": wl.M, "N": wl.N, "K": wl.K,
                   "l2": "flushed between timed steps (256 MB write, then a 256 MB read so that "
                         "L2 is left clean; outside the timed events)",
                   "timing": "CUDA graph replay per step, CUDA events on the launching stream",
                   "parallelism": "replicas x%d" % world},
        "gemm_tflops": gemm_tflops,
        "gemm_frac_of_fp8_peak": gemm_tflops / fp8_peak,
        "quant_gbs": q_gbs,
        "quant_frac_of_hbm": [q / peaks["hbm_gbs"] for q in q_gbs],
        # the same against the ~8 TB/s nominal HBM3e figure, for context
        "quant_frac_of_nominal_hbm_8tbs": [q / 8000.0 for q in q_gbs],
        # the same quantizers launched back to back over copies of their input
        # (together 3x L2), ramp and tail amortised; null for inputs >= 256 MB
        "quant_back_to_back": [None if b is None else {
            "launches": b["launches"], "ms": b["ms_per_launch"],
            "gbs": wl.quant_bytes[i] / (b["ms_per_launch"] * 1e-3) / 1e9,
            "frac_of_hbm": wl.quant_bytes[i] / (b["ms_per_launch"] * 1e-3) / 1e9 / peaks["hbm_gbs"]}
            for i, b in enumerate(q_b2b)],
        "kernel_ms": {"quant_a": kt[0][0], "quant_b": kt[1][0], "gemm": gemm_ms,
                      "gemm_min": kt[2][1], "gemm_mean": kt[2][2], "replays": KERNEL_REPLAYS,
                      "statistic": "median"},
        "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": gemm_tflops / fp8_peak,
                     "traffic": profiled_traffic("gemm_" + args.workload),
                     "kernel": "k_gemm",
                     "peak_source": "2 x bf16 burst (%s)" % peaks["source"],
                     "algorithmic_bytes": wl.gemm_bytes,
                     "frac_of_mma_peak_measured": gemm_tflops / mma_meas if mma_meas else None},
        "fp8_mma_peak_measured": peak_probe,
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": clocks,
        "wall_ms_timed_region": wall_ms,
    }
    if fused:
        out["fused_quant_gemm"] = fused
    if dense:
        dense["gemm_frac_of_fp8_peak"] = dense["gemm_tflops"] / fp8_peak
        dense["gemm_frac_of_mma_peak_measured"] = (dense["gemm_tflops"] / mma_meas
                                                   if mma_meas else None)
        dense["quant_frac_of_hbm"] = [q / peaks["hbm_gbs"] for q in dense["quant_gbs"]]
        out["dense_headline"] = dense
    if e2e:
        out["e2e"] = {"value": job_tflops(world, wl.flops, e2e_ms), "unit": "TFLOPS",
                      "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                      "ms_per_step": e2e_ms}
    if world == 1 and not args.no_cpu_baseline:
        # size the oracle's sample to about 12 s of CPU work (cost ~ rows^2)
        probe = oracle_sample(args.workload, 128, data=wl.host)
        rows = int(128 * (12.0 / max(probe["sample_s"], 1e-3)) ** 0.5) // 128 * 128
        rows = max(128, min(rows, wl.M, wl.N))
        cb = oracle_sample(args.workload, rows, data=wl.host)
        out["cpu_baseline"] = {"value": cb["tflops"], "unit": "TFLOPS", "cores": cb["cores"],
                               "kind": "oracle", "sample": cb["sample"],
                               "sample_seconds": cb["sample_s"]}
    print(json.dumps(out))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["fp8q", "reference"], default="fp8q")
    ap.add_argument("--workload", choices=["forward", "wgrad", "accum", "grouped", "backward",
                                           "mlp_down", "forward_norm"],
                    default="grouped")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-dense-headline", action="store_true",
                    help="skip the weight-gradient figures added to the grouped workload's line")
    ap.add_argument("--no-mma-peak", action="store_true",
                    help="skip the tensor-pipe probe")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "fp8q" and args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_fp8q(args)


if __name__ == "__main__":
    main()
