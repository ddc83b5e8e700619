"""Benchmark of the FP8 W8A8 decode hot path on GB300.

One step = one pass of the decode fused path over one batch: for each
M in {1, 2, 4, 8, 16, 32}, the fused RMSNorm -> static E4M3 quantisation of
x[:M] ([M, 5120] bf16) followed by the merged-QKV FP8 GEMM (N=10240, K=5120,
per-output-channel weight scales, bf16 out).  Every M uses its own weight copy,
so a step streams six distinct 52.4 MB weights (315 MB, more than twice the
129 MB L2) and each GEMM reads its weight from HBM.

The value is algorithmic bytes per step / device time per step, in TB/s
(weights N*K, activations, outputs, scales, the norm's x and gamma).  The
step is captured in a CUDA graph and replayed.  See `python bench.py -h`.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas; no data-path collective) and rank 0 prints one JSON line.
"""
import argparse
import json
import os
import platform
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "fp8_scaled_mm HBM TB/s (M≤32) & FP8 TFLOPS (prefill), % of GB300 roofline"
MS = workloads.DECODE_FUSED_MS
N_QKV, K_HID = workloads.QKV_N, workloads.HIDDEN
WORKLOAD = ("decode fused path: RMSNorm(eps 1e-6) -> static per-tensor E4M3 quant -> merged-QKV FP8 GEMM "
            "N=10240 K=5120, per-channel weight scales, bf16 out; one pass per M in {1,2,4,8,16,32}; "
            "kernels chained with programmatic dependent launch, weights flagged static")
INNER = 20  # steps captured per CUDA graph


def gemm_bytes(M, N=N_QKV, K=K_HID):
    """Algorithmic bytes of one decode GEMM: weights, activations, bf16 output,
    per-channel weight scales and the scalar activation scale."""
    return N * K + M * K + 2 * M * N + 4 * N + 4


def norm_bytes(M, K=K_HID):
    """Algorithmic bytes of one fused RMSNorm -> quant: bf16 x and gamma in,
    E4M3 out, the scale."""
    return 2 * M * K + 2 * K + M * K + 4


def step_bytes():
    return sum(gemm_bytes(m) + norm_bytes(m) for m in MS)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fp8_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.dev), "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[4:8]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


DECODE_KERNEL_SOURCES = ("fp8_w8a8_scaled_gb300/csrc/gemm_decode.cu", "fp8_w8a8_scaled_gb300/csrc/splitk.cuh",
                         "fp8_w8a8_scaled_gb300/csrc/ptx.cuh")
TRAFFIC_RECORD = "profiles/decode_gemm_qkv_10240x5120.md"


def decode_kernel_digest():
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per GEMM launch from the committed ncu summary, or None when
    the summary is missing or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, TRAFFIC_RECORD)
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.split(":", 1)[0] in ("traffic_bytes_per_launch", "kernel_source_digest"):
                k, v = line.split(":", 1)
                fields[k] = v.strip()
    if fields.get("kernel_source_digest") != decode_kernel_digest():
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- our arm

class DecodeFusedStep:
    """Device buffers and the captured CUDA graph of the decode fused step."""

    def __init__(self, torch, fp8, device, seed=0):
        self.torch, self.fp8, self.device = torch, fp8, device
        g = workloads.rng(seed)
        x = workloads.bf16_normal(g, (32, K_HID))
        gamma = workloads.bf16_normal(g, (K_HID,), mean=1.0, std=0.1)
        self.x = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        self.gamma = torch.from_numpy(gamma.view(np.int16)).view(torch.bfloat16).to(device)
        self.s_a = torch.tensor([float(workloads.STATIC_INPUT_SCALE)], dtype=torch.float32, device=device)
        self.W, self.sb, self.A = [], [], []
        # the outputs of all M are rows of one buffer, so that one copy reads
        # them back; two such buffers, so that a step's read-back can overlap
        # the next step (the end-to-end loop alternates them)
        self.Y_all = [torch.empty((sum(MS), N_QKV), dtype=torch.bfloat16, device=device) for _ in range(2)]
        self.Y2 = [[], []]
        row = 0
        for i, m in enumerate(MS):
            self.W.append(workloads.device_e4m3_codes(torch, (N_QKV, K_HID), seed=100 + i, device=device)
                          .view(torch.float8_e4m3fn))
            self.sb.append(workloads.device_uniform_f32(torch, (N_QKV,), 0.5e-3, 2e-3, seed=200 + i, device=device))
            self.A.append(torch.empty((m, K_HID), dtype=torch.float8_e4m3fn, device=device))
            for b in range(2):
                self.Y2[b].append(self.Y_all[b][row:row + m])
            row += m
        self.Y = self.Y2[0]

    def launch_step(self, buf=0, x=None):
        fp8 = self.fp8
        x = self.x if x is None else x
        for i, m in enumerate(MS):
            fp8.rmsnorm_quant_fp8(x[:m], self.gamma, workloads.RMS_EPS, self.s_a, out=self.A[i])
            fp8.fp8_scaled_mm(self.A[i], self.W[i], self.s_a, self.sb[i], fp8.GRAN_PER_CHANNEL,
                              out=self.Y2[buf][i], flags=fp8.FLAG_WEIGHTS_STATIC)

    def decode_ms(self):
        """The M values the weight-streaming decode kernel serves."""
        return [m for m in MS if self.fp8.describe_dispatch(m, N_QKV, K_HID, 1) == self.fp8.KERNEL_DECODE_SPLITK]

    def launch_gemms(self):
        """The decode-kernel GEMM launches of one step alone (the roofline's
        dominant kernel)."""
        fp8 = self.fp8
        for i, m in enumerate(MS):
            if m not in self.decode_ms():
                continue
            fp8.fp8_scaled_mm(self.A[i], self.W[i], self.s_a, self.sb[i], fp8.GRAN_PER_CHANNEL, out=self.Y[i],
                              flags=fp8.FLAG_WEIGHTS_STATIC)

    def capture_once(self, fn):
        """fn (which records INNER steps itself) run once, then captured."""
        torch = self.torch
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        return graph

    def capture(self, fn, inner):
        torch = self.torch
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(inner):
                fn()
        return graph


def time_graph(torch, graph, reps, dist_barrier):
    """Device time of `reps` replays (CUDA events on the replay stream), max over ranks."""
    stream = torch.cuda.current_stream()
    dist_barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(reps):
        graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    dist_barrier()
    return t0.elapsed_time(t1)


def segment_bounds(reps, segments):
    """Replay counts at the segment boundaries: `segments` (at most `reps`,
    at least one) runs of replays whose lengths differ by at most one."""
    segments = max(1, min(segments, reps))
    return [reps * i // segments for i in range(segments + 1)]


def time_graph_segments(torch, graph, reps, segments, dist_barrier):
    """Like time_graph, with CUDA events also between `segments` equal runs of
    replays (no synchronisation inside the timed region): returns the total
    and each segment's time in ms."""
    stream = torch.cuda.current_stream()
    bounds = segment_bounds(reps, segments)
    segments = len(bounds) - 1
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(segments + 1)]
    dist_barrier()
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(segments):
        for _ in range(bounds[i + 1] - bounds[i]):
            graph.replay()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    dist_barrier()
    seg = [ev[i].elapsed_time(ev[i + 1]) / (bounds[i + 1] - bounds[i]) for i in range(segments)]
    return ev[0].elapsed_time(ev[-1]), seg


def cpu_model(cpuinfo="/proc/cpuinfo"):
    """The host CPU as /proc/cpuinfo names it (model name, or implementer and
    part on Arm), with the machine type and the logical CPU count."""
    name = ""
    try:
        fields = {}
        with open(cpuinfo) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        name = fields.get("model name") or ""
        if not name and "CPU part" in fields:
            arm = {"0xd40": "Neoverse V1", "0xd4f": "Neoverse V2", "0xd84": "Neoverse V3", "0xd0c": "Neoverse N1",
                   "0xd49": "Neoverse N2", "0xd8e": "Neoverse N3"}
            part = fields["CPU part"].lower()
            known = arm.get(part, "") if fields.get("CPU implementer", "").lower() == "0x41" else ""
            name = f"{known + ' ' if known else ''}(implementer {fields.get('CPU implementer', '?')} part {part})"
    except OSError:
        pass
    return f"{name or platform.processor() or 'unknown'} ({platform.machine()}, {os.cpu_count()} logical CPUs)"


def cpu_baseline_sample(budget_s=10.0):
    """The oracle, as it stands, on the decode fused step (all six M values,
    full N), repeated until about `budget_s` seconds of wall time."""
    import oracle
    d = workloads.decode_fused(seed=0)
    nthreads = oracle.default_threads()
    steps, t0 = 0, time.perf_counter()
    while True:
        for m in MS:
            A = oracle.rmsnorm_quant(d["x"][:m], d["gamma"], d["eps"], float(d["s_a"]))
            oracle.scaled_mm(A, d["B"], d["s_a"], d["sb"], 1, nthreads=nthreads)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    # the same oracle on one thread, over a quarter of the budget
    steps1, t1 = 0, time.perf_counter()
    while True:
        for m in MS:
            A = oracle.rmsnorm_quant(d["x"][:m], d["gamma"], d["eps"], float(d["s_a"]))
            oracle.scaled_mm(A, d["B"], d["s_a"], d["sb"], 1, nthreads=1)
        steps1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= budget_s / 4:
            break
    return {"value": steps * step_bytes() / el / 1e12, "unit": "TB/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{steps} full decode-fused steps (6 norm-quants + 6 GEMMs 10240x5120, M=1..32), "
                      f"{el:.1f} s wall",
            "one_thread": {"value": steps1 * step_bytes() / el1 / 1e12, "unit": "TB/s", "cores": 1,
                           "sample": f"{steps1} steps, {el1:.1f} s wall"},
            "cpu_model": cpu_model()}


PREFILL_SHAPES = [(m, n) for m in workloads.PREFILL_MS for n in workloads.PREFILL_NS]


def fp8_dense_peak():
    """FP8 dense tensor peak (TFLOP/s): the measured bf16 GEMM rate times the
    nominal FP8 / bf16 ratio (4.5 / 2.25 PFLOP/s dense)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return 2.0 * float(p["bf16_tflops"]), "measured bf16 burst x 2 (nominal fp8/bf16 ratio)"
    return 2.0 * 1900.0, "fallback bf16 1.9 PFLOP/s x 2 (nominal fp8/bf16 ratio)"


def run_prefill(torch, fp8, device, dist_barrier, dist_max, seconds_per_shape=0.25):
    """The prefill-chunk GEMMs (M in {2048, 8192} x N in {10240, 34816},
    K = 5120, per-token x per-channel scales, bf16 out), each timed alone as a
    CUDA graph of launches rotating over three weight copies (so inputs plus
    outputs exceed L2), and the per-token activation quantisation of the same
    chunks.  Returns the prefill object of the JSON line."""
    K = K_HID
    shapes, tot_flop, tot_ms = [], 0.0, 0.0
    quant = []
    launches = 0
    for (M, N) in PREFILL_SHAPES:
        x = workloads.device_bf16_normal(torch, (M, K), seed=500 + M, device=device)
        A = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=device)
        sa = torch.empty((M,), dtype=torch.float32, device=device)
        Bs = [workloads.device_e4m3_codes(torch, (N, K), seed=600 + i, device=device).view(torch.float8_e4m3fn)
              for i in range(3)]
        sb = workloads.device_uniform_f32(torch, (N,), 0.5e-3, 2e-3, seed=700, device=device)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        fp8.quant_fp8_per_token(x, out=A, scale_out=sa)

        def gemms():
            for i in range(3):
                fp8.fp8_scaled_mm(A, Bs[i], sa, sb, fp8.GRAN_PER_TOKEN_CHANNEL, out=Y)

        def quants():
            for _ in range(3):
                fp8.quant_fp8_per_token(x, out=A, scale_out=sa)

        flop = 2.0 * M * N * K
        res = {}
        for name, fn, per in (("gemm", gemms, 3), ("quant", quants, 3)):
            s = torch.cuda.Stream(device=device)
            s.wait_stream(torch.cuda.current_stream(device))
            with torch.cuda.stream(s):
                fn()
            torch.cuda.current_stream(device).wait_stream(s)
            torch.cuda.synchronize(device)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                fn()
            for _ in range(3):
                graph.replay()
            torch.cuda.synchronize(device)
            t = time_graph(torch, graph, 1, dist_barrier) / per
            reps = max(3, int(seconds_per_shape * 1e3 / max(t * per, 1e-3)))
            res[name] = dist_max(time_graph(torch, graph, reps, dist_barrier)) / (reps * per)
            launches += reps * per
        ms = res["gemm"]
        shapes.append({"M": M, "N": N, "K": K, "ms": round(ms, 5), "tflops": round(flop / ms / 1e9, 1),
                       "frac": round(flop / ms / 1e9 / fp8_dense_peak()[0], 4)})
        quant.append({"M": M, "K": K, "us": round(res["quant"] * 1e3, 2),
                      "tbps": round(3.0 * M * K / (res["quant"] * 1e-3) / 1e12, 3)})
        tot_flop += flop
        tot_ms += ms
        del x, A, sa, Bs, sb, Y
    peak, src = fp8_dense_peak()
    achieved = tot_flop / tot_ms / 1e9
    return {
        "metric": "prefill FP8 GEMM TFLOP/s (M in {2048, 8192}, K 5120, N in {10240, 34816}, per-token x "
                  "per-channel scales, bf16 out)",
        "value": round(achieved, 1), "unit": "TFLOP/s", "shapes": shapes,
        "roofline": {"kernel": "prefill_gemm_kernel (tcgen05 128x256 tiles, persistent)", "bound": "tensor",
                     "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_source": src, "traffic": None},
        "quant_per_token": quant,
        "gpu_launches": launches,
        "l2": "three weight copies rotated per graph (inputs + outputs > 129 MB L2)",
        "data": "synthetic: device-random N(0,1) activations (quantised per token in the graph) and uniform "
                "E4M3 weight codes; values do not change the tensor-core time",
    }


def gemm_bytes_gran(M, N, K, per_token):
    """Algorithmic bytes of one GEMM whose activation scale is per token
    (M floats) or per tensor (one float); per-channel weight scales."""
    return N * K + M * K + 2 * M * N + 4 * N + (4 * M if per_token else 4)


def quant_bytes(M, K):
    """Per-token quantisation: bf16 in, E4M3 out, one f32 scale per row."""
    return 2 * M * K + M * K + 4 * M


def silu_quant_bytes(M, I):
    """SiLU(gate) * up -> per-token quant: bf16 [M, 2I] in, E4M3 [M, I] out, scales."""
    return 2 * M * 2 * I + M * I + 4 * M


def graph_of(torch, device, fn, inner):
    s = torch.cuda.Stream(device=device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        fn(0)
    torch.cuda.current_stream(device).wait_stream(s)
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(inner):
            fn(i)
    return graph


def run_gate_up(torch, fp8, device, dist_barrier, dist_max, reps=40):
    """Merged gate_up decode GEMM (N 34816, K 5120, per-channel weight scales,
    per-tensor activation scale) at M in {1, 8, 32, 64}: 20 launches per graph
    alternating two 178 MB weights (inputs > L2)."""
    N, K = workloads.GATE_UP_N, K_HID
    W = [workloads.device_e4m3_codes(torch, (N, K), seed=800 + i, device=device).view(torch.float8_e4m3fn)
         for i in range(2)]
    sb = workloads.device_uniform_f32(torch, (N,), 0.5e-3, 2e-3, seed=802, device=device)
    s_a = torch.tensor([float(workloads.STATIC_INPUT_SCALE)], dtype=torch.float32, device=device)
    peak, _ = measured_peaks()
    rows, launches = [], 0
    for M in workloads.GATE_UP_MS:
        A = workloads.device_e4m3_codes(torch, (M, K), seed=803, device=device).view(torch.float8_e4m3fn)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        g = graph_of(torch, device, lambda i: fp8.fp8_scaled_mm(A, W[i % 2], s_a, sb, fp8.GRAN_PER_CHANNEL, out=Y,
                                                                 flags=fp8.FLAG_WEIGHTS_STATIC), 20)
        for _ in range(3):
            g.replay()
        us = dist_max(time_graph(torch, g, reps, dist_barrier)) * 1e3 / (20 * reps)
        launches += 20 * reps
        b = gemm_bytes_gran(M, N, K, False)
        gbps = b / (us * 1e-6) / 1e9
        rows.append({"M": M, "us": round(us, 3), "GBps": round(gbps, 1), "frac": round(gbps / peak, 4),
                     "kernel": "decode" if fp8.describe_dispatch(M, N, K, 1) == fp8.KERNEL_DECODE_SPLITK else "prefill"})
    del W
    return {"workload": "merged gate_up decode GEMM N=34816 K=5120, per-channel weight scales, per-tensor "
                        "activation scale, bf16 out; two 178 MB weights alternated", "unit": "GB/s",
            "peak": peak, "per_M": rows, "gpu_launches": launches}


def run_w8a16(torch, fp8, device, dist_barrier, dist_max, reps=40):
    """Weight-only FP8 GEMM on the merged QKV shape (N 10240, K 5120, bf16
    activations, per-channel weight scales): the CUDA-core GEMV at M in {1, 4}
    and the widen-on-chip decode kernel at M in {8, 16, 32} (weight bytes per
    launch / time, against the HBM peak; 20 launches per graph over eight 52.4
    MB weights) and the large-M tile kernel (weight widened on chip, bf16
    MMAs) at M 2048 in TFLOP/s."""
    N, K = N_QKV, K_HID
    W = [workloads.device_e4m3_codes(torch, (N, K), seed=900 + i, device=device).view(torch.float8_e4m3fn)
         for i in range(8)]
    sb = workloads.device_uniform_f32(torch, (N,), 0.5e-3, 2e-3, seed=908, device=device)
    peak, _ = measured_peaks()
    rows, launches = [], 0
    for M in (1, 4, 8, 16, 32):
        x = workloads.device_bf16_normal(torch, (M, K), seed=909, device=device)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        g = graph_of(torch, device, lambda i: fp8.w8a16_mm(x, W[i % 8], sb, fp8.GRAN_PER_CHANNEL, out=Y,
                                                          flags=fp8.FLAG_WEIGHTS_STATIC), 20)
        for _ in range(3):
            g.replay()
        us = dist_max(time_graph(torch, g, reps, dist_barrier)) * 1e3 / (20 * reps)
        launches += 20 * reps
        b = N * K + 2 * M * K + 2 * M * N + 4 * N
        gbps = b / (us * 1e-6) / 1e9
        kind = fp8.w8a16_describe_dispatch(M, N, K)
        rows.append({"M": M, "us": round(us, 3), "GBps": round(gbps, 1), "frac": round(gbps / peak, 4),
                     "kernel": "gemv" if kind == fp8.KERNEL_W16_GEMV else "decode"})
    M = 2048
    x = workloads.device_bf16_normal(torch, (M, K), seed=910, device=device)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    # eager launches: each call is ~100 us of GPU work, far above the host's
    # enqueue time, so the events time the GPU
    for i in range(3):
        fp8.w8a16_mm(x, W[i % 8], sb, fp8.GRAN_PER_CHANNEL, out=Y)
    torch.cuda.synchronize(device)
    dist_barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(40):
        fp8.w8a16_mm(x, W[i % 8], sb, fp8.GRAN_PER_CHANNEL, out=Y)
    e1.record()
    torch.cuda.synchronize(device)
    us = dist_max(e0.elapsed_time(e1)) * 1e3 / 40
    dense = {"M": M, "us": round(us, 2), "tflops": round(2.0 * M * N * K / (us * 1e-6) / 1e12, 1),
             "path": "tile kernel: E4M3 weight boxes widened to bf16 in TMEM, tcgen05 kind::f16 MMAs, "
                     "per-channel scale in the epilogue"}
    del W
    return {"workload": "weight-only FP8 (W8A16) merged QKV N=10240 K=5120, bf16 activations, per-channel "
                        "weight scales, bf16 out; eight 52.4 MB weights rotated", "unit": "GB/s", "peak": peak,
            "per_M": rows, "dense_m2048": dense, "gpu_launches": launches}


def decode_step_weights(torch, device):
    """Distinct weights and per-channel scales of the 64 layers of the
    synthetic decode step: (QKV, O, gate_up, down) per layer, 23.15 GB."""
    shapes = workloads.LayerShapes()
    Wl = []
    for layer in range(workloads.STEP_LAYERS):
        ws = []
        for j, (n, k) in enumerate((shapes.qkv, shapes.o, shapes.gate_up, shapes.down)):
            w = workloads.device_e4m3_codes(torch, (n, k), seed=10000 + 8 * layer + j, device=device)
            ws.append((w.view(torch.float8_e4m3fn),
                       workloads.device_uniform_f32(torch, (n,), 0.5e-3, 2e-3, seed=20000 + 8 * layer + j,
                                                    device=device)))
        Wl.append(ws)
    return Wl


def decode_step_fn(torch, fp8, device, Wl, M, buffers=None):
    """One synthetic decode step at M tokens over the layers' weights Wl:
    per layer RMSNorm -> static quant -> QKV, per-token quant of an [M, 8192]
    stub (the attention output, not on this path) -> O, gate_up on the same
    normalised input, SiLU(gate) * up -> per-token quant -> down (7 launches
    per layer).  If `buffers` is a dict, the step's inputs, intermediates and
    outputs are put in it (for checking one layer against the oracle)."""
    shapes = workloads.LayerShapes()
    K = K_HID
    gamma = workloads.device_bf16_normal(torch, (K,), seed=30000, device=device, std=0.1, mean=1.0)
    s_a = torch.tensor([float(workloads.STATIC_INPUT_SCALE)], dtype=torch.float32, device=device)
    x = workloads.device_bf16_normal(torch, (M, K), seed=30001, device=device)
    o_in = workloads.device_bf16_normal(torch, (M, workloads.O_K), seed=30002, device=device)
    a = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=device)
    a_o = torch.empty((M, workloads.O_K), dtype=torch.float8_e4m3fn, device=device)
    a_d = torch.empty((M, workloads.DOWN_K), dtype=torch.float8_e4m3fn, device=device)
    s_o = torch.empty((M,), dtype=torch.float32, device=device)
    s_d = torch.empty((M,), dtype=torch.float32, device=device)
    y = [torch.empty((M, n), dtype=torch.bfloat16, device=device)
         for (n, _) in (shapes.qkv, shapes.o, shapes.gate_up, shapes.down)]
    st = fp8.FLAG_WEIGHTS_STATIC
    if buffers is not None:
        buffers.update(x=x, gamma=gamma, s_a=s_a, o_in=o_in, a=a, a_o=a_o, s_o=s_o, a_d=a_d, s_d=s_d, y=y)

    def step(_i):
        for ws in Wl:
            fp8.rmsnorm_quant_fp8(x, gamma, workloads.RMS_EPS, s_a, out=a)
            fp8.fp8_scaled_mm(a, ws[0][0], s_a, ws[0][1], fp8.GRAN_PER_CHANNEL, out=y[0], flags=st)
            fp8.quant_fp8_per_token(o_in, out=a_o, scale_out=s_o)
            fp8.fp8_scaled_mm(a_o, ws[1][0], s_o, ws[1][1], fp8.GRAN_PER_TOKEN_CHANNEL, out=y[1], flags=st)
            fp8.fp8_scaled_mm(a, ws[2][0], s_a, ws[2][1], fp8.GRAN_PER_CHANNEL, out=y[2], flags=st)
            fp8.silu_mul_quant_per_token(y[2], out=a_d, scale_out=s_d)
            fp8.fp8_scaled_mm(a_d, ws[3][0], s_d, ws[3][1], fp8.GRAN_PER_TOKEN_CHANNEL, out=y[3], flags=st)

    return step


def run_decode_step(torch, fp8, device, dist_barrier, dist_max, reps=20):
    """Synthetic 64-layer decode step at M in {1, 4, 8} (decode_step_fn),
    distinct weights per layer (23.15 GB), the whole step one CUDA graph."""
    L_ = workloads.STEP_LAYERS
    shapes = workloads.LayerShapes()
    Wl = decode_step_weights(torch, device)
    peak, _ = measured_peaks()
    rows, launches = [], 0
    for M in workloads.STEP_MS:
        step = decode_step_fn(torch, fp8, device, Wl, M)
        g = graph_of(torch, device, step, 1)
        for _ in range(3):
            g.replay()
        ms = dist_max(time_graph(torch, g, reps, dist_barrier)) / reps
        launches += reps * 7 * L_
        layer_bytes = (norm_bytes(M) + gemm_bytes_gran(M, *shapes.qkv, False)
                       + quant_bytes(M, workloads.O_K) + gemm_bytes_gran(M, *shapes.o, True)
                       + gemm_bytes_gran(M, *shapes.gate_up, False)
                       + silu_quant_bytes(M, workloads.DOWN_K) + gemm_bytes_gran(M, *shapes.down, True))
        tbps = L_ * layer_bytes / (ms * 1e-3) / 1e12
        rows.append({"M": M, "ms_per_step": round(ms, 4), "bytes_per_step": L_ * layer_bytes, "TBps": round(tbps, 4),
                     "frac": round(tbps * 1e3 / peak, 4)})
    del Wl
    torch.cuda.empty_cache()
    return {"workload": "64-layer synthetic decode step (norm-quant, QKV, per-token quant of an attention-output "
                        "stub, O, gate_up, SiLU(gate)*up -> per-token quant, down per layer; 361.76 MB of distinct "
                        "weights per layer), one CUDA graph",
            "unit": "TB/s", "peak_GBps": peak, "per_M": rows, "gpu_launches": launches}


def run_tiny(torch, fp8, device, dist_barrier, dist_max, reps=200):
    """The tiny GEMM (M 4, K 256, N 512, per-tensor scales): microseconds per
    call inside a CUDA graph of 20 calls."""
    A = workloads.device_e4m3_codes(torch, (4, 256), seed=900, device=device).view(torch.float8_e4m3fn)
    B = workloads.device_e4m3_codes(torch, (512, 256), seed=901, device=device).view(torch.float8_e4m3fn)
    s = torch.tensor([1e-2], dtype=torch.float32, device=device)
    Y = torch.empty((4, 512), dtype=torch.bfloat16, device=device)
    g = graph_of(torch, device, lambda i: fp8.fp8_scaled_mm(A, B, s, s, fp8.GRAN_PER_TENSOR, out=Y), 20)
    for _ in range(3):
        g.replay()
    us = dist_max(time_graph(torch, g, reps, dist_barrier)) * 1e3 / (20 * reps)
    return {"workload": "tiny GEMM M=4 K=256 N=512 per-tensor", "us_per_call": round(us, 3),
            "gpu_launches": 20 * reps}


def run_ours(args, rank, world, dist_barrier, dist_max):
    import torch
    import fp8_w8a8_scaled_gb300 as fp8

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    fp8.clear_device_error()
    step = DecodeFusedStep(torch, fp8, device)
    step_graph = step.capture(step.launch_step, INNER)
    gemm_graph = step.capture(step.launch_gemms, INNER)
    reps = max(1, (args.steps + INNER - 1) // INNER)
    steps = reps * INNER
    warm = max(1, (args.warmup + INNER - 1) // INNER)

    for _ in range(warm):
        step_graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms, seg = time_graph_segments(torch, step_graph, reps, 5, dist_barrier)
    ms = dist_max(ms)
    clk = clocks.stop()
    ms_step = ms / steps
    seg_steps = [dist_max(t) / INNER for t in seg]  # ms per step of each fifth of the timed replays
    value = whole_job_tbps(world, step_bytes(), ms_step)

    # roofline of the dominant kernel: the GEMM launches alone, same rotation
    for _ in range(warm):
        gemm_graph.replay()
    ms_g = dist_max(time_graph(torch, gemm_graph, reps, dist_barrier))
    dms = step.decode_ms()
    per_launch_ms = ms_g / (steps * len(dms))
    gbytes = sum(gemm_bytes(m) for m in dms) / len(dms)
    achieved = gbytes / (per_launch_ms * 1e-3) / 1e9
    peak, peak_src = measured_peaks()

    # end to end through the public API with host buffers: every step copies
    # its x in from pinned host memory, runs and copies all its outputs back
    # (one copy each way), captured with the steps in the replayed graph.  The
    # copies run on a second stream and overlap the neighbouring steps' work,
    # as a serving loop would: step j reads input buffer j % 2 (copied in
    # while step j - 1 computes) and writes output buffer j % 2 (copied out
    # while step j + 1 computes).
    x_host = step.x.cpu().pin_memory()
    x_dev = [step.x, torch.empty_like(step.x)]
    y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in step.Y_all]
    side = torch.cuda.Stream(device=device)
    read_back = [torch.cuda.Event(), torch.cuda.Event()]  # output buffer b copied to the host
    loaded = [torch.cuda.Event(), torch.cuda.Event()]     # input buffer b copied from the host
    consumed = [torch.cuda.Event(), torch.cuda.Event()]   # the step that read input buffer b is done

    def copy_in(j):
        b = j % 2
        with torch.cuda.stream(side):
            if j >= 2:
                side.wait_event(consumed[b])  # step j - 2 has finished reading buffer b
            x_dev[b].copy_(x_host, non_blocking=True)
            loaded[b].record(side)

    def e2e_step(j):
        b = j % 2
        main = torch.cuda.current_stream(device)
        main.wait_event(loaded[b])
        if j >= 2:
            main.wait_event(read_back[b])  # step j - 2's outputs have left output buffer b
        if j + 1 < INNER:
            copy_in(j + 1)                 # the next step's input, while this step computes
        step.launch_step(b, x_dev[b])
        consumed[b].record(main)
        side.wait_event(consumed[b])
        with torch.cuda.stream(side):
            y_host[b].copy_(step.Y_all[b], non_blocking=True)
            read_back[b].record(side)

    def e2e_steps():
        side.wait_stream(torch.cuda.current_stream(device))
        copy_in(0)
        for j in range(INNER):
            e2e_step(j)
        torch.cuda.current_stream(device).wait_stream(side)
    one = step.capture_once(e2e_steps)
    for _ in range(warm):
        one.replay()
    e2e_reps = max(1, min(reps, 2000 // INNER))
    dist_barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(e2e_reps):
        one.replay()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = dist_max(e0.elapsed_time(e1)) / (e2e_reps * INNER)
    h2d = step.x.numel() * 2
    d2h = step.Y_all[0].numel() * 2
    err = fp8.get_device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x}")

    out = {
        "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": world, "steps": steps,
        "warmup": warm * INNER, "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
        "spread": {"segments": len(seg_steps), "min_ms_per_step": round(min(seg_steps), 6),
                   "max_ms_per_step": round(max(seg_steps), 6),
                   "min_value": round(whole_job_tbps(world, step_bytes(), max(seg_steps)), 4),
                   "max_value": round(whole_job_tbps(world, step_bytes(), min(seg_steps)), 4)},
        "config": {"workload": WORKLOAD, "bytes_per_step": step_bytes(), "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: six distinct 52.4 MB weights per step (315 MB)",
                   "graph": f"{INNER} steps per CUDA graph replay"},
        "roofline": {"kernel": "decode_gemm_kernel (tcgen05 swap-AB; 3-CTA clusters per 128-channel tile on QKV, "
                               "partial sums reduced through distributed shared memory), the M = "
                               + "/".join(str(m) for m in dms) + " GEMMs of the step",
                     "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src, "traffic": recorded_traffic(),
                     "traffic_source": TRAFFIC_RECORD,
                     "bytes_per_launch": gbytes, "us_per_launch": round(per_launch_ms * 1e3, 3)},
        "e2e": {"value": round(whole_job_tbps(world, step_bytes(), e2e_ms), 4), "unit": "TB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 6)},
        "gpu_launches": steps * 2 * len(MS),
        "clocks": clk,
    }
    if not args.no_prefill:
        clocks_p = ClockSampler(local)
        clocks_p.start()
        time.sleep(0.2)
        out["prefill"] = run_prefill(torch, fp8, device, dist_barrier, dist_max)
        out["prefill"]["clocks"] = clocks_p.stop()
        err = fp8.get_device_error()
        if err:
            raise RuntimeError(f"device error word {err:#x}")
    if not args.no_extras:
        out["gate_up"] = run_gate_up(torch, fp8, device, dist_barrier, dist_max)
        out["w8a16"] = run_w8a16(torch, fp8, device, dist_barrier, dist_max)
        out["decode_step"] = run_decode_step(torch, fp8, device, dist_barrier, dist_max)
        out["tiny"] = run_tiny(torch, fp8, device, dist_barrier, dist_max)
        err = fp8.get_device_error()
        if err:
            raise RuntimeError(f"device error word {err:#x}")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_sample(args.cpu_seconds)
    return out


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle timed on the host cores on the same workload and metric: each
    step is a bounded sample (the first `cols` output channels of every
    M's GEMM, plus the full norm-quants), sized so the whole run takes about
    `--ref-seconds` of wall time."""
    import oracle
    d = workloads.decode_fused(seed=0)
    nthreads = oracle.default_threads()
    A_by_m = {}

    def one_step(cols):
        for m in MS:
            A_by_m[m] = oracle.rmsnorm_quant(d["x"][:m], d["gamma"], d["eps"], float(d["s_a"]))
            oracle.scaled_mm(A_by_m[m], d["B"][:cols], d["s_a"], d["sb"][:cols], 1, nthreads=nthreads)

    def sample_bytes(cols):
        return sum(gemm_bytes(m, N=cols) + norm_bytes(m) for m in MS)

    t0 = time.perf_counter()
    one_step(256)
    per_col = (time.perf_counter() - t0) / 256
    total = max(1, args.steps + args.warmup)
    cols = int(max(8, min(N_QKV, args.ref_seconds / total / max(per_col, 1e-9))))
    cols -= cols % 8
    for _ in range(args.warmup):
        one_step(cols)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step(cols)
    el = time.perf_counter() - t0
    value = args.steps * sample_bytes(cols) / el / 1e12
    sample = f"{args.steps} steps, each the norm-quants plus the first {cols} of 10240 GEMM output channels for M=1..32"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 8), "unit": "TB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": round(value, 8), "unit": "TB/s", "cores": nthreads, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 8), "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile_case(args):
    """Small eager case for profilers: `--steps` launches of one GEMM shape
    (plus the norm-quant that feeds it) rotating over three weight copies
    (more than L2 in total), without CUDA graphs or timing claims."""
    import torch
    import fp8_w8a8_scaled_gb300 as fp8
    M, N, K = (int(v) for v in args.profile.split(","))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    if args.profile_kind == "step":  # the 64-layer decode step at M tokens (N, K unused), eagerly
        step = decode_step_fn(torch, fp8, dev, decode_step_weights(torch, dev), M)
        for i in range(args.steps):
            step(i)
        torch.cuda.synchronize()
        err = fp8.get_device_error()
        print(json.dumps({"profile_case": [M, N, K], "kind": "step", "device_error": err}))
        if err:
            raise SystemExit(1)
        return
    g = workloads.rng(0)
    x = torch.from_numpy(workloads.bf16_normal(g, (M, K)).view(np.int16)).view(torch.bfloat16).to(dev)
    gamma = torch.from_numpy(workloads.bf16_normal(g, (K,), mean=1.0, std=0.1).view(np.int16)).view(
        torch.bfloat16).to(dev)
    s_a = torch.tensor([float(workloads.STATIC_INPUT_SCALE)], dtype=torch.float32, device=dev)
    W = [workloads.device_e4m3_codes(torch, (N, K), seed=300 + i, device=dev).view(torch.float8_e4m3fn)
         for i in range(3)]
    sb = workloads.device_uniform_f32(torch, (N,), 0.5e-3, 2e-3, seed=400, device=dev)
    A = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    kind = args.profile_kind
    if kind == "blockwise":  # per-token-group activations x 128x128-block weights
        sag = torch.empty((M, (K + 127) // 128), dtype=torch.float32, device=dev)
        sbb = workloads.device_uniform_f32(torch, ((N + 127) // 128, (K + 127) // 128), 0.5e-3, 2e-3, seed=401,
                                           device=dev)
    for i in range(args.steps):
        if kind == "w8a16":  # bf16 activations, E4M3 weights: no activation quantisation
            fp8.w8a16_mm(x, W[i % 3], sb, fp8.GRAN_PER_CHANNEL, out=Y)
        elif kind == "blockwise":
            fp8.quant_per_token_group(x, out=A, scale_out=sag)
            fp8.fp8_scaled_mm(A, W[i % 3], sag, sbb, fp8.GRAN_BLOCK_128, out=Y)
        else:
            fp8.rmsnorm_quant_fp8(x, gamma, workloads.RMS_EPS, s_a, out=A)
            fp8.fp8_scaled_mm(A, W[i % 3], s_a, sb, fp8.GRAN_PER_CHANNEL, out=Y)
    torch.cuda.synchronize()
    err = fp8.get_device_error()
    print(json.dumps({"profile_case": [M, N, K], "kind": kind, "device_error": err}))
    if err:
        raise SystemExit(1)


def whole_job_tbps(world, bytes_per_step, ms_per_step):
    """The whole job's rate: every rank runs the same step (replicas), so the
    bytes of all ranks over the slowest rank's step time."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e12


def dist_ops(dist, device):
    """A barrier and a max over ranks of one float, through the process group
    `dist` (None: one process); `device` holds the reduced tensor ("cuda" for
    NCCL, "cpu" for gloo)."""
    def barrier():
        if dist is not None:
            dist.barrier()

    def dmax(v):
        if dist is None:
            return v
        import torch
        t = torch.tensor([float(v)], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, dmax


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="wall-time budget of the oracle CPU baseline")
    ap.add_argument("--ref-seconds", type=float, default=60.0, help="wall-time budget of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill-chunk GEMM measurement")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the gate_up decode, 64-layer decode step and tiny GEMM measurements")
    ap.add_argument("--profile", metavar="M,N,K", help="run a small eager case for a profiler and exit")
    ap.add_argument("--profile-kind", choices=("w8a8", "w8a16", "blockwise", "step"), default="w8a8",
                    help="the GEMM of the --profile case: per-channel W8A8 after the norm-quant (default), "
                         "weight-only W8A16, or blockwise-scaled W8A8 after the per-token-group quant; or "
                         "'step': the 64-layer decode step at M tokens (N, K ignored)")
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args)
        return
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")

    barrier, dmax = dist_ops(dist, "cuda")
    out = run_ours(args, rank, world, barrier, dmax)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
