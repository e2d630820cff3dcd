#!/usr/bin/env python3
"""Benchmark of the fused MoE layer forward on one GB300 (per rank).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-sweep]

A step is one call of the whole layer (routing, permutation, grouped gate+up
GEMM with SiLU, grouped down GEMM with the weighted combine, output cast)
over one batch whose inputs are already resident in HBM.  Between timed
steps a 256 MiB buffer is written to flush L2, outside the per-step CUDA
events.  Rank 0 prints one JSON line.

After the headline's timed region, rank 0 also measures the batch sweep of
the metric: every workload (decode, sparse E=400 with and without the old
estimate and the EP8 slice, the FP8 batch sweep T=1..4096, skewed prefill)
timed as µs per call over 24 CUDA-graph replays after 5 warm-ups, each with
its roofline fractions, plus the routing micro-benchmark (--no-sweep skips
both).

Under torchrun every rank runs an independent replica of the layer on its
own GPU (tokens are independent; there is no exchange step), so the work
per GPU is fixed as N grows ("weak" scaling).

--impl reference times the CPU oracle (the plain C restatement of the
method) on the host cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused-MoE layer µs/call & tokens/s vs batch; % of HBM/tensor roofline, 1 GB300"
HBM_ROOFLINE_GBS = 8000.0
FLUSH_BYTES = 256 << 20
SWEEP = ["decode_bf16", "decode_grouped_bf16", "sparse_uniform_bf16", "sparse_concentrated_bf16",
         "sparse_uniform_bf16_old_est", "sparse_concentrated_bf16_old_est",
         "sparse_uniform_bf16_ep8", "sparse_uniform_bf16_ep8_old_est",
         "fp8_T1", "fp8_T2", "fp8_T4", "fp8_T16", "fp8_T64", "fp8_T128", "fp8_T256", "fp8_T1024",
         "fp8_T4096", "skewed_prefill_bf16", "skewed_prefill_sigmoid_bf16", "tiny_f32"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_bf16")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the per-workload sweep and the routing micro-benchmark")
    ap.add_argument("--sweep-samples", type=int, default=24)
    ap.add_argument("--sweep-only", default="",
                    help="comma-separated workload names: sweep only these")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def strip_c_comments(text):
    """C/C++ source without comments and with runs of whitespace collapsed,
    so that comment-only edits leave the code's fingerprint unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal, copied as is
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_fingerprint():
    """sha256 over the CUDA sources (csrc/*.cu, *.cuh) with comments removed."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "serving_moe_route_gb300", "csrc")
    for fn in sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh"))):
        with open(fn, encoding="utf-8") as f:
            h.update(strip_c_comments(f.read()).encode())
    return h.hexdigest()


def ncu_traffic(workload):
    """DRAM bytes (read + write) per launch of the dominant GEMM kernel from
    the committed ncu summary, if it was taken from the current kernel code
    (the comment-free source fingerprint matches); else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get("entries", {}).get(workload)
    if e is None or d.get("source_sha256") != kernel_source_fingerprint():
        return None
    return int(e["dram_read_bytes"] + e["dram_write_bytes"])


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def measure_fp8_peak(dev, n=8192, reps=10):
    """Dense FP8 (e4m3 x e4m3 -> bf16) matmul throughput of this GPU: the
    best of `reps` CUDA-event-timed torch._scaled_mm calls on n x n x n
    (2 n^3 FLOP each), after three warm-up calls.  Returns TFLOP/s, or None
    when the call is unavailable."""
    import torch
    try:
        g = torch.Generator(device="cpu")
        g.manual_seed(8)
        a = torch.randn(n, n, generator=g).to(dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, generator=g).to(dev).to(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize(dev)
        best = None
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b
        return round(2.0 * n ** 3 / (best * 1e-3) / 1e12, 1)
    except (RuntimeError, AttributeError, TypeError):
        return None


def tensor_peak(wl, pk):
    """Dense tensor peak (TFLOP/s) for the workload's operand type: bf16
    measured; FP8 measured by the probe when it ran, else 2 x bf16 (the
    nominal ratio); TF32 half of bf16 (nominal ratio)."""
    from serving_moe_route_gb300 import workloads as W
    if wl.dtype == W.FP8:
        if pk.get("fp8_tflops"):
            return pk["fp8_tflops"], "measured (torch._scaled_mm e4m3 8192^3 probe)"
        return 2.0 * pk["bf16_tflops"], "2 x measured bf16 (nominal ratio; fp8 probe unavailable)"
    if wl.dtype == W.F32:
        return pk["bf16_tflops"] / 2.0, "measured bf16 / 2 (nominal tf32 ratio)"
    return pk["bf16_tflops"], pk["source"]


# ------------------------------------------------------------ accounting
def bytes_per_elem(dtype):
    from serving_moe_route_gb300 import workloads as W
    return {W.F32: 4, W.BF16: 2, W.FP8: 1}[dtype]


def algorithmic(wl, counts):
    """Algorithmic FLOPs and bytes of one layer call and of each GEMM launch.

    FLOPs = 6*T*k*H*I.  Layer bytes = touched experts x (w13 + w2 + scales)
    + logits + x + out.  GEMM1 bytes = touched x (w13 + scales) + permuted
    x rows + act rows; GEMM2 bytes = touched x (w2 + scales) + act rows +
    the fp32 combine accumulator written once."""
    from serving_moe_route_gb300 import workloads as W
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    bw = bytes_per_elem(wl.dtype)
    bx = 4 if wl.dtype == W.F32 else 2
    touched = int(sum(1 for c in counts if c > 0))
    s13 = (2 * I // 128) * (H // 128) * 4 if wl.dtype == W.FP8 else 0
    s2 = (H // 128) * (I // 128) * 4 if wl.dtype == W.FP8 else 0
    w13 = 2 * I * H * bw + s13
    w2 = H * I * bw + s2
    R = T * k
    layer = touched * (w13 + w2) + T * E * bx + T * H * bx + T * H * bx
    g1 = touched * w13 + R * H * bw + R * I * bw
    g2 = touched * w2 + R * I * bw + T * H * 4
    return {"flops": 6.0 * T * k * H * I, "layer_bytes": layer, "g1_bytes": g1, "g2_bytes": g2,
            "touched": touched, "w13_bytes_per_expert": w13, "w2_bytes_per_expert": w2}


# ------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
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
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ GPU arm
class Runner:
    """One workload resident on the GPU, timed per stage with CUDA events."""

    def __init__(self, wl, inp, dev):
        import torch

        from serving_moe_route_gb300 import MoELayer
        self.torch = torch
        self.wl = wl
        self.dev = dev
        s13 = inp["s13"].to(dev) if inp["s13"] is not None else None
        s2 = inp["s2"].to(dev) if inp["s2"] is not None else None
        self.layer = MoELayer(inp["w13"].to(dev), inp["w2"].to(dev), k=wl.k, dtype=wl.dtype,
                              scoring=wl.scoring, renorm=wl.renorm, s13=s13, s2=s2,
                              force_est=wl.force_est, ep_size=wl.ep_size, ep_rank=wl.ep_rank,
                              n_group=wl.n_group, topk_group=wl.topk_group,
                              gemm_pair=wl.gemm_pair, gemm_tm=wl.gemm_tm)
        self.x = inp["x"].to(dev)
        self.lg = inp["logits"].to(dev)
        self.out = torch.empty(wl.T, wl.H, dtype=self.x.dtype, device=dev)
        self.flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.plan = self.layer.plan(wl.T)
        self.ws = self.layer.workspace(wl.T)
        self.x_h = inp["x"].pin_memory()
        self.lg_h = inp["logits"].pin_memory()
        self.out_h = torch.empty(wl.T, wl.H, dtype=self.x.dtype).pin_memory()

    def _events(self, n):
        # torch creates the CUDA event lazily: record each once so that its
        # handle exists before the library records it again
        evs = [[self.torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(n)]
        for row in evs:
            for e in row:
                e.record(self.stream)
        return evs

    def step_timed(self, ev):
        from serving_moe_route_gb300 import _binding as B
        L = self.layer
        rc = B.moe_forward_timed(self.plan, self.x.data_ptr(), self.lg.data_ptr(),
                                 L.w13.data_ptr(), 0 if L.s13 is None else L.s13.data_ptr(),
                                 L.w2.data_ptr(), 0 if L.s2 is None else L.s2.data_ptr(),
                                 self.out.data_ptr(), self.ws.data_ptr(), self.ws.numel(),
                                 self.stream.cuda_stream, [e.cuda_event for e in ev])
        B._check(rc, "moe_forward_timed")

    def capture(self):
        """One CUDA graph of the whole forward for this call shape (the
        library's launches and its error-word memset become graph nodes)."""
        torch = self.torch
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(side):
            for _ in range(2):  # first calls set kernel attributes outside capture
                self.layer.forward(self.x, self.lg, self.out)
        torch.cuda.current_stream(self.dev).wait_stream(side)
        torch.cuda.synchronize(self.dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.layer.forward(self.x, self.lg, self.out)
        torch.cuda.synchronize(self.dev)

    def run(self, steps, warmup):
        """Timed region: `steps` graph replays, each bracketed by CUDA events
        on the replay stream; L2 flushed before each, outside the events."""
        torch = self.torch
        if getattr(self, "graph", None) is None:
            self.capture()
        for i in range(warmup):
            self.flush.fill_(i & 0xFF)
            self.graph.replay()
        torch.cuda.synchronize(self.dev)
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(steps)]
        for i in range(steps):
            self.flush.fill_(i & 0xFF)
            pairs[i][0].record()
            self.graph.replay()
            pairs[i][1].record()
        torch.cuda.synchronize(self.dev)
        rc, bits = self.layer.check(self.wl.T)
        if rc != 0:
            raise RuntimeError(f"device error word {bits:#x} after the timed steps")
        return [a.elapsed_time(b) for a, b in pairs]

    def run_stages(self, steps, warmup=2):
        """Per-launch times from moe_forward_timed (events between the
        library's launches; not graphed, so launch gaps are included)."""
        torch = self.torch
        for i in range(warmup):
            self.flush.fill_(i & 0xFF)
            self.step_timed(self._events(1)[0])
        torch.cuda.synchronize(self.dev)
        evs = self._events(steps)
        for i in range(steps):
            self.flush.fill_(i & 0xFF)
            self.step_timed(evs[i])
        torch.cuda.synchronize(self.dev)
        stages = {"route": (0, 1), "scan": (1, 2), "gather": (2, 3), "gemm1": (3, 4),
                  "gemm2": (4, 5), "combine": (5, 6), "step": (0, 6)}
        return {name: [evs[i][a].elapsed_time(evs[i][b]) for i in range(steps)]
                for name, (a, b) in stages.items()}

    def run_e2e(self, steps, warmup):
        """Host buffers in, host buffer out: H2D of x and logits, the layer
        through the public API, D2H of the output, all inside the events."""
        torch = self.torch
        times = []
        for i in range(warmup + steps):
            self.flush.fill_(i & 0xFF)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            self.x.copy_(self.x_h, non_blocking=True)
            self.lg.copy_(self.lg_h, non_blocking=True)
            self.layer.forward(self.x, self.lg, self.out)
            self.out_h.copy_(self.out, non_blocking=True)
            b.record()
            if i >= warmup:
                times.append((a, b))
        torch.cuda.synchronize(self.dev)
        ms = [a.elapsed_time(b) for a, b in times]
        h2d = self.x_h.numel() * self.x_h.element_size() + self.lg_h.numel() * \
            self.lg_h.element_size()
        d2h = self.out_h.numel() * self.out_h.element_size()
        return ms, h2d, d2h

    def counts(self):
        return self.layer.intermediates(self.wl.T)["counts"].cpu().tolist()

    def family(self):
        """The GEMM kernel family the last call picked on the device (1 one
        CTA per tile, 2 CTA pairs), or None for plans that fix it."""
        if not self.plan.gemm_dyn:
            return None
        return int(self.layer.intermediates(self.wl.T)["family"][0])


def job_throughput(local_seconds, units_per_rank, device=None):
    """Whole-job throughput of independent replicas: every rank processed
    units_per_rank units; the job's time is the max over ranks of their timed
    regions (all_reduce MAX).  Returns (units/s over all ranks, job seconds)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    t = float(local_seconds)
    if world > 1:
        x = torch.tensor([t], dtype=torch.float64, device=device)
        dist.all_reduce(x, op=dist.ReduceOp.MAX)
        t = float(x.item())
    return world * units_per_rank / t, t


def pct(v, q):
    s = sorted(v)
    return s[min(len(s) - 1, max(0, int(round(q * (len(s) - 1)))))]


def gemm_roofline(wl, stage_ms, acc, pk, family=None, plan=None):
    """The dominant kernel (the GEMM with the larger mean time) against the
    measured HBM copy bandwidth (decode-sized batches) or bf16 tensor peak.
    family: the kernel family a per-call plan picked (stage 'gemm1' then
    spans the single-CTA launch, 'gemm2' the CTA-pair ones), else None.
    plan: the layer's plan, which names the kernel."""
    from serving_moe_route_gb300 import workloads as W
    kern = "moe_gemm_kernel"
    if plan is not None and wl.dtype == W.FP8 and plan.gemm_tm:
        kern = "moe_gemm_tm_kernel"
    elif plan is not None and wl.dtype != W.FP8 and (plan.gemm_pair or family == 2):
        kern = "moe_gemm_pair_kernel"
    g1 = statistics.mean(stage_ms["gemm1"])
    g2 = statistics.mean(stage_ms["gemm2"])
    both = acc["g1_bytes"] + acc["g2_bytes"]
    if family == 2:
        name, ms, nbytes, flops = "gemm1+gemm2 on CTA pairs (picked per call)", g2, both, \
            acc["flops"]
    elif family == 1:
        name, ms, nbytes, flops = "gemm1+gemm2 fused (picked per call)", g1, both, acc["flops"]
    elif g2 < 0.02 * g1:  # both GEMMs ran as one launch (shared tile list)
        name, ms, nbytes, flops = "gemm1+gemm2 fused", g1, both, acc["flops"]
    elif g1 >= g2:
        name, ms, nbytes, flops = "gemm1", g1, acc["g1_bytes"], acc["flops"] * 2.0 / 3.0
    else:
        name, ms, nbytes, flops = "gemm2", g2, acc["g2_bytes"], acc["flops"] / 3.0
    t_mem = nbytes / (pk["hbm_gbs"] * 1e9)
    tensor_pk, tensor_src = tensor_peak(wl, pk)
    t_cmp = flops / (tensor_pk * 1e12)
    if t_mem >= t_cmp:
        achieved = nbytes / (ms * 1e-3) / 1e9
        return name, {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                      "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                      "traffic": None, "kernel": f"{kern} ({name})",
                      "algorithmic_bytes": int(nbytes), "mean_ms": round(ms, 5),
                      "peak_source": pk["source"]}
    achieved = flops / (ms * 1e-3) / 1e12
    return name, {"bound": "tensor", "achieved": round(achieved, 1), "peak": tensor_pk,
                  "unit": "TFLOP/s", "frac": round(achieved / tensor_pk, 4), "traffic": None,
                  "kernel": f"{kern} ({name})", "algorithmic_flops": flops,
                  "mean_ms": round(ms, 5), "peak_source": tensor_src}


def layer_roofline(wl, step_ms, acc, pk):
    """Roofline of the whole layer: max(FLOPs / tensor peak,
    bytes / 8 TB/s); also against the measured copy bandwidth."""
    tp, _ = tensor_peak(wl, pk)
    t_c = acc["flops"] / (tp * 1e12)
    t_ns = max(t_c, acc["layer_bytes"] / (HBM_ROOFLINE_GBS * 1e9))
    t_meas = max(t_c, acc["layer_bytes"] / (pk["hbm_gbs"] * 1e9))
    s = step_ms * 1e-3
    return {"floor_us_8tbs": round(t_ns * 1e6, 2), "frac_8tbs": round(t_ns / s, 4),
            "floor_us_measured_hbm": round(t_meas * 1e6, 2), "frac_measured_hbm": round(t_meas / s, 4),
            "bound": "tensor" if t_c * 1e0 >= acc["layer_bytes"] / (pk["hbm_gbs"] * 1e9) else "hbm",
            "flops": acc["flops"], "bytes": acc["layer_bytes"], "touched_experts": acc["touched"]}


def oracle_args(wl, inp):
    from serving_moe_route_gb300 import workloads as W
    return dict(T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, dtype=wl.dtype, scoring=wl.scoring,
                renorm=wl.renorm, x=W.storage_numpy(inp["x"]),
                logits=W.storage_numpy(inp["logits"]), w13=W.storage_numpy(inp["w13"]),
                w2=W.storage_numpy(inp["w2"]), s13=W.storage_numpy(inp["s13"]),
                s2=W.storage_numpy(inp["s2"]), ep_size=wl.ep_size, ep_rank=wl.ep_rank,
                n_group=wl.n_group, topk_group=wl.topk_group)


def time_oracle(args, n_tokens, seconds):
    """Passes of the oracle over the first n_tokens tokens until about
    `seconds` have gone by (at least one).  Returns (tokens/s, passes, s)."""
    import numpy as np

    import oracle
    toks = np.arange(n_tokens, dtype=np.int32)
    t0 = time.perf_counter()
    passes = 0
    while True:
        oracle.moe_forward(**args, tokens=toks)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            return n_tokens * passes / dt, passes, dt


def cpu_baseline(wl, inp, seconds):
    """The oracle as it stands, on the host cores: OpenMP over tokens on
    every core, passes over a token sample for about `seconds`; for batches
    of at most 128 tokens also one thread on a smaller sample."""
    import numpy as np

    import oracle
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    args = oracle_args(wl, inp)
    n = min(wl.T, max(1, cores))
    t0 = time.perf_counter()
    oracle.moe_forward(**args, tokens=np.arange(n, dtype=np.int32))
    dt = max(time.perf_counter() - t0, 1e-6)
    n = int(min(wl.T, max(n, n * seconds / dt)))  # one pass of about `seconds` at most
    rate, passes, dt = time_oracle(args, n, seconds)
    out = {"value": round(rate, 3), "unit": "tokens/s", "cores": oracle.threads(),
           "kind": "oracle",
           "sample": f"first {n} of {wl.T} tokens of {wl.name} (routing, expert MLPs and combine "
                     f"for those tokens) x {passes} passes, {dt:.2f} s, OpenMP over tokens"}
    if wl.T <= 128:
        oracle.set_threads(1)
        n1 = min(wl.T, 16)
        r1, p1, d1 = time_oracle(args, n1, seconds / 4)
        out["single_thread"] = {"value": round(r1, 3), "unit": "tokens/s", "cores": 1,
                                "sample": f"first {n1} tokens x {p1} passes, {d1:.2f} s"}
        oracle.set_threads(cores)
    return out


def routing_bench(dev, calls=500):
    """The routing micro-benchmark of PR #39593 ("Test Plan", item 3): 128
    tokens x 128 experts, top-8, bf16 logits with 10% all-NaN rows.  moe_route_topk
    (NaN sanitised in registers) against the same call behind a separate
    nan_to_num launch; per-call CUDA-event times, p20/p50/p80 in µs."""
    import torch

    from serving_moe_route_gb300 import route_topk
    from serving_moe_route_gb300 import workloads as W
    wl = W.workloads()["decode_bf16"]
    lg = W.make_logits(wl).to(dev)
    out = {}
    for scoring, sname in ((W.SOFTMAX, "topk_softmax"), (W.SIGMOID, "topk_sigmoid")):
        for variant in ("fused", "separate_nan_to_num"):
            def call():
                x = lg
                if variant != "fused":
                    x = torch.nan_to_num(lg, nan=float("-inf"))
                return route_topk(x, wl.k, scoring=scoring, renorm=True)
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                for _ in range(3):
                    call()
            torch.cuda.current_stream(dev).wait_stream(side)
            torch.cuda.synchronize(dev)
            # one graph per variant, replayed: device time per call without
            # the host's per-call launch cost
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call()
            for _ in range(20):
                g.replay()
            torch.cuda.synchronize(dev)
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(calls)]
            for a, b in pairs:
                a.record()
                g.replay()
                b.record()
            torch.cuda.synchronize(dev)
            us = [a.elapsed_time(b) * 1e3 for a, b in pairs]
            out[f"{sname}_{variant}"] = {"p20": round(pct(us, 0.2), 2),
                                         "p50": round(pct(us, 0.5), 2),
                                         "p80": round(pct(us, 0.8), 2)}
    out["config"] = ("T=128, E=128, top-8, bf16 logits, 13 all-NaN rows; CUDA-graph replays, "
                     "events around each replay")
    return out


def sweep(dev, samples, pk, only=()):
    """Every workload (or those in `only`): median/p20/p80 us per call,
    tokens/s, roofline."""
    import torch

    from serving_moe_route_gb300 import workloads as W
    wls = W.workloads()
    wkey, weights = None, None
    rows = []
    for name in (only or SWEEP):
        wl = wls[name]
        key = (wl.H, wl.I, wl.E, wl.dtype, wl.seed, wl.ep_size, wl.ep_rank)
        if key != wkey:  # weights depend on (H, I, E, dtype, seed, ep slice) only
            weights = None
            torch.cuda.empty_cache()
            wkey, weights = key, W.make_weights(wl)
        inp = dict(weights)
        inp.update(W.make_activations(wl))
        r = Runner(wl, inp, dev)
        steps = r.run(samples, 5)
        st = r.run_stages(samples)
        acc = algorithmic(wl, r.counts())
        med = statistics.median(steps)
        gname, groof = gemm_roofline(wl, st, acc, pk, r.family(), r.plan)
        rows.append({
            "workload": name, "T": wl.T, "E": wl.E, "k": wl.k, "dtype": W.DTYPE_NAMES[wl.dtype],
            "scoring": "sigmoid" if wl.scoring else "softmax", "est_tile": [r.plan.est,
                                                                             r.plan.tile_n],
            "us_median": round(med * 1e3, 2), "us_p20": round(pct(steps, 0.2) * 1e3, 2),
            "us_p80": round(pct(steps, 0.8) * 1e3, 2),
            "tokens_per_s": round(wl.T / (med * 1e-3), 1),
            "stage_us_eager": {k2: round(statistics.median(v) * 1e3, 2) for k2, v in st.items()},
            "layer_roofline": layer_roofline(wl, med, acc, pk),
            "gemm_roofline": groof,
            "routing": {"touched_experts": acc["touched"], "max_rows": max(r.counts()),
                        "mean_rows_touched": round(wl.T * wl.k / max(1, acc["touched"]), 2)},
        })
        del r
    return rows


def estimate_ablation(rows):
    """The H20 article's comparison on each workload that the sweep also ran
    with the old token-count estimate: µs per call of each, and old / new
    (above 1: the rows-per-expert estimate is faster)."""
    us = {r["workload"]: r["us_median"] for r in rows}
    out = {}
    for name, new in us.items():
        old = us.get(name + "_old_est")
        if old:
            out[name] = {"us_estimate": new, "us_old_estimate": old,
                         "old_over_new": round(old / new, 3)}
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    from serving_moe_route_gb300 import _build
    from serving_moe_route_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group(backend="nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()

    pk = peaks()
    wl = W.workloads()[args.workload]
    inp = W.make_inputs(wl)
    r = Runner(wl, inp, dev)
    steps, warmup = args.steps, max(3, args.warmup)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
    step_ms = r.run(steps, warmup)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    st = r.run_stages(min(steps, 100))

    value, total_s = job_throughput(sum(step_ms) * 1e-3, steps * wl.T, dev)
    ms_per_step = total_s * 1e3 / steps

    e2e_steps = max(10, min(steps, 200))
    e2e_ms, h2d, d2h = r.run_e2e(e2e_steps, 3)
    e2e_val, _ = job_throughput(sum(e2e_ms) * 1e-3, e2e_steps * wl.T, dev)

    acc = algorithmic(wl, r.counts())
    gname, groof = gemm_roofline(wl, st, acc, pk, r.family(), r.plan)
    groof["traffic"] = ncu_traffic(wl.name)
    groof["traffic_source"] = ("profiles/ncu_traffic.json (ncu --set full, same kernel sources)"
                               if groof["traffic"] is not None else None)
    fused = statistics.mean(st["gemm2"]) < 0.02 * statistics.mean(st["gemm1"])
    # route, scan, gather, the GEMM launch(es), combine; a per-call plan
    # queues both families (two CTA-pair launches and one single-CTA launch)
    launches_per_step = 7 if r.plan.gemm_dyn else 5 if fused else 6
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_call_median": round(statistics.median(step_ms) * 1e3, 2),
        "us_per_call_p20": round(pct(step_ms, 0.2) * 1e3, 2),
        "us_per_call_p80": round(pct(step_ms, 0.8) * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": W.DTYPE_NAMES[wl.dtype], "data": "synthetic (seeded; see workloads.py)",
        "config": {"workload": wl.name, "T": wl.T, "hidden": wl.H, "intermediate": wl.I,
                   "experts": wl.E, "top_k": wl.k,
                   "scoring": "sigmoid" if wl.scoring else "softmax", "renorm": wl.renorm,
                   "est": r.plan.est, "tile_n": r.plan.tile_n,
                   "parallelism": f"replicas x{world} (independent token batches)",
                   "l2": "256 MiB buffer written between timed steps, outside the step events; "
                         "touched weights also exceed L2",
                   "timing": "one CUDA graph of moe_forward per call shape, replayed; per-step "
                             "CUDA events on the replay stream"},
        "stage_us_eager": {k: round(statistics.median(v) * 1e3, 2) for k, v in st.items()},
        "roofline": groof,
        "layer_roofline": layer_roofline(wl, statistics.median(step_ms), acc, pk),
        "e2e": {"value": round(e2e_val, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "us_per_call_median": round(statistics.median(e2e_ms) * 1e3, 2)},
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_seconds)
    if rank == 0 and not args.no_sweep:
        # the batch sweep of the metric (every workload, 24 samples after 5
        # warm-ups each) and the routing micro-benchmark, after the headline's
        # timed region; FP8 rooflines divide by the measured FP8 peak
        del r
        pk["fp8_tflops"] = measure_fp8_peak(dev)
        line["peaks"] = {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                         "fp8_tflops": pk["fp8_tflops"],
                         "fp8_source": "torch._scaled_mm e4m3 8192^3, best of 10 (this run)"
                         if pk["fp8_tflops"] else "unavailable: 2 x bf16 used",
                         "source": pk["source"]}
        line["routing_microbench"] = routing_bench(dev)
        t0 = time.perf_counter()
        only = tuple(n for n in args.sweep_only.split(",") if n)
        line["sweep"] = sweep(dev, args.sweep_samples, pk, only)
        line["sweep_wall_s"] = round(time.perf_counter() - t0, 1)
        line["estimate_ablation"] = estimate_ablation(line["sweep"])
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_reference(args):
    """The oracle (plain C, OpenMP) timed on the host cores: each step is a
    bounded sample of the workload's tokens."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    import oracle
    from serving_moe_route_gb300 import workloads as W
    wl = W.workloads()[args.workload]
    inp = W.make_inputs(wl)
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    fa = oracle_args(wl, inp)
    n = min(wl.T, max(1, cores))  # tokens per step: one per host core
    toks = np.arange(n, dtype=np.int32)
    for _ in range(max(0, args.warmup)):
        oracle.moe_forward(**fa, tokens=toks)
    steps = max(1, args.steps)
    budget = 120.0  # keep the reference arm within a few minutes
    t0 = time.perf_counter()
    done = 0
    for _ in range(steps):
        oracle.moe_forward(**fa, tokens=toks)
        done += 1
        if time.perf_counter() - t0 > budget:
            break
    dt = time.perf_counter() - t0
    value = done * n / dt
    sample = f"{n} of {wl.T} tokens of {wl.name} per step, {done} steps, OpenMP over tokens"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": done, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / done, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (fp32 values, double accumulation)",
        "data": "synthetic (seeded; see workloads.py)",
        "config": {"workload": wl.name, "T": wl.T, "hidden": wl.H, "intermediate": wl.I,
                   "experts": wl.E, "top_k": wl.k},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
