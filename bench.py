#!/usr/bin/env python
"""MoE-layer throughput on GB300: tokens/s and fraction of roofline.

Default workload (one step = forward + backward of one MoE layer):
  bf16, T=2048 tokens, d=2048, E=64 experts, f=1408, top-6 softmax router
  renormalised over the top-6, router bias giving a Zipf(s=1.0) expert load.
Extra workloads in the same JSON line (key "extra"): the DeepSeek-V3-shaped
bf16 forward (T=8192, d=7168, 256 routed + 1 shared expert, f=2048, top-8
sigmoid x 2.5; uniform and Zipf s=1.2 routing) and small-batch decode B=1/4/16.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0. Inputs are synthetic (moe_synth), resident in
HBM before the timed region; the expert weights (1.1 GB) exceed L2 and stream
from HBM every step, so no L2 flush is inserted. "e2e" repeats the step
through the C ABI with host-resident x and dy copied in and y and dx copied out
every step. The step itself is timed as a replay of one CUDA graph holding its
C-ABI calls ("eager_ms_per_step": the same calls launched one by one).
"roofline" is for the kernel group with the largest time share.
The reference arm (--impl reference) times the CPU oracle on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth  # noqa: E402

METRIC = "MoE-layer tokens/s fwd, fwd+bwd, decode on 1×GB300; % of roofline"
# The pages' own figures, on their hardware (multi-GPU NVL72 systems, relative speedups of their
# kernels over their previous ones): context for the reader, not a target or a ratio of ours.
PAGES_CONTEXT = {
    "warp decoding, Blackwell": "1.84x decode throughput (toolnavs.com, 'Cursor a reecrit le decodage de MoE')",
    "MoE layer, 64 GPUs of a GB300 NVL72, 2048 tokens/GPU": "MXFP8 2.37x fwd / 1.78x bwd, BF16 1.92x fwd / 1.58x bwd",
    "training at 512 GB300 GPUs": "760.9 -> 1070.2 tokens/s/GPU",
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled while running: through NVML (read-only
    queries, every 2 ms, so that a timed region of a few milliseconds still gets samples) when
    libnvidia-ml loads, else nvidia-smi every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons (nvml.h)
    NVML_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.samples = []        # NVML: (sm MHz, max sm MHz, reason bits)
        self.stop = threading.Event()
        self.thread = None

    def _nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
                return None
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            return lib, h, reasons
        except (OSError, AttributeError):
            return None

    def _poll(self, lib, h, reasons):
        import ctypes
        clk, mx, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                    reasons(h, ctypes.byref(bits)) == 0):
                self.samples.append((clk.value, mx.value, bits.value))
            time.sleep(0.002)

    def __enter__(self):
        nv = self._nvml()
        if nv:
            self.thread = threading.Thread(target=self._poll, args=nv, daemon=True)
            self.thread.start()
            time.sleep(0.005)
            return self
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        if self.samples:
            for c, m, bits in self.samples:
                sm.append(float(c))
                mx.append(float(m))
                reasons.update(n for n, b in self.NVML_BITS.items() if bits & b)
            src = "nvml, 2 ms"
        else:
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in self.lines:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
            src = "nvidia-smi, 200 ms"
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm), "source": src}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------- algorithmic work per group

def work_per_group(spec, cnt, training=True):
    """Algorithmic (flops, bytes) of one launch of each kernel group for the realised expert loads.

    Bytes count what each step must move at least once: weights of experts that
    received tokens, activations read and written once.
    """
    T, d, E, S, f, k = spec.T, spec.d, spec.E, spec.S, spec.f, spec.k
    A = T * k
    R = A + S * T
    active = int(np.count_nonzero(cnt)) + S
    w13 = active * 2 * f * d * 2
    wd = active * d * f * 2
    g = {}
    g["router_logits"] = (2 * T * E * d, T * d * 2 + E * d * 2 + T * E * 4)
    g["gateup"] = (2 * R * 2 * f * d, w13 + T * d * 2 + R * f * 2 + (R * 2 * f * 2 if training else 0))
    g["down"] = (2 * R * d * f, wd + R * f * 2 + R * d * 2)
    g["combine"] = (R * d, R * d * 2 + T * d * 2)
    g["bwd_dh"] = (2 * R * f * d, wd + T * d * 2 + R * 2 * f * 2 * 2 + R * f * 2)
    g["bwd_dx"] = (2 * R * d * 2 * f, w13 + R * 2 * f * 2 + R * d * 2)
    g["bwd_dw13"] = (2 * R * 2 * f * d, (E + S) * 2 * f * d * 2 + R * 2 * f * 2 + T * d * 2)
    g["bwd_dwd"] = (2 * R * d * f, (E + S) * f * d * 2 + R * f * 2 + T * d * 2)
    g["dx_gather"] = (R * d, R * d * 2 + T * d * 2)
    g["decode_gateup"] = (2 * R * 2 * f * d, w13 + T * d * 2)
    g["decode_down"] = (2 * R * d * f, wd + R * f * 4 + T * d * 2)
    return g


def layer_work(spec, cnt, kind="fwd"):
    """Algorithmic (flops, bytes) of one whole call, from the method's definition.

    FLOPs: the routed expert products (shared expert included; never the dense E-expert FFN that
    routing avoids) and the router GEMM. Bytes that must move at least once: the weights of the
    experts that received tokens, the router weight, the activations in and out. What an
    implementation writes and reads back between its kernels (h, the gated expert outputs before
    the combine) is not algorithmic work; it shows in the ncu traffic instead.
    kind "fwd" (also decode: the forward of B tokens) or "fwd+bwd": the backward reads the used
    experts' weights once more, writes every expert's weight gradients once, reads x and dy, writes
    dx, and reads the u, v pre-activations the forward saved (written once by the forward).
    """
    T, d, E, S, f, k = spec.T, spec.d, spec.E, spec.S, spec.f, spec.k
    eb = 4 if spec.dtype == "fp32" else 2
    R = T * k + S * T
    active = int(np.count_nonzero(np.asarray(cnt)[:E])) + S
    w_used = active * 3 * f * d * eb
    fl = 2 * R * 3 * f * d + 2 * T * E * d
    by = w_used + E * d * eb + 2 * T * d * eb
    if kind == "fwd":
        return fl, by
    fl += 2 * (2 * R * 3 * f * d) + 2 * (2 * T * E * d)
    by += w_used + (E + S) * 3 * f * d * eb + 3 * T * d * eb + 2 * R * 2 * f * eb
    return fl, by


def roof_line(ms, flops, nbytes, pk, tensor_peak=None):
    """Whole-call roofline: t_roof = max(flops / tensor peak, bytes / HBM bandwidth), and ms's fraction."""
    tp = tensor_peak or pk["bf16_tflops"]
    t_t, t_h = flops / (tp * 1e12), nbytes / (pk["hbm_gbs"] * 1e9)
    t_roof = max(t_t, t_h)
    return {"GB": nbytes / 1e9, "TFLOP": flops / 1e12, "roofline_ms": t_roof * 1e3,
            "bound": "tensor" if t_t >= t_h else "hbm", "frac_of_roofline": t_roof * 1e3 / ms}


def host_cpu():
    """Host CPU model and online core count (the oracle's machine)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as fh:
                for line in fh:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"model": model or platform.machine(), "nproc": os.cpu_count()}


def roofline_entry(group, ms_per_launch, flops, nbytes, pk, traffic=None):
    t_tensor = flops / (pk["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        achieved = flops / (ms_per_launch * 1e-3) / 1e12
        return {"kernel": group, "bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"], "traffic": traffic,
                "peak_source": pk["source"] + " (burst)"}
    achieved = nbytes / (ms_per_launch * 1e-3) / 1e9
    return {"kernel": group, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": traffic, "peak_source": pk["source"]}


def written_bytes(spec):
    """Bytes the weight-gradient kernels write (bf16 gradients of every expert)."""
    nseg = spec.E + spec.S
    return {"bwd_dw13": nseg * 2 * spec.f * spec.d * 2, "bwd_dwd": nseg * spec.f * spec.d * 2}


def write_bandwidth(dev, nbytes=1 << 30, reps=10):
    """HBM write rate (GB/s): time of filling a buffer larger than L2, CUDA events."""
    buf = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        buf.fill_(1.0)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        buf.fill_(1.0)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    del buf
    return nbytes / (ms * 1e-3) / 1e9


def stored_traffic(group):
    """dram bytes per launch from the committed ncu summary, if its kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as fh:
            tab = json.load(fh)
        ent = tab.get(group)
        if not ent:
            return None
        h = hashlib.sha256()
        for src in ent["sources"]:
            with open(os.path.join(ROOT, src), "rb") as fh:
                h.update(fh.read())
        if h.hexdigest()[:16] != ent["source_sha256_16"]:
            return None
        return ent["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------ our GPU path

class TrainStep:
    """Preallocated buffers for forward (saving ctx) + backward through the C ABI."""

    def __init__(self, spec, dev):
        from mixture_experts_layer_routing_gb300 import MoeLayer, moe_backward, moe_forward
        self._fwd, self._bwd = moe_forward, moe_backward
        self.spec = spec
        inp = moe_synth.make_inputs(spec, dev, grad=True)
        self.inp = inp
        self.layer = MoeLayer.from_spec(spec, device=dev)
        self.layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
        torch.cuda.synchronize()
        del inp["Wg"], inp["Wu"], inp["Wd"]
        torch.cuda.empty_cache()
        T, d, E, S, f = spec.T, spec.d, spec.E, spec.S, spec.f
        sz = self.layer.sizes(T)
        self.ctx = self.layer.new_ctx(T)
        self.ws = self.layer.buffer("fwd", sz["fwd_ws"])
        self.bws = self.layer.buffer("bwd", sz["bwd_ws"])
        bf = torch.bfloat16
        self.y = torch.empty((T, d), dtype=bf, device=dev)
        self.dx = torch.empty((T, d), dtype=bf, device=dev)
        self.dWr = torch.empty((E, d), dtype=torch.float32, device=dev)
        self.dWg = torch.empty((E + S, f, d), dtype=bf, device=dev)
        self.dWu = torch.empty((E + S, f, d), dtype=bf, device=dev)
        self.dWd = torch.empty((E + S, d, f), dtype=bf, device=dev)

    def __call__(self, x=None, dy=None, y=None, dx=None):
        x = self.inp["x"] if x is None else x
        dy = self.inp["dy"] if dy is None else dy
        y = self.y if y is None else y
        dx = self.dx if dx is None else dx
        h, T = self.layer.h, self.spec.T
        self._fwd(h, x, T, y, self.ctx, self.ws)
        self._bwd(h, x, dy, T, self.ctx, dx, self.dWr, self.dWg, self.dWu, self.dWd, self.bws)


class PipelinedE2E:
    """End-to-end steps through the C ABI with host-resident inputs and outputs, as a training loop
    would run them: step i's x and dy are copied in from pinned host memory on a copy stream while
    step i-1 computes, and step i's y and dx are copied back on another stream while step i+1
    computes (device buffers alternate between two sets). Every step's copies are inside the timed
    region; the region ends when the last step's results are on the host."""

    def __init__(self, step, n_batches=2):
        self.step = step
        src_x, src_dy = step.inp["x"], step.inp["dy"]
        self.x_h = [src_x.cpu().pin_memory() for _ in range(n_batches)]
        self.dy_h = [src_dy.cpu().pin_memory() for _ in range(n_batches)]
        self.y_h = [torch.empty_like(self.x_h[0]).pin_memory() for _ in range(2)]
        self.dx_h = [torch.empty_like(self.x_h[0]).pin_memory() for _ in range(2)]
        self.x_d = [torch.empty_like(src_x) for _ in range(2)]
        self.dy_d = [torch.empty_like(src_dy) for _ in range(2)]
        self.y_d = [torch.empty_like(src_x) for _ in range(2)]
        self.dx_d = [torch.empty_like(src_x) for _ in range(2)]
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        self.bytes_in = self.x_h[0].numel() * 2 + self.dy_h[0].numel() * 2
        self.bytes_out = self.y_h[0].numel() * 2 + self.dx_h[0].numel() * 2

    def run(self, steps):
        comp = torch.cuda.current_stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        nb = len(self.x_h)
        self.s_in.wait_stream(comp)    # nothing of this run starts before the caller's start event

        def copy_in(i):
            b = i % 2
            with torch.cuda.stream(self.s_in):
                if i >= 2:
                    self.s_in.wait_event(ev_done[b])          # step i-2 no longer reads this set
                self.x_d[b].copy_(self.x_h[i % nb], non_blocking=True)
                self.dy_d[b].copy_(self.dy_h[i % nb], non_blocking=True)
                ev_in[b].record(self.s_in)

        copy_in(0)
        for i in range(steps):
            b = i % 2
            if i + 1 < steps:
                copy_in(i + 1)
            comp.wait_event(ev_in[b])
            if i >= 2:
                comp.wait_event(ev_out[b])                    # step i-2's results are on the host
            self.step(self.x_d[b], self.dy_d[b], self.y_d[b], self.dx_d[b])
            ev_done[b].record(comp)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_done[b])
                self.y_h[b].copy_(self.y_d[b], non_blocking=True)
                self.dx_h[b].copy_(self.dx_d[b], non_blocking=True)
                ev_out[b].record(self.s_out)
        for e in ev_out:
            comp.wait_event(e)


def time_steps(fn, steps, warmup, world, stats=None):
    """Mean milliseconds per step over `steps` timed steps (CUDA events on the current stream, after
    `warmup` untimed steps, synchronised and barriered on both sides; max over ranks). With a dict
    `stats`, also fills in the median and the min of the per-step times (an event between steps)."""
    for _ in range(warmup):
        fn()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for i in range(steps):
        fn()
        ev[i + 1].record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    ms = ev[0].elapsed_time(ev[steps]) / steps
    if world > 1:
        ms = reduce_max(ms, "cuda")
    if stats is not None:
        stats.update(ms_mean=ms, ms_median=float(np.median(per)), ms_min=float(min(per)), steps=steps)
    return ms


def reduce_max(value: float, device) -> float:
    """The largest value over all ranks (the slowest rank sets the step time)."""
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def profile_groups(layer_h, fn, steps):
    from mixture_experts_layer_routing_gb300 import moe_profile_enable, moe_profile_read
    moe_profile_read(layer_h)
    moe_profile_enable(layer_h, True)
    for _ in range(steps):
        fn()
    torch.cuda.synchronize()
    moe_profile_enable(layer_h, False)
    return moe_profile_read(layer_h)


def oracle_inputs(inp_cpu):
    """Host float32 copies of the inputs (bf16 values widened exactly); prepared outside any timer."""
    return {k: v.float().numpy() for k, v in inp_cpu.items()}


def cpu_baseline(spec, n, n_tokens, training=True):
    """Seconds the oracle, as it stands, takes for the first n_tokens tokens of the workload (host cores)."""
    from oracle import moe_oracle as oracle
    x = n["x"][:n_tokens]
    kw = dict(k=spec.k, router=spec.router, renorm=spec.renorm, scale=spec.route_scale, n_shared=spec.S)
    t0 = time.perf_counter()
    oracle.forward(x, n["Wr"], n["b"], n["Wg"], n["Wu"], n["Wd"], **kw)
    if training:
        oracle.backward(x, n["Wr"], n["b"], n["Wg"], n["Wu"], n["Wd"], n["dy"][:n_tokens], **kw)
    return time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return int(max(i.get("num_threads", 1) for i in info))
    except Exception:
        pass
    return os.cpu_count() or 1


def bench_config(spec, world):
    """The bench line's "config" (the same dict on both arms)."""
    return {"workload": spec.name + " fwd+bwd", "T": spec.T, "d": spec.d, "E": spec.E, "f": spec.f, "k": spec.k,
            "router": "softmax top-6 renorm, Zipf(1.0) load bias", "global_batch": spec.T * world,
            "parallelism": f"replicas x{world}",
            "l2": "no flush: expert weights (1.11 GB) exceed L2 and stream from HBM every step"}


def capture(fn):
    """fn's launches captured once in a CUDA graph (fn only enqueues work)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        fn()
    return graph


def r4(v):
    """v rounded to 4 significant digits (the summary is read from the tail of the output)."""
    return float(f"{v:.4g}") if isinstance(v, float) else v


def summary_row(st, tokens, rl):
    """One line of the per-workload summary: mean / median / min ms per call, tokens/s from the mean,
    the algorithmic work (GB, TFLOP), the whole-call roofline and the mean's fraction of it."""
    row = {"ms": st["ms_mean"], "med": st["ms_median"], "min": st["ms_min"], "tok_s": tokens / (st["ms_mean"] * 1e-3),
           "GB": rl["GB"], "TF": rl["TFLOP"], "roof_ms": rl["roofline_ms"], "bound": rl["bound"],
           "frac": rl["frac_of_roofline"]}
    return {k: r4(v) for k, v in row.items()}


def run_ours(args):
    world, rank, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    from mixture_experts_layer_routing_gb300 import moe_forward, moe_launch_count
    pk = peaks()
    spec = moe_synth.BF16_T2048
    step = TrainStep(spec, dev)
    r = step.layer.route(step.inp["x"])
    cnt = r["cnt"].cpu().numpy()
    # the step's C-ABI calls captured once in a CUDA graph and replayed (the calls only enqueue
    # work, so a training loop can do the same); the eager time of the same calls is reported too
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    n0 = moe_launch_count(step.layer.h)
    graph = capture(step)
    launches_per_step = (moe_launch_count(step.layer.h) - n0) // 2
    st = {}
    with ClockSampler(local) as clk:
        ms = time_steps(graph.replay, args.steps, args.warmup, world, st)
    launches = launches_per_step * args.steps
    ms_eager = time_steps(step, args.steps, args.warmup, world)
    value = world * spec.T / (ms * 1e-3)

    # end to end through the C ABI: host x, dy in; host y, dx out; every step (copies overlapped
    # with the neighbouring steps' compute, as in a training loop)
    pipe = PipelinedE2E(step)
    pipe.run(args.warmup)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record()
    pipe.run(args.steps)
    eb.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_e2e = ea.elapsed_time(eb) / args.steps
    if world > 1:
        ms_e2e = reduce_max(ms_e2e, "cuda")
    e2e = {"value": world * spec.T / (ms_e2e * 1e-3), "unit": "tokens/s",
           "h2d_bytes_per_step": pipe.bytes_in, "d2h_bytes_per_step": pipe.bytes_out,
           "overlap": "inputs of step i+1 copied in and results of step i copied out while step i / i+1 compute"}

    # per-kernel-group times (events on the launching stream), dominant group's roofline
    prof = profile_groups(step.layer.h, step, args.steps)
    work = work_per_group(spec, cnt, training=True)
    tot = sum(v[1] for v in prof.values())
    groups = {}
    for g, (nk, gms) in prof.items():
        per_launch = gms / args.steps
        ent = {"ms_per_step": per_launch, "share": gms / tot if tot else None}
        if g in work:
            fl, by = work[g]
            ent.update(tflops=fl / (per_launch * 1e-3) / 1e12, gbs=by / (per_launch * 1e-3) / 1e9)
        groups[g] = ent
    dom = max((g for g in prof if g in work), key=lambda g: prof[g][1])
    dom_ms = prof[dom][1] / args.steps
    roof = roofline_entry(dom, dom_ms, *work[dom], pk, stored_traffic(dom))
    wbytes = written_bytes(spec).get(dom)
    if wbytes:
        # a weight-gradient kernel mostly writes: its bound is the HBM write rate, measured here
        wpk = write_bandwidth(dev)
        roof["write_bound"] = {"written_bytes": wbytes, "achieved_write_gbs": wbytes / (dom_ms * 1e-3) / 1e9,
                               "measured_write_peak_gbs": wpk,
                               "frac": wbytes / (dom_ms * 1e-3) / 1e9 / wpk,
                               "peak_source": "fill of a 1 GiB buffer, CUDA events, this run"}

    # the per-workload summary (last key of the line): the step above, its forward alone, the tiny fp32
    # layer, and (rank 0) the DeepSeek-V3-shaped workloads
    summary = {}
    if rank == 0:
        fst = {}
        fwd_graph = capture(lambda: moe_forward(step.layer.h, step.inp["x"], spec.T, step.y, None, step.ws))
        time_steps(fwd_graph.replay, args.steps, args.warmup, 1, fst)
        del fwd_graph
        summary["c0 fp32 T64 fwd"] = tiny_forward_line(dev, pk, args)
        summary["c1 bf16 T2048 fwd"] = summary_row(fst, spec.T, roof_line(fst["ms_mean"], *layer_work(spec, cnt), pk))
    summary["c1 bf16 T2048 fwd+bwd (headline)"] = summary_row(st, spec.T, roof_line(
        ms, *layer_work(spec, cnt, "fwd+bwd"), pk))

    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms, "ms_median": st["ms_median"], "ms_min": st["ms_min"],
           "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, moe_synth)",
           "config": bench_config(spec, world),
           "routing": {"active_experts": int(np.count_nonzero(cnt)), "max_expert_load": int(cnt.max())},
           "launch": "CUDA graph of the step's C-ABI calls, replayed", "eager_ms_per_step": ms_eager,
           "e2e": e2e, "gpu_launches": int(launches), "kernel_groups": groups,
           "pages_context": PAGES_CONTEXT}
    out["clocks"] = clk.summary()

    if rank == 0 and not args.no_extra:
        out["extra"] = run_extra(args, dev, pk, summary)
    if rank == 0 and not args.no_cpu_baseline:
        n = oracle_inputs(moe_synth.make_inputs(spec, "cpu", grad=True))
        ntok = min(args.cpu_tokens, spec.T)
        # whole passes over the sample until at least --cpu-seconds of host time have gone by
        times = []
        while not times or (sum(times) < args.cpu_seconds and len(times) < 16):
            times.append(cpu_baseline(spec, n, ntok))
        dt = float(np.mean(times))
        what = f"the whole {spec.T}-token" if ntok == spec.T else f"the first {ntok} of {spec.T} tokens'"
        out["cpu_baseline"] = {"value": ntok / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                               "host": host_cpu(),
                               "sample": f"{what} fwd+bwd (all experts' weights), {len(times)} passes of "
                                         f"{dt:.1f} s each, mean"}
    out["roofline"] = roof
    out["configs"] = summary
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def tiny_forward_line(dev, pk, args):
    """The tiny fp32 layer's forward (launch-bound; reported without a target): one C-ABI forward per
    step, replayed from a CUDA graph, and the eager calls' time beside it."""
    from mixture_experts_layer_routing_gb300 import MoeLayer, moe_forward
    spec = moe_synth.TINY_FP32
    inp = moe_synth.make_inputs(spec, dev)
    layer = MoeLayer.from_spec(spec, device=dev)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    cnt = layer.route(inp["x"])["cnt"].cpu().numpy()
    y = torch.empty_like(inp["x"])
    ws = layer.buffer("fwd", layer.sizes(spec.T)["fwd_ws"])
    fn = lambda: moe_forward(layer.h, inp["x"], spec.T, y, None, ws)  # noqa: E731
    eager = {}
    time_steps(fn, args.steps, args.warmup, 1, eager)
    g = capture(fn)
    st = {}
    time_steps(g.replay, args.steps, args.warmup, 1, st)
    row = summary_row(st, spec.T, roof_line(st["ms_mean"], *layer_work(spec, cnt), pk))
    row["eager_ms"] = r4(eager["ms_mean"])
    row["note"] = "launch-bound; no target"
    del g
    layer.close()
    return row


def run_extra(args, dev, pk, summary):
    """DeepSeek-V3-shaped forward (uniform, Zipf 1.2), decode B=1/4/16, the MXFP8 chunked step;
    their summary rows go into `summary`."""
    from mixture_experts_layer_routing_gb300 import MoeLayer, moe_decode, moe_forward
    extra = {}
    steps, warm = args.steps, 5
    for spec in (moe_synth.DSV3_UNIFORM, moe_synth.DSV3_ZIPF):
        inp = moe_synth.make_inputs(spec, dev)
        layer = MoeLayer.from_spec(spec, device=dev)
        layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
        del inp["Wg"], inp["Wu"], inp["Wd"]
        torch.cuda.empty_cache()
        cnt = layer.route(inp["x"])["cnt"].cpu().numpy()
        y = torch.empty_like(inp["x"])
        ws = layer.buffer("fwd", layer.sizes(spec.T)["fwd_ws"])
        fn = lambda: moe_forward(layer.h, inp["x"], spec.T, y, None, ws)  # noqa: E731
        # the forward's C-ABI call replayed from a CUDA graph, as the headline step; eager beside it
        graph = capture(fn)
        for _ in range(warm):
            graph.replay()
        st = {}
        with ClockSampler(dev.index or 0) as clk:
            ms = time_steps(graph.replay, steps, 0, 1, st)
        del graph
        eager = {}
        time_steps(fn, steps, warm, 1, eager)
        prof = profile_groups(layer.h, fn, steps)
        fl, by = layer_work(spec, cnt)
        rl = roof_line(ms, fl, by, pk)
        # a loop of these 6 ms steps can draw ~1.4 kW and meet the power cap: the sustained bf16 peak
        # is the denominator for a kernel timed inside such a loop when the clocks show the cap
        rl_s = roof_line(ms, fl, by, dict(pk, bf16_tflops=pk["bf16_tflops_sustained"]))
        groups_ms = {g: v[1] / steps for g, v in prof.items()}
        work = work_per_group(spec, cnt, training=False)
        dom = max((g for g in groups_ms if g in work), key=lambda g: groups_ms[g])
        row = summary_row(st, spec.T, rl)
        dent = roofline_entry(dom, groups_ms[dom], *work[dom], pk, stored_traffic("dsv3_" + dom))
        cl = clk.summary()
        row["frac_sustained_peak"] = r4(rl_s["frac_of_roofline"])
        row["sm_mhz"] = cl["sm_mhz"]
        row["clock_reasons"] = cl["reasons"]
        row["dominant"] = {"kernel": dom, "bound": dent["bound"], "frac": r4(dent["frac"])}
        row["eager_ms"] = r4(eager["ms_mean"])
        summary["c2 bf16 " + ("uniform" if spec.zipf_s is None else f"zipf{spec.zipf_s}") + " fwd"] = row
        extra[spec.name + " fwd"] = {
            "tokens_per_s": spec.T / (ms * 1e-3), **st, **rl, "eager_ms": eager["ms_mean"],
            "launch": "CUDA graph of the forward's C-ABI call, replayed",
            "frac_of_roofline_sustained_peak": rl_s["frac_of_roofline"],
            "clocks": clk.summary(), "active_experts": int(np.count_nonzero(cnt)) + spec.S,
            "groups_ms": groups_ms}
        # decode on the same weights
        if spec is moe_synth.DSV3_UNIFORM:
            dl = decode_lines(layer, spec, dev, pk, "dsv3_bf16", 3 * spec.f * spec.d * 2)
            extra.update(dl)
            for key, v in dl.items():
                summary["c4 bf16 decode B" + key.rsplit("B", 1)[1]] = decode_row(v)
            extra["dsv3_bf16_decode_vs_grouped_gemm"] = decode_crossover(layer, spec, dev)
        layer.close()
        del layer, inp
        torch.cuda.empty_cache()
    extra.update(run_extra_mxfp8(dev, pk, summary))
    extra["bf16_T128_d2048_E64_f1408_top6 fwd+bwd, eager vs CUDA graph"] = graph_vs_eager(dev)
    extra["forward as one persistent kernel (expert GEMMs / whole forward) vs separate launches"] = fused_vs_separate(dev)
    return extra


def decode_lines(layer, spec, dev, pk, tag, expert_bytes, n_batches=16):
    """Decode B=1/4/16 over n_batches independent token batches taken in turn (consecutive steps route
    to different experts, so the weights come from HBM); bytes = the router weight plus, per batch,
    expert_bytes for each distinct expert it uses (routed ones plus the shared expert)."""
    from mixture_experts_layer_routing_gb300 import moe_decode
    out = {}
    for B in (1, 4, 16):
        xs = [t.contiguous() for t in moe_synth.make_tokens(spec.with_(T=B), n_batches, dev)]
        yb = torch.empty_like(xs[0])
        wsb = layer.buffer("fwd", layer.sizes(B)["fwd_ws"])
        it = [0]

        def fnb():
            moe_decode(layer.h, xs[it[0] % n_batches], B, yb, wsb)
            it[0] += 1

        stb = {}
        msb = time_steps(fnb, 64, 8, 1, stb)
        profb = profile_groups(layer.h, fnb, 32)
        nact = [int(np.count_nonzero(layer.route(x)["cnt"].cpu().numpy())) + spec.S for x in xs]
        nbytes = float(np.mean(nact)) * expert_bytes + spec.E * spec.d * 2
        t_roof = nbytes / (pk["hbm_gbs"] * 1e9)
        out[f"{tag}_decode_B{B}"] = {
            "path": ("warp-per-output kernels" if B < 4
                     else "grouped-GEMM forward (from the crossover batch)"),
            "tokens_per_s": B / (msb * 1e-3), "ms": msb, "ms_median": stb["ms_median"], "ms_min": stb["ms_min"],
            "weight_gbs": nbytes / (msb * 1e-3) / 1e9,
            "roofline_ms": t_roof * 1e3, "frac_of_roofline": t_roof * 1e3 / msb,
            "experts_read_mean": float(np.mean(nact)), "batches": n_batches,
            "groups_ms": {g: v[1] / 32 for g, v in profb.items()}}
    return out


def decode_row(v):
    """Summary line of a decode workload (bytes: the router weight and the used experts' weights)."""
    return {"ms": r4(v["ms"]), "med": r4(v["ms_median"]), "min": r4(v["ms_min"]), "tok_s": r4(v["tokens_per_s"]),
            "weight_GBs": r4(v["weight_gbs"]), "roof_ms": r4(v["roofline_ms"]), "frac": r4(v["frac_of_roofline"]),
            "path": "warp" if v["path"].startswith("warp") else "grouped GEMM"}


def graph_vs_eager(dev, T=128, steps=50):
    """Launch overhead at a small batch: the 2048-token bench layer's forward + backward on T tokens,
    eager through the C ABI and replayed from one captured CUDA graph (same calls, same buffers)."""
    spec = moe_synth.BF16_T2048.with_(T=T)
    step = TrainStep(spec, dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    from mixture_experts_layer_routing_gb300 import moe_launch_count
    n0 = moe_launch_count(step.layer.h)
    eager = time_steps(step, steps, 5, 1)
    launches = (moe_launch_count(step.layer.h) - n0) // (steps + 5)
    replay = time_steps(graph.replay, steps, 5, 1)
    step.layer.close()
    return {"T": T, "eager_ms": eager, "graph_ms": replay, "kernel_launches_per_step": launches}


def fused_vs_separate(dev, steps=30):
    """Forward milliseconds (CUDA-graph replay, so launch gaps are the graph's) with the gate/up and
    down GEMMs as one persistent kernel (moe_set_fused 1), the whole forward as one persistent kernel
    (2), and separate launches (0), on the 2048-token bench layer at several T and on the
    DeepSeek-V3-shaped layer (uniform routing) at T=8192."""
    from mixture_experts_layer_routing_gb300 import MoeLayer, moe_forward, moe_set_fused
    out = {}
    for spec, Ts in ((moe_synth.BF16_T2048, (64, 256, 2048)), (moe_synth.DSV3_UNIFORM, (8192,))):
        inp = moe_synth.make_inputs(spec, dev)
        layer = MoeLayer.from_spec(spec, device=dev)
        layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
        for T in Ts:
            x = inp["x"][:T].contiguous()
            y = torch.empty_like(x)
            ws = layer.buffer("fwd", layer.sizes(T)["fwd_ws"])
            row = {}
            for fused in (0, 1, 2):
                moe_set_fused(layer.h, fused)
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    moe_forward(layer.h, x, T, y, None, ws)
                torch.cuda.current_stream().wait_stream(s)
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    moe_forward(layer.h, x, T, y, None, ws)
                row[("separate_ms", "fused_experts_ms", "fused_forward_ms")[fused]] = time_steps(graph.replay, steps, 5, 1)
                del graph
            row["speedup_experts"] = row["separate_ms"] / row["fused_experts_ms"]
            row["speedup_forward"] = row["separate_ms"] / row["fused_forward_ms"]
            out[f"{spec.name.split('_')[0]}_d{spec.d}_E{spec.E}_T{T}"] = row
        moe_set_fused(layer.h, 0)
        layer.close()
        del layer, inp
        torch.cuda.empty_cache()
    return out


def decode_crossover(layer, spec, dev, n_batches=8):
    """Milliseconds per step of the warp-per-output decode kernels and of the grouped-GEMM forward on
    the same B tokens (independent batches in turn), and the smallest B where the GEMM path wins."""
    from mixture_experts_layer_routing_gb300 import moe_decode, moe_forward, moe_set_decode_crossover
    moe_set_decode_crossover(layer.h, 65)   # every batch on the warp kernels for this comparison
    rows = {}
    cross = None
    for B in (1, 2, 4, 8, 16, 32, 64):
        xs = [t.contiguous() for t in moe_synth.make_tokens(spec.with_(T=B), n_batches, dev, seed_offset=11)]
        yb = torch.empty_like(xs[0])
        ws = layer.buffer("fwd", layer.sizes(B)["fwd_ws"])
        it = [0]

        def dec():
            moe_decode(layer.h, xs[it[0] % n_batches], B, yb, ws)
            it[0] += 1

        def gemm():
            moe_forward(layer.h, xs[it[0] % n_batches], B, yb, None, ws)
            it[0] += 1

        md = time_steps(dec, 24, 4, 1)
        mg = time_steps(gemm, 24, 4, 1)
        rows[str(B)] = {"decode_ms": md, "grouped_gemm_ms": mg}
        if cross is None and mg < md:
            cross = B
    default = 4
    moe_set_decode_crossover(layer.h, default)
    return {"ms": rows, "gemm_faster_from_B": cross,
            "note": f"decode_ms: warp-per-output kernels forced; moe_decode itself switches to the GEMMs from B = {default}"}


def mx_step_work(spec, n_chunks, slots, fl_fwd, fl_bwd):
    """Algorithmic (flops, bytes) of the chunked MXFP8 step: "ideal once" (each quantised weight copy
    read once, E4M3 codes + one E8M0 byte per 32; bf16 weight gradients written once; activations in
    and out once) and "per chunk" (the chunked method's own cost: every chunk's forward, and the
    recomputed forwards of the chunks the ring does not hold, read the forward weight copies; every
    chunk's backward reads the backward copies)."""
    nseg, d, f = spec.E + spec.S, spec.d, spec.f
    w_axis = 3 * nseg * f * d * (1 + 1 / 32)          # W13 + Wd, one quantisation axis
    grads = 3 * nseg * f * d * 2
    acts = 4 * spec.T * spec.d * 2                     # x, dy in; y, dx out
    recompute = max(0, n_chunks - slots)
    ideal = (fl_fwd + fl_bwd, 2 * w_axis + grads + acts)
    per_chunk = (fl_fwd * (1 + recompute / n_chunks) + fl_bwd,
                 (n_chunks + recompute) * w_axis + n_chunks * w_axis + grads + acts)
    return ideal, per_chunk


def run_extra_mxfp8(dev, pk, summary):
    """DeepSeek-V3-shaped MXFP8 forward + backward, T=8192 in 2368-token chunks over a 512 MB ring."""
    from mixture_experts_layer_routing_gb300 import MoeLayer, moe_train_chunked, moe_train_chunked_sizes
    spec = moe_synth.DSV3_MXFP8
    inp = moe_synth.make_inputs(spec, dev, grad=True)
    layer = MoeLayer.from_spec(spec, device=dev)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    torch.cuda.synchronize()
    del inp["Wg"], inp["Wu"], inp["Wd"]
    torch.cuda.empty_cache()
    cnt = layer.route(inp["x"])["cnt"].cpu().numpy()
    z = moe_train_chunked_sizes(layer.h, spec.T)
    ring_bytes = (512 << 20) // z["slot"] * z["slot"]
    ring = layer.buffer("ring", ring_bytes)
    ws = layer.buffer("chunk_ws", z["workspace"])
    g = layer.grads_like(inp["x"])
    y = torch.empty_like(inp["x"])
    rec = []
    fn = lambda: rec.append(moe_train_chunked(layer.h, inp["x"], inp["dy"], spec.T, y, g["dx"], g["dWr"],  # noqa: E731
                                              g["dWg"], g["dWu"], g["dWd"], ring, ring_bytes, ws))
    st = {}
    ms = time_steps(fn, 5, 3, 1, st)
    prof = profile_groups(layer.h, fn, 2)
    fl_fwd, _ = layer_work(spec, cnt, "fwd")
    fl_all, _ = layer_work(spec, cnt, "fwd+bwd")
    slots = ring_bytes // z["slot"]
    (fi, bi), (fc, bc) = mx_step_work(spec, z["n_chunks"], slots, fl_fwd, fl_all - fl_fwd)
    mx_peak = 2 * pk["bf16_tflops"]          # MXFP8 dense = 2x bf16 (nominal ratio) of the measured bf16 peak
    once = roof_line(ms, fi, bi, pk, mx_peak)
    chunked = roof_line(ms, fc, bc, pk, mx_peak)
    key = spec.name + " fwd+bwd"
    out = {key: {
        "tokens_per_s": spec.T / (ms * 1e-3), **st, "roofline_ms": once["roofline_ms"],
        "frac_of_roofline": once["frac_of_roofline"], "ideal_once": once, "per_chunk": chunked,
        "chunks": z["n_chunks"], "ring_slots": slots,
        "recomputed_chunks": rec[-1] if rec else None, "peak_mxfp8_tflops": mx_peak,
        "groups_ms": {k: v[1] / 2 for k, v in prof.items()}}}
    row = summary_row(st, spec.T, once)
    row["frac_per_chunk"] = r4(chunked["frac_of_roofline"])
    row["roof_ms_per_chunk"] = r4(chunked["roofline_ms"])
    summary["c3 mxfp8 T8192 chunked fwd+bwd (frac: ideal once)"] = row
    # decode on the E4M3 weights: per expert W13 and Wd codes plus one scale byte per 32
    dl = decode_lines(layer, spec, dev, pk, "dsv3_mxfp8", 3 * spec.f * spec.d * (1 + 1 / 32))
    out.update(dl)
    for k, v in dl.items():
        summary["c4 mxfp8 decode B" + k.rsplit("B", 1)[1]] = decode_row(v)
    out["dsv3_mxfp8_decode_vs_grouped_gemm"] = decode_crossover(layer, spec, dev)
    layer.close()
    del layer, inp, g, y
    torch.cuda.empty_cache()
    return out


# Small workloads for profiler captures (a few GB on the device): DeepSeek-V3 shapes with 32 routed
# experts (+1 shared) instead of 256.
PROFILE_CASES = {
    "dsv3_e32_bf16_decode_b4": (moe_synth.DSV3_UNIFORM.with_(name="dsv3_e32_bf16", E=32, T=64, seed=12), "decode", 4),
    "dsv3_e32_mxfp8_decode_b4": (moe_synth.DSV3_MXFP8.with_(name="dsv3_e32_mxfp8", E=32, T=64, chunk=0, seed=12),
                                 "decode", 4),
    "dsv3_e32_bf16_fwd_t4096": (moe_synth.DSV3_UNIFORM.with_(name="dsv3_e32_bf16", E=32, T=4096, seed=9), "fwd", 4096),
    "dsv3_e32_mxfp8_chunked_t4096": (moe_synth.DSV3_MXFP8.with_(name="dsv3_e32_mxfp8", E=32, T=4096, chunk=2048,
                                                                seed=11), "chunked", 4096),
    "bf16_t2048_fused_fwd": (moe_synth.BF16_T2048, "fwd_fused", 2048),
    "bf16_t2048_fused_whole_fwd": (moe_synth.BF16_T2048, "fwd_fused_whole", 2048),
    # ~256 rows per routed expert (2-3 row tiles), as in the 256-expert, 8192-token forward; 2.9 GB of weights
    "dsv3_e32_bf16_fwd_t1024": (moe_synth.DSV3_UNIFORM.with_(name="dsv3_e32_T1024", E=32, T=1024, seed=9), "fwd", 1024),
    "dsv3_e32_bf16_fwd_t1024_rowtiles2": (moe_synth.DSV3_UNIFORM.with_(name="dsv3_e32_T1024", E=32, T=1024, seed=9),
                                          "fwd_rowtiles2", 1024),
    # decode at B = 1 (the warp-per-output kernels; from B = 4 moe_decode takes the grouped GEMMs)
    "dsv3_e32_bf16_decode_b1": (moe_synth.DSV3_UNIFORM.with_(name="dsv3_e32_bf16", E=32, T=64, seed=12), "decode", 1),
    "dsv3_e32_mxfp8_decode_b1": (moe_synth.DSV3_MXFP8.with_(name="dsv3_e32_mxfp8", E=32, T=64, chunk=0, seed=12),
                                 "decode", 1),
    # 256 + 1 experts and four 1024-token chunks: ~4 token-axis K groups per expert in the weight gradients, as in
    # the 8192-token DeepSeek-V3 step, at d = 1024, f = 512 (~4 GB on the device)
    "mxfp8_e256_d1024_chunked_t4096": (moe_synth.LayerSpec("mxfp8_T4096_d1024_E256+1_f512_top8_chunk1024", 4096, 1024,
                                                           256, 1, 512, 8, "sigmoid", True, 2.5, "mxfp8", None, 81,
                                                           1024), "chunked", 4096),
}


def run_profile_case(args):
    from mixture_experts_layer_routing_gb300 import MoeLayer, moe_decode, moe_set_fused, moe_set_pairs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    spec, kind, n = PROFILE_CASES[args.profile_case]
    inp = moe_synth.make_inputs(spec, dev, grad=kind == "chunked")
    layer = MoeLayer.from_spec(spec, device=dev)
    layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
    if kind == "decode":
        xs = [t.contiguous() for t in moe_synth.make_tokens(spec.with_(T=n), 8, dev)]
        y = torch.empty_like(xs[0])
        ws = layer.buffer("fwd", layer.sizes(n)["fwd_ws"])
        it = [0]

        def fn():
            moe_decode(layer.h, xs[it[0] % 8], n, y, ws)
            it[0] += 1
    elif kind in ("fwd", "fwd_fused", "fwd_fused_whole", "fwd_rowtiles2"):
        moe_set_fused(layer.h, {"fwd_fused": 1, "fwd_fused_whole": 2}.get(kind, 0))
        moe_set_pairs(layer.h, 2 if kind == "fwd_rowtiles2" else 0)
        fn = lambda: layer.forward(inp["x"])  # noqa: E731
    else:
        fn = lambda: layer.train_chunked(inp["x"], inp["dy"], slots=1)  # noqa: E731
    ms = time_steps(fn, args.steps, args.warmup, 1)
    print(json.dumps({"profile_case": args.profile_case, "ms": ms, "status": layer.status()}), flush=True)
    layer.close()


def run_chunk_sweep(args):
    """The DeepSeek-V3 MXFP8 forward + backward of T=8192 tokens for several chunk sizes, each with a
    512 MB ring of saved activations: ms per step, chunks, ring slots and recomputed chunk forwards.
    Prints one JSON line."""
    from mixture_experts_layer_routing_gb300 import MoeLayer, moe_train_chunked, moe_train_chunked_sizes
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    base = moe_synth.DSV3_MXFP8
    inp = moe_synth.make_inputs(base, dev, grad=True)
    rows = {}
    for chunk in (1024, 2048, 2368, 4096, 8192):
        spec = base.with_(chunk=chunk)
        layer = MoeLayer.from_spec(spec, device=dev)
        layer.set_weights(inp["Wr"], inp["b"], inp["Wg"], inp["Wu"], inp["Wd"])
        z = moe_train_chunked_sizes(layer.h, spec.T)
        slots = max(1, (512 << 20) // z["slot"])
        ring = layer.buffer("ring", slots * z["slot"])
        ws = layer.buffer("chunk_ws", z["workspace"])
        g = layer.grads_like(inp["x"])
        y = torch.empty_like(inp["x"])
        rec = []
        fn = lambda: rec.append(moe_train_chunked(layer.h, inp["x"], inp["dy"], spec.T, y, g["dx"], g["dWr"],  # noqa: E731
                                                  g["dWg"], g["dWu"], g["dWd"], ring, slots * z["slot"], ws))
        ms = time_steps(fn, args.steps, args.warmup, 1)
        rows[str(chunk)] = {"ms": ms, "tokens_per_s": spec.T / (ms * 1e-3), "chunks": z["n_chunks"],
                            "ring_slots": slots, "slot_mb": z["slot"] / 2**20, "recomputed_chunks": rec[-1]}
        layer.close()
        del layer, g, y, ring, ws
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": "dsv3 mxfp8 fwd+bwd, T=8192, 512 MB ring", "steps": args.steps,
                      "warmup": args.warmup, "by_chunk_tokens": rows}), flush=True)


# -------------------------------------------------------- reference arm

def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return
    spec = moe_synth.BF16_T2048
    n = oracle_inputs(moe_synth.make_inputs(spec, "cpu", grad=True))
    ntok = min(args.ref_tokens, spec.T)
    for _ in range(args.warmup):
        cpu_baseline(spec, n, ntok)
    times = [cpu_baseline(spec, n, ntok) for _ in range(args.steps)]
    ms = 1e3 * float(np.mean(times))
    value = ntok / (ms * 1e-3)
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, moe_synth)",
           "config": bench_config(spec, world),
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                            "host": host_cpu(),
                            "sample": (f"the whole {spec.T}-token fwd+bwd per step" if ntok == spec.T else
                                       f"fwd+bwd of the first {ntok} of {spec.T} tokens per step")},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=2048,
                    help="tokens of the workload the oracle runs for cpu_baseline (default: all of them)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="cpu_baseline repeats whole oracle passes until this much host time has gone by")
    ap.add_argument("--ref-tokens", type=int, default=2048,
                    help="tokens of the workload the oracle runs per reference-arm step (default: all of them)")
    ap.add_argument("--chunk-sweep", action="store_true",
                    help="instead of the bench line: the DeepSeek-V3 MXFP8 fwd+bwd over chunk sizes 1024..8192")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES),
                    help="instead of the bench line: run one small workload --steps times (for a profiler)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.profile_case:
        run_profile_case(args)
    elif args.chunk_sweep:
        run_chunk_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
