#!/usr/bin/env python3
"""Benchmark of the vocabulary cross-entropy hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload linear|logits|both]

One step is one forward + backward pass over one batch of synthetic inputs:

* linear form (headline): lce_forward + lce_backward, N=4096 tokens, H=4096,
  V=131072, BF16 X ~ N(0,1), W ~ N(0, 1/H), uniform targets, mean reduction.
  Throughput counts four classifier GEMMs per step (8 N H V flops: forward
  logits, backward recomputation, dX, dW), the convention of the Liger SM100
  pull request ("Performance methodology").
* logits form: ce_forward + ce_backward, N = 4 x 4096 rows, V = 128256 BF16
  logits ~ N(0, 9), 5% ignored, label smoothing 0.1, mean reduction; reported
  as HBM GB/s of algorithmic bytes in the ``logits_ce`` object.

Both workloads are larger than the 129 MB L2 (W is 1 GiB, the logits 4.2 GB),
so no L2 flush is needed between steps.  Device timing uses CUDA events on the
launching stream; ``e2e`` repeats the step through the same public calls with
the inputs copied from pinned host memory and the loss read back every step.
With ``--gpus N`` (torchrun) every rank runs an independent replica: the path
has no exchange step, so there is no collective on the data path.

``--impl reference`` times the FP64 CPU oracle on a bounded sample of the same
workload (a few tokens / rows per step) on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wk  # noqa: E402

PUBLISHED_TP1_FB_TFLOPS = 1606.5  # Liger SM100 PR, M=4096 F+B, TP1, NVIDIA B300 (context)
# Liger SM100 PR "Model-shape campaign", TP1 forward+backward ms on NVIDIA B300 (context)
PUBLISHED_MODEL_SHAPES_FB_MS = {"qwen3_30b_a3b_8192x2048x151936": 13.692,
                                "llama4_8192x5120x202048": 50.180,
                                "deepseek_v3_8192x7168x129280": 43.588}


CSRC = os.path.join(ROOT, "vocabulary_cross_entropy_gb300", "csrc")

# Kernel sources behind each traffic figure below and their SHA-256 (first 16 hex
# digits) when the counters were taken.  A traffic figure is reported only while
# the sources still hash to that digest; after any change it is null until the
# counters are taken again.
TRAFFIC_SOURCES = {
    "gemm": (("lce_tc.cu", "sm100_ptx.cuh", "vce_internal.cuh"), "c918968bd6e5a2a3"),
    "rows": (("ce_rows.cu", "sm100_ptx.cuh", "vce_internal.cuh"), "5283450d5db6766c"),
}


def source_digest(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_current(kind) -> bool:
    """Whether the kernels behind the ``kind`` traffic figures are unchanged since their capture."""
    names, digest = TRAFFIC_SOURCES[kind]
    try:
        return source_digest(names) == digest
    except OSError:
        return False


def FWD_GEMM_TRAFFIC_BYTES(wl):
    """DRAM bytes (read + write) per launch of the forward GEMM, from a one-pass ncu
    capture (dram__bytes_read.sum, dram__bytes_write.sum) of a full-size launch at
    N = H = 4096, V = 131072, scaled to this workload's V: the X bytes stay, the W
    bytes and the per-tile partials grow with V.  None for workloads outside that
    N = H = 4096 family."""
    captured_v, read_bytes, write_bytes = 131072, 1.108277e+09, 1.997773e+07
    if wl.n != 4096 or wl.hidden != 4096 or not traffic_current("gemm"):
        return None
    x_bytes = wl.n * wl.hidden * 2
    scale = wl.vocab / captured_v
    return x_bytes + (read_bytes - x_bytes) * scale + write_bytes * scale


# DRAM bytes (read, write) per launch of the logits-form row kernels, from ncu
# captures (dram__bytes_read.sum, dram__bytes_write.sum) of 2048 rows of
# V = 128256 BF16 with 5% of the rows ignored
LOGITS_CAPTURED_TRAFFIC = {
    "forward": (502.379264e6, 2.996736e6),
    "backward": (502.401280e6, 464.565504e6),
    "fused": (505.392128e6, 464.131584e6),
}


def LOGITS_TRAFFIC_BYTES(wl, kernel):
    """Read + write DRAM bytes per launch of one row kernel, scaled from the 2048-row
    capture by the row count.  None for other vocabularies or dtypes."""
    if wl.vocab != 128256 or wl.dtype != "bf16" or not traffic_current("rows"):
        return None
    read_bytes, write_bytes = LOGITS_CAPTURED_TRAFFIC[kernel]
    return (read_bytes + write_bytes) * wl.n_rows / 2048


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------

def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        pg = dist
    return rank, world, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class Clocks:
    """nvidia-smi sampling (every 20 ms) around a timed region.

    Each sample carries nvidia-smi's own timestamp, and the summary keeps only the
    samples taken between entering and leaving the ``with`` block, so that idle
    readings just before or after the region never enter the median.
    """
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def _reader(self):
        for line in self.proc.stdout:
            if line.strip():
                self.lines.append(line.strip())

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", str(self.INTERVAL_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()
        t = time.time()
        while not self.lines and time.time() - t < 5.0:
            time.sleep(0.02)
        self.t0 = time.time()
        return self

    def __exit__(self, *exc):
        self.t1 = time.time()
        if self.proc is not None:
            time.sleep(0.25)  # let samples taken inside the region arrive
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)
        return False

    @staticmethod
    def _when(stamp):
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = [[x.strip() for x in l.split(",")] for l in self.lines]
        rows = [f for f in rows if len(f) >= 10]
        # if nvidia-smi's timestamps cannot be read, every sample counts (window unknown)
        stamped = any(self._when(f[0]) is not None for f in rows)
        for f in rows:
            when = self._when(f[0])
            if stamped and (when is None or self.t0 is None or not (self.t0 <= when <= self.t1)):
                continue
            try:
                sm.append(float(f[2]))
                mx.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
               "samples": len(sm)}
        if not stamped:
            out["window"] = "unfiltered"
        return out


# ---------------------------------------------------------------------------
# GPU arms
# ---------------------------------------------------------------------------

def _torch_inputs_linear(wl, dev):
    import torch
    inp = wk.make_linear_inputs(wl)
    host = dict(
        X=torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16),
        W=torch.from_numpy(inp.w.view(np.int16)).view(torch.bfloat16),
        target=torch.from_numpy(inp.target),
        grad=torch.from_numpy(inp.grad),
    )
    devt = {k: v.to(dev) for k, v in host.items()}
    return host, devt, inp


class LinearStep:
    """lce_forward + lce_backward with every buffer preallocated (no allocation per step)."""

    def __init__(self, wl, dev, max_slab_bytes=0):
        import torch
        import vocabulary_cross_entropy_gb300 as vce
        self.vce = vce
        self.wl = wl
        self.max_slab_bytes = max_slab_bytes
        self.host, self.d, _ = _torch_inputs_linear(wl, dev)
        n, h, v = wl.n, wl.hidden, wl.vocab
        self.loss = torch.empty(1 if wl.reduce_loss else n, dtype=torch.float32, device=dev)
        self.lse = torch.empty(n, dtype=torch.float32, device=dev)
        self.n_valid = torch.empty(1, dtype=torch.int64, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.dX = torch.empty(n, h, dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty(v, h, dtype=torch.bfloat16, device=dev)
        self.ws_bytes = vce.lce_workspace_size(n, h, v, wl.reduce_loss, max_slab_bytes)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.n_valid_count = int((self.host["target"] != wk.IGNORE_IDX).sum())

    def forward(self):
        wl = self.wl
        self.vce.lce_forward(self.d["X"], self.d["W"], self.d["target"], wl.label_smoothing,
                             wl.reduce_loss, loss=self.loss, lse=self.lse, n_valid=self.n_valid,
                             workspace=self.ws, dev_status=self.status)

    def backward(self):
        wl = self.wl
        self.vce.lce_backward(self.d["X"], self.d["W"], self.d["target"], self.lse, self.n_valid,
                              self.d["grad"], wl.label_smoothing, wl.reduce_loss, dX=self.dX,
                              dW=self.dW, workspace=self.ws, dev_status=self.status)

    def flops(self):
        wl = self.wl
        return 8.0 * wl.n * wl.hidden * wl.vocab

    def units(self):
        return self.flops() / 1e12  # TFLOP per step


class LogitsStep:
    def __init__(self, wl, dev):
        import torch
        import vocabulary_cross_entropy_gb300 as vce
        self.vce = vce
        self.wl = wl
        inp = wk.make_logits_inputs(wl)
        logits = (torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16) if wl.dtype == "bf16"
                  else torch.from_numpy(inp.logits))
        self.host = dict(logits=logits, target=torch.from_numpy(inp.target), grad=torch.from_numpy(inp.grad))
        del inp
        self.d = {k: v.to(dev) for k, v in self.host.items()}
        n, v = wl.n_rows, wl.vocab
        self.loss = torch.empty(1 if wl.reduce_loss else n, dtype=torch.float32, device=dev)
        self.stats = torch.empty(n, 2, dtype=torch.float32, device=dev)
        self.n_valid = torch.empty(1, dtype=torch.int64, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.dlogits = torch.empty_like(self.d["logits"])
        self.ws = torch.empty(max(1, vce.ce_workspace_size(n, v, wl.reduce_loss)), dtype=torch.uint8,
                              device=dev)
        self.n_valid_count = int((self.host["target"] != wk.IGNORE_IDX).sum())

    def forward(self):
        wl = self.wl
        self.vce.ce_forward(self.d["logits"], self.d["target"], wl.label_smoothing, wl.reduce_loss,
                            loss=self.loss, stats=self.stats, n_valid=self.n_valid, workspace=self.ws,
                            dev_status=self.status)

    def backward(self):
        wl = self.wl
        self.vce.ce_backward(self.d["logits"], self.d["target"], self.stats, self.n_valid,
                             self.d["grad"], wl.label_smoothing, wl.reduce_loss, dlogits=self.dlogits,
                             dev_status=self.status)

    def bytes_fwd(self):
        return float(self.n_valid_count) * self.wl.vocab * self.d["logits"].element_size()

    def bytes_bwd(self):
        es = self.d["logits"].element_size()
        return float(self.n_valid_count) * self.wl.vocab * es + float(self.wl.n_rows) * self.wl.vocab * es

    def units(self):
        return (self.bytes_fwd() + self.bytes_bwd()) / 1e9  # GB per step


def time_steps(step, steps, warmup, pg, phase_events=True):
    """Returns (total_ms max over ranks, {phase: mean ms per launch}); the library's kernel
    launches inside the timed region are left in ``step.timed_launches``.  With
    ``phase_events`` False only the region is timed (no per-call events: for steps of a
    few microseconds, where recording events would add to the host time measured)."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        step.forward()
        step.backward()
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    phases = ("forward", "backward") if phase_events else ()
    ev = {p: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)] for p in phases}
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    launches0 = step.vce.vce_kernel_launches()
    start.record(stream)
    if phase_events:
        for i in range(steps):
            ev["forward"][i][0].record(stream)
            step.forward()
            ev["forward"][i][1].record(stream)
            ev["backward"][i][0].record(stream)
            step.backward()
            ev["backward"][i][1].record(stream)
    else:
        for i in range(steps):
            step.forward()
            step.backward()
    end.record(stream)
    step.timed_launches = step.vce.vce_kernel_launches() - launches0
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    total = max_over_ranks(pg, start.elapsed_time(end))
    out = {p: statistics.mean(a.elapsed_time(b) for a, b in ev[p]) for p in phases}
    return total, out


MIN_REGION_S = 0.5  # the sub-measurements time at least this long: 20+ clock samples each


def steps_for(fn, min_steps, min_s=MIN_REGION_S, pg=None):
    """Step count whose timed region lasts at least ``min_s``, from the wall time of a
    short untimed probe of ``fn`` (one step); the same count on every rank."""
    import torch
    fn()
    torch.cuda.synchronize()
    k = 3
    t0 = time.perf_counter()
    for _ in range(k):
        fn()
    torch.cuda.synchronize()
    per = max((time.perf_counter() - t0) / k, 1e-6)
    return int(max_over_ranks(pg, float(max(min_steps, math.ceil(min_s / per)))))


def both(step):
    """One forward + backward of ``step`` (for steps_for)."""
    def fn():
        step.forward()
        step.backward()
    return fn


def time_graph_replay(step, k, warmup):
    """Mean us of one forward + backward step captured once in a CUDA graph and
    replayed ``k`` times (every library call is capturable: no allocation, no host
    synchronisation); the replays show the device time without the per-call host
    overhead of the Python binding."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warmup):
            step.forward()
            step.backward()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.forward()
        step.backward()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(k):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return 1e3 * a.elapsed_time(b) / k


def peak_extra_memory(step):
    """Peak device memory one forward + backward call adds beyond inputs, weights and final
    outputs (loss, dX, dW): workspace, lse and the small state, allocated on demand through
    torch's caching allocator inside the calls (the library itself allocates nothing)."""
    import torch
    wl = step.wl
    vce = step.vce
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    f = vce.lce_forward(step.d["X"], step.d["W"], step.d["target"], wl.label_smoothing, wl.reduce_loss,
                        loss=step.loss, max_slab_bytes=step.max_slab_bytes)
    vce.lce_backward(step.d["X"], step.d["W"], step.d["target"], f.lse, f.n_valid, step.d["grad"],
                     wl.label_smoothing, wl.reduce_loss, dX=step.dX, dW=step.dW,
                     max_slab_bytes=step.max_slab_bytes)
    torch.cuda.synchronize()
    return torch.cuda.max_memory_allocated() - base


def fused_logits_call(step):
    wl = step.wl
    step.vce.ce_forward_backward(step.d["logits"], step.d["target"], step.d["grad"], wl.label_smoothing,
                                 wl.reduce_loss, dlogits=step.dlogits, loss=step.loss, stats=step.stats,
                                 n_valid=step.n_valid, workspace=step.ws, dev_status=step.status)


def time_fused_logits(step, steps, warmup, pg):
    """Mean ms of ce_forward_backward over ``steps`` timed calls (separate output buffer)."""
    import torch
    stream = torch.cuda.current_stream()

    def one():
        fused_logits_call(step)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    barrier(pg)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        one()
    e.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    return max_over_ranks(pg, s.elapsed_time(e)) / steps


# vocabularies of common models (BF16 logits, 16384 rows; 8192 rows above 150K)
VOCAB_SWEEP = (32000, 32768, 50257, 65536, 100352, 128256, 151936, 202048, 256000)


def vocab_sweep(dev, args, pg, pk):
    """ce_forward, ce_backward and ce_forward_backward over common vocabulary sizes:
    BF16 logits ~ N(0, 9) drawn on the device from a seeded generator, 5% ignored
    rows, eps = 0.1, mean reduction.  GB/s counts the algorithmic bytes."""
    import torch
    import vocabulary_cross_entropy_gb300 as vce
    out = []
    for v in VOCAB_SWEEP:
        n = 16384 if v <= 150000 else 8192
        g = torch.Generator(device=dev).manual_seed(v)
        z = (torch.randn(n, v, device=dev, generator=g) * 3).to(torch.bfloat16)
        t = torch.randint(0, v, (n,), device=dev, generator=g)
        t[torch.rand(n, device=dev, generator=g) < 0.05] = wk.IGNORE_IDX
        dz = torch.empty_like(z)
        grad = torch.ones(1, device=dev)
        loss, stats = torch.empty(1, device=dev), torch.empty(n, 2, device=dev)
        nv = torch.empty(1, dtype=torch.int64, device=dev)
        ws = torch.empty(vce.ce_workspace_size(n, v, True), dtype=torch.uint8, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        calls = {
            "forward": lambda: vce.ce_forward(z, t, 0.1, True, loss=loss, stats=stats, n_valid=nv, workspace=ws,
                                              dev_status=status),
            "backward": lambda: vce.ce_backward(z, t, stats, nv, grad, 0.1, True, dlogits=dz, dev_status=status),
            "fused": lambda: vce.ce_forward_backward(z, t, grad, 0.1, True, dlogits=dz, loss=loss, stats=stats,
                                                     n_valid=nv, workspace=ws, dev_status=status),
        }
        calls["forward"]()
        torch.cuda.synchronize()
        n_valid = int(nv.item())
        read, write = float(n_valid) * v * 2, float(n) * v * 2
        nbytes = {"forward": read, "backward": read + write, "fused": read + write}
        row = {"vocab": v, "n_rows": n}
        stream = torch.cuda.current_stream()
        for name, fn in calls.items():
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            barrier(pg)
            s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            k = 20
            s_.record(stream)
            for _ in range(k):
                fn()
            e_.record(stream)
            torch.cuda.synchronize()
            ms = max_over_ranks(pg, s_.elapsed_time(e_)) / k
            row[name + "_ms"] = ms
            row[name + "_frac_hbm"] = nbytes[name] / (ms / 1e3) / 1e9 / pk["hbm"]
        assert int(status.item()) == 0, "device status reported an error"
        out.append(row)
        del z, dz, t
        torch.cuda.empty_cache()
    return out


TOKEN_SWEEP = (512, 1024, 2048, 4096, 8192, 16384)


def token_sweep(dev, args, pg, pk):
    """lce_forward + lce_backward at H = 4096, V = 131072 over token counts: X ~ N(0, 1)
    and W ~ N(0, 1/H) in BF16 drawn on the device from a seeded generator, uniform
    targets, mean reduction.  TFLOP/s counts the four classifier GEMMs, 8 N H V."""
    import torch
    import vocabulary_cross_entropy_gb300 as vce
    h, v = 4096, 131072
    g = torch.Generator(device=dev).manual_seed(1)
    w = (torch.randn(v, h, device=dev, generator=g) * h ** -0.5).to(torch.bfloat16)
    dw = torch.empty_like(w)
    out = []
    for n in TOKEN_SWEEP:
        x = torch.randn(n, h, device=dev, generator=g).to(torch.bfloat16)
        y = torch.randint(0, v, (n,), device=dev, generator=g)
        dx = torch.empty_like(x)
        grad = torch.ones(1, device=dev)
        loss, lse = torch.empty(1, device=dev), torch.empty(n, device=dev)
        nv = torch.empty(1, dtype=torch.int64, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = torch.empty(vce.lce_workspace_size(n, h, v, True), dtype=torch.uint8, device=dev)

        def step():
            vce.lce_forward(x, w, y, 0.0, True, loss=loss, lse=lse, n_valid=nv, workspace=ws, dev_status=status)
            vce.lce_backward(x, w, y, lse, nv, grad, 0.0, True, dX=dx, dW=dw, workspace=ws, dev_status=status)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        barrier(pg)
        k = max(3, args.steps // 3)
        stream = torch.cuda.current_stream()
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record(stream)
        for _ in range(k):
            step()
        e_.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(pg, s_.elapsed_time(e_)) / k
        assert int(status.item()) == 0, "device status reported an error"
        tf = 8.0 * n * h * v / (ms / 1e3) / 1e12
        out.append({"n": n, "ms_per_step": ms, "value": tf, "unit": "TFLOP/s", "frac_of_burst": tf / pk["bf16"]})
        del x, dx, ws
        torch.cuda.empty_cache()
    return out


def time_forward_entropy(step, steps, warmup, pg):
    """lce_forward without and with the per-token entropy output (one more multiply-add
    per logit and a third partial per vocabulary tile).  The two kinds of call alternate
    one by one, each timed by its own pair of events, and the medians are compared: the
    power-capped SM clock drifts over tens of milliseconds, so two separate loops of each
    kind can see different clocks, while neighbouring calls see the same one."""
    import torch
    wl = step.wl
    stream = torch.cuda.current_stream()
    ent = torch.empty(wl.n, dtype=torch.float32, device=step.lse.device)

    def one(with_entropy):
        step.vce.lce_forward(step.d["X"], step.d["W"], step.d["target"], wl.label_smoothing, wl.reduce_loss,
                             loss=step.loss, lse=step.lse, n_valid=step.n_valid, workspace=step.ws,
                             dev_status=step.status, entropy=ent if with_entropy else None)

    for _ in range(warmup):
        one(False)
        one(True)
    torch.cuda.synchronize()
    barrier(pg)
    ev = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
          for k in (False, True)}
    for i in range(steps):
        for k in ((False, True) if i % 2 == 0 else (True, False)):
            ev[k][i][0].record(stream)
            one(k)
            ev[k][i][1].record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    med = {k: max_over_ranks(pg, statistics.median(a.elapsed_time(b) for a, b in ev[k])) for k in ev}
    return {"forward_ms": med[False], "forward_with_entropy_ms": med[True],
            "overhead": med[True] / med[False] - 1.0,
            "note": "medians over %d calls of each kind, the two kinds alternating call by call" % steps}


H2D_STREAMS = 1  # copy streams that share one step's host-to-device copy (--h2d-streams)


def copy_inputs(dst, pinned, streams, after):
    """Issues the copy of every pinned host tensor into ``dst``: with several streams,
    tensors of 64 MiB or more are cut into equal row ranges, one per stream, so that
    several copy engines can share them; each stream first waits for ``after``.
    Returns one event per stream.  (Measured on shared boxes, 1, 2 and 4 streams gave
    the same spread of end-to-end times: the host's copy bandwidth varies between runs.)"""
    import torch
    events = []
    for i, st in enumerate(streams):
        with torch.cuda.stream(st):
            st.wait_event(after)
            for k, t in pinned.items():
                if t.dim() >= 1 and t.numel() * t.element_size() >= (64 << 20):
                    lo, hi = t.shape[0] * i // len(streams), t.shape[0] * (i + 1) // len(streams)
                    dst[k][lo:hi].copy_(t[lo:hi], non_blocking=True)
                elif i == 0:
                    dst[k].copy_(t, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(st)
            events.append(ev)
    return events


def time_e2e_linear(step, steps, warmup, pg, h2d_streams=H2D_STREAMS):
    """The same step through the public calls, inputs copied from pinned host memory
    each step, then forward, backward and the loss read, one after another."""
    import torch
    stream = torch.cuda.current_stream()
    copy_streams = [torch.cuda.Stream() for _ in range(max(1, h2d_streams))]
    pinned = {k: v.pin_memory() for k, v in step.host.items()}
    loss_host = torch.empty_like(step.loss, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = loss_host.numel() * loss_host.element_size()

    def one():
        prev = torch.cuda.Event()
        prev.record(stream)  # the previous step no longer reads the inputs
        for ev in copy_inputs(step.d, pinned, copy_streams, prev):
            stream.wait_event(ev)
        step.forward()
        step.backward()
        loss_host.copy_(step.loss, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    barrier(pg)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        one()
    e.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    return max_over_ranks(pg, s.elapsed_time(e)), h2d, d2h


def time_e2e_linear_pipelined(step, steps, warmup, pg, h2d_streams=H2D_STREAMS):
    """End to end with the host copies overlapped: while step i computes, step i+1's
    inputs are copied from pinned host memory into the other of two device input
    buffers (the usual prefetch of a training loop), and
    step i's loss is read back on its own stream, so that the 4-byte read never waits
    on the compute stream behind a copy engine that is busy with the next step's
    inputs (two loss buffers by step parity keep a step from overwriting a loss still
    being read).  Every step still copies all of its inputs and reads its loss back;
    the timed region runs from before the first copy to after the last loss read."""
    import torch
    vce, wl = step.vce, step.wl
    comp = torch.cuda.current_stream()
    copy_streams = [torch.cuda.Stream() for _ in range(max(1, h2d_streams))]
    read_stream = torch.cuda.Stream()
    pinned = {k: v.pin_memory() for k, v in step.host.items()}
    bufs = [step.d, {k: torch.empty_like(v) for k, v in step.d.items()}]
    losses = [step.loss, torch.empty_like(step.loss)]
    ready = [[], []]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    read = [torch.cuda.Event(), torch.cuda.Event()]
    loss_host = [torch.empty_like(step.loss, device="cpu").pin_memory() for _ in range(2)]

    def copy_into(b):
        ready[b] = copy_inputs(bufs[b], pinned, copy_streams, done[b])

    def compute(b):
        d = bufs[b]
        for ev in ready[b]:
            comp.wait_event(ev)
        comp.wait_event(read[b])  # the loss buffer's previous read has finished
        vce.lce_forward(d["X"], d["W"], d["target"], wl.label_smoothing, wl.reduce_loss, loss=losses[b],
                        lse=step.lse, n_valid=step.n_valid, workspace=step.ws, dev_status=step.status)
        vce.lce_backward(d["X"], d["W"], d["target"], step.lse, step.n_valid, d["grad"], wl.label_smoothing,
                         wl.reduce_loss, dX=step.dX, dW=step.dW, workspace=step.ws, dev_status=step.status)
        done[b].record(comp)
        with torch.cuda.stream(read_stream):
            read_stream.wait_event(done[b])
            loss_host[b].copy_(losses[b], non_blocking=True)
            read[b].record(read_stream)

    def run(n):
        copy_into(0)
        for i in range(n):
            if i + 1 < n:
                copy_into((i + 1) % 2)
            compute(i % 2)
        comp.wait_stream(read_stream)  # every loss read is inside the region

    run(warmup)
    torch.cuda.synchronize()
    barrier(pg)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(comp)
    for st in copy_streams:
        st.wait_event(s)
    read_stream.wait_event(s)
    run(steps)
    e.record(comp)
    torch.cuda.synchronize()
    barrier(pg)
    return max_over_ranks(pg, s.elapsed_time(e))


# ---------------------------------------------------------------------------
# CPU baseline (the oracle, timed on a bounded sample)
# ---------------------------------------------------------------------------

class OracleLinearSample:
    """The FP64 oracle's forward + backward on the first ``tokens`` tokens of a linear
    workload against its full W; inputs are generated once, outside the timing."""

    def __init__(self, wl, tokens: int):
        self.wl = wl
        self.tokens = min(tokens, wl.n)
        self.x = wk.normal_rows(wl.seed, wk.TID_X, np.arange(self.tokens), wl.hidden, 1.0, True)
        self.w = wk.normal_matrix(wl.seed, wk.TID_W, wl.vocab, wl.hidden, wk.linear_w_std(wl), True)
        self.t = wk.linear_targets(wl)[:self.tokens]
        self.g = np.ones(1) if wl.reduce_loss else wk.grad_rows(wl.seed, wl.n)[:self.tokens]
        self.flops = 8.0 * self.tokens * wl.hidden * wl.vocab

    def run(self) -> float:
        import oracle
        wl = self.wl
        t0 = time.perf_counter()
        f = oracle.lce_forward(self.x, self.w, self.t, wl.label_smoothing, wl.reduce_loss)
        oracle.lce_backward(self.x, self.w, self.t, f["lse"], f["n_valid"], self.g, wl.label_smoothing,
                            wl.reduce_loss, z=f["z"])
        return time.perf_counter() - t0


def oracle_logits_sample(wl, rows: int):
    import oracle
    r = np.arange(rows)
    z = wk.logits_rows(wl, r)
    t = wk.uniform_targets(wl.seed, wl.n_rows, wl.vocab, wl.ignore_frac)[:rows]
    t0 = time.perf_counter()
    f = oracle.ce_forward(z, t, wl.label_smoothing, wl.reduce_loss, dtype=wl.dtype)
    oracle.ce_backward(z, t, f["lse"], f["n_valid"], np.ones(1), wl.label_smoothing, wl.reduce_loss,
                       dtype=wl.dtype)
    dt = time.perf_counter() - t0
    nv = int((t != wk.IGNORE_IDX).sum())
    nbytes = nv * wl.vocab * 2 * 2 + rows * wl.vocab * 2
    return dt, nbytes


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


LIN_SAMPLE_TOKENS = 32
LARGE_SLAB_CAP = 1 << 30  # dZ slab cap for the large workload: 1 GiB of BF16 gradient per slab
LOGITS_SAMPLE_ROWS = 256


def cpu_baseline_linear(wl, full=False):
    """The oracle's forward + backward timed on the host cores: on every token of the
    workload (``full``), else on its first LIN_SAMPLE_TOKENS tokens against the full W."""
    smp = OracleLinearSample(wl, wl.n if full else LIN_SAMPLE_TOKENS)
    dt = smp.run()
    what = (f"every token ({smp.tokens})" if smp.tokens == wl.n else f"the first {smp.tokens} tokens")
    return {"value": smp.flops / dt / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"FP64 NumPy oracle forward+backward on {what} of the workload against the full W "
                      f"({wl.vocab}x{wl.hidden}); flops counted as 8*tokens*H*V", "seconds": dt}


def cpu_baseline_logits(wl):
    dt, nb = oracle_logits_sample(wl, LOGITS_SAMPLE_ROWS)
    return {"value": nb / dt / 1e9, "unit": "GB/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"FP64 NumPy oracle forward+backward on the first {LOGITS_SAMPLE_ROWS} rows",
            "seconds": dt}


# ---------------------------------------------------------------------------
# memory / speed trade of the dZ slab cap
# ---------------------------------------------------------------------------

# (workload, max_slab_bytes): the headline with one 1 GiB slab over the whole
# vocabulary and at 64 MiB slabs (16), against the library's default cap of 256
# MiB (4 slabs) that the headline line uses; the large workload at 256 MiB (16
# slabs) against the 1 GiB slabs of its own line
SLAB_UNCAPPED = (1 << 64) - 1


def parse_slab_cap(text):
    """--slab-cap: 'default' -> 0 (the library's 256 MiB), 'uncapped' -> SLAB_UNCAPPED,
    else a positive number of bytes."""
    special = {"default": 0, "uncapped": SLAB_UNCAPPED}
    if text in special:
        return special[text]
    cap = int(text)
    if cap <= 0:
        raise ValueError("--slab-cap takes 'default', 'uncapped' or a positive number of bytes")
    return cap


def slab_cap_label(cap):
    return {0: "library default (256 MiB)", SLAB_UNCAPPED: "uncapped"}.get(cap, cap)
SLAB_CAPS = (("headline", SLAB_UNCAPPED), ("headline", 64 << 20), ("large", 256 << 20))


def slab_cap_sweep(dev, args, pg, local, headline_ms):
    """lce_forward + lce_backward with other dZ slab caps: time, TFLOP/s and the peak
    extra device memory of one call pair, against the headline step (the library's
    default 256 MiB cap)."""
    import torch
    out = {"headline_default_cap_ms": headline_ms, "runs": []}
    for name, cap in SLAB_CAPS:
        wl = wk.LINEAR_HEADLINE if name == "headline" else wk.LINEAR_LARGE
        stp = LinearStep(wl, dev, max_slab_bytes=cap)
        k = steps_for(both(stp), 3, pg=pg)
        with Clocks(local) as ck:
            t, ph = time_steps(stp, k, args.warmup, pg)
        assert int(stp.status.item()) == 0, "device status reported an error"
        ms = t / k
        out["runs"].append({
            "workload": wl.name, "max_slab_bytes": "uncapped" if cap == SLAB_UNCAPPED else cap,
            "slabs": -(-wl.vocab // max(256, cap // (wl.n * 2) // 256 * 256)),
            "ms_per_step": ms, "value": stp.units() / (ms / 1e3), "unit": "TFLOP/s",
            "fwd_ms": ph["forward"], "bwd_ms": ph["backward"], "steps": k,
            "workspace_bytes": stp.ws_bytes, "peak_extra_memory_bytes": peak_extra_memory(stp),
            "vs_default_cap": (ms / headline_ms - 1.0) if name == "headline" else None,
            "clocks": ck.summary()})
        del stp
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def linear_workload(args):
    if args.shape:
        n_, h_, v_ = (int(x) for x in args.shape.split(","))
        return wk.LinearWorkload(f"linear_{n_}x{h_}x{v_}", n_, h_, v_, reduce_loss=True)
    return wk.LINEAR_HEADLINE


def run_reference(args, rank, world, pg):
    """The oracle as it stands, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return 0
    wl = linear_workload(args)
    smp = OracleLinearSample(wl, LIN_SAMPLE_TOKENS)
    times = []
    for i in range(args.warmup + args.steps):
        dt = smp.run()
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = smp.flops * len(times) / total / 1e12
    cb = {"value": value, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
          "sample": f"each step: FP64 NumPy oracle forward+backward on {smp.tokens} tokens of the "
                    f"workload against the full W; flops counted as 8*tokens*H*V"}
    line = {
        "impl": "reference",
        "metric": "linear-CE fwd+bwd TFLOP/s (4 classifier GEMMs)",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / len(times) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "n": wl.n, "h": wl.hidden, "v": wl.vocab,
                   "sample_tokens": smp.tokens},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="both", choices=["linear", "logits", "both"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--h2d-streams", type=int, default=H2D_STREAMS,
                    help="copy streams that share each step's host-to-device copy in the e2e timing")
    ap.add_argument("--token-sweep", action="store_true",
                    help="also time the linear form at H=4096, V=131072 over token counts 512..16384")
    ap.add_argument("--vocab-sweep", action="store_true",
                    help="also time the logits form (forward, backward, fused) over common vocabulary sizes")
    ap.add_argument("--sweep", action="store_true",
                    help="also time the model-shape sweep (Qwen3-30B-A3B, Llama 4, DeepSeek-V3 heads at M=8192)")
    ap.add_argument("--no-large", dest="large", action="store_false",
                    help="skip the 16384x4096x128256 workload (throughput and peak extra memory)")
    ap.add_argument("--slab-cap", default="default",
                    help="dZ slab cap of the linear step: 'default' (the library's 256 MiB), 'uncapped' "
                         "(one slab over the whole vocabulary) or a number of bytes")
    ap.add_argument("--shape", default=None,
                    help="linear workload N,H,V instead of the headline (e.g. a small profiling case)")
    ap.add_argument("--logits-rows", type=int, default=None,
                    help="rows of the logits workload instead of 4 x 4096 (profiling)")
    ap.add_argument("--logits-vocab", type=int, default=None,
                    help="vocabulary of the logits workload instead of 128256 (profiling)")
    ap.add_argument("--logits-dtype", choices=("bf16", "f32"), default=None,
                    help="logits dtype instead of bf16 (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local, pg = dist_setup(args.gpus)
    if args.impl == "reference":
        return run_reference(args, rank, world, pg)

    import torch
    from vocabulary_cross_entropy_gb300 import build as vbuild
    if rank == 0:
        vbuild.build()
    barrier(pg)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk = peaks()
    out = {}

    logits_obj = None
    if args.workload in ("logits", "both"):
        lwl = wk.LOGITS_MEMBOUND
        if args.logits_rows or args.logits_vocab or args.logits_dtype:
            import dataclasses
            lwl = dataclasses.replace(lwl, n_rows=args.logits_rows or lwl.n_rows,
                                      vocab=args.logits_vocab or lwl.vocab, dtype=args.logits_dtype or lwl.dtype)
            lwl = dataclasses.replace(lwl, name=f"logits_{lwl.n_rows}x{lwl.vocab}" +
                                      ("" if lwl.dtype == "bf16" else "_" + lwl.dtype))
        st = LogitsStep(lwl, dev)
        # as the headline (--workload logits) exactly K steps; as a sub-number, enough
        # steps for a timed region of at least MIN_REGION_S
        kl = args.steps if args.workload == "logits" else steps_for(both(st), args.steps, pg=pg)
        with Clocks(local) as ck:
            total, ph = time_steps(st, kl, args.warmup, pg)
        clocks_l = ck.summary()
        gb = st.units() * world * kl / (total / 1e3)
        bwd_gbs = st.bytes_bwd() / (ph["backward"] / 1e3) / 1e9
        fwd_gbs = st.bytes_fwd() / (ph["forward"] / 1e3) / 1e9
        assert int(st.status.item()) == 0, "device status reported an error"
        kf = steps_for(lambda: fused_logits_call(st), args.steps, pg=pg)
        with Clocks(local) as ckf:
            fused_ms = time_fused_logits(st, kf, args.warmup, pg)
        fused_gbs = st.bytes_bwd() / (fused_ms / 1e3) / 1e9
        logits_obj = {
            "metric": "logits-CE fwd+bwd HBM GB/s", "value": gb, "unit": "GB/s", "steps": kl,
            "ms_per_step": total / kl, "fwd_gbs": fwd_gbs, "bwd_gbs": bwd_gbs,
            "fwd_ms": ph["forward"], "bwd_ms": ph["backward"],
            "config": {"workload": st.wl.name, "n_rows": st.wl.n_rows, "vocab": st.wl.vocab,
                       "dtype": st.wl.dtype, "label_smoothing": st.wl.label_smoothing,
                       "reduce_loss": st.wl.reduce_loss, "n_valid": st.n_valid_count,
                       "l2": "inputs larger than L2 (%.2f GB logits), no flush" % (
                           st.wl.n_rows * st.wl.vocab * st.d["logits"].element_size() / 1e9)},
            "roofline": {"kernel": "ce_backward_rows", "bound": "hbm", "achieved": bwd_gbs,
                         "peak": pk["hbm"], "unit": "GB/s", "frac": bwd_gbs / pk["hbm"],
                         "traffic": LOGITS_TRAFFIC_BYTES(st.wl, "backward"),
                         "peak_source": pk["source"] + " hbm_gbs (copy)",
                         "algorithmic_bytes": st.bytes_bwd()},
            "roofline_fwd": {"kernel": "ce_forward_rows", "bound": "hbm", "achieved": fwd_gbs,
                             "peak": pk["hbm"], "unit": "GB/s", "frac": fwd_gbs / pk["hbm"],
                             "traffic": LOGITS_TRAFFIC_BYTES(st.wl, "forward"),
                             "algorithmic_bytes": st.bytes_fwd()},
            "gpu_launches": st.timed_launches,
            "clocks": clocks_l,
            # ce_forward_backward: the same results as one forward + backward step with
            # one HBM read and one write per logit (timed separately, same workload)
            "fused": {"ms_per_step": fused_ms, "value": fused_gbs, "unit": "GB/s", "steps": kf,
                      "algorithmic_bytes": st.bytes_bwd(), "frac": fused_gbs / pk["hbm"],
                      "traffic": LOGITS_TRAFFIC_BYTES(st.wl, "fused"),
                      "speedup_vs_separate": (total / kl) / fused_ms, "clocks": ckf.summary()},
        }
        if rank == 0 and not args.no_cpu_baseline:
            logits_obj["cpu_baseline"] = cpu_baseline_logits(st.wl)
        del st
        torch.cuda.empty_cache()

    if args.workload == "logits":
        line = dict(logits_obj)
        line.update({"n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                     "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                     "dtype": lwl.dtype, "data": "synthetic"})
        if args.vocab_sweep:
            torch.cuda.empty_cache()
            line["vocab_sweep"] = vocab_sweep(dev, args, pg, pk)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0

    lin = linear_workload(args)
    slab_cap = parse_slab_cap(args.slab_cap)
    st = LinearStep(lin, dev, max_slab_bytes=slab_cap)
    with Clocks(local) as ck:
        total, ph = time_steps(st, args.steps, args.warmup, pg)
    clocks = ck.summary()
    assert int(st.status.item()) == 0, "device status reported an error"
    value = st.units() * world * args.steps / (total / 1e3)
    fwd_flops = 2.0 * st.wl.n * st.wl.hidden * st.wl.vocab
    fwd_tf = fwd_flops / (ph["forward"] / 1e3) / 1e12
    bwd_tf = 3 * fwd_flops / (ph["backward"] / 1e3) / 1e12
    e2e_steps = max(3, args.steps)  # as many steps as the device loop: the first copy (pipeline fill) counts once
    if args.no_e2e:
        e2e_obj = None
    else:
        ser_ms, h2d, d2h = time_e2e_linear(st, e2e_steps, 3, pg, args.h2d_streams)
        with Clocks(local) as cke:
            pip_ms = time_e2e_linear_pipelined(st, e2e_steps, 3, pg, args.h2d_streams)
        e2e_obj = {"value": st.units() * world * e2e_steps / (pip_ms / 1e3), "unit": "TFLOP/s",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": pip_ms / e2e_steps,
                   "pipeline": f"step i+1's inputs copied from pinned host memory (W cut over "
                               f"{args.h2d_streams} copy streams) while step i computes (two device input "
                               "buffers); each loss read on its own stream",
                   "clocks": cke.summary(),
                   "serial": {"value": st.units() * world * e2e_steps / (ser_ms / 1e3),
                              "ms_per_step": ser_ms / e2e_steps,
                              "pipeline": f"copy (W cut over {args.h2d_streams} copy streams), forward, "
                                          "backward, loss read, one after another"}}
    line = {
        "metric": "linear-CE fwd+bwd TFLOP/s (4 classifier GEMMs)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": value / world / PUBLISHED_TP1_FB_TFLOPS,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": st.wl.name, "n": st.wl.n, "h": st.wl.hidden, "v": st.wl.vocab,
                   "reduce_loss": True, "label_smoothing": 0.0,
                   "l2": "inputs larger than L2 (W is 1 GiB), no flush",
                   "max_slab_bytes": slab_cap_label(slab_cap),
                   "workspace_bytes": st.ws_bytes},
        "fwd_ms": ph["forward"], "bwd_ms": ph["backward"], "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
        # the timed region is K steps of ~10 ms, far shorter than the seconds-long loop
        # behind the sustained figure, so the denominator is the burst figure; the
        # sustained fraction is kept beside it
        "roofline": {"kernel": "tc_gemm_kernel<FwdEpi> (lce_forward: X W^T + softmax partials; "
                               "the combine and mean kernels add <2%)", "bound": "tensor",
                     "achieved": fwd_tf, "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": fwd_tf / pk["bf16"], "traffic": FWD_GEMM_TRAFFIC_BYTES(st.wl),
                     "peak_source": pk["source"] + " bf16_tflops (cuBLAS burst; timed region %.2f s)" % (
                         total / 1e3),
                     "frac_of_sustained_peak": fwd_tf / pk["bf16_sustained"],
                     "step_frac_of_burst_peak": value / world / pk["bf16"],
                     # against the dense BF16 rate of the SMs at the clock they ran at:
                     # 8192 flops per SM per cycle x SM count x median SM clock
                     "frac_of_tensor_peak_at_clock": (
                         fwd_tf / (torch.cuda.get_device_properties(dev).multi_processor_count * 8192.0
                                   * clocks["sm_mhz"] * 1e6 / 1e12)) if clocks.get("sm_mhz") else None,
                     "algorithmic_flops": fwd_flops},
        "e2e": e2e_obj,
        "gpu_launches": st.timed_launches,
        "clocks": clocks,
    }
    # pairs of forwards (without, with the entropy output) filling at least MIN_REGION_S
    ke = steps_for(lambda: (st.forward(), st.forward()), max(3, args.steps), pg=pg)
    with Clocks(local) as ckent:
        line["entropy_cost"] = time_forward_entropy(st, ke, 3, pg)
    line["entropy_cost"]["clocks"] = ckent.summary()
    line["config"]["peak_extra_memory_bytes"] = peak_extra_memory(st)
    if logits_obj is not None:
        line["logits_ce"] = logits_obj
    headline_ms = total / args.steps
    if args.large and lin is wk.LINEAR_HEADLINE:
        del st
        torch.cuda.empty_cache()
        big = LinearStep(wk.LINEAR_LARGE, dev, max_slab_bytes=LARGE_SLAB_CAP)
        ksteps = steps_for(both(big), max(3, args.steps // 3), pg=pg)
        with Clocks(local) as ckb:
            tb, phb = time_steps(big, ksteps, args.warmup, pg)
        assert int(big.status.item()) == 0, "device status reported an error"
        nv = big.n_valid_count
        line["linear_large"] = {
            "metric": "linear-CE fwd+bwd TFLOP/s (4 classifier GEMMs)",
            "value": big.units() * world * ksteps / (tb / 1e3), "unit": "TFLOP/s",
            "value_valid_tokens": 8.0 * nv * big.wl.hidden * big.wl.vocab * world * ksteps / (tb / 1e3) / 1e12,
            "ms_per_step": tb / ksteps, "fwd_ms": phb["forward"], "bwd_ms": phb["backward"], "steps": ksteps,
            "config": {"workload": big.wl.name, "n": big.wl.n, "h": big.wl.hidden, "v": big.wl.vocab,
                       "n_valid": nv, "label_smoothing": big.wl.label_smoothing, "targets": "zipf(1.1)",
                       "max_slab_bytes": LARGE_SLAB_CAP, "workspace_bytes": big.ws_bytes,
                       "peak_extra_memory_bytes": peak_extra_memory(big)},
            "clocks": ckb.summary(),
        }
        if rank == 0 and not args.no_cpu_baseline:
            line["linear_large"]["cpu_baseline"] = cpu_baseline_linear(big.wl)
        del big
        torch.cuda.empty_cache()
        if slab_cap == 0:  # the sweep's runs are compared with the default cap
            line["slab_caps"] = slab_cap_sweep(dev, args, pg, local, headline_ms)
    if args.large and lin is wk.LINEAR_HEADLINE:
        # the two small configurations: the tiny FP32 logits case (launch latency)
        # and the 4096 x 2048 x 32000 linear case (per-token loss, 2% ignored)
        torch.cuda.empty_cache()
        tiny = LogitsStep(wk.LOGITS_TINY[3], dev)
        kt = 100
        _, pht = time_steps(tiny, kt, args.warmup, pg)
        ktl = steps_for(both(tiny), kt, pg=pg)
        with Clocks(local) as ckt:
            tt, _ = time_steps(tiny, ktl, args.warmup, pg, phase_events=False)
        graph_us = time_graph_replay(tiny, ktl, args.warmup)
        assert int(tiny.status.item()) == 0, "device status reported an error"
        sm = LinearStep(wk.LINEAR_SMALL, dev)
        ks = steps_for(both(sm), max(3, args.steps // 3), pg=pg)
        with Clocks(local) as ckm:
            tsm, phm = time_steps(sm, ks, args.warmup, pg)
        assert int(sm.status.item()) == 0, "device status reported an error"
        line["small_configs"] = {
            "logits_tiny": {"workload": tiny.wl.name, "n_rows": tiny.wl.n_rows, "vocab": tiny.wl.vocab,
                            "dtype": "f32", "us_per_step": 1e3 * tt / ktl, "steps": ktl,
                            "fwd_us": 1e3 * pht["forward"], "bwd_us": 1e3 * pht["backward"],
                            "phase_steps": kt, "graph_us_per_step": graph_us, "clocks": ckt.summary(),
                            "note": "ce_forward (+ mean) + ce_backward called from Python one by one "
                                    "(us_per_step: no per-call events; fwd_us/bwd_us: a separate run with "
                                    "events around each call); graph_us_per_step replays the step "
                                    "captured in a CUDA graph"},
            "linear_small": {"workload": sm.wl.name, "value": sm.units() * world * ks / (tsm / 1e3),
                             "unit": "TFLOP/s", "ms_per_step": tsm / ks, "fwd_ms": phm["forward"],
                             "bwd_ms": phm["backward"], "steps": ks, "clocks": ckm.summary()},
        }
        if rank == 0 and not args.no_cpu_baseline:
            line["small_configs"]["linear_small"]["cpu_baseline"] = cpu_baseline_linear(sm.wl, full=True)
        del tiny, sm
    if args.sweep and lin is wk.LINEAR_HEADLINE:
        torch.cuda.empty_cache()
        line["sweep"] = []
        for shp in wk.MODEL_SHAPES:
            stp = LinearStep(shp, dev, max_slab_bytes=slab_cap)
            ks = max(3, args.steps // 3)
            with Clocks(local) as cks:
                ts, phs = time_steps(stp, ks, args.warmup, pg)
            assert int(stp.status.item()) == 0, "device status reported an error"
            line["sweep"].append({
                "workload": shp.name, "n": shp.n, "h": shp.hidden, "v": shp.vocab,
                "value": stp.units() * world * ks / (ts / 1e3), "unit": "TFLOP/s", "ms_per_step": ts / ks,
                "fwd_ms": phs["forward"], "bwd_ms": phs["backward"], "steps": ks,
                "pages_tp1_fb_ms_b300": PUBLISHED_MODEL_SHAPES_FB_MS.get(shp.name),
                "max_slab_bytes": slab_cap_label(slab_cap),
                "workspace_bytes": stp.ws_bytes, "clocks": cks.summary()})
            del stp
            torch.cuda.empty_cache()
    if args.token_sweep and lin is wk.LINEAR_HEADLINE:
        torch.cuda.empty_cache()
        line["token_sweep"] = token_sweep(dev, args, pg, pk)
    if args.vocab_sweep and lin is wk.LINEAR_HEADLINE:
        torch.cuda.empty_cache()
        line["vocab_sweep"] = vocab_sweep(dev, args, pg, pk)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_linear(lin)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
