#!/usr/bin/env python
"""Forward-convolution benchmark on one GB300: TFLOPS, roofline fraction and
workspace bytes against im2col.

One step is one conv2d_fwd call of the ResNet-style 3x3 layer (N=32,
C_in=64 -> C_out=128, 56x56, stride 1, pad 1, bf16 in, fp32 accumulate, bf16
out): the indirection-buffer build plus the tcgen05 implicit-GEMM kernel.
Inputs are seeded synthetic tensors already resident in HBM; successive steps
rotate through enough input/output sets that each step's data has left the
129 MB L2 before it is used again.  The K timed steps are captured once into a
CUDA graph and replayed, so host-side call overhead is not timed.

The JSON line (rank 0) also carries:
  roofline      the implicit-GEMM kernel alone (CUDA events around launches of
                conv2d_fwd_indirect on a prebuilt indirection buffer)
  e2e           the same metric through the C ABI from pinned host buffers,
                host->device and device->host copies inside the timed region
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same layer
  sweep         every benchmark configuration (and im2win_transform) timed
                the same way, with its roofline fraction
  clocks        SM clocks and throttle reasons sampled during the timed region

--impl reference times the CPU oracle instead (there is no reference code to
install: the pages are abstracts and a tutorial), on host cores.
Multi-GPU: independent replicas, one per rank, no collective in the data path.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "conv2d fwd TFLOPS & % of GB300 bf16 roofline; workspace bytes vs im2col"
HEADLINE = workloads.RESNET_3X3
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
# bf16 tcgen05 rate per SM per cycle: a 128x128x16 MMA (524,288 flop) issues
# every 64 cycles (measured with back-to-back MMAs on one SM)
TC_FLOP_PER_CLK_SM = 8192


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def reduce_max(value: float, dist=None, device="cpu") -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------------------------------- shape arithmetic
def shape_numbers(g, c: workloads.ConvShape):
    """FLOPs, algorithmic bytes and footprints of one convolution (metric arithmetic)."""
    Ho, Wo = g.output_dims(c.H, c.W, c.KH, c.KW, c.stride, c.pad, c.dilation)
    M = c.N * Ho * Wo
    K = c.C_in * c.KH * c.KW
    flops = 2 * M * c.C_out * K
    x_b = c.N * c.H * c.W * c.C_in * 2
    if c.KH == 1 and c.KW == 1 and c.pad == 0 and c.stride > 1:
        x_b = c.N * Ho * Wo * c.C_in * 2  # only the sampled pixels are needed
    y_b = M * c.C_out * (4 if c.out_f32 else 2)
    alg_bytes = x_b + c.C_out * K * 2 + (c.C_out * 2 if c.bias else 0) + y_b
    return dict(H_out=Ho, W_out=Wo, M=M, K=K, flops=flops, bytes=alg_bytes,
                x_bytes=x_b, y_bytes=y_b,
                workspace_bytes=g.workspace_size(c.N, c.C_in, c.H, c.W, c.C_out, c.KH, c.KW,
                                                 c.stride, c.pad, c.dilation),
                im2col_bytes=g.im2col_bytes(c.N, c.C_in, c.H, c.W, c.KH, c.KW, c.stride, c.pad,
                                            c.dilation),
                im2win_bytes=g.im2win_bytes(c.N, c.C_in, c.H, c.W, c.KH, c.KW, c.stride, c.pad,
                                            c.dilation),
                path={1: "gather", 2: "dense", 3: "stem", 4: "window", 5: "plane", 6: "im2win",
                      7: "stemwin", 8: "winfold"}.get(
                    g.select_path(c.N, c.C_in, c.H, c.W, c.C_out, c.KH, c.KW, c.stride, c.pad,
                                  c.dilation), "?"))


KERNEL_SOURCES = ("indirect_implicit_gemm_gb300/csrc/igemm.cu",
                  "indirect_implicit_gemm_gb300/csrc/api.cu",
                  "indirect_implicit_gemm_gb300/csrc/internal.h",
                  "indirect_implicit_gemm_gb300/csrc/ptx.cuh")


def strip_comments(src: str) -> str:
    """C/C++ source without // and /* */ comments, trailing spaces and blank lines
    (string and character literals are kept as they are), so that editing a
    comment does not change what the hash below says about the code."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            while i < n and src[i] != "\n":
                i += 1
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def kernel_source_hash():
    """sha256 over the sources that define the implicit-GEMM kernel and its plan,
    comments and blank lines removed."""
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()


def profiled_traffic(workload):
    """DRAM bytes per launch of the GEMM kernel on `workload` ({"total", "read",
    "write"}), from the committed ncu summary under profiles/, or None when no
    summary covers this workload or the kernel sources changed since it was
    taken.  The summary carries lines `workload: <name>`, `source_sha256:
    <hex>`, `dram_bytes_per_launch: <int>` and optionally
    `dram_read_bytes_per_launch` / `dram_write_bytes_per_launch`."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    want = kernel_source_hash()
    for fn in sorted(os.listdir(d)):
        if not fn.endswith(".md"):
            continue
        kv = {}
        with open(os.path.join(d, fn)) as f:
            for line in f:
                if ":" in line and line.split(":", 1)[0].strip() in (
                        "workload", "source_sha256", "dram_bytes_per_launch",
                        "dram_read_bytes_per_launch", "dram_write_bytes_per_launch"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip().strip("`")
        if kv.get("workload") == workload and kv.get("source_sha256") == want:
            try:
                tot = int(kv["dram_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
            rd, wr = kv.get("dram_read_bytes_per_launch"), kv.get("dram_write_bytes_per_launch")
            return {"total": tot, "read": int(rd) if rd else None,
                    "write": int(wr) if wr else None}
    return None


def sweep_summary(sweep):
    """The per-configuration results as they ride on the headline line: one
    short entry per workload (path, us, TFLOP/s, fraction of its roofline and
    what bounds it, workspace bytes), so the line stays a few KB; each full
    entry is printed on its own `sweep` line ahead of the headline line."""
    out = {}
    for ent in sweep:
        if "error" in ent:
            out[ent["workload"]] = {"error": ent["error"][:80]}
            continue
        out[ent["workload"]] = {"path": ent["path"], "us": round(ent["us"], 2),
                                "tflops": round(ent["tflops"], 1),
                                "frac": round(ent["frac_of_roofline"], 3), "bound": ent["bound"],
                                "ws_B": ent["workspace_bytes"]}
    return out


def roofline_time_s(num, peaks):
    t_tc = num["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_hbm = num["bytes"] / (peaks["hbm_gbs"] * 1e9)
    return max(t_tc, t_hbm), ("tensor" if t_tc >= t_hbm else "hbm")


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the GPU works (100 ms period)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]),
                                 float(parts[4]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [r for r in rows if r[3] > 0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[4]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows),
                "samples_busy": len(busy), "reasons": reasons}


# --------------------------------------------------------------------------- GPU timing
def rotation_sets(per_set_bytes, cap_bytes=8 << 30):
    """Enough input/output sets that one step's data is out of L2 when reused."""
    n = max(2, math.ceil(2 * L2_BYTES / max(per_set_bytes, 1)) + 1)
    return int(max(1, min(n, cap_bytes // max(per_set_bytes, 1))))


def graph_time_ms(fn, steps, stream):
    """Time `steps` calls of fn(i) replayed from one CUDA graph (no host overhead).

    The calls are captured once, replayed once untimed, then timed as one
    replay bracketed by CUDA events on the capturing stream.
    """
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(steps):
                fn(i)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    s = torch.cuda.current_stream()
    start.record(s)
    graph.replay()
    end.record(s)
    torch.cuda.synchronize()
    del graph
    return start.elapsed_time(end)


def single_launch_us(layer, stream, reps=21):
    """One conv2d_fwd on an idle GPU, issued eagerly through the binding (host
    call included), bracketed by events: the latency a lone call sees, apart
    from the graph-replayed throughput figure.  Median of `reps`."""
    times = []
    for i in range(reps):
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        layer.step(i)
        end.record(stream)
        torch.cuda.synchronize()
        times.append(start.elapsed_time(end) * 1e3)
    times.sort()
    return {"median_us": times[len(times) // 2], "min_us": times[0],
            "note": "one eager conv2d_fwd through the Python binding on an idle GPU, "
                    "events around it; the headline value is CUDA-graph replay"}


def event_time_ms(fn, steps, stream):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        fn(i)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


class Layer:
    """Device-resident inputs (rotated) and outputs for one configuration.

    path: the CONVGB_PATH_* value to run (0: the library's choice); cin_pad: run
    the layer with its channels zero-padded to this many (ablation of the stem
    paths against the gather path, which needs C_in % 8 == 0).  FLOPs and
    algorithmic bytes are always those of the unpadded layer."""

    def __init__(self, g, c, dev, sets=None, path=0, cin_pad=0):
        self.g, self.c, self.dev, self.path = g, c, dev, path
        x, w, b = workloads.make_inputs(c, device=dev)
        if cin_pad and cin_pad > c.C_in:
            x = torch.nn.functional.pad(x, (0, cin_pad - c.C_in)).contiguous()
            w = torch.nn.functional.pad(w, (0, cin_pad - c.C_in)).contiguous()
        self.cin = x.shape[3]
        self.w, self.b = w, b
        self.out_dtype = torch.float32 if c.out_f32 else torch.bfloat16
        self.num = shape_numbers(g, c)
        per_set = self.num["x_bytes"] + self.num["y_bytes"]
        self.sets = sets or rotation_sets(per_set)
        self.xs = [x] + [torch.randn_like(x, dtype=torch.float32).to(torch.bfloat16)
                         for _ in range(self.sets - 1)]
        Ho, Wo = self.num["H_out"], self.num["W_out"]
        self.ys = [torch.empty((c.N, Ho, Wo, c.C_out), dtype=self.out_dtype, device=dev)
                   for _ in range(self.sets)]
        ws = g.workspace_size(c.N, self.cin, c.H, c.W, c.C_out, c.KH, c.KW, c.stride, c.pad,
                              c.dilation, path=path)
        self.ws = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        self.ibuf = None

    def step(self, i):
        c = self.c
        self.g.conv2d_fwd_path(self.path, self.xs[i % self.sets], self.w, self.b, c.stride, c.pad,
                               c.dilation, out_dtype=self.out_dtype, y=self.ys[i % self.sets],
                               workspace=self.ws)

    def plan(self):
        c = self.c
        return self.g.plan_info(c.N, self.cin, c.H, c.W, c.C_out, c.KH, c.KW, c.stride, c.pad,
                                c.dilation, path=self.path, out_dtype=self.out_dtype)

    def gemm_only(self, i):
        """The implicit-GEMM kernel alone (indirection buffer prebuilt)."""
        c = self.c
        self.g.conv2d_fwd_indirect(self.xs[i % self.sets], self.w, self.b, self.ibuf, c.stride,
                                   c.pad, c.dilation, out_dtype=self.out_dtype,
                                   y=self.ys[i % self.sets])

    def launches_per_step(self):
        """Kernels of this library one conv2d_fwd launches, from its plan: the
        implicit GEMM, plus the indirection-buffer build (gather modes), the weight
        re-pack (stem modes), the window-order re-layout (im2win mode) and the
        split-K finishing pass."""
        p = self.plan()
        a = p["a_mode"]
        n = 1
        n += 1 if a in (1, 2, 3, 12) else 0      # build_indirection_kernel
        n += 1 if a in (2, 5, 10) else 0         # weight re-pack
        n += 1 if a == 10 else 0                 # im2win re-layout
        n += 1 if p["splits"] > 1 or p["stream_k"] else 0  # finish_split_kernel
        return n


def time_layer(layer, steps, warmup, stream):
    for i in range(warmup):
        layer.step(i)
    ms = graph_time_ms(layer.step, steps, stream)
    return ms / steps


def time_gemm_kernel(layer, steps, warmup, stream):
    c = layer.c
    if layer.num["path"] != "gather":
        return None
    layer.ibuf = layer.g.build_indirection_buffer(c.H, c.W, c.C_in, c.KH, c.KW, c.stride, c.pad,
                                                  c.dilation, device=layer.dev)
    for i in range(warmup):
        layer.gemm_only(i)
    return graph_time_ms(layer.gemm_only, steps, stream) / steps


def time_e2e(g, c, steps, warmup, dev, stream):
    """conv2d_fwd_host (the C ABI's host-buffer entry point) from pinned host buffers:
    every step copies x, w and bias in and y out, pipelined in chunks of the batch
    against the convolution."""
    x, w, b = workloads.make_inputs(c, device=dev)
    xh = x.cpu().pin_memory()
    wh = w.cpu().pin_memory()
    bh = b.cpu().pin_memory()
    num = shape_numbers(g, c)
    out_dtype = torch.float32 if c.out_f32 else torch.bfloat16
    yh = torch.empty((c.N, num["H_out"], num["W_out"], c.C_out), dtype=out_dtype).pin_memory()
    scratch = torch.empty(g.conv2d_fwd_host_scratch_size(
        c.N, c.C_in, c.H, c.W, c.C_out, c.KH, c.KW, c.stride, c.pad, c.dilation, out_dtype, True),
        dtype=torch.uint8, device=dev)

    def one(_):
        g.conv2d_fwd_host(xh, wh, bh, c.stride, c.pad, c.dilation, out_dtype=out_dtype, y=yh,
                          scratch=scratch)

    for i in range(warmup):
        one(i)
    ms = event_time_ms(one, steps, stream) / steps
    h2d = xh.numel() * 2 + wh.numel() * 2 + bh.numel() * 2
    d2h = yh.numel() * yh.element_size()
    return ms, h2d, d2h


def time_link(h2d_bytes, d2h_bytes, steps, dev):
    """Plain pinned copies of the e2e step's bytes, no convolution: the host->device
    and device->host legs on two streams at once (what a perfect overlap of the
    copies could reach), and each alone.  Milliseconds per step."""
    hin = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    hout = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    din = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    dout = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def run(which):
        for _ in range(3):
            _copies(which, hin, hout, din, dout, s1, s2)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            _copies(which, hin, hout, din, dout, s1, s2)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / steps * 1e3

    return {"both_ms": run("both"), "h2d_ms": run("h2d"), "d2h_ms": run("d2h")}


def _copies(which, hin, hout, din, dout, s1, s2):
    if which in ("both", "h2d"):
        with torch.cuda.stream(s1):
            din.copy_(hin, non_blocking=True)
    if which in ("both", "d2h"):
        with torch.cuda.stream(s2):
            hout.copy_(dout, non_blocking=True)


def time_im2win(g, c, steps, warmup, dev, stream):
    if c.C_in % 8 != 0:
        return None
    x, _, _ = workloads.make_inputs(c, device=dev)
    nb = g.im2win_bytes(c.N, c.C_in, c.H, c.W, c.KH, c.KW, c.stride, c.pad, c.dilation)
    if nb > (4 << 30):
        return None
    sets = rotation_sets(x.numel() * 2 + nb, cap_bytes=12 << 30)
    xs = [x] + [torch.randn_like(x, dtype=torch.float32).to(torch.bfloat16) for _ in range(sets - 1)]
    wins = [torch.empty(nb // 2, dtype=torch.bfloat16, device=dev) for _ in range(sets)]

    def one(i):
        g.im2win_transform(xs[i % sets], c.KH, c.KW, c.stride, c.pad, c.dilation,
                           win=wins[i % sets])

    for i in range(warmup):
        one(i)
    ms = graph_time_ms(one, steps, stream) / steps
    moved = x.numel() * 2 + nb  # read x once, write the buffer once
    return ms, moved


# --------------------------------------------------------------------------- CPU oracle
def cpu_baseline(c: workloads.ConvShape, budget_s=10.0):
    """fp64 oracle on the host cores over whole images of the batch, for about budget_s."""
    import oracle  # test/benchmark infrastructure only
    x, w, b = workloads.make_inputs(c)
    xb, wb, bb = workloads.bits(x), workloads.bits(w), workloads.bits(b)
    Ho = oracle.output_size(c.H, c.KH, c.stride, c.pad, c.dilation)
    Wo = oracle.output_size(c.W, c.KW, c.stride, c.pad, c.dilation)
    per_image = 2 * Ho * Wo * c.C_out * c.C_in * c.KH * c.KW
    t0 = time.perf_counter()
    n = 0
    while n < c.N and (time.perf_counter() - t0) < budget_s:
        oracle.conv2d_direct(xb[n:n + 1], wb, bb, c.stride, c.pad, c.dilation)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": per_image * n / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": "images 0..%d of the N=%d batch (%d of %d outputs), fp64 7-loop" % (
                n - 1, c.N, n * Ho * Wo * c.C_out, c.N * Ho * Wo * c.C_out)}


def run_reference(args):
    """--impl reference: the CPU oracle, timed per step on a bounded sample (one image)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    c = HEADLINE
    x, w, b = workloads.make_inputs(c)
    xb, wb, bb = workloads.bits(x), workloads.bits(w), workloads.bits(b)
    Ho = oracle.output_size(c.H, c.KH, c.stride, c.pad, c.dilation)
    Wo = oracle.output_size(c.W, c.KW, c.stride, c.pad, c.dilation)
    per_image = 2 * Ho * Wo * c.C_out * c.C_in * c.KH * c.KW
    for i in range(args.warmup):
        oracle.conv2d_direct(xb[i % c.N:i % c.N + 1], wb, bb, c.stride, c.pad, c.dilation)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.conv2d_direct(xb[i % c.N:i % c.N + 1], wb, bb, c.stride, c.pad, c.dilation)
    dt = time.perf_counter() - t0
    value = per_image * args.steps / dt / 1e12
    sample = "one image (1/%d of the batch) per step, fp64 7-loop oracle" % c.N
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": c.name, "N": c.N, "C_in": c.C_in, "H": c.H, "W": c.W,
                       "C_out": c.C_out, "KH": c.KH, "KW": c.KW, "stride": c.stride,
                       "pad": c.pad, "dilation": c.dilation, "step_sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- ablations
# (layer, label, tuning bn, tuning max_stages, path, cin_pad): each group runs in
# one process, one after another, so its rows compare like with like.
def ablation_rows():
    R = workloads.BY_NAME
    rows = []
    for st in (2, 3, 0):
        rows.append(("resnet_3x3_64to128_56", "stages<=%d" % st if st else "default", 0, st, 0, 0))
    for st in (2, 3, 0):
        rows.append(("sweep_3x3_256c_28", "stages<=%d" % st if st else "default", 0, st, 0, 0))
    for st in (2, 3, 4, 6, 0):
        rows.append(("pointwise_1x1_256to64_56", "stages<=%d" % st if st else "default", 0, st,
                     0, 0))
    for st in (4, 5, 0):  # the TMA gather's four warps take turns: at least four stages
        rows.append(("strided_3x3_s2_128to256_56", "stages<=%d" % st if st else "default", 0,
                     st, 0, 0))
    for st in (2, 4, 0):
        rows.append(("sweep_3x3_32c_150", "stages<=%d" % st if st else "default", 0, st, 0, 0))
    # taps folded into the MMA's columns (default) against the gather path's N=32 MMAs
    rows.append(("sweep_3x3_32c_150", "gather path", 0, 0, 1, 0))
    for bn in (64, 128, 256):
        rows.append(("sweep_3x3_256c_28", "bn=%d" % bn, bn, 0, 0, 0))
        rows.append(("strided_3x3_s2_128to256_56", "bn=%d" % bn, bn, 0, 0, 0))
        rows.append(("sweep_1x1_512to2048_7", "bn=%d" % bn, bn, 0, 0, 0))
    for name in ("stem_7x7_s2_3to64_224", "sweep_11x11_s4_3to64_224"):
        rows.append((name, "staged-window stem path (default)", 0, 0, 0, 0))
        rows.append((name, "im2win path", 0, 0, 6, 0))
        rows.append((name, "staged-row stem path", 0, 0, 3, 0))
        rows.append((name, "gather path, C_in padded to 8", 0, 0, 1, 8))
    rows.append(("sweep_3x3_512c_7", "whole units (default)", 0, 0, 0, 0))
    rows.append(("sweep_3x3_512c_7", "stream-K", 0, 0, 0, 0, 1))
    return [(R[r[0]],) + tuple(r[1:]) + ((0,) if len(r) == 6 else ()) for r in rows]


def run_ablation(g, dev, stream, steps):
    out = []
    for c, label, bn, st, path, cin_pad, sk in ablation_rows():
        g.set_tuning(bn, st, sk)
        try:
            L = Layer(g, c, dev, path=path, cin_pad=cin_pad)
            ms = time_layer(L, steps, 3, stream)
            plan = L.plan()
            st_, code = g.check_device_errors()
            ent = {"workload": c.name, "variant": label, "us": ms * 1e3,
                   "tflops": L.num["flops"] / (ms * 1e-3) / 1e12,
                   "plan": {k: plan[k] for k in ("path", "a_mode", "bn", "stages",
                                                 "weights_resident", "cta_pair", "splits",
                                                 "stream_k")},
                   "device_status": st_}
            del L
            torch.cuda.empty_cache()
        except Exception as e:
            ent = {"workload": c.name, "variant": label, "error": str(e)[:200]}
        finally:
            g.set_tuning(0, 0)
        print("ablation " + json.dumps(ent), flush=True)
        out.append(ent)
    return out


# --------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=HEADLINE.name, help="workload name (workloads.py)")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-configuration sweep")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--sweep-steps", type=int, default=30)
    ap.add_argument("--profile-launches", type=int, default=0,
                    help="profiling mode: run this many eager conv2d_fwd calls of --config "
                         "(batch --batch) and exit without timing or output")
    ap.add_argument("--batch", type=int, default=0, help="override N of --config (profiling)")
    ap.add_argument("--profile-op", choices=["conv", "im2win"], default="conv",
                    help="profiling mode: conv2d_fwd (default) or the exported im2win_transform")
    ap.add_argument("--ablate", action="store_true",
                    help="run the ablation study (tile width, ring depth, stem paths) and exit; "
                         "one 'ablation {json}' line per row")
    ap.add_argument("--clock-probe-s", type=float, default=0.5,
                    help="seconds of untimed steps before the timed region, so the clock "
                         "sampler sees the GPU under load (0 disables)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    world, rank, local = dist_env()
    import indirect_implicit_gemm_gb300 as g
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    g.load()
    peaks, peak_src = load_peaks()
    c = workloads.BY_NAME[args.config]
    if args.batch:
        c = c.scaled(args.batch, "_n%d" % args.batch)
    if args.profile_launches:
        if args.profile_op == "im2win":
            x, _, _ = workloads.make_inputs(c, device=dev)
            for i in range(args.profile_launches):
                g.im2win_transform(x, c.KH, c.KW, c.stride, c.pad, c.dilation)
        else:
            layer = Layer(g, c, dev, sets=1)
            for i in range(args.profile_launches):
                layer.step(i)
        torch.cuda.synchronize()
        st, code = g.check_device_errors()
        return 0 if st == 0 else 1
    stream = torch.cuda.current_stream()
    if args.ablate:
        run_ablation(g, dev, stream, args.sweep_steps)
        return 0
    layer = Layer(g, c, dev)
    num = layer.num

    # headline: whole conv2d_fwd per step, clocks sampled around the timed region
    for i in range(args.warmup):
        layer.step(i)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    with ClockSampler(local) as clk:
        # keep the GPU busy long enough for the sampler to see load
        t_end = time.perf_counter() + args.clock_probe_s
        i = 0
        while time.perf_counter() < t_end and i < 20000:
            layer.step(i)
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        ms_total = graph_time_ms(layer.step, args.steps, stream)
        if pg:
            pg.barrier()
    clocks = clk.summary()
    ms_step = reduce_max(ms_total / args.steps, pg, dev)
    value = world * num["flops"] / (ms_step * 1e-3) / 1e12

    # the dominant kernel alone (implicit GEMM), for the roofline: timed on its
    # own on the gather path (whose step also builds the indirection buffer);
    # on single-launch paths the step is that kernel
    k_ms = time_gemm_kernel(layer, max(args.steps, 50), 5, stream)
    if k_ms is None and layer.launches_per_step() == 1:
        k_ms = time_layer(layer, max(args.steps, 50), 5, stream)
    t_roof, bound = roofline_time_s(num, peaks)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    roof = None
    if k_ms is not None:
        if bound == "tensor":
            achieved = num["flops"] / (k_ms * 1e-3) / 1e12
            peak = peaks["bf16_tflops"]
            unit = "TFLOP/s"
        else:
            achieved = num["bytes"] / (k_ms * 1e-3) / 1e9
            peak = peaks["hbm_gbs"]
            unit = "GB/s"
        tr = profiled_traffic(c.name)
        roof = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": tr["total"] if tr else None,
                "traffic_read": tr["read"] if tr else None,
                "traffic_write": tr["write"] if tr else None,
                "traffic_note": "DRAM bytes read + written while the launch runs (ncu); "
                                "output lines still dirty in L2 when it ends are written "
                                "back later and are not in the figure",
                "algorithmic_bytes": num["bytes"],
                "kernel": "igemm_kernel (%s path, tcgen05)" % num["path"],
                "kernel_us": k_ms * 1e3,
                "peak_source": "%s (MEASURED_PEAKS.json %s)" % (
                    peak_src, "bf16_tflops burst" if bound == "tensor" else "hbm_gbs"),
                "roofline_us": t_roof * 1e6,
                "frac_of_roofline": (t_roof * 1e3) / k_ms}
        if clocks.get("sm_mhz"):
            # the tensor cores' rate at the clock the kernel ran at: 8192 bf16
            # flop per SM per cycle (a 128x128x16 MMA issues every 64 cycles)
            clk_peak = sms * TC_FLOP_PER_CLK_SM * clocks["sm_mhz"] * 1e6 / 1e12
            roof["tensor_peak_at_clock_tflops"] = clk_peak
            roof["tensor_frac_at_clock"] = num["flops"] / (k_ms * 1e-3) / 1e12 / clk_peak

    single = single_launch_us(layer, stream)
    e2e_ms, h2d, d2h = time_e2e(g, c, max(10, args.steps // 10), 3, dev, stream)
    link = time_link(h2d, d2h, max(10, args.steps // 10), dev)
    e2e = {"value": world * num["flops"] / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "link_ms_per_step": link["both_ms"], "link_h2d_ms": link["h2d_ms"],
           "link_d2h_ms": link["d2h_ms"], "frac_of_link": link["both_ms"] / e2e_ms,
           "link_note": "plain pinned cudaMemcpyAsync of the same bytes, both directions "
                        "at once on two streams, no convolution"}

    sweep = []
    if not args.no_sweep:
        for sc in workloads.ALL:
            try:
                L = Layer(g, sc, dev)
                ms = time_layer(L, args.sweep_steps, 3, stream)
                tr, bd = roofline_time_s(L.num, peaks)
                ent = {"workload": sc.name, "path": L.num["path"], "us": ms * 1e3,
                       "tflops": L.num["flops"] / (ms * 1e-3) / 1e12,
                       "gbs": L.num["bytes"] / (ms * 1e-3) / 1e9,
                       "bound": bd, "roofline_us": tr * 1e6, "frac_of_roofline": tr * 1e3 / ms,
                       "workspace_bytes": L.num["workspace_bytes"],
                       "im2col_bytes": L.num["im2col_bytes"],
                       "im2win_bytes": L.num["im2win_bytes"]}
                kms = time_gemm_kernel(L, args.sweep_steps, 3, stream)
                if kms is not None:
                    ent["gemm_kernel_us"] = kms * 1e3
                    ent["gemm_frac_of_roofline"] = tr * 1e3 / kms
                iw = time_im2win(g, sc, args.sweep_steps, 3, dev, stream)
                if iw is not None:
                    ent["im2win_us"] = iw[0] * 1e3
                    ent["im2win_gbs"] = iw[1] / (iw[0] * 1e-3) / 1e9
                    ent["im2win_frac_hbm"] = ent["im2win_gbs"] / peaks["hbm_gbs"]
                del L
                torch.cuda.empty_cache()
            except Exception as e:  # keep the headline line even if one sweep entry fails
                ent = {"workload": sc.name, "error": str(e)[:200]}
            sweep.append(ent)
            if rank == 0:  # one line per configuration, ahead of the headline line
                print("sweep " + json.dumps(ent), flush=True)

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(c)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded normal x, fan-in-scaled w, N(0,0.1) bias; bf16)",
        "config": {"workload": c.name, "N": c.N, "C_in": c.C_in, "H": c.H, "W": c.W,
                   "C_out": c.C_out, "KH": c.KH, "KW": c.KW, "stride": c.stride, "pad": c.pad,
                   "dilation": c.dilation, "out_dtype": "fp32" if c.out_f32 else "bf16",
                   "path": num["path"], "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2: %d rotating x/y sets of %.1f MB" % (
                       layer.sets, (num["x_bytes"] + num["y_bytes"]) / 1e6),
                   "workspace_bytes": num["workspace_bytes"], "im2col_bytes": num["im2col_bytes"],
                   "roofline_us": t_roof * 1e6,
                   "frac_of_roofline": t_roof * 1e3 / ms_step},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": layer.launches_per_step() * args.steps,
        "single_launch": single,
        "clocks": clocks, "sweep": sweep_summary(sweep),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
