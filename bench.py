#!/usr/bin/env python
"""Benchmark of the W4A16 group-quantized matmul on GB300.

Headline (one JSON line on stdout): the decode GEMV of the Llama-3-8B MLP up-projection
(M = 1, N = 14336, K = 4096, group 128) -- a step is one ``w4a16_matmul`` launch on
weights already resident in HBM. Throughput is the effective HBM bandwidth on weight +
scale bytes (the pages' "effective GB/s": format bytes / time), timed with CUDA events
around CUDA-graph replays that rotate over 12 weight copies (374 MB, more than twice the
129 MB L2), so no launch finds its weights in L2.

The same line carries the other steps of the hot path as "rows": GPU quantize and pack,
the batch sweep M = 1..4096 against a BF16 cuBLAS matmul at the same M, the Q4 block-32
quantize and GEMV (16384 x 16384), the zero-point format (quantize, layout move, matmul at
M = 1, 16, 4096), the W8A16 per-row INT8, NVFP4A16 and MXFP4A16 quantize and GEMV, and the
196-matmul Qwen2.5-1.5B-shaped decode stack in one CUDA graph (also with q/k/v and gate/up
concatenated: 112 matmuls); each with its roofline fraction.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-rows]
  python bench.py --case gemv_m1 --launches 6     # a few untimed launches, for ncu

With --impl reference the CPU oracle is timed instead (bounded samples of the same
workload, same metric). Under torchrun each rank runs an independent replica on its own
GPU (the GEMV does not shard); rank 0 prints the line with the max time over ranks.
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

METRIC = "W4A16 µs & effective HBM GB/s at M=1; TFLOPS vs M=1..4096; % of roofline"
PAGES_M1_GBPS = 169.0  # the pages' M=1 effective bandwidth for this shape (RTX 4060 Laptop)
ROTATE = 12            # weight copies in rotation (12 x 31.2 MB > 2 x L2)
GRAPH_LEN = 96         # launches per captured graph in the timed loop
EVENT_GRAPH_MAX = 2048  # up to this many steps a region is one graph with its events inside
EVENT_GRAPH_PRE = 8     # untimed launches at the head of such a graph
ROUNDS = 3             # timed regions per run; the median is reported
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- #
# distributed plumbing (replicas only)
# --------------------------------------------------------------------------- #

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- #
# peaks, clocks
# --------------------------------------------------------------------------- #

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except OSError:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------------- #
# timing helpers
# --------------------------------------------------------------------------- #

def capture(fn, count: int, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(count):
            fn(i)
    return g


def graph_time_us(fn, launches: int, reps: int, stream) -> float:
    """Average device time per launch of fn(i), i = 0..launches-1 captured once and
    replayed `reps` times (CUDA events on the capture stream)."""
    with torch.cuda.stream(stream):
        for i in range(3):
            fn(i)
    torch.cuda.synchronize()
    g = capture(fn, launches, stream)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) * 1e3 / (launches * reps)


def w4a16_bytes(M, N, K, group=128):
    """Algorithmic bytes of one matmul: packed codes + BF16 scale/min + x + y."""
    return N * K // 2 + 4 * N * (K // group) + 2 * M * K + 2 * M * N


def weight_bytes(N, K, group=128):
    return N * K // 2 + 4 * N * (K // group)


def roofline_us(bytes_, flops, peaks):
    return max(bytes_ / (peaks["hbm_gbs"] * 1e3), flops / (peaks["bf16_tflops"] * 1e6))


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #

def workspace_for(M, N, K, device):
    """The workspace the library asks for at this shape (zero-filled), or None: split-K
    partials and counters, or the skinny kernel's converted activations."""
    import gemv_w4a16_group_gb300 as w4

    need = w4.w4a16_matmul_workspace_bytes(M, N, K)
    return torch.zeros(need, dtype=torch.uint8, device=device) if need else None


def prepared_workspace_for(M, N, K, device):
    """The workspace w4a16_matmul_prepared asks for at this shape (zero-filled), or None."""
    import gemv_w4a16_group_gb300 as w4

    need = w4.w4a16_matmul_prepared_workspace_bytes(M, N, K)
    return torch.zeros(need, dtype=torch.uint8, device=device) if need else None


def quantized_on_device(N, K, seed, device, outlier_frac=0.0):
    import gemv_w4a16_group_gb300 as w4

    w = workloads.weights(N, K, seed=seed, outlier_frac=outlier_frac).to(device)
    codes, s, m = w4.w4a16_quantize(w)
    qw = w4.w4a16_pack(codes)
    return w, codes, qw, s, m


def run_ours(args, world, rank, local):
    import gemv_w4a16_group_gb300 as w4

    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    peaks, peaks_src = load_peaks()
    stream = torch.cuda.Stream(device)
    cfg = workloads.LLAMA_UP
    M, N, K = cfg["M"], cfg["N"], cfg["K"]

    w, codes, qw, s, m = quantized_on_device(N, K, 0, device)
    del w, codes
    copies = [(qw.clone(), s.clone(), m.clone()) for _ in range(ROTATE)]
    x = workloads.activations_bf16(M, K, seed=0).to(device)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
    bytes_w = weight_bytes(N, K)

    ws = workspace_for(M, N, K, device)

    def step(i):
        c = copies[i % ROTATE]
        w4.w4a16_matmul(x, c[0], c[1], c[2], y=y, workspace=ws)

    # warm-up: W untimed steps, then capture the timed loop
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize()
    in_graph = args.steps <= EVENT_GRAPH_MAX
    if in_graph:
        # One graph per region: EVENT_GRAPH_PRE untimed launches, then exactly --steps timed
        # ones. The start and end events are recorded inside the graph on a branch forked
        # from the launch stream after the last untimed and the last timed launch, so the
        # chain of dependent launches is not broken and the region runs from the completion
        # of the last untimed launch to that of the last timed one: --steps launches in the
        # steady state, with no host latency inside.
        side = torch.cuda.Stream(device)
        ev0 = torch.cuda.Event(enable_timing=True, external=True)
        ev1 = torch.cuda.Event(enable_timing=True, external=True)
        fork0, fork1, join = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        g_main = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_main, stream=stream):
            for i in range(EVENT_GRAPH_PRE):
                step(i)
            fork0.record(stream)
            side.wait_event(fork0)
            ev0.record(side)
            for i in range(args.steps):
                step(EVENT_GRAPH_PRE + i)
            fork1.record(stream)
            side.wait_event(fork1)
            ev1.record(side)
            join.record(side)
            stream.wait_event(join)
        g_tail = None
    else:
        glen = min(GRAPH_LEN, args.steps)
        g_main = capture(step, glen, stream)
        tail = args.steps % glen
        g_tail = capture(step, tail, stream) if tail else None
    with torch.cuda.stream(stream):
        g_main.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.25)
    # ROUNDS timed regions of exactly --steps launches each; the median is reported. For long
    # runs (several graphs per region) an untimed replay is already queued before each
    # region, so that its start event fires when the GPU reaches it rather than when the host
    # gets there.
    region_s = []
    for _ in range(ROUNDS):
        barrier(world)
        torch.cuda.synchronize()
        if in_graph:
            with torch.cuda.stream(stream):
                g_main.replay()
            torch.cuda.synchronize()
            barrier(world)
            region_s.append(ev0.elapsed_time(ev1) / 1e3)
            continue
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            g_main.replay()  # untimed: keeps the GPU busy while the timed region is queued
            ev0.record(stream)
            for _ in range(args.steps // glen):
                g_main.replay()
            if g_tail is not None:
                g_tail.replay()
            ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        region_s.append(ev0.elapsed_time(ev1) / 1e3)
    sampler.stop()
    local_s = statistics.median(region_s)
    max_s = reduce_max(local_s, world, device)
    clocks = sampler.summary()
    us_per_step = local_s / args.steps * 1e6

    result = None
    if rank == 0:
        value = world * bytes_w * args.steps / max_s / 1e9
        achieved = bytes_w / (us_per_step * 1e3)
        traffic = read_traffic("gemv_w4a16_kernel", w4a16_bytes(M, N, K))
        result = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(max_s / args.steps * 1e3, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": round(value / world / PAGES_M1_GBPS, 2),
            "vs_baseline_ref": "169 GB/s at M=1 on this shape, RTX 4060 Laptop (pages)",
            "dtype": "bf16", "accumulate": "fp32", "weights": "int4 group-128 (4.25 bit)",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) BF16 x)",
            "config": {"workload": cfg["name"], "M": M, "N": N, "K": K, "group": cfg["group"]},
            "timing": {"l2": f"rotating {ROTATE} weight copies ({ROTATE * bytes_w / 1e6:.0f} MB "
                             "> 2x L2), CUDA-graph replay",
                       "statistic": (f"median of {ROUNDS} timed regions of {args.steps} launches, "
                                     + (f"each one graph of {EVENT_GRAPH_PRE} untimed + "
                                        f"{args.steps} timed launches with its events recorded "
                                        "inside on a forked branch" if in_graph else
                                        "each started behind an untimed replay")),
                       "us_per_step": round(us_per_step, 3),
                       "regions_us_per_step": [round(t / args.steps * 1e6, 3) for t in region_s],
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": traffic, "peak_source": f"{peaks_src} copy bandwidth",
                         "algorithmic_bytes_per_launch": bytes_w},
            "gpu_launches": args.steps,
            "clocks": clocks,
        }
        result["e2e"] = e2e_ours(copies, x, y, M, N, K, device, stream)
    del copies
    if rank == 0 and world == 1 and not args.no_rows:
        result["rows"] = rows_ours(peaks, device, stream)
    if rank == 0 and world == 1:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    barrier(world)
    return result


def kernel_source_digest(files) -> str:
    """sha256 over the CUDA sources a kernel is built from (to tell stale counters)."""
    import hashlib

    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gemv_w4a16_group_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def read_traffic(kernel: str, algorithmic: int):
    """DRAM bytes (read + write) per launch from the committed ncu summary
    (profiles/traffic.json), or None when the kernel's sources changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f).get(kernel)
        if entry and entry["source_sha256"] == kernel_source_digest(entry["sources"]):
            return entry["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        pass
    return None


def e2e_ours(copies, x_dev, y_dev, M, N, K, device, stream, steps=2000):
    """Same metric through the C-ABI call with host buffers (w4a16_matmul_host): each step
    copies x from pinned host memory, runs the matmul and copies y back to pinned host
    memory (one library call), then waits for the result on the host."""
    import gemv_w4a16_group_gb300 as w4

    ws = workspace_for(M, N, K, device)
    x_host = x_dev.cpu().pin_memory()
    y_host = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    bytes_w = weight_bytes(N, K)
    for i in range(20):
        c = copies[i % ROTATE]
        w4.w4a16_matmul_host(x_host, c[0], c[1], c[2], y_host=y_host, x_dev=x_dev, y_dev=y_dev,
                             workspace=ws, stream=stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        c = copies[i % ROTATE]
        w4.w4a16_matmul_host(x_host, c[0], c[1], c[2], y_host=y_host, x_dev=x_dev, y_dev=y_dev,
                             workspace=ws, stream=stream)
        stream.synchronize()  # the step's result is on the host
    t1 = time.perf_counter()
    return {"value": round(bytes_w * steps / (t1 - t0) / 1e9, 1), "unit": "GB/s",
            "us_per_step": round((t1 - t0) / steps * 1e6, 2),
            "h2d_bytes_per_step": x_host.numel() * 2, "d2h_bytes_per_step": y_host.numel() * 2}


def rows_ours(peaks, device, stream):
    """Every step of the hot path on its own workload, with its roofline fraction."""
    import gemv_w4a16_group_gb300 as w4

    rows = {}
    hbm = peaks["hbm_gbs"]
    # quantize + pack on the Llama up-projection weights
    N, K = workloads.LLAMA_UP["N"], workloads.LLAMA_UP["K"]
    w, codes, qw, s, m = quantized_on_device(N, K, 0, device)
    us = graph_time_us(lambda i: w4.w4a16_quantize(w, codes=codes, scales=s, mins=m), 4, 5, stream)
    b = N * K * 4 + N * K + 4 * N * (K // 128)
    rows["w4a16_quantize"] = {"shape": [N, K], "us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                              "frac_hbm": round(b / us / 1e3 / hbm, 3)}
    us = graph_time_us(lambda i: w4.w4a16_pack(codes, qw=qw), 4, 5, stream)
    b = N * K + N * K // 2
    rows["w4a16_pack"] = {"shape": [N, K], "us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                          "frac_hbm": round(b / us / 1e3 / hbm, 3)}
    # prepared (reordered) copy of the same packed weights
    prep = w4.w4a16_prepare(qw, s, m)
    us = graph_time_us(lambda i: w4.w4a16_prepare(qw, s, m, prepared=prep), 4, 5, stream)
    b = 2 * weight_bytes(N, K)  # canonical bytes read, the same bytes written reordered
    rows["w4a16_prepare"] = {"shape": [N, K], "us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                             "frac_hbm": round(b / us / 1e3 / hbm, 3)}
    del w, codes, qw, s, m, prep

    # batch sweep with outliers, against BF16 cuBLAS at the same M
    cfg = workloads.BATCH_SWEEP
    N, K = cfg["N"], cfg["K"]
    w, codes, qw, s, m = quantized_on_device(N, K, 0, device, outlier_frac=cfg["outlier_frac"])
    w_bf16 = w.to(torch.bfloat16)
    del w, codes
    cps = [(qw.clone(), s.clone(), m.clone()) for _ in range(ROTATE)]
    preps = [w4.w4a16_prepare(*c) for c in cps]
    bf_cps = [w_bf16.clone() for _ in range(3)]  # 3 x 117 MB > 2 x L2
    sweep = []
    for M in cfg["Ms"]:
        x = workloads.activations_bf16(M, K, seed=M).to(device)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
        ws = workspace_for(M, N, K, device)
        big = M >= 1024
        us = graph_time_us(lambda i: w4.w4a16_matmul(x, *cps[i % ROTATE], y=y, workspace=ws),
                           ROTATE if big else 4 * ROTATE, 2 if big else 10, stream)
        us_bf = graph_time_us(lambda i: torch.matmul(x, bf_cps[i % 3].T, out=y),
                              6 if big else 12, 2 if big else 10, stream)
        bts, fl = w4a16_bytes(M, N, K), 2 * M * N * K
        roof = roofline_us(bts, fl, peaks)
        prepared = None
        if w4.w4a16_matmul_prepared_uses_prepared(M):
            wsp = prepared_workspace_for(M, N, K, device)
            us_p = graph_time_us(
                lambda i: w4.w4a16_matmul_prepared(x, *cps[i % ROTATE], preps[i % ROTATE], y=y,
                                                   workspace=wsp),
                ROTATE if big else 4 * ROTATE, 2 if big else 10, stream)
            prepared = {"us": round(us_p, 2), "frac": round(roof / us_p, 3),
                        "speedup_vs_bf16": round(us_bf / us_p, 2) if us_bf else None}
        sweep.append({"M": M, "us": round(us, 2), "TFLOPS": round(fl / us / 1e6, 1),
                      "GBps": round(bts / us / 1e3, 1), "roofline_us": round(roof, 2),
                      "frac": round(roof / us, 3),
                      "bound": "hbm" if bts / (peaks["hbm_gbs"] * 1e3) >= fl / (peaks["bf16_tflops"] * 1e6) else "tensor",
                      "bf16_cublas_us": round(us_bf, 2),
                      "bf16_cublas_TFLOPS": round(fl / us_bf / 1e6, 1),
                      "speedup_vs_bf16": round(us_bf / us, 2),
                      "prepared_layout": prepared})
        del x, y
    del cps, preps, bf_cps, w_bf16
    rows["batch_sweep"] = sweep
    def best_us(r):
        p = r.get("prepared_layout")
        return min(r["us"], p["us"]) if p else r["us"]

    even = [r["M"] for r in sweep if r["bf16_cublas_us"] <= best_us(r)]
    bpw = 4.25 / 8
    rows["crossover"] = {
        "predicted_4bit_ridge_M": round(peaks["bf16_tflops"] * 1e12 * bpw / (2 * peaks["hbm_gbs"] * 1e9), 1),
        "predicted_bf16_ridge_M": round(peaks["bf16_tflops"] * 1e12 * 2 / (2 * peaks["hbm_gbs"] * 1e9), 1),
        "measured_breakeven_vs_bf16_M": even[0] if even else None,
        "pages": "~28 (4-bit) and ~100 (BF16) at a ridge of 102 FLOP/B; break-even at 128 measured"}

    # zero-point format on the up-projection: quantize, move to the matmul's layout, and the
    # matmul at M = 1, 16 and 4096 (same kernels as the minimum form, FP16 scale and zero)
    N, K = workloads.LLAMA_UP["N"], workloads.LLAMA_UP["K"]
    w = workloads.weights(N, K, seed=0).to(device)
    qr, zs, zz = w4.w4a16zp_quantize(w)
    us = graph_time_us(lambda i: w4.w4a16zp_quantize(w, qw_rows=qr, scales=zs, zeros=zz), 4, 5,
                       stream)
    b = N * K * 4 + N * K // 2 + 4 * N * (K // 128)
    zp = {"shape": [N, K],
          "quantize": {"us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                       "frac_hbm": round(b / us / 1e3 / hbm, 3)}}
    del w
    qk, sk, zk = w4.w4a16zp_prepare(qr, zs, zz)
    us = graph_time_us(lambda i: w4.w4a16zp_prepare(qr, zs, zz, qw=qk, scales_t=sk, zeros_t=zk),
                       4, 5, stream)
    b = 2 * (N * K // 2 + 4 * N * (K // 128))
    zp["prepare"] = {"us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                     "frac_hbm": round(b / us / 1e3 / hbm, 3)}
    del qr, zs, zz
    cps = [(qk.clone(), sk.clone(), zk.clone()) for _ in range(ROTATE)]
    mm = []
    for M in (1, 16, 4096):
        x = workloads.activations_bf16(M, K, seed=M).to(device)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
        ws = workspace_for(M, N, K, device)
        big = M >= 1024
        us = graph_time_us(lambda i: w4.w4a16zp_matmul(x, *cps[i % ROTATE], y=y, workspace=ws),
                           ROTATE if big else 4 * ROTATE, 2 if big else 10, stream)
        bts, fl = w4a16_bytes(M, N, K), 2 * M * N * K
        roof = roofline_us(bts, fl, peaks)
        mm.append({"M": M, "us": round(us, 2), "TFLOPS": round(fl / us / 1e6, 1),
                   "GBps": round(bts / us / 1e3, 1), "roofline_us": round(roof, 2),
                   "frac": round(roof / us, 3)})
        del x, y
    zp["matmul"] = mm
    rows["zero_point"] = zp
    del cps, qk, sk, zk

    # W8A16 (per-row INT8) on the up-projection: quantize and the M = 1 GEMV
    N, K = workloads.LLAMA_UP["N"], workloads.LLAMA_UP["K"]
    w = workloads.weights(N, K, seed=0).to(device)
    q8, s8 = w4.w8a16_quantize(w)
    us = graph_time_us(lambda i: w4.w8a16_quantize(w, q=q8, scales=s8), 4, 5, stream)
    b = N * K * 4 + N * K + 4 * N
    w8 = {"shape": [N, K], "quantize": {"us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                                         "frac_hbm": round(b / us / 1e3 / hbm, 3)}}
    del w
    cps8 = [(q8.clone(), s8.clone()) for _ in range(8)]  # 8 x 58.7 MB > 2 x L2
    x8 = workloads.activations_bf16(1, K, seed=1)[0].to(device)
    y8 = torch.empty(N, dtype=torch.bfloat16, device=device)
    us = graph_time_us(lambda i: w4.w8a16_gemv(x8, *cps8[i % 8], y=y8), 16, 10, stream)
    b = N * K + 4 * N
    w8["gemv"] = {"us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                  "frac_hbm": round(b / us / 1e3 / hbm, 3), "roofline_us": round(b / hbm / 1e3, 2)}
    rows["w8a16"] = w8
    del cps8, q8, s8

    # NVFP4A16 on the up-projection: quantize and the M = 1 GEMV
    w = workloads.weights(N, K, seed=0).to(device)
    c4, s4, S4 = w4.nvfp4_quantize(w)
    us = graph_time_us(lambda i: w4.nvfp4_quantize(w, codes=c4, scales=s4, tensor_scale=S4), 4, 5,
                       stream)
    b = N * K * 4 * 2 + N * K // 2 + N * K // 16  # two reads of w (amax, then codes)
    nv = {"shape": [N, K], "quantize": {"us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                                         "frac_hbm": round(b / us / 1e3 / hbm, 3)}}
    del w
    cps4 = [(c4.clone(), s4.clone(), S4.clone()) for _ in range(ROTATE)]
    us = graph_time_us(lambda i: w4.nvfp4_gemv(x8, *cps4[i % ROTATE], y=y8), 2 * ROTATE, 10, stream)
    b = N * K // 2 + N * K // 16
    nv["gemv"] = {"us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                  "frac_hbm": round(b / us / 1e3 / hbm, 3), "roofline_us": round(b / hbm / 1e3, 2)}
    for Mb in (8, 32):  # the M > 1 matmul (x prepared once, one pass per 32 rows)
        xb = workloads.activations_bf16(Mb, K, seed=Mb).to(device)
        yb = torch.empty(Mb, N, dtype=torch.bfloat16, device=device)
        wsb = torch.empty(w4.fp4_matmul_workspace_bytes(Mb, K), dtype=torch.uint8, device=device)
        us = graph_time_us(lambda i: w4.nvfp4_matmul(xb, *cps4[i % ROTATE], y=yb, workspace=wsb),
                           2 * ROTATE, 10, stream)
        bb = b + 2 * Mb * K + 2 * Mb * N
        nv[f"matmul_m{Mb}"] = {"us": round(us, 2), "GBps": round(bb / us / 1e3, 1),
                               "frac_hbm": round(bb / us / 1e3 / hbm, 3)}
        del xb, yb, wsb
    rows["nvfp4a16"] = nv
    del cps4, c4, s4, S4

    # MXFP4A16 on the up-projection: quantize and the M = 1 GEMV
    w = workloads.weights(N, K, seed=0).to(device)
    cm, sm_ = w4.mxfp4_quantize(w)
    us = graph_time_us(lambda i: w4.mxfp4_quantize(w, codes=cm, scales=sm_), 4, 5, stream)
    b = N * K * 4 + N * K // 2 + N * K // 32
    mx = {"shape": [N, K], "quantize": {"us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                                         "frac_hbm": round(b / us / 1e3 / hbm, 3)}}
    del w
    cpsm = [(cm.clone(), sm_.clone()) for _ in range(ROTATE)]
    us = graph_time_us(lambda i: w4.mxfp4_gemv(x8, *cpsm[i % ROTATE], y=y8), 2 * ROTATE, 10, stream)
    b = N * K // 2 + N * K // 32
    mx["gemv"] = {"us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                  "frac_hbm": round(b / us / 1e3 / hbm, 3), "roofline_us": round(b / hbm / 1e3, 2)}
    for Mb in (8, 32):
        xb = workloads.activations_bf16(Mb, K, seed=Mb).to(device)
        yb = torch.empty(Mb, N, dtype=torch.bfloat16, device=device)
        wsb = torch.empty(w4.fp4_matmul_workspace_bytes(Mb, K), dtype=torch.uint8, device=device)
        us = graph_time_us(lambda i: w4.mxfp4_matmul(xb, *cpsm[i % ROTATE], y=yb, workspace=wsb),
                           2 * ROTATE, 10, stream)
        bb = b + 2 * Mb * K + 2 * Mb * N
        mx[f"matmul_m{Mb}"] = {"us": round(us, 2), "GBps": round(bb / us / 1e3, 1),
                               "frac_hbm": round(bb / us / 1e3 / hbm, 3)}
        del xb, yb, wsb
    rows["mxfp4a16"] = mx
    del cpsm, cm, sm_, x8, y8

    # Q4 block-32, 16384 x 16384
    qc_cfg = workloads.Q4_SQUARE
    N, K = qc_cfg["N"], qc_cfg["K"]
    w = workloads.weights(N, K, seed=0).to(device)
    qc, qsc = w4.q4b32_quantize(w)
    us = graph_time_us(lambda i: w4.q4b32_quantize(w, codes=qc, scales=qsc), 2, 3, stream)
    b = N * K * 4 + N * K // 2 + N * K // 16
    rows["q4b32_quantize"] = {"shape": [N, K], "us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                              "frac_hbm": round(b / us / 1e3 / hbm, 3)}
    del w
    xq = workloads.activations_fp16(K, seed=0).to(device)
    yq = torch.empty(N, dtype=torch.float16, device=device)
    qcps = [(qc.clone(), qsc.clone()) for _ in range(2)] + [(qc, qsc)]
    us = graph_time_us(lambda i: w4.q4b32_gemv(xq, *qcps[i % 3], y=yq), 12, 10, stream)
    b = N * K * 18 // 32
    rows["q4b32_gemv"] = {"shape": [N, K], "us": round(us, 2), "GBps": round(b / us / 1e3, 1),
                          "frac_hbm": round(b / us / 1e3 / hbm, 3), "roofline_us": round(b / hbm / 1e3, 2),
                          "pages": "93.0 us (1,624 GB/s) on an RTX 5090"}
    del qcps, qc, qsc

    # Qwen2.5-1.5B-shaped decode stack: 196 matmuls in one CUDA graph
    stack = []
    tot_bytes = 0
    for layer in range(workloads.QWEN_STACK["layers"]):
        for name, Nl, Kl in workloads.QWEN_STACK["block"]:
            g = torch.Generator(device=device)
            g.manual_seed(layer * 16 + len(stack))
            wl = torch.randn(Nl, Kl, generator=g, device=device) * workloads.WEIGHT_STD
            cl, sl, ml = w4.w4a16_quantize(wl)
            ql = w4.w4a16_pack(cl)
            del wl, cl
            xl = torch.randn(1, Kl, generator=g, device=device).to(torch.bfloat16)
            yl = torch.empty(1, Nl, dtype=torch.bfloat16, device=device)
            stack.append((xl, ql, sl, ml, yl, workspace_for(1, Nl, Kl, device)))
            tot_bytes += w4a16_bytes(1, Nl, Kl)

    def token(i):
        for (xl, ql, sl, ml, yl, wsl) in stack:
            w4.w4a16_matmul(xl, ql, sl, ml, y=yl, workspace=wsl)

    us_tok = graph_time_us(token, 1, 50, stream)
    rows["qwen_stack"] = {"matmuls": len(stack), "us_per_token": round(us_tok, 2),
                          "bytes": tot_bytes, "roofline_us": round(tot_bytes / hbm / 1e3, 2),
                          "frac": round(tot_bytes / hbm / 1e3 / us_tok, 3),
                          "note": "weights (698 MB) > L2; one graph of 196 launches per token",
                          "pages": "3.68 ms for 197 matmuls (tinygemm, RTX 4060 Laptop)"}

    # The same weights with the projections that share an input concatenated along N (q, k, v
    # and gate, up: the quantization is per output column, so the fused matmul computes the
    # same numbers): 4 launches per layer instead of 7.
    per = len(workloads.QWEN_STACK["block"])
    fused = []
    for layer in range(workloads.QWEN_STACK["layers"]):
        blk = stack[layer * per:(layer + 1) * per]
        for group in ((0, 1, 2), (3,), (4, 5), (6,)):
            parts = [blk[j] for j in group]
            ql = torch.cat([p[1] for p in parts], dim=1).contiguous()
            sl = torch.cat([p[2] for p in parts], dim=1).contiguous()
            ml = torch.cat([p[3] for p in parts], dim=1).contiguous()
            Kl, Nl = ql.shape[0] * 8, ql.shape[1]
            yl = torch.empty(1, Nl, dtype=torch.bfloat16, device=device)
            fused.append((parts[0][0], ql, sl, ml, yl, workspace_for(1, Nl, Kl, device)))
    del stack

    def token_fused(i):
        for (xl, ql, sl, ml, yl, wsl) in fused:
            w4.w4a16_matmul(xl, ql, sl, ml, y=yl, workspace=wsl)

    us_f = graph_time_us(token_fused, 1, 50, stream)
    rows["qwen_stack_fused_qkv_gateup"] = {
        "matmuls": len(fused), "us_per_token": round(us_f, 2), "bytes": tot_bytes,
        "roofline_us": round(tot_bytes / hbm / 1e3, 2),
        "frac": round(tot_bytes / hbm / 1e3 / us_f, 3),
        "note": "same weights, q/k/v and gate/up concatenated along N: 112 launches per token"}
    del fused
    return rows


# --------------------------------------------------------------------------- #
# CPU oracle (baseline and reference arm)
# --------------------------------------------------------------------------- #

def oracle_inputs():
    import oracle

    cfg = workloads.LLAMA_UP
    w = workloads.weights(cfg["N"], cfg["K"], seed=0).numpy()
    codes, s, m = oracle.w4a16_quantize(w)
    qw = oracle.w4a16_pack(codes)
    x = workloads.bits16(workloads.activations_bf16(1, cfg["K"], seed=0))
    return x, qw, s, m


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_matmul_threads(x, qw, s, m, cols, threads: int):
    """The unchanged oracle over disjoint slices of the output columns, one host thread per
    slice (the oracle is C behind ctypes, which releases the GIL during the call)."""
    import concurrent.futures as cf

    import numpy as np

    import oracle

    cols = np.asarray(cols, dtype=np.int32)
    parts = [p for p in np.array_split(cols, threads) if len(p)]
    with cf.ThreadPoolExecutor(max_workers=len(parts)) as ex:
        list(ex.map(lambda p: oracle.w4a16_matmul(x, qw, s, m, cols=p), parts))
    return len(parts)


def cpu_baseline(seconds: float):
    """The oracle as it stands (scalar C, fp64 sums) on the full M=1 workload, its output
    columns split over every host core, repeated until at least `seconds` have passed."""
    x, qw, s, m = oracle_inputs()
    N, K = qw.shape[1], qw.shape[0] * 8
    cores = host_cores()
    cols = list(range(N))
    reps, t0 = 0, time.perf_counter()
    used = cores
    while True:
        used = oracle_matmul_threads(x, qw, s, m, cols, cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": round(weight_bytes(N, K) * reps / el / 1e9, 3), "unit": "GB/s",
            "cores": used, "kind": "oracle",
            "sample": f"full M=1 workload (all {N} columns, K={K}) x {reps} repetitions, "
                      f"{el:.1f} s, columns split over {used} host threads"}


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm, on bounded samples of the same workload, its
    output columns split over every host core."""
    if rank != 0:
        return None
    import oracle

    x, qw, s, m = oracle_inputs()
    N, K = qw.shape[1], qw.shape[0] * 8
    cores = host_cores()
    t0 = time.perf_counter()
    oracle.w4a16_matmul(x, qw, s, m, cols=list(range(0, N, 64)))
    t_col = (time.perf_counter() - t0) / len(range(0, N, 64))
    budget = 90.0  # seconds for warmup + timed steps together
    per_step = budget / max(1, args.steps + args.warmup)
    ncols = int(max(8 * cores, min(N, per_step * cores / max(t_col, 1e-9))))
    ncols = min(N, ncols)
    cols = list(range(0, N, max(1, N // ncols)))[:ncols]
    used = cores
    for _ in range(args.warmup):
        oracle_matmul_threads(x, qw, s, m, cols, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        used = oracle_matmul_threads(x, qw, s, m, cols, cores)
    el = time.perf_counter() - t0
    bytes_step = weight_bytes(N, K) * len(cols) / N
    value = bytes_step * args.steps / el / 1e9
    sample = (f"{len(cols)} of {N} output columns (all K={K}) per step, split over {used} "
              "host threads")
    cfg = workloads.LLAMA_UP
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg["name"], "M": 1, "N": N, "K": K, "group": 128},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": used,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


PROFILE_CASES = ("gemv_m1", "gemv_m8", "skinny_m16", "skinny_m32", "tc_m16", "tc_m64",
                 "tc_m4096", "q4b32_gemv", "quantize", "pack", "w8a16_gemv", "zp_m1",
                 "nvfp4_gemv", "nvfp4_gemv_plain", "mxfp4_gemv", "prep_m64", "prep_m128",
                 "tc_m128", "prepare", "qwen_layer", "nvfp4_mm32")


def profile_case(args):
    """A few launches of one workload, untimed, for a profiler (ncu -k ... -c ...): the
    Llama-3-8B up-projection (14336 x 4096) at M = 1, 8, 16 or 32 (skinny kernel), 16
    (tensor-core kernel) or 4096 with 6 rotating weight copies (174 MB > L2), the Q4
    block-32 GEMV (16384 x 16384), quantize / pack, the W8A16, NVFP4 or MXFP4 GEMV or the zero-point
    matmul at M = 1 on the same layer."""
    import gemv_w4a16_group_gb300 as w4

    device = torch.device("cuda:0")
    torch.cuda.set_device(device)
    case, n = args.case, args.launches
    if case in ("w8a16_gemv", "zp_m1", "nvfp4_gemv", "nvfp4_gemv_plain", "mxfp4_gemv"):
        N, K = workloads.LLAMA_UP["N"], workloads.LLAMA_UP["K"]
        w = workloads.weights(N, K, seed=0).to(device)
        x = workloads.activations_bf16(1, K, seed=1).to(device)
        if case == "nvfp4_gemv_plain":  # the plain-load kernel, not the ring the shape picks
            w4.testing_set_fp4_variant(0)
        if case in ("nvfp4_gemv", "nvfp4_gemv_plain"):
            c4, s4, S4 = w4.nvfp4_quantize(w)
            del w
            cps = [(c4.clone(), s4.clone(), S4.clone()) for _ in range(6)]
            for i in range(n):
                w4.nvfp4_gemv(x[0], *cps[i % 6])
        elif case == "mxfp4_gemv":
            cm, sm_ = w4.mxfp4_quantize(w)
            del w
            cps = [(cm.clone(), sm_.clone()) for _ in range(6)]
            for i in range(n):
                w4.mxfp4_gemv(x[0], *cps[i % 6])
        elif case == "w8a16_gemv":
            q8, s8 = w4.w8a16_quantize(w)
            del w
            cps = [(q8.clone(), s8.clone()) for _ in range(4)]
            for i in range(n):
                w4.w8a16_gemv(x[0], *cps[i % 4])
        else:
            qk, sk, zk = w4.w4a16zp_prepare(*w4.w4a16zp_quantize(w))
            del w
            cps = [(qk.clone(), sk.clone(), zk.clone()) for _ in range(6)]
            for i in range(n):
                w4.w4a16zp_matmul(x, *cps[i % 6])
    elif case == "nvfp4_mm32":
        # the NVFP4 matmul at M = 32 on the up-projection (one pass of 32 rows)
        N, K = workloads.LLAMA_UP["N"], workloads.LLAMA_UP["K"]
        w = workloads.weights(N, K, seed=0).to(device)
        c4, s4, S4 = w4.nvfp4_quantize(w)
        del w
        cps = [(c4.clone(), s4.clone(), S4.clone()) for _ in range(6)]
        x = workloads.activations_bf16(32, K, seed=32).to(device)
        y = torch.empty(32, N, dtype=torch.bfloat16, device=device)
        ws = torch.empty(w4.fp4_matmul_workspace_bytes(32, K), dtype=torch.uint8, device=device)
        for i in range(n):
            w4.nvfp4_matmul(x, *cps[i % 6], y=y, workspace=ws)
    elif case == "qwen_layer":
        # one Qwen2.5-1.5B-shaped layer (7 matmuls, each with its own weights and x, the
        # workspace the library asks for), the layer repeated n times
        layer = []
        for name, Nl, Kl in workloads.QWEN_STACK["block"]:
            g = torch.Generator(device=device)
            g.manual_seed(len(layer))
            wl = torch.randn(Nl, Kl, generator=g, device=device) * workloads.WEIGHT_STD
            cl, sl, ml = w4.w4a16_quantize(wl)
            ql = w4.w4a16_pack(cl)
            xl = torch.randn(1, Kl, generator=g, device=device).to(torch.bfloat16)
            yl = torch.empty(1, Nl, dtype=torch.bfloat16, device=device)
            layer.append((xl, ql, sl, ml, yl, workspace_for(1, Nl, Kl, device)))
        for _ in range(n):
            for (xl, ql, sl, ml, yl, wsl) in layer:
                w4.w4a16_matmul(xl, ql, sl, ml, y=yl, workspace=wsl)
    elif case in ("prep_m64", "prep_m128", "prepare"):
        N, K = workloads.LLAMA_UP["N"], workloads.LLAMA_UP["K"]
        w, codes, qw, s, m = quantized_on_device(N, K, 0, device)
        del w, codes
        if case == "prepare":
            prep = w4.w4a16_prepare(qw, s, m)
            for _ in range(n):
                w4.w4a16_prepare(qw, s, m, prepared=prep)
        else:
            M = 64 if case == "prep_m64" else 128
            cps = [(qw.clone(), s.clone(), m.clone()) for _ in range(6)]
            preps = [w4.w4a16_prepare(*c) for c in cps]
            x = workloads.activations_bf16(M, K, seed=M).to(device)
            y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
            ws = prepared_workspace_for(M, N, K, device)
            for i in range(n):
                w4.w4a16_matmul_prepared(x, *cps[i % 6], preps[i % 6], y=y, workspace=ws)
    elif case in ("gemv_m1", "gemv_m8", "skinny_m16", "skinny_m32", "tc_m16", "tc_m64",
                  "tc_m128", "tc_m4096", "quantize", "pack"):
        N, K = workloads.LLAMA_UP["N"], workloads.LLAMA_UP["K"]
        w, codes, qw, s, m = quantized_on_device(N, K, 0, device)
        if case == "quantize":
            for _ in range(n):
                w4.w4a16_quantize(w, codes=codes, scales=s, mins=m)
        elif case == "pack":
            for _ in range(n):
                w4.w4a16_pack(codes, qw=qw)
        else:
            del w, codes
            M = {"gemv_m1": 1, "gemv_m8": 8, "skinny_m16": 16, "skinny_m32": 32, "tc_m16": 16,
                 "tc_m64": 64, "tc_m128": 128, "tc_m4096": 4096}[case]
            if case.startswith("tc_"):  # the tensor-core kernel whatever the size picks
                w4.testing_force_kernel(2)
            cps = [(qw.clone(), s.clone(), m.clone()) for _ in range(6)]
            x = workloads.activations_bf16(M, K, seed=M).to(device)
            y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
            ws = workspace_for(M, N, K, device)
            for i in range(n):
                w4.w4a16_matmul(x, *cps[i % 6], y=y, workspace=ws)
    else:
        N = K = workloads.Q4_SQUARE["N"]
        w = workloads.weights(N, K, seed=0).to(device)
        qc, qsc = w4.q4b32_quantize(w)
        del w
        x = workloads.activations_fp16(K, seed=0).to(device)
        cps = [(qc.clone(), qsc.clone()) for _ in range(2)] + [(qc, qsc)]
        for i in range(n):
            w4.q4b32_gemv(x, *cps[i % 3])
    torch.cuda.synchronize()
    status = w4.w4a16_device_status()
    return {"case": case, "launches": n, "device_status": status}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=96000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-rows", action="store_true", help="headline line only")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--case", choices=PROFILE_CASES, default=None,
                    help="run a few untimed launches of one workload (for ncu) and exit")
    ap.add_argument("--launches", type=int, default=6, help="launches for --case")
    args = ap.parse_args(argv)
    if args.case is not None:
        print(json.dumps(profile_case(args)), flush=True)
        return
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    world, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
