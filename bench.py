#!/usr/bin/env python3
"""Benchmark of the Q8_0 linear layer on GB300 (one JSON line on stdout, from rank 0).

Headline workload: the decode GEMV of a dense ~9B-class FFN up-projection, M = 1 token,
K = 4096, N = 12288, Q8_0 weights, bf16 activations.  One step = one q8_linear call (fused
activation quantization, int8 block dots, binary32 rescale, y store).  Metric: HBM GB/s
of the algorithmic bytes (weight codes + binary16 scales + activations + y) per second.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Timing: W warm-up steps, then exactly K steps, bracketed by a barrier and
torch.cuda.synchronize(); CUDA events on the launching stream; steps run as replays of a
CUDA graph that holds one step per weight copy; the weights rotate over enough copies to
exceed twice the L2 size, so every step reads its weights from HBM.  SM clocks are sampled
with nvidia-smi during the timed region.

--impl reference times the CPU oracle (oracle/, the plain C definition of the layer) on the
host cores, on the same workload and metric, each step a bounded sample of the rows.
Under torchrun (N > 1) each rank runs an independent replica on its own GPU (the layer's
batch is independent per replica: weak scaling); rank 0 prints the aggregate.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "Q8_0 GEMM int8 TOPS (prefill) & GEMV HBM GB/s (decode), % of roofline"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------------- #
# distributed plumbing (replicas)                                                      #
# ----------------------------------------------------------------------------------- #

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value: float) -> float:
    """Largest value over all ranks (timings: the slowest replica decides)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------------- #
# peaks, clocks, profile-derived traffic                                              #
# ----------------------------------------------------------------------------------- #

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while it runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="q8clk_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def kernel_source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "q8_int8_block_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary_md, sources):
    """DRAM bytes per launch recorded by an ncu capture, if that capture was taken on the
    current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", summary_md)
    try:
        txt = open(path).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", txt)
    m_b = re.search(r"dram_bytes_per_launch_full_size:\s*([0-9.eE+]+)", txt)
    if not m_sha or not m_b or m_sha.group(1) != kernel_source_sha(sources):
        return None
    return float(m_b.group(1))


# ----------------------------------------------------------------------------------- #
# GPU arm                                                                              #
# ----------------------------------------------------------------------------------- #

def l2_bytes(torch):
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 129 * 1024 * 1024


def time_graph_steps(torch, step_fns, steps, warmup):
    """Captures one CUDA graph holding len(step_fns) steps, runs `warmup` steps, then times
    exactly `steps` steps (whole replays, plus a prefix replay of a partial graph).
    Returns (total seconds, seconds per step) measured with CUDA events."""
    R = len(step_fns)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for f in step_fns:  # eager once (allocations, attributes) before capture
            f()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    full = torch.cuda.CUDAGraph()
    with torch.cuda.graph(full):
        for f in step_fns:
            f()
    rem = steps % R
    part = None
    if rem:
        part = torch.cuda.CUDAGraph()
        with torch.cuda.graph(part):
            for f in step_fns[:rem]:
                f()
    for _ in range((warmup + R - 1) // R):
        full.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(steps // R):
        full.replay()
    if part is not None:
        part.replay()
    ev1.record()
    torch.cuda.synchronize()
    barrier()
    total = ev0.elapsed_time(ev1) / 1e3
    return total, total / steps


def gpu_arm(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist_init("nccl")
    import __graft_entry__ as g
    g.build()
    import q8_int8_block_gb300 as q8

    pk, pk_src = peaks()
    dev = torch.device("cuda", local)
    wl = workloads.WORKLOADS["decode"]
    pr = wl.projections[0]
    M, K, N = 1, pr.K, pr.N
    W = wl.make_weights(0)
    x_np, _ = wl.make_act(0, 0)  # M = 1
    Wq0, Wd0 = q8.q8_quantize_weights(torch.from_numpy(W).to(dev))
    wbytes = N * K + 2 * N * (K // 32)
    copies = max(2, -(-(2 * l2_bytes(torch) + wbytes) // wbytes))
    Wqs = [Wq0] + [Wq0.clone() for _ in range(copies - 1)]
    Wds = [Wd0] + [Wd0.clone() for _ in range(copies - 1)]
    x = torch.from_numpy(x_np.view(np.int16).copy()).to(dev).view(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    fns = [lambda i=i: q8.q8_linear(x, Wqs[i], Wds[i], y=y) for i in range(copies)]
    bytes_step = workloads.algorithmic_bytes(M, N, K)

    with ClockSampler(local) as clk:
        total, per_step = time_graph_steps(torch, fns, args.steps, args.warmup)
    clocks = clk.summary()
    t_max = max_over_ranks(total)
    value = sum_over_ranks(bytes_step * args.steps) / t_max / 1e9
    achieved = bytes_step / per_step / 1e9
    traffic = profiled_traffic("decode_kernel_m1_k4096_n12288.md", ["q8_decode.cu", "q8_ptx.cuh",
                                                                     "q8_quant_dev.cuh"])

    # end to end through the public API: H2D of x from pinned memory, the call, D2H of y
    e2e_steps = min(args.steps, 2000)
    xh = torch.from_numpy(x_np.view(np.int16).copy()).pin_memory()
    yh = torch.empty((M, N), dtype=torch.float32).pin_memory()
    xd = torch.empty((M, K), dtype=torch.int16, device=dev)
    for i in range(max(3, args.warmup // 100)):
        xd.copy_(xh, non_blocking=True)
        q8.q8_linear(xd.view(torch.bfloat16), Wqs[i % copies], Wds[i % copies], y=y)
        yh.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host = time.perf_counter()
    e0.record()
    for i in range(e2e_steps):
        xd.copy_(xh, non_blocking=True)
        q8.q8_linear(xd.view(torch.bfloat16), Wqs[i % copies], Wds[i % copies], y=y)
        yh.copy_(y, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    t_host = time.perf_counter() - t_host
    barrier()
    e2e_t = max_over_ranks(max(e0.elapsed_time(e1) / 1e3, t_host))
    e2e_value = sum_over_ranks(bytes_step * e2e_steps) / e2e_t / 1e9

    extra = {}
    if not args.no_extra:
        extra = extra_measurements(torch, q8, dev, pk, args)

    err = q8.q8_device_error()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_max / args.steps * 1e3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded N(0,0.02) weights quantized to Q8_0, N(0,1) bf16 activations)",
        "config": {"workload": "decode GEMV, FFN up-projection of a dense ~9B-class layer",
                   "M": M, "K": K, "N": N, "weights": "Q8_0 (int8 codes + binary16 scale per 32)",
                   "activations": "bf16, quantized per call inside the kernel",
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {copies} rotating weight copies "
                         f"({copies * wbytes / 1e6:.0f} MB > 2 x L2)",
                   "timing": "CUDA graph replays, CUDA events"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                     "traffic": traffic, "kernel": "q8::decode_kernel<1,false,true>",
                     "algorithmic_bytes_per_launch": bytes_step,
                     "peak_source": f"hbm_gbs of {pk_src} peaks"},
        "clocks": clocks,
        "e2e": {"value": round(e2e_value, 3), "unit": "GB/s",
                "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 4,
                "steps": e2e_steps, "api": "q8_int8_block_gb300.q8_linear (C ABI q8_linear)"},
        "gpu_launches": args.steps,
        "device_error_word": err,
    }
    if extra:
        line["extra"] = extra
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(Wq0, Wd0, x_np, M, N, K, args.cpu_seconds)
    return rank, line


def extra_measurements(torch, q8, dev, pk, args):
    """Secondary lines: batched decode and the prefill GEMM (not part of the headline)."""
    out = {}
    # batched decode, same weights, M = 4, 16, 64
    wl = workloads.WORKLOADS["decode"]
    pr = wl.projections[0]
    W = wl.make_weights(0)
    Wq, Wd = q8.q8_quantize_weights(torch.from_numpy(W).to(dev))
    K, N = pr.K, pr.N
    wbytes = N * K + 2 * N * (K // 32)
    copies = max(2, -(-(2 * l2_bytes(torch) + wbytes) // wbytes))
    Wqs = [Wq] + [Wq.clone() for _ in range(copies - 1)]
    Wds = [Wd] + [Wd.clone() for _ in range(copies - 1)]
    for mi, M in enumerate(wl.Ms):
        if M == 1:
            continue
        x_np, _ = wl.make_act(0, mi)
        x = torch.from_numpy(x_np.view(np.int16).copy()).to(dev).view(torch.bfloat16)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        fns = [lambda i=i: q8.q8_linear(x, Wqs[i], Wds[i], y=y) for i in range(copies)]
        steps = 2000
        _, per = time_graph_steps(torch, fns, steps, 60)
        b = workloads.algorithmic_bytes(M, N, K)
        ops = workloads.algorithmic_ops(M, N, K)
        out[f"decode_M{M}"] = {"GB/s": round(b / per / 1e9, 2), "TOPS": round(ops / per / 1e12, 3),
                               "us_per_step": round(per * 1e6, 3),
                               "hbm_frac": round(b / per / 1e9 / pk["hbm_gbs"], 4)}
    del Wqs, Wds
    # prefill: 9B-class up and down projections, M = 2048
    wl = workloads.WORKLOADS["prefill9b"]
    for p, pr in enumerate(wl.projections):
        W = wl.make_weights(p)
        Wq, Wd = q8.q8_quantize_weights(torch.from_numpy(W).to(dev))
        x_np, _ = wl.make_act(p, 0)
        M = x_np.shape[0]
        x = torch.from_numpy(x_np.view(np.int16).copy()).to(dev).view(torch.bfloat16)
        y = torch.empty((M, pr.N), dtype=torch.float32, device=dev)
        fns = [lambda: q8.q8_linear(x, Wq, Wd, y=y)]
        steps = 50
        _, per = time_graph_steps(torch, fns, steps, 5)
        ops = workloads.algorithmic_ops(M, pr.N, pr.K)
        tops = ops / per / 1e12
        out[f"prefill9b_{pr.name}_M{M}"] = {
            "TOPS": round(tops, 2), "us_per_step": round(per * 1e6, 2),
            "K": pr.K, "N": pr.N,
            "tensor_frac_of_f16_peak": round(tops / pk["bf16_tflops"], 4),
            "note": "int8-equivalent ops 2MNK on the kind::f16 pipe (binary16 codes); peak = "
                    "dense bf16/f16 burst rate; per step = activation quantize + weight code "
                    "widening + GEMM"}
    return out


# ----------------------------------------------------------------------------------- #
# CPU baseline and the reference arm (the oracle, as it stands)                        #
# ----------------------------------------------------------------------------------- #

def _oracle_cores():
    return os.cpu_count() or 1


def cpu_baseline(Wq_t, Wd_t, x_np, M, N, K, seconds):
    from oracle import oracle as O
    Wq = Wq_t.cpu().numpy()
    Wd = Wd_t.cpu().numpy().view(np.uint16)
    cores = _oracle_cores()
    O.linear(x_np, Wq, Wd, bf16=True, nthreads=cores)  # warm
    passes, t0 = 0, time.perf_counter()
    while True:
        O.linear(x_np, Wq, Wd, bf16=True, nthreads=cores)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= seconds or passes >= 100000:
            break
    b = workloads.algorithmic_bytes(M, N, K) * passes
    return {"value": round(b / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{passes} full passes of the M={M} K={K} N={N} layer (activation "
                      f"quantization + all {N} outputs) in {dt:.1f} s"}


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0, None  # the oracle is timed once, on rank 0
    from oracle import oracle as O
    wl = workloads.WORKLOADS["decode"]
    pr = wl.projections[0]
    M, K, N = 1, pr.K, pr.N
    W = wl.make_weights(0)
    x_np, _ = wl.make_act(0, 0)
    Wq, Wd = O.quantize_weights(W)
    cores = _oracle_cores()
    t0 = time.perf_counter()
    O.linear(x_np, Wq, Wd, bf16=True, nthreads=cores)
    t_full = time.perf_counter() - t0
    # each step: the layer on a contiguous slice of output rows, sized so that all steps
    # fit in about a minute
    budget = 60.0
    rows = int(max(64, min(N, N * budget / max(1, args.steps + args.warmup) / max(t_full, 1e-6))))
    starts = [(i * rows) % (N - rows + 1) for i in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        s = starts[i]
        O.linear(x_np, Wq[s:s + rows], Wd[s:s + rows], bf16=True, nthreads=cores)
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        s = starts[i]
        O.linear(x_np, Wq[s:s + rows], Wd[s:s + rows], bf16=True, nthreads=cores)
    dt = time.perf_counter() - t0
    b = workloads.algorithmic_bytes(M, rows, K) * args.steps
    value = b / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded N(0,0.02) weights quantized to Q8_0, N(0,1) bf16 activations)",
        "config": {"workload": "decode GEMV, FFN up-projection of a dense ~9B-class layer",
                   "M": M, "K": K, "N": N, "parallelism": "CPU oracle, rank 0 only"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {rows} of {N} output rows (activation quantization + "
                                   f"those rows), rotating over the matrix"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return rank, line


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1:
        ap.error("--steps must be >= 1")
    return a


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        rank, line = reference_arm(args)
    else:
        rank, line = gpu_arm(args)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    try:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass


if __name__ == "__main__":
    main()
