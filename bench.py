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
        out = {k: float(p[k]) for k in FALLBACK}
        if "sm_max_mhz" in p:
            out["sm_max_mhz"] = float(p["sm_max_mhz"])
        return out, "measured"
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


def recorded_traffic(name):
    """DRAM bytes per launch from the committed ncu capture record of workload `name`
    (profiles/traffic.json), if that capture was taken on the current kernel sources (else
    None: the kernel has changed since the counters were taken)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)["records"][name]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_sha256_16") != kernel_source_sha(rec["sources"]):
        return None
    return float(rec["dram_bytes_per_launch"])


def measured_rates():
    """Per-SM unit rates measured by bench_rates.py on this GPU type (committed record), or
    None."""
    try:
        with open(os.path.join(ROOT, "profiles", "rates_gb300.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def unit_peak(torch, pk, key, ops_per_unit, fallback):
    """Peak in T-ops/s of a unit rate (per clock per SM) x ops per unit x SMs x maximum SM
    clock; the rate from the measured record, else `fallback`.  Returns (peak, source)."""
    rec = measured_rates()
    rate, src = fallback, "assumed rate"
    if rec and key in rec.get("rates", {}):
        rate, src = rec["rates"][key], "bench_rates.py record"
    sms = sm_count(torch)
    return rate * ops_per_unit * sms * pk.get("sm_max_mhz", 2070.0) * 1e6 / 1e12, (
        f"{rate} {key} ({src}) x {ops_per_unit} ops x {sms} SMs x maximum SM clock")


def sm_count(torch):
    return int(torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count)


# ----------------------------------------------------------------------------------- #
# GPU arm                                                                              #
# ----------------------------------------------------------------------------------- #

def l2_bytes(torch):
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 129 * 1024 * 1024


# Named workloads: (workload, projection index, M index) of workloads.WORKLOADS.
CASES = {
    "decode_m1": ("decode", 0, 0), "decode_m4": ("decode", 0, 1), "decode_m16": ("decode", 0, 2),
    "decode_m64": ("decode", 0, 3), "tiny": ("tiny", 0, 0),
    "prefill9b_up": ("prefill9b", 0, 0), "prefill9b_down": ("prefill9b", 1, 0),
    "prefill27b_up": ("prefill27b", 0, 0), "prefill27b_down": ("prefill27b", 1, 0),
    "gate_m128": ("sweep", 4, 3), "gate_m512": ("sweep", 4, 4),
}
_WEIGHTS = {}


def quantized_weights(torch, q8, dev, wname, p):
    """Q8_0 weights (codes, binary16 scales) of projection p of a workload, quantized by the
    library on the device; the most recent shapes are kept so that cases sharing a projection
    draw and quantize it once."""
    key = (wname, p)
    if key not in _WEIGHTS:
        if len(_WEIGHTS) >= 4:
            _WEIGHTS.pop(next(iter(_WEIGHTS)))
        W = workloads.WORKLOADS[wname].make_weights(p)
        _WEIGHTS[key] = q8.q8_quantize_weights(torch.from_numpy(W).to(dev))
        del W
    return _WEIGHTS[key]


def time_graph_steps(torch, q8, step_fns, steps, warmup, instrument=True):
    """Runs `warmup` untimed steps, then times exactly `steps` steps, all as replays of CUDA
    graphs that rotate over step_fns (one step per weight copy).  Up to 48 steps the timed
    region is one replay of a graph holding exactly `steps` steps; longer runs replay a graph
    of whole rotations (at least 48 steps) and then one holding the remainder.  Every graph
    the timed region replays has been replayed during the warm-up (a graph's first launch
    also uploads it).  Returns (seconds for the timed steps, mean seconds of the main kernel),
    all from CUDA events on the launching stream.  With `instrument`, the library records
    event nodes around each step's main kernel and the mean is over the launches of one
    graph; without it (one kernel per step, consecutive launches overlapping through
    programmatic dependent launch, which event nodes between them would serialize), the main
    kernel's time per launch is the timed region's time per step."""
    if steps <= 48:
        R = steps
    else:
        R = len(step_fns) * max(1, -(-48 // len(step_fns)))
    fns = [step_fns[i % len(step_fns)] for i in range(R)]
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(R)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(R)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for f in step_fns:  # eager once (attributes, workspace)
            f()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    if instrument:
        q8.q8_set_timing_events(starts, stops)
    try:
        full = torch.cuda.CUDAGraph()
        with torch.cuda.graph(full):
            for f in fns:
                f()
        rem = steps % R
        part = None
        if rem:
            if instrument:
                q8.q8_set_timing_events(starts, stops)
            part = torch.cuda.CUDAGraph()
            with torch.cuda.graph(part):
                for f in fns[:rem]:
                    f()
    finally:
        q8.q8_set_timing_events()
    for _ in range(max(1, -(-warmup // R))):
        full.replay()
    if part is not None:
        part.replay()
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
    if instrument:
        n = rem if part is not None else R
        kern = statistics.mean(a.elapsed_time(b) for a, b in zip(starts[:n], stops[:n])) / 1e3
    else:
        kern = total / steps
    return total, kern


def run_case(torch, q8, dev, name, steps, warmup, pk, pk_src, clocks=False, e2e=False, spec=None,
             force_path=None, gated=None, norm=False, prepared=False):
    """gated: None (the plain layer, float32 y), "fused" (q8_linear_fused: y = silu(gate) *
    x.W^T stored as bfloat16 by the GEMM's own epilogue) or "unfused" (the plain layer, then
    torch's silu, multiply and bfloat16 cast as separate kernels).  norm (with "fused"): x is
    the un-normalised hidden state and its RMSNorm runs inside the layer's quantizer.
    prepared: the tensor-core path on weights widened once (q8_linear_prepared)."""
    wname, p, mi = spec if spec is not None else CASES[name]
    wl = workloads.WORKLOADS[wname]
    Wq0, Wd0 = quantized_weights(torch, q8, dev, wname, p)
    x_np, _ = wl.make_act(p, mi)
    M, K = x_np.shape
    N = Wq0.shape[0]
    wbytes = N * K + 2 * N * (K // 32)
    copies = max(2, -(-(2 * l2_bytes(torch)) // wbytes))
    Wqs = [Wq0] + [Wq0.clone() for _ in range(copies - 1)]
    Wds = [Wd0] + [Wd0.clone() for _ in range(copies - 1)]
    xdt = torch.bfloat16 if wl.bf16 else torch.float32
    xsize = 2 if wl.bf16 else 4
    if wl.bf16:
        x = torch.from_numpy(x_np.view(np.int16).copy()).to(dev).view(torch.bfloat16)
    else:
        x = torch.from_numpy(x_np).to(dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    wsz = (q8.q8_linear_prepared_workspace_size(M, N, K) if prepared
           else q8.q8_linear_workspace_size(M, N, K, force_path or "auto"))
    ws = torch.empty(max(wsz, 1), dtype=torch.uint8, device=dev) if wsz else None
    if prepared:
        path = "tensor"
    elif force_path:
        path = force_path
    else:
        wsz_batch = q8.q8_linear_workspace_size(M, N, K, "batch") if M <= 64 else 0
        path = "decode" if wsz == 0 else ("batch" if wsz == wsz_batch else "tensor")
    if prepared:
        B16s = [q8.q8_weights_to_f16(w) for w in Wqs]
        fns = [lambda i=i: q8.q8_linear_prepared(x, B16s[i], Wds[i], y=y, workspace=ws)
               for i in range(copies)]
    elif gated is None:
        fns = [lambda i=i: q8.q8_linear_ex(x, Wqs[i], Wds[i], y=y, path=path, workspace=ws)
               for i in range(copies)]
    else:
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        gate = torch.randn((M, N), device=dev, generator=gen) * 2.5
        yb = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        if gated == "fused":
            nw = torch.rand(K, device=dev, generator=gen) + 0.5 if norm else None
            fns = [lambda i=i: q8.q8_linear_fused(x, Wqs[i], Wds[i], epi="silu_mul", aux=gate, y=yb,
                                                  out_dtype=torch.bfloat16, path=path, workspace=ws,
                                                  norm_weight=nw, norm_eps=1e-6)
                   for i in range(copies)]
        else:
            def unfused(i):
                q8.q8_linear_ex(x, Wqs[i], Wds[i], y=y, path=path, workspace=ws)
                yb.copy_(torch.nn.functional.silu(gate).mul_(y))
            fns = [lambda i=i: unfused(i) for i in range(copies)]
    bytes_step = workloads.algorithmic_bytes(M, N, K, x_bytes=xsize)
    if gated is not None:  # the gate is read (4 bytes), y is stored as bfloat16 (2, not 4)
        bytes_step += M * N * 2
    ops_step = workloads.algorithmic_ops(M, N, K)
    t_hbm = bytes_step / (pk["hbm_gbs"] * 1e9)
    t_tc = ops_step / (pk["bf16_tflops"] * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    # the tensor path's steps hold three kernels: time the GEMM itself with event nodes; the
    # streaming paths (one kernel, or the activation quantizer chained by programmatic
    # dependent launch to the batched kernel) are timed per step
    inst = path in ("tensor", "dp4a") or gated == "unfused"
    if clocks:
        with ClockSampler(torch.cuda.current_device()) as clk:
            total, kern = time_graph_steps(torch, q8, fns, steps, warmup, instrument=inst)
        clk_summary = clk.summary()
    else:
        total, kern = time_graph_steps(torch, q8, fns, steps, warmup, instrument=inst)
        clk_summary = None
    t_max = max_over_ranks(total)
    if bound == "hbm":
        unit = "GB/s"
        value = sum_over_ranks(bytes_step * steps) / t_max / 1e9
        roof = {"bound": "hbm", "achieved": round(bytes_step / kern / 1e9, 2), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(bytes_step / kern / 1e9 / pk["hbm_gbs"], 4),
                "algorithmic_bytes_per_launch": bytes_step,
                "peak_source": f"hbm_gbs of the {pk_src} peaks"}
    else:
        unit = "TOPS"
        value = sum_over_ranks(ops_step * steps) / t_max / 1e12
        roof = {"bound": "tensor", "achieved": round(ops_step / kern / 1e12, 2),
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(ops_step / kern / 1e12 / pk["bf16_tflops"], 4),
                "algorithmic_flops_per_launch": ops_step,
                "peak_source": f"bf16_tflops (burst) of the {pk_src} peaks: the kernel runs on "
                               "the dense kind::f16 tensor pipe (int8 codes as binary16)"}
    if path == "dp4a":
        # CUDA-core integer path: peak from unit counts, 64 dp4a per clock per SM (measured),
        # 4 int8 MACs each, at the maximum SM clock
        dp4a_peak, dp4a_src = unit_peak(torch, pk, "dp4a_per_clk_sm", 8, 64.0)
        roof = {"bound": "alu", "achieved": round(ops_step / kern / 1e12, 2),
                "peak": round(dp4a_peak, 1), "unit": "TOPS",
                "frac": round(ops_step / kern / 1e12 / dp4a_peak, 4),
                "algorithmic_flops_per_launch": ops_step,
                "peak_source": "dp4a: " + dp4a_src}
    if path == "tensor":
        # the GPU's int8 tensor path (mma.sync s8, what an int8 GEMM runs on here), for reference
        i8, i8_src = unit_peak(torch, pk, "imma_mac_per_clk_sm", 2, 252.0)
        roof["int8_mma_sync_peak_tops"] = round(i8, 1)
        roof["int8_equivalent_tops"] = round(ops_step / kern / 1e12, 2)
        roof["frac_of_int8_mma_sync_peak"] = round(ops_step / kern / 1e12 / i8, 3)
    roof["kernel"] = {"decode": "q8::decode_kernel", "batch": "q8::batch_kernel",
                      "dp4a": "q8::dp4a_gemm_kernel"}.get(path, "q8::gemm_tc_kernel")
    roof["kernel_us"] = round(kern * 1e6, 3)
    roof["kernel_time"] = ("time per step of the timed region (one kernel per step; "
                           "consecutive launches overlap by programmatic dependent launch)"
                           if path == "decode" else
                           "time per step of the timed region (activation quantizer + batched "
                           "kernel, chained by programmatic dependent launch)"
                           if path == "batch" else "mean of event-node pairs around the GEMM launches")
    # the committed captures are of the library's own choice of kernel on the plain layer
    roof["traffic"] = (recorded_traffic(name) if force_path is None and gated is None and not prepared
                       else None)
    out = {"name": name, "M": M, "K": K, "N": N, "path": path, "unit": unit, "value": value,
           "steps": steps,
           "t_max": t_max, "roofline": roof, "copies": copies, "wbytes": wbytes,
           "launches_per_step": {"decode": 1, "batch": 2, "dp4a": 2}.get(path, 3), "clocks": clk_summary,
           "bytes_step": bytes_step, "xsize": xsize, "bf16": wl.bf16}
    if e2e:
        out["e2e"] = e2e_measure(torch, q8, dev, x_np, wl.bf16, Wqs, Wds, M, N, K, steps, warmup,
                                 bytes_step, ops_step, bound, path=force_path)
        out["Wq0"], out["Wd0"], out["x_np"] = Wq0, Wd0, x_np
    return out


def run_kv3(torch, q8, dev, steps, warmup, pk, pk_src):
    """The 3-bit KV-cache codec on one attention layer's keys at a 256K-token context
    (262144 tokens x 4 heads x 256 channels, bf16): encode and decode, each timed alone.
    Algorithmic bytes per group: 256 (bf16 values) + 48 (codes) + 4 (scale)."""
    rng = np.random.default_rng(12)
    x_np = workloads.kv_groups(rng, **workloads.KV3_LAYER_256K)
    x = torch.from_numpy(x_np.view(np.int16)).to(dev).view(torch.bfloat16)
    n = x.shape[0]
    codes = torch.empty((n, 12), dtype=torch.int32, device=dev)
    scales = torch.empty((n,), dtype=torch.float32, device=dev)
    out = torch.empty((n, 128), dtype=torch.bfloat16, device=dev)
    bytes_step = n * (256 + 48 + 4)
    res = {}
    for name, fn in (("kv3_encode_256k", lambda: q8.q8_kv3_encode(x, codes=codes, scales=scales)),
                     ("kv3_decode_256k", lambda: q8.q8_kv3_decode(codes, scales, torch.bfloat16, out=out))):
        fn()
        total, kern = time_graph_steps(torch, q8, [fn], steps, warmup, instrument=False)
        gbs = bytes_step / kern / 1e9
        res[name] = {"value": round(gbs, 2), "unit": "GB/s", "us_per_step": round(kern * 1e6, 3),
                     "groups": n, "algorithmic_bytes_per_launch": bytes_step,
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": pk["hbm_gbs"],
                                  "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                                  "peak_source": f"hbm_gbs of the {pk_src} peaks",
                                  "kernel": "q8::kv3_" + name.split("_")[1] + "_kernel",
                                  "traffic": recorded_traffic(name)},
                     "steps": steps}
    return res


def run_bsa(torch, q8, dev, steps, warmup, pk, pk_src):
    """Block-sparse causal attention at a 32K-token prefill (32 query heads over 8
    key/value heads, head dim 128, ~10 % of the causal key blocks).  Algorithmic flops:
    4 * d per visible (query, key) pair, counted from the block lists (a listed block
    below the diagonal holds 64 x 64 pairs, the diagonal block 64 * 65 / 2)."""
    cfg = workloads.BSA_32K
    rng = np.random.default_rng(13)
    q, k, v = workloads.bsa_qkv(rng, cfg["H"], cfg["Hkv"], cfg["T"], cfg["d"])
    rp, ci = workloads.bsa_mask(rng, cfg["H"], cfg["T"], cfg["density"])
    nb = cfg["T"] // 64
    rows = np.repeat(np.tile(np.arange(nb), cfg["H"]), np.diff(rp))
    pairs = int(np.sum(np.where(ci == rows, 64 * 65 // 2, 64 * 64)))
    flops = 4 * cfg["d"] * pairs
    dt = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    qt, kt, vt = dt(q), dt(k), dt(v)
    rpt, cit = torch.from_numpy(rp).to(dev), torch.from_numpy(ci).to(dev)
    o = torch.empty((cfg["H"], cfg["T"], cfg["d"]), dtype=torch.bfloat16, device=dev)
    fn = lambda: q8.q8_bsa_attention(qt, kt, vt, rpt, cit, out_dtype=torch.bfloat16, o=o)
    fn()
    total, kern = time_graph_steps(torch, q8, [fn], steps, warmup, instrument=False)
    tf = flops / kern / 1e12
    # the ceiling of this formulation: every MMA of the kernel is M = 64 (one query block), a
    # shape the tensor pipe runs at half its rate; the recorded cycles per key block per CTA
    # with two CTAs per SM (bench_rates.py) give two blocks of 4 d 64 64 flops per SM
    rec = measured_rates() or {}
    blk_cycles = rec.get("rates", {}).get("umma_attn_block_2cta_cycles")
    m64_ceiling = (2 * 4 * cfg["d"] * 64 * 64 / blk_cycles * sm_count(torch) *
                   pk.get("sm_max_mhz", 2070.0) * 1e6 / 1e12) if blk_cycles else None
    return {"bsa_32k": {"value": round(tf, 2), "unit": "TFLOP/s", "us_per_step": round(kern * 1e6, 2),
                        "algorithmic_flops_per_launch": flops, "visible_pairs": pairs,
                        "block_density": round(len(ci) / (cfg["H"] * nb * (nb + 1) / 2), 4),
                        "roofline": {"bound": "tensor", "achieved": round(tf, 2),
                                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                                     "frac": round(tf / pk["bf16_tflops"], 4),
                                     "peak_source": f"bf16_tflops (burst) of the {pk_src} peaks",
                                     "m64_mma_ceiling_tflops": round(m64_ceiling, 1) if m64_ceiling else None,
                                     "frac_of_m64_ceiling": round(tf / m64_ceiling, 4) if m64_ceiling else None,
                                     "kernel": "q8::bsa_tc_kernel",
                                     "traffic": recorded_traffic("bsa_32k")},
                        "steps": steps,
                        "note": ("block-sparse causal attention (MInference-style): tcgen05 "
                                 "M=64 MMAs with S and O in TMEM, K/V by TMA, online softmax")}}


def e2e_measure(torch, q8, dev, x_np, bf16, Wqs, Wds, M, N, K, steps, warmup, bytes_step, ops_step,
                bound, path=None):
    """End to end through the public call q8_linear / q8_linear_ex: per step the H2D copy of x
    from pinned memory, the call, and the D2H copy of y into pinned memory."""
    copies = len(Wqs)
    n = max(1, min(steps, 2000 if bound == "hbm" else 50))
    if bf16:
        xh = torch.from_numpy(x_np.view(np.int16).copy()).pin_memory()
        xd = torch.empty((M, K), dtype=torch.int16, device=dev)
        if path is None:
            call = lambda i: q8.q8_linear(xd.view(torch.bfloat16), Wqs[i % copies], Wds[i % copies], y=yd)
        else:
            call = lambda i: q8.q8_linear_ex(xd.view(torch.bfloat16), Wqs[i % copies], Wds[i % copies],
                                             y=yd, path=path)
    else:
        xh = torch.from_numpy(x_np.copy()).pin_memory()
        xd = torch.empty((M, K), dtype=torch.float32, device=dev)
        call = lambda i: q8.q8_linear_ex(xd, Wqs[i % copies], Wds[i % copies], y=yd, path=path or "auto")
    yh = torch.empty((M, N), dtype=torch.float32).pin_memory()
    yd = torch.empty((M, N), dtype=torch.float32, device=dev)
    for i in range(3):
        xd.copy_(xh, non_blocking=True)
        call(i)
        yh.copy_(yd, non_blocking=True)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t = time.perf_counter()
    e0.record()
    for i in range(n):
        xd.copy_(xh, non_blocking=True)
        call(i)
        yh.copy_(yd, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    t = time.perf_counter() - t
    barrier()
    t = max_over_ranks(max(t, e0.elapsed_time(e1) / 1e3))
    if bound == "hbm":
        v, u = sum_over_ranks(bytes_step * n) / t / 1e9, "GB/s"
    else:
        v, u = sum_over_ranks(ops_step * n) / t / 1e12, "TOPS"
    return {"value": round(v, 3), "unit": u, "h2d_bytes_per_step": int(xh.numel() * xh.element_size()),
            "d2h_bytes_per_step": M * N * 4, "steps": n,
            "api": "q8_int8_block_gb300.q8_linear (C ABI q8_linear), host-timed"}


def int8_library_reference(torch, dev, M=2048, K=4096, N=12288, steps=20):
    """Speed reference only (not this library's path): the int8 x int8 -> int32 GEMM of
    PyTorch's torch._int_mm (a vendor-library int8 GEMM) on the 9B up-projection shape, in
    int8 TOPS.  It tells what the GPU's int8 GEMM route delivers; None if unavailable."""
    try:
        g = torch.Generator(device=dev)
        g.manual_seed(5)
        a = torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev, generator=g)
        b = torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev, generator=g).t()
        for _ in range(3):
            torch._int_mm(a, b)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            torch._int_mm(a, b)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / steps
        return {"tops": round(2 * M * N * K / t / 1e12, 1), "us": round(t * 1e6, 1),
                "shape": f"M={M} K={K} N={N}", "what": "torch._int_mm (library int8 GEMM), "
                "speed reference only"}
    except Exception as e:  # noqa: BLE001
        return {"unavailable": f"{type(e).__name__}: {str(e)[:80]}"}


# The configurations measured in every default run, after the headline: (case name, steps).
CONFIG_CASES = (("tiny", 20000), ("decode_m4", 20000), ("decode_m16", 20000), ("decode_m64", 20000),
                ("prefill9b_up", 200), ("prefill9b_down", 200), ("prefill27b_up", 20),
                ("prefill27b_down", 20))


def compact(e):
    """[value of the whole call, unit, roofline frac of the main kernel, us per call, us of the
    main kernel, path]"""
    return [round(e["value"], 2 if e["value"] < 1000 else 1), e["unit"], e["roofline"]["frac"],
            round(e["t_max"] / e["steps"] * 1e6, 2), e["roofline"]["kernel_us"], e["path"]]


def sweep_points(torch, q8, dev, pk, pk_src, budget_s=1.0):
    """Every (projection shape, M) point of the dense-layer sweep workload, timed like the
    headline (graph replays, rotating weight copies > 2 x L2), with the whole call's fraction
    of max(bytes / HBM peak, ops / tensor peak)."""
    wl = workloads.WORKLOADS["sweep"]
    points, seen = [], set()
    for p, proj in enumerate(wl.projections):
        if (proj.K, proj.N) in seen:  # q, k, v, o share one shape; so do gate and up
            continue
        seen.add((proj.K, proj.N))
        for mi, M in enumerate(wl.Ms):
            ops = workloads.algorithmic_ops(M, proj.N, proj.K)
            b = workloads.algorithmic_bytes(M, proj.N, proj.K, x_bytes=2)
            t_roof = max(b / (pk["hbm_gbs"] * 1e9), ops / (pk["bf16_tflops"] * 1e12))
            steps = int(max(20, min(2000, budget_s / max(t_roof * 4, 1e-9))))
            r = run_case(torch, q8, dev, f"sweep_{proj.name}_m{M}", steps, max(3, steps // 20), pk,
                         pk_src, spec=("sweep", p, mi))
            t = r["t_max"] / steps
            points.append({"projection": proj.name, "K": proj.K, "N": proj.N, "M": M,
                           "path": r["path"], "us_per_call": round(t * 1e6, 3),
                           "GBps": round(b / t / 1e9, 1), "TOPS": round(ops / t / 1e12, 2),
                           "bound": "hbm" if b / (pk["hbm_gbs"] * 1e9) >= ops / (pk["bf16_tflops"] * 1e12)
                           else "tensor",
                           "roofline_frac": round(t_roof / t, 4),
                           "kernel_frac": r["roofline"]["frac"]})
    return points


def sweep_compact(points):
    """{"M": [...], "<proj> KxN": [whole-call roofline fraction per M]}"""
    out = {"M": sorted({pt["M"] for pt in points})}
    for pt in points:
        key = f"{pt['projection']} {pt['K']}>{pt['N']}"
        out.setdefault(key, []).append(pt["roofline_frac"])
    return out


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
    r = run_case(torch, q8, dev, args.workload, args.steps, args.warmup, pk, pk_src, clocks=True,
                 e2e=True, force_path=None if args.path == "auto" else args.path)
    extra, configs = {}, {}
    if not args.no_extra and args.workload == "decode_m1":
        for name, st, fp in (("prefill9b_up", 50, "dp4a"),
                             ("decode_m1", 20000, "gated_fused"), ("decode_m1", 20000, "gated_unfused"),
                             ("prefill9b_up", 200, "gated_fused"), ("prefill9b_up", 200, "gated_unfused"),
                             ("decode_m1", 20000, "norm_gated_fused"),
                             ("prefill9b_up", 200, "norm_gated_fused"),
                             ("prefill9b_up", 200, "prepared"), ("gate_m128", 2000, None),
                             ("gate_m128", 2000, "prepared"), ("gate_m512", 500, None),
                             ("gate_m512", 500, "prepared")):
            norm = bool(fp) and fp.startswith("norm_")
            tag = fp[5:] if norm else fp
            gated = tag[6:] if tag and tag.startswith("gated_") else None
            prep = fp == "prepared"
            e = run_case(torch, q8, dev, name, st, max(3, st // 50), pk, pk_src,
                         force_path=None if (gated or prep) else fp, gated=gated, norm=norm,
                         prepared=prep)
            key = name if fp is None else f"{name}_{fp}"
            extra[key] = {"value": round(e["value"], 3), "unit": e["unit"], "path": e["path"],
                          "us_per_step": round(e["t_max"] / st * 1e6, 3),
                          "roofline": e["roofline"], "steps": st}
            if fp == "dp4a":
                extra[key]["note"] = ("the post's own design (dp4a int8 GEMM on CUDA cores), "
                                      "kept as the prior-art comparison on this GPU")
            if gated == "fused":
                extra[key]["note"] = ("gated FFN unit: y = silu(gate) * x.W^T, bfloat16 y, "
                                      "stored by the layer's epilogue (q8_linear_fused)")
                if norm:
                    extra[key]["note"] = ("RMSNorm + linear + SiLU gate + bfloat16 y in one call "
                                          "(q8_linear_fused with norm_weight)")
            if prep:
                extra[key]["note"] = ("tensor-core path on weights widened to binary16 once "
                                      "(q8_weights_to_f16 + q8_linear_prepared): no per-call "
                                      "widening pass")
            if gated == "unfused":
                extra[key]["note"] = ("the same unit as the plain layer (float32 y) followed by "
                                      "torch silu, multiply and bfloat16 cast; us_per_step is "
                                      "the whole step, roofline the layer's kernel alone")
        extra.update(run_kv3(torch, q8, dev, 200, 10, pk, pk_src))
        extra.update(run_bsa(torch, q8, dev, 20, 3, pk, pk_src))
        for k in ("kv3_encode_256k", "kv3_decode_256k"):
            extra[k]["note"] = ("3-bit KV-cache codec (Walsh-Hadamard rotation + Lloyd-Max), "
                                "one attention layer's keys at a 256K-token context")
        # every configured workload, compact: the prefill half of the metric with the rest
        configs["legend"] = ("[call value, unit, kernel roofline frac, us/call, kernel us, path]; "
                             f"peaks {pk['hbm_gbs']} GB/s, {pk['bf16_tflops']} TFLOP/s ({pk_src})")
        configs["decode_m1"] = compact(dict(r, steps=args.steps))
        for name, st in CONFIG_CASES:
            e = run_case(torch, q8, dev, name, st, max(3, st // 50), pk, pk_src)
            configs[name] = compact(dict(e, steps=st))
            extra.setdefault("configs_roofline", {})[name] = e["roofline"]
        pts = sweep_points(torch, q8, dev, pk, pk_src)
        extra["sweep_points"] = pts
        configs["sweep_call_frac"] = sweep_compact(pts)
        ref = int8_library_reference(torch, dev)
        extra["int8_library_ref"] = ref
        configs["int8_library_ref_tops"] = ref.get("tops")
    err = q8.q8_device_error()
    desc = workload_desc(args.workload)
    line = {
        "metric": METRIC, "value": round(r["value"], 3), "unit": r["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(r["t_max"] / args.steps * 1e3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded N(0,0.02) weights quantized to Q8_0, N(0,1) activations)",
        "config": {"workload": desc, "M": r["M"], "K": r["K"], "N": r["N"],
                   "weights": "Q8_0 (int8 codes + binary16 scale per 32 along K)",
                   "activations": ("bf16" if r["bf16"] else "float32") +
                                  ", quantized per call inside the library",
                   "kernel_path": r["path"], "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {r['copies']} rotating weight copies "
                         f"({r['copies'] * r['wbytes'] / 1e6:.0f} MB > 2 x L2)",
                   "timing": "CUDA graph replays timed by CUDA events; " +
                             ("the GEMM kernel timed by event nodes around each launch"
                              if r["path"] in ("tensor", "dp4a") else
                              "kernel time = the timed region's time per step (the streaming "
                              "kernel, chained to its neighbours by programmatic dependent "
                              "launch; event nodes would serialize the overlapping launches)")},
        "roofline": r["roofline"],
        "clocks": r["clocks"],
        "e2e": r["e2e"],
        "gpu_launches": args.steps * r["launches_per_step"],
        "device_error_word": err,
    }
    if extra:
        line["extra"] = extra
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(r["Wq0"], r["Wd0"], r["x_np"], r["bf16"], r["M"], r["N"],
                                            r["K"], r["xsize"], args.cpu_seconds)
    if configs:
        line["configs"] = configs  # last: the end of the line holds every config's summary
    return rank, line


# ----------------------------------------------------------------------------------- #
# CPU baseline and the reference arm (the oracle, as it stands)                        #
# ----------------------------------------------------------------------------------- #

def _oracle_cores():
    return os.cpu_count() or 1


def cpu_baseline(Wq_t, Wd_t, x_np, bf16, M, N, K, xsize, seconds):
    from oracle import oracle as O
    Wq = Wq_t.cpu().numpy()
    Wd = Wd_t.cpu().numpy().view(np.uint16)
    cores = _oracle_cores()
    rows = N
    t0 = time.perf_counter()
    O.linear(x_np, Wq, Wd, bf16=bf16, nthreads=cores)
    t_full = time.perf_counter() - t0
    if t_full > seconds:  # large layers: a contiguous slice of the output rows
        rows = max(64, int(N * seconds / t_full / 2))
    passes, t0 = 0, time.perf_counter()
    while True:
        O.linear(x_np, Wq[:rows], Wd[:rows], bf16=bf16, nthreads=cores)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= seconds or passes >= 100000:
            break
    b = workloads.algorithmic_bytes(M, rows, K, x_bytes=xsize) * passes
    ops = workloads.algorithmic_ops(M, rows, K) * passes
    tensor = workloads.algorithmic_ops(M, N, K) / 1.9e15 > workloads.algorithmic_bytes(M, N, K) / 6.8e12
    val, unit = (ops / dt / 1e12, "TOPS") if tensor else (b / dt / 1e9, "GB/s")
    return {"value": round(val, 6), "unit": unit, "cores": cores, "kind": "oracle",
            "sample": f"{passes} passes of the M={M} K={K} layer over {rows} of {N} output rows "
                      f"(activation quantization + those outputs) in {dt:.1f} s"}


def workload_desc(name):
    """The config's workload string, the same on both arms."""
    wname = CASES[name][0]
    desc = {"decode": "decode GEMV, FFN up-projection of a dense ~9B-class layer",
            "tiny": "tiny Q8_0 linear (float32 activations)",
            "prefill9b": "prefill GEMM, 9B-class projection",
            "prefill27b": "prefill GEMM, 27B-class projection, 1% activation channels x20",
            "sweep": "dense-layer sweep point, hidden-5120 hybrid layer"}[wname]
    return f"{desc}: {name}"


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0, None  # the oracle is timed once, on rank 0
    from oracle import oracle as O
    wname, p, mi = CASES[args.workload]
    wl = workloads.WORKLOADS[wname]
    W = wl.make_weights(p)
    x_np, _ = wl.make_act(p, mi)
    M, K = x_np.shape
    N = W.shape[0]
    xsize = 2 if wl.bf16 else 4
    Wq, Wd = O.quantize_weights(W)
    del W
    cores = _oracle_cores()
    # time a slice first, to size each step so that all steps fit in about a minute
    probe = min(N, 256)
    t0 = time.perf_counter()
    O.linear(x_np, Wq[:probe], Wd[:probe], bf16=wl.bf16, nthreads=cores)
    t_row = (time.perf_counter() - t0) / probe
    budget = 60.0
    rows = int(max(16, min(N, budget / max(1, args.steps + args.warmup) / max(t_row, 1e-9))))
    starts = [(i * rows) % (N - rows + 1) for i in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        s = starts[i]
        O.linear(x_np, Wq[s:s + rows], Wd[s:s + rows], bf16=wl.bf16, nthreads=cores)
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        s = starts[i]
        O.linear(x_np, Wq[s:s + rows], Wd[s:s + rows], bf16=wl.bf16, nthreads=cores)
    dt = time.perf_counter() - t0
    b = workloads.algorithmic_bytes(M, rows, K, x_bytes=xsize) * args.steps
    ops = workloads.algorithmic_ops(M, rows, K) * args.steps
    tensor = workloads.algorithmic_ops(M, N, K) / 1.9e15 > workloads.algorithmic_bytes(M, N, K) / 6.8e12
    value, unit = (ops / dt / 1e12, "TOPS") if tensor else (b / dt / 1e9, "GB/s")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded N(0,0.02) weights quantized to Q8_0, N(0,1) activations)",
        "config": {"workload": workload_desc(args.workload), "M": M, "K": K, "N": N,
                   "parallelism": "CPU oracle, rank 0 only"},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": f"each step: the layer over {rows} of {N} output rows "
                                   f"(activation quantization + those outputs), rotating over W"},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return rank, line


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=sorted(CASES), default="decode_m1",
                    help="which configured shape to time (default: decode GEMV, M=1)")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--path", choices=["auto", "decode", "batch", "tensor", "dp4a"], default="auto",
                    help="force a kernel family for --workload (default: the library's choice)")
    ap.add_argument("--sweep", action="store_true",
                    help="time every point of the dense-layer sweep workload (one GPU) and exit")
    ap.add_argument("--bsa", action="store_true",
                    help="time only block-sparse attention (32K-token prefill) and exit")
    ap.add_argument("--kv3", action="store_true",
                    help="time only the 3-bit KV-cache codec (one layer's keys at a 256K-token "
                         "context: encode and decode) and exit")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1:
        ap.error("--steps must be >= 1")
    return a


def sweep_arm(args):
    """Every (projection, M) point of the dense-layer sweep workload, each timed like the
    headline workload, with its roofline fraction against max(bytes / HBM, ops / tensor
    peak).  One JSON line with all points."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__ as g
    g.build()
    import q8_int8_block_gb300 as q8
    pk, pk_src = peaks()
    pts = sweep_points(torch, q8, torch.device("cuda", 0), pk, pk_src)
    return {"metric": METRIC, "sweep": "dense-layer sweep, hidden 5120 (q/k/v/o 5120x5120, "
            "gate/up 5120x17408, down 17408x5120, GDN in-proj 5120x10240)",
            "time": "whole call per step (all kernels of the path), CUDA graph replays",
            "peaks": {k: pk[k] for k in ("hbm_gbs", "bf16_tflops")}, "peak_source": pk_src,
            "points": pts, "call_frac": sweep_compact(pts),
            "device_error_word": q8.q8_device_error()}


def main(argv=None):
    args = parse_args(argv)
    if args.sweep:
        print(json.dumps(sweep_arm(args)), flush=True)
        return
    if args.bsa:
        import torch
        import __graft_entry__ as g
        g.build()
        import q8_int8_block_gb300 as q8
        torch.cuda.set_device(0)
        pk, pk_src = peaks()
        r = run_bsa(torch, q8, torch.device("cuda", 0), args.steps, args.warmup, pk, pk_src)
        print(json.dumps({"bsa": r, "device_error_word": q8.q8_device_error()}), flush=True)
        return
    if args.kv3:
        import torch
        import __graft_entry__ as g
        g.build()
        import q8_int8_block_gb300 as q8
        torch.cuda.set_device(0)
        pk, pk_src = peaks()
        r = run_kv3(torch, q8, torch.device("cuda", 0), args.steps, args.warmup, pk, pk_src)
        print(json.dumps({"kv3": r, "device_error_word": q8.q8_device_error()}), flush=True)
        return
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
