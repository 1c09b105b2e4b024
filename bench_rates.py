#!/usr/bin/env python3
"""Per-SM rate microbenchmarks of the GPU (bench_rates.cu), one JSON line on stdout.

These are the unit rates that the secondary rooflines of bench.py rest on (the dp4a GEMM's
integer-ALU peak, the mma.sync ceiling of the batched and attention kernels) and that the
analysis of the prefill GEMM uses (the FP32 rescale rate against the tcgen05 MMA rate, the
broadcast shared-memory load rate of the rescale's column scales, the commit round trip) and
the block-sparse attention kernel's (the rates of its M = 64 MMA shapes).

    python bench_rates.py [--record profiles/rates_gb300.json]

--record also writes the line (with the command and the GPU's name) to that file, which
bench.py then reads for its dp4a and mma.sync peaks.
"""
import argparse
import ctypes
import json
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(ROOT, "bench_rates.cu")
LIB = os.path.join(ROOT, "_build", "libq8rates.so")

NAMES = [
    ("ffma_per_clk_sm", "binary32 FMA per clock per SM, scalar FFMA"),
    ("ffma2_per_clk_sm", "binary32 FMA per clock per SM, packed f32x2 (2 per instruction)"),
    ("dp4a_per_clk_sm", "dp4a (4 int8 MACs each) per clock per SM"),
    ("hmma_mac_per_clk_sm", "mma.sync m16n8k16 f16->f32 MACs per clock per SM"),
    ("imma_mac_per_clk_sm", "mma.sync m16n8k32 s8->s32 MACs per clock per SM"),
    ("lds_bcast_per_clk_sm", "warp-wide one-address LDS.128 per clock per SM"),
    ("umma_mac_per_clk_sm", "tcgen05.mma kind::f16 M128 N256 K16 MACs per clock per SM"),
    ("umma_pair_commit_rt_cycles", "cycles: 2 x M128 N256 K16, tcgen05.commit, mbarrier wait"),
    ("umma_m64n64_1cta_cycles", "cycles per tcgen05.mma M64 N64 K16 in a dependent chain, one CTA per SM"),
    ("umma_m64n64_2cta_mac_per_clk_sm", "tcgen05.mma M64 N64 K16 MACs per clock per SM, two CTAs per SM"),
    ("umma_m128n64_2cta_mac_per_clk_sm", "tcgen05.mma M128 N64 K16 MACs per clock per SM, two CTAs per SM"),
    ("umma_attn_block_2cta_cycles", "cycles per attention key block per CTA (8 x M64 N64 + 4 x M64 N128 K16), "
                                    "two CTAs per SM"),
]


def build():
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I" + ROOT, "-Xcompiler", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp"],
                   check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


def measure():
    import torch
    lib = ctypes.CDLL(build())
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    res = (ctypes.c_double * len(NAMES))()
    n = lib.q8_rates(sms, res)
    if n != len(NAMES):
        raise RuntimeError(f"q8_rates failed ({n})")
    rates = {k: round(res[i], 2) for i, (k, _) in enumerate(NAMES)}
    mhz = None
    try:
        out = subprocess.run(["nvidia-smi", "-i", "0", "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True)
        mhz = float(out.stdout.strip().splitlines()[0])
    except Exception:  # noqa: BLE001
        pass
    line = {"gpu": props.name, "sms": sms, "sm_max_mhz": mhz, "rates": rates,
            "what": {k: d for k, d in NAMES}}
    if mhz:
        f = sms * mhz * 1e6 / 1e12
        line["peaks_at_max_clock"] = {
            "dp4a_int8_tops": round(rates["dp4a_per_clk_sm"] * 8 * f, 1),
            "mma_sync_f16_tflops": round(rates["hmma_mac_per_clk_sm"] * 2 * f, 1),
            "mma_sync_s8_tops": round(rates["imma_mac_per_clk_sm"] * 2 * f, 1),
            "tcgen05_f16_tflops": round(rates["umma_mac_per_clk_sm"] * 2 * f, 1),
            "fp32_tflops": round(rates["ffma_per_clk_sm"] * 2 * f, 1),
        }
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--record", default=None, help="also write the JSON line to this file")
    a = ap.parse_args(argv)
    line = measure()
    print(json.dumps(line), flush=True)
    if a.record:
        line = dict(line, command="python bench_rates.py --record " + a.record)
        with open(os.path.join(ROOT, a.record) if not os.path.isabs(a.record) else a.record, "w") as f:
            json.dump(line, f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    sys.exit(main())
