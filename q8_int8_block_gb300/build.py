"""Builds libq8.so (the CUDA library behind include/q8.h) in-tree, for sm_103a only.

Each .cu file is compiled by its own nvcc process (in parallel), then linked into
q8_int8_block_gb300/libq8.so.  A rebuild happens only when a source or header is newer
than the library.  Usage: python -m q8_int8_block_gb300.build [--force] [--jobs N]
"""
import concurrent.futures as cf
import glob
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(ROOT, "_build", "obj")
LIB = os.path.join(HERE, "libq8.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")
    return path


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


# Kernels whose warp roles resize their registers with setmaxnreg: the split is exact only for
# the register count the kernel was written for (the constant named here, in the same file).
# The build reads ptxas's report and stops if the compiled count differs, rather than leave
# the library to refuse every launch of that kernel at run time.
REG_PINS = {"q8_gemm.cu": ("gemm_tc_kernel", "kLaunchRegs")}


def _check_reg_pin(src: str, ptxas_report: str) -> None:
    name = os.path.basename(src)
    if name not in REG_PINS:
        return
    kernel, const = REG_PINS[name]
    m = re.search(r"constexpr int " + const + r" = (\d+);", open(src).read())
    if not m:
        raise RuntimeError(f"{name}: constant {const} not found")
    want = int(m.group(1))
    current, seen = None, 0
    for line in ptxas_report.splitlines():
        e = re.search(r"Compiling entry function '([^']+)'", line)
        if e:
            current = e.group(1)
            continue
        u = re.search(r"Used (\d+) registers", line)
        if u and current and kernel in current:
            seen += 1
            if int(u.group(1)) != want:
                raise RuntimeError(f"{name}: {current} compiled to {u.group(1)} registers per thread, "
                                   f"but its setmaxnreg split assumes {const} = {want}")
    if seen == 0:
        raise RuntimeError(f"{name}: no ptxas register report for {kernel}")


def _compile(src: str, extra) -> str:
    obj = os.path.join(OBJ, os.path.basename(src) + ".o")
    verbose = ["-Xptxas", "-v"] if os.path.basename(src) in REG_PINS else []
    cmd = [nvcc()] + ARCH + CFLAGS + verbose + list(extra) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    _check_reg_pin(src, r.stdout + r.stderr)
    return obj


def build(force: bool = False, jobs: int = 0, extra=()) -> str:
    if not force and not extra and up_to_date():
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    srcs = sources()
    jobs = jobs or min(len(srcs), os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), srcs))
    tmp = LIB + ".tmp"
    # the driver API is reached through cudaGetDriverEntryPointByVersion: no -lcuda
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    jobs = 0
    if "--jobs" in sys.argv:
        jobs = int(sys.argv[sys.argv.index("--jobs") + 1])
    print(build(force="--force" in sys.argv, jobs=jobs))
