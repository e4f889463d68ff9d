"""Builds libmie.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each translation unit is compiled in parallel; the CUDA runtime is linked statically
so the library has no runtime search-path requirements.
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "libmie.so")
BUILD_DIR = os.path.join(PKG, "_build", platform.machine())
STAMP = os.path.join(BUILD_DIR, "libmie.so.stamp")
SOURCES = ["gemv.cu", "gemv_slots.cu", "attn.cu", "step.cu", "quant.cu", "model.cu", "probe.cu", "sample.cu", "gemm.cu", "prefill.cu", "pool.cpp", "spec.cpp"]
HEADERS = ["common.cuh", "internal.h", "device.cuh", "attn_core.cuh", "attn_mma.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# MIE_STAGE_TRACE=1 builds the instrumented library whose persistent step also stamps
# every ring stage (mie_set_trace); its objects live in their own build folder.
DEFINES = ["-DMIE_STAGE_TRACE"] if os.environ.get("MIE_STAGE_TRACE") == "1" else []
if DEFINES:
    BUILD_DIR = BUILD_DIR + "-stage-trace"
    STAMP = os.path.join(BUILD_DIR, "libmie.so.stamp")


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmie.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    header_paths = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "mie.h")]
    cc = nvcc()
    jobs = []
    objs = []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [sp] + header_paths):
            cmd = [cc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                   "-I", os.path.join(ROOT, "include"), *DEFINES, "-c", sp, "-o", obj + ".tmp"]
            if src.endswith(".cu"):
                cmd[1:1] = ["-Xptxas", "-v"] if verbose else []
            jobs.append((cmd, obj))

    def run(job):
        cmd, obj = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return r.stderr

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            logs = list(ex.map(run, jobs))
        if verbose:
            for lg in logs:
                print(lg)
    if force or jobs or _stale(STAMP, objs) or not os.path.exists(OUT):
        tmp = OUT + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, OUT)
        with open(STAMP, "w") as f:
            f.write(platform.machine() + "\n")
    return OUT


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
