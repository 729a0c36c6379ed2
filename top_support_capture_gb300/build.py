"""Build libsfc.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in its own nvcc process (in parallel), then linked into
``top_support_capture_gb300/libsfc.so``. No CMake, no torch extension machinery.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libsfc.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["sfc_api.cu", "sfc_launch_bf16.cu", "sfc_launch_f32.cu", "sfc_replay.cu", "sfc_pack.cu",
           "sfc_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]
# Shared cudart: when PyTorch is loaded first, its libcudart.so.13 is reused (one runtime instance,
# one notion of the current device); otherwise the toolkit's copy is found through the rpath.
LINK = ["-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the sm_103a CUDA toolkit is required to build libsfc.so")


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        jobs.append((obj, [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]))
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(lambda j: _run(j[1]), jobs))
    if verbose or ptxas_info:
        for (obj, _), out in zip(jobs, outs):
            sys.stdout.write(f"--- {os.path.basename(obj)}\n{out}")
    tmp = OUT + ".tmp"
    _run([cc, *ARCH, *LINK, "-o", tmp, *[o for o, _ in jobs]])
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
