"""Builds libconvrot.so in-tree with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then linked into a shared
library next to this file (`_build/libconvrot.so`).  Only the CUDA runtime is
linked; the driver entry point for tensor-map encoding is resolved at run time.
"""
from __future__ import annotations

import concurrent.futures
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libconvrot.so")
# The same sources with -DCONVROT_CHECKED: every instrumented kernel access is checked against its tensor.
CHECKED_LIB_PATH = os.path.join(OUT_DIR, "libconvrot_checked.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["rotq.cu", "rotq_wide.cu", "lora_rotq.cu", "bwd_prep.cu", "bwd_r2.cu", "gemm_tc.cu", "convrot_api.cu",
           "noalloc.cu", "selftest.cu", "peak_probe.cu", "lora_down.cu",
           "bwd_weight.cu"]
HEADERS = ["common.cuh", "fwht.cuh", "mbar.cuh", "wide.cuh", "internal.h", "launch_cache.h", "tcgen05.cuh", "dfloat.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "convrot.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Builds the release library and its checked variant (all objects compiled in parallel)."""
    targets = [(LIB_PATH, [], ""), (CHECKED_LIB_PATH, ["-DCONVROT_CHECKED"], "_checked")]
    todo = [t for t in targets if force or _stale(t[0])]
    if not todo:
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(job):
        src, flags, suffix = job
        obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + suffix + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *flags, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    jobs = [(src, flags, suffix) for _, flags, suffix in todo for src in SOURCES]
    with concurrent.futures.ThreadPoolExecutor(min(len(jobs), os.cpu_count() or 8)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for i, (path, _, _) in enumerate(todo):
        mine = objs[i * len(SOURCES):(i + 1) * len(SOURCES)]
        tmp = path + f".tmp{os.getpid()}"
        cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *mine, "-o", tmp, "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
