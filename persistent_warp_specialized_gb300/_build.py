"""Builds libtg.so (the C ABI of include/tg.h) in-tree with nvcc for sm_103a.

    python -m persistent_warp_specialized_gb300._build [--force] [-v]

Two translation units compile in parallel (the kernels, and the C-ABI host code) and are
linked into ``persistent_warp_specialized_gb300/libtg.so`` with the CUDA runtime linked
statically.  A stamp of the sources and flags skips rebuilding when nothing changed.
"""

import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libtg.so")
STAMP = os.path.join(BUILD_DIR, "libtg.stamp")

SOURCES = ["tg_gemm.cu", "tg_api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-Wall", "-diag-suppress", "177"]


def nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand) and not shutil.which(cand):
        raise RuntimeError("nvcc not found; set NVCC or put the CUDA toolkit on PATH")
    return cand


def _inputs():
    files = [os.path.join(ROOT, "include", "tg.h")]
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            files.append(os.path.join(CSRC, name))
    return files


def _stamp():
    """sha256 of the library's sources (by path relative to the repository) and flags: the
    same on every machine for the same sources."""
    h = hashlib.sha256()
    for path in _inputs():
        h.update(os.path.relpath(path, ROOT).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(FLAGS).encode())
    return h.hexdigest()


# The sources each GEMM kernel's device code is built from (a profile taken of a kernel stays
# valid while these and the flags are unchanged).
KERNEL_SOURCES = {
    "gemm_persistent_ws": ["tg_config.h", "tg_ptx.cuh", "tg_tile_scheduler.cuh",
                           "tg_gemm_kernel.cuh"],
    "gemm_pair_ws": ["tg_config.h", "tg_ptx.cuh", "tg_tile_scheduler.cuh", "tg_gemm_kernel.cuh",
                     "tg_gemm_pair_kernel.cuh"],
    "gemm_pair_wide_ws": ["tg_config.h", "tg_ptx.cuh", "tg_tile_scheduler.cuh", "tg_gemm_kernel.cuh",
                          "tg_gemm_pair_kernel.cuh", "tg_wide_config.h",
                          "tg_gemm_pair_wide_kernel.cuh"],
    "gemm_mxfp8_ws": ["tg_config.h", "tg_ptx.cuh", "tg_tile_scheduler.cuh", "tg_gemm_kernel.cuh",
                      "tg_mx_kernel.cuh"],
    "gemm_mxfp8_pair_ws": ["tg_config.h", "tg_ptx.cuh", "tg_tile_scheduler.cuh",
                           "tg_gemm_kernel.cuh", "tg_gemm_pair_kernel.cuh", "tg_mx_kernel.cuh",
                           "tg_mx_pair_kernel.cuh"],
}


def kernel_stamp(kernel):
    """sha256 of one kernel's device sources and the flags."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        h.update(name.encode())
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    h.update(" ".join(FLAGS).encode())
    return h.hexdigest()


def build(force=False, verbose=False, ptxas_info=False):
    """Compile libtg.so if its sources changed; returns its path."""
    stamp = _stamp()
    if not force and os.path.exists(LIB_PATH) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == stamp:
                return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc] + FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(f"--- {src}\n{text}")
        elif verbose or ptxas_info:
            print(text, end="", flush=True)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIB_PATH + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, LIB_PATH)
    with open(STAMP, "w") as f:
        f.write(stamp)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv)
    print(LIB_PATH)
