"""Build libwoq.so in-tree with nvcc for sm_103a.

Each source compiles to an object in parallel; the link exports only the
woq_* C ABI (a linker version script), with the CUDA runtime linked
statically so the library's kernels are registered with its own runtime.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libwoq.so")
SOURCES = ["woq_api.cu", "woq_gemv_w4.cu", "woq_gemv_w4_pro.cu", "woq_gemv_w4_mma.cu", "woq_gemv_w4_mma_pro.cu",
           "woq_gemv_w6.cu", "woq_gemv_w6_pro.cu", "woq_small_kernels.cu", "woq_pack.cpp", "woq_tree.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (set NVCC or put CUDA 13 on PATH)")
    return cand


def _deps_mtime() -> float:
    inc = os.path.join(ROOT, "include")
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(inc, f) for f in os.listdir(inc)] + [__file__]
    return max(os.path.getmtime(p) for p in paths)


def needs_build() -> bool:
    return not os.path.exists(LIB) or os.path.getmtime(LIB) < _deps_mtime()


def _compile(src: str, verbose_ptxas: bool, out_dir: str = OUT_DIR, defines=()) -> str:
    obj = os.path.join(out_dir, src + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden,-O2",
           *[f"-D{d}" for d in defines],
           "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd[1:1] = ["-x", "cu"]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, trace: bool = False) -> str:
    """Build libwoq.so; trace=True builds libwoq_trace.so with per-CTA phase stamps instead."""
    lib = os.path.join(PKG, "libwoq_trace.so") if trace else LIB
    out_dir = os.path.join(OUT_DIR, "trace") if trace else OUT_DIR
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    os.makedirs(out_dir, exist_ok=True)
    defines = ("WOQ_TRACE",) if trace else ()
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, out_dir, defines), SOURCES))
    vs = os.path.join(out_dir, "exports.map")
    with open(vs, "w") as f:
        f.write("{ global: woq_*; local: *; };\n")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, f"-Xlinker=--version-script={vs}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, trace="--trace" in sys.argv))
