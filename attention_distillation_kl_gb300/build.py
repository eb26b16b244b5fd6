"""Builds libstreamkl.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel, then linked with the
static CUDA runtime into ``attention_distillation_kl_gb300/libstreamkl.so``.
"""

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libstreamkl.so")
DEBUG_LIB = os.path.join(PKG, "libstreamkl_debug.so")
SOURCES = ["api.cu", "fwd.cu", "fwd_wide.cu", "bwd.cu", "dq_fixed.cu", "bwd_wide_p0.cu", "bwd_wide_p1.cu", "bwd_both.cu",
           "static_ws.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set CUDA_HOME or NVCC")


def cflags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                   "-I", CSRC, "--expt-relaxed-constexpr", *extra]


def build(verbose=False, extra_flags=(), debug=True):
    """Compiles libstreamkl.so and, with debug=True, libstreamkl_debug.so (the
    same sources with STREAMKL_DEBUG: in-kernel bounds checks that record a
    failed check in the device status word), all translation units of both
    in parallel."""
    nvcc = nvcc_path()
    variants = [("", LIB, [])]
    if debug:
        variants.append(("debug", DEBUG_LIB, ["-DSTREAMKL_DEBUG"]))
    for sub, _, _ in variants:
        os.makedirs(os.path.join(BUILD, sub), exist_ok=True)

    def one(job):
        sub, flags, src = job
        obj = os.path.join(BUILD, sub, src.replace(".cu", ".o"))
        cmd = [nvcc, *cflags([*extra_flags, *flags]), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    jobs = [(sub, flags, src) for sub, _, flags in variants for src in SOURCES]
    with ThreadPoolExecutor(min(len(jobs), max(4, os.cpu_count() or 4))) as ex:
        objs = list(ex.map(one, jobs))
    for k, (sub, lib, _) in enumerate(variants):
        tmp = lib + ".tmp"
        part = objs[k * len(SOURCES):(k + 1) * len(SOURCES)]
        cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *part]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else []))
