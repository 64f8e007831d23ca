"""Builds libsse.so in-tree (``_build/``) from ``csrc/*.cu`` with nvcc for
sm_103a.  Translation units compile in parallel; the link uses the static CUDA
runtime so the library has no runtime dependency beyond the driver."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libsse.so")
# Checked build for the failure-detection test: the persistent tensor-core
# kernels compiled with -DSSE_FAULT_INJECT (short bounded waits, a switch
# that withholds one barrier arrival or one product round), linked with the
# same objects as libsse.so otherwise.
LIB_CHECKED = os.path.join(BUILD, "libsse_checked.so")
CHECKED_SRCS = ("fwd_chunked.cu", "delta_chunked.cu", "backward_chunked.cu")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", INCLUDE]
if os.environ.get("SSE_NVTX") == "1":   # NVTX ranges around every entry point
    FLAGS.append("-DSSE_NVTX")


def _nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: libsse needs the CUDA toolkit to build")
    return p


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdrs = sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "sse.h")]
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(job):
        src, checked = job
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ("_checked.o" if checked else ".o"))
        if force or _stale(obj, [src] + hdrs):
            cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, *(["-DSSE_FAULT_INJECT"] if checked else []), "-c", src,
                   "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose:
                print(r.stdout + r.stderr)
        return obj

    checked_srcs = [os.path.join(CSRC, n) for n in CHECKED_SRCS]
    jobs = [(src, False) for src in srcs] + [(src, True) for src in checked_srcs]
    # the largest translation units first, so the parallel compile ends sooner
    jobs.sort(key=lambda j: -os.path.getsize(j[0]))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        done = dict(zip(jobs, ex.map(compile_one, jobs)))
    objs = [done[(src, False)] for src in srcs]
    checked_objs = [done[(src, src in checked_srcs)] for src in srcs]
    for lib, lib_objs in ((LIB, objs), (LIB_CHECKED, checked_objs)):
        if force or _stale(lib, lib_objs):
            tmp = lib + ".tmp.%d" % os.getpid()
            r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *lib_objs], capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
