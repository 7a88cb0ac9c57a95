"""Build libpkv.so in-tree for sm_103a with nvcc.

Each translation unit under ``csrc/`` compiles in parallel to an object in
``_build/``; the objects link into ``paged_kv_gqa_nx_gb300/libpkv.so``
(CUDA runtime linked statically, only the ``pkv_*`` C ABI exported).

    python paged_kv_gqa_nx_gb300/build.py [--force] [--verbose]

(Run by path: importing the package itself needs the built library.)
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libpkv.so")
HEADERS = [os.path.join(ROOT, "include", "pkv.h"), os.path.join(CSRC, "pkv_internal.h"),
           os.path.join(CSRC, "pkv_tcgen05.h")]
SOURCES = ["pkv_kernels.cu", "pkv_decode_mma.cu", "pkv_prefill.cu", "pkv_host.cpp", "pkv_noalloc.cu",
           "pkv_probe.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
          "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpkv")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)



def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link.  Extra nvcc flags (e.g. -DPKV_FAST_STAGES=3) may be
    given in the PKV_NVCC_FLAGS environment variable."""
    nvcc = _nvcc()
    extra = os.environ.get("PKV_NVCC_FLAGS", "").split()
    os.makedirs(BUILD, exist_ok=True)
    jobs = []
    objs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + HEADERS):
            cmd = [nvcc] + ARCH + COMMON + extra + ["-c", path, "-o", obj]
            if src.endswith(".cu"):
                cmd += ["-Xptxas", "-v"] if verbose else []
            else:
                cmd = [nvcc] + COMMON + extra + ["-x", "c++", "-c", path, "-o", obj]
            jobs.append(cmd)
    with cf.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
    for cmd, r in zip(jobs, results):
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on " + cmd[-3])
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lrt", "-ldl", "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            raise RuntimeError("link of libpkv.so failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
