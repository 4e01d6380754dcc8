"""Build libssd_gb300.so (the C-ABI library) in-tree with nvcc for sm_103a.

The translation units compile in parallel, then link with the shared
CUDA runtime.  Nothing is installed outside this directory.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libssd_gb300.so")
SOURCES = ["ssd_stats.cu", "ssd_residual.cu", "ssd_topk.cu", "ssd_filter.cu", "ssd_tree.cu",
           "ssd_cache.cu", "ssd_chain.cu", "ssd_step.cu", "ssd_api.cu"]
HEADERS = ["ssd_device.cuh", "ssd_scan.cuh", "ssd_merge.cuh", "ssd_cache.cuh", "ssd_draw.cuh", "ssd_pass.cuh",
           "ssd_layout.h", "exp2_table.inc"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def cuda_lib_dir() -> str:
    base = os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))
    for d in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        p = os.path.join(base, d)
        if os.path.exists(os.path.join(p, "libcudart.so")):
            return p
    return os.path.join(base, "lib64")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "ssd.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    cc = nvcc()
    tmp = tempfile.mkdtemp(prefix="ssd_build_")
    try:
        procs = []
        objs = []
        for src in SOURCES:
            obj = os.path.join(tmp, src.replace(".cu", ".o"))
            objs.append(obj)
            cmd = [cc, "-std=c++17", *ARCH, "-O3", "-lineinfo", "-Xcompiler", "-fPIC",
                   "-Xcompiler", "-fvisibility=hidden", "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        failed = []
        for src, p in procs:
            out, _ = p.communicate()
            if verbose or p.returncode:
                sys.stderr.write(out.decode(errors="replace"))
            if p.returncode:
                failed.append(src)
        if failed:
            raise RuntimeError("nvcc failed on " + ", ".join(failed))
        out = LIB + ".tmp%d" % os.getpid()
        libdir = cuda_lib_dir()
        link = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", out, *objs,
                "-Xlinker", "-rpath=" + libdir, "-L" + libdir]
        r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode:
            sys.stderr.write(r.stdout.decode(errors="replace"))
            raise RuntimeError("link of libssd_gb300.so failed")
        os.replace(out, LIB)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
