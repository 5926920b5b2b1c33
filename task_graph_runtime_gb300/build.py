"""Compile ``libmpk.so`` in-tree for sm_103a (nvcc + g++, no cmake).

The translation units compile in parallel; the shared library lands
next to this file.  ``python -m task_graph_runtime_gb300.build`` runs it."""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "libmpk.so")
BUILD_DIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if not os.path.isdir(home):
        nvcc = shutil.which("nvcc")
        if nvcc:
            home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return home


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                       text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" +
                           r.stdout)
    return r.stdout


def build(verbose: bool = False) -> str:
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(BUILD_DIR, exist_ok=True)
    inc = ["-I" + INCLUDE, "-I" + CSRC, "-I" + os.path.join(cuda, "include")]
    jobs = [
        [nvcc] + ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler",
                         "-fPIC", "-c", os.path.join(CSRC, "kernels.cu"),
                         "-o", os.path.join(BUILD_DIR, "kernels.o")] + inc,
        [nvcc] + ARCH + ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-c",
                         os.path.join(CSRC, "noalloc.cu"), "-o",
                         os.path.join(BUILD_DIR, "noalloc.o")] + inc,
        ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-c",
         os.path.join(CSRC, "capi.cpp"), "-o",
         os.path.join(BUILD_DIR, "capi.o")] + inc,
        ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-c",
         os.path.join(CSRC, "tgraph_builder.cpp"), "-o",
         os.path.join(BUILD_DIR, "tgraph_builder.o")] + inc,
        ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-c",
         os.path.join(CSRC, "layout.cpp"), "-o",
         os.path.join(BUILD_DIR, "layout.o")] + inc,
        ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-pthread", "-c",
         os.path.join(CSRC, "protocol_sim.cpp"), "-o",
         os.path.join(BUILD_DIR, "protocol_sim.o")] + inc,
    ]
    with concurrent.futures.ThreadPoolExecutor(len(jobs)) as ex:
        for out in ex.map(_run, jobs):
            if verbose and out.strip():
                print(out)
    tmp = OUT + ".tmp"
    _run([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp,
                          os.path.join(BUILD_DIR, "kernels.o"),
                          os.path.join(BUILD_DIR, "noalloc.o"),
                          os.path.join(BUILD_DIR, "capi.o"),
                          os.path.join(BUILD_DIR, "tgraph_builder.o"),
                          os.path.join(BUILD_DIR, "layout.o"),
                          os.path.join(BUILD_DIR, "protocol_sim.o"),
                          "-Xcompiler", "-pthread",
                          "-Xlinker", "-rpath=" + os.path.join(cuda, "lib64")])
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
