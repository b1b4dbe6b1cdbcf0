"""Compile libswiglu.so for sm_103a with nvcc, in-tree.

    python gate_up_swiglu_gb300/build.py [--ptxas-info]

Run it as a script (or load it by path): importing the package itself needs
the built library.

The library is three translation units (the C ABI with the streaming kernel
templates it instantiates, the tensor-core linear_fc1 + SwiGLU kernel, and the
host-buffer pipeline),
compiled in parallel and linked against the static CUDA runtime so the .so depends on
nothing but the NVIDIA driver (libcuda).  No fast-math: the kernels choose every approximate
operation explicitly and must keep subnormal results.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libswiglu.so")
SOURCES = [os.path.join(CSRC, "swiglu_abi.cu"), os.path.join(CSRC, "fc1_swiglu.cu"),
           os.path.join(CSRC, "host_pipeline.cu")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libswiglu needs the CUDA toolkit to build")


COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2"]


def compile_commands(out: str = LIB, ptxas_info: bool = False):
    """One nvcc -c per translation unit (run in parallel), then one link."""
    objs, cmds = [], []
    for src in SOURCES:
        obj = out + "." + os.path.splitext(os.path.basename(src))[0] + ".o"
        cmd = [nvcc(), *ARCH, *COMMON, "-I", INCLUDE, "-I", CSRC, "-c", "-o", obj, src]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        cmds.append(cmd)
    link = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", out, *objs]
    return cmds, link, objs


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    deps = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, ptxas_info: bool = False, out: str = LIB) -> str:
    if force or ptxas_info or _stale(out):
        tmp = out + ".tmp%d" % os.getpid()
        cmds, link, objs = compile_commands(tmp, ptxas_info)
        procs = [subprocess.Popen(c) for c in cmds]
        codes = [p.wait() for p in procs]
        try:
            if any(codes):
                raise subprocess.CalledProcessError(max(codes), cmds[codes.index(max(codes))])
            subprocess.run(link, check=True)
            os.replace(tmp, out)
        finally:
            for o in objs:
                if os.path.exists(o):
                    os.remove(o)
    return out


if __name__ == "__main__":
    print(build(force=True, ptxas_info="--ptxas-info" in sys.argv))
