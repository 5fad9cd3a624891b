"""Build libkitty.so in-tree for sm_103a (nvcc + g++, translation units in parallel)."""

from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libkitty.so")
INCLUDE = os.path.join(ROOT, "include")

CU = ["quantize.cu", "decode.cu", "fp16kv.cu"]
CPP = ["host.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def _sources():
    return [os.path.join(CSRC, f) for f in CU + CPP + ["kitty_common.cuh", "quant_tile.cuh", "host_common.h"]] + [
        os.path.join(INCLUDE, "kitty.h")]


def build(force: bool = False, verbose: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(s) for s in _sources())):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    cmds = []
    objs = []
    for f in CU:
        o = os.path.join(OUT_DIR, f + ".o")
        objs.append(o)
        cmds.append([nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-c", os.path.join(CSRC, f), "-o", o])
    for f in CPP:
        o = os.path.join(OUT_DIR, f + ".o")
        objs.append(o)
        cmds.append(["g++", "-O2", "-std=c++17", "-fPIC", "-I" + INCLUDE,
                     "-c", os.path.join(CSRC, f), "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("build failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(len(cmds)) as ex:
        list(ex.map(run, cmds))
    tmp = LIB + ".tmp%d" % os.getpid()
    run([nvcc, *ARCH, "-shared", "--cudart=static", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
