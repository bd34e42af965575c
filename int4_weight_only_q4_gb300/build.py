"""Build libq4.so in-tree with nvcc for sm_103a (GB300).

Four translation units (the GEMV/GEMM kernels, the attention kernels, the
tensor-memory prefill GEMM and the host packer) are compiled in parallel and
linked into one shared library next to this file.  The CUDA runtime is linked
statically, so the library needs only the NVIDIA driver.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "libq4.so")
BUILD_DIR = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-I", INCLUDE, "-Xcompiler", "-fPIC,-ffp-contract=off"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or install the CUDA toolkit)")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(verbose: bool = False, extra: list[str] | None = None) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    nv = nvcc()
    extra = list(extra or [])
    srcs = [("q4_gemv.cu", ARCH), ("q4_attn.cu", ARCH), ("q4_prefill_tc.cu", ARCH), ("q4_host.cpp", [])]
    objs = []
    cmds = []
    for name, arch in srcs:
        obj = os.path.join(BUILD_DIR, name + ".o")
        objs.append(obj)
        lang = [] if name.endswith(".cu") else ["-x", "c++"]
        cmds.append([nv, *arch, *COMMON, *extra, *lang, "-c", os.path.join(CSRC, name), "-o", obj])
    with ThreadPoolExecutor(len(cmds)) as ex:
        logs = list(ex.map(_run, cmds))
    tmp = OUT + ".tmp"
    logs.append(_run([nv, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fPIC", "-lpthread"]))
    os.replace(tmp, OUT)
    if verbose:
        print("\n".join(l for l in logs if l.strip()))
    return OUT


if __name__ == "__main__":
    v = "-v" in sys.argv
    xs = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(verbose=v or bool(xs), extra=xs))
