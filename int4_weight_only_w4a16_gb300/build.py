"""Build the C-ABI library ``libw4a16.so`` in-tree for sm_103a.

Each CUDA translation unit is compiled in parallel with nvcc, then linked into
one shared object next to this file.  Run as ``python -m
int4_weight_only_w4a16_gb300.build`` or through ``__graft_entry__.build()``.
No fast-math: the packer's codes must match IEEE fp32 division and rintf.
"""

import hashlib
import os
import platform
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libw4a16.so")
SOURCES = ["common.cu", "pack.cu", "gemv.cu", "attention.cu", "decode.cu", "prefill.cu", "gemm.cu", "container.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr"]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: %s\n%s" % (" ".join(cmd), r.stdout))
    return r.stdout


def build(verbose=False, force=False):
    """Compile and link; returns the path of the shared library."""
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    deps = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC))
    deps.append(os.path.join(os.path.dirname(HERE), "include", "w4a16.h"))
    h = hashlib.sha256(platform.machine().encode())
    for d in deps:
        with open(d, "rb") as f:
            h.update(f.read())
    stamp_path = os.path.join(OUT_DIR, "stamp")
    stamp = h.hexdigest()
    if not force and os.path.exists(LIB) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read().strip() == stamp:
                return LIB

    def compile_one(src):
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        out = _run([nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj])
        if verbose and out.strip():
            print(out)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
