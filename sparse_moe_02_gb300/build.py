"""Builds sparse_moe_02_gb300/libmoe.so in-tree: every .cu in csrc/ compiled for sm_103a in
parallel, then linked into one shared library with the CUDA runtime linked statically."""
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe.so")
SOURCES = ["api.cu", "route.cu", "experts.cu", "decode.cu", "decode_q4.cu", "noalloc.cu", "probe.cu",
           "hostio.cu", "gdn.cu"]
HEADERS = ["layer.cuh", "plan.cuh", "ptx.cuh", "select.cuh", "q4.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + CSRC,
         "-I" + os.path.join(ROOT, "include")]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps += [os.path.join(ROOT, "include", h) for h in ("moe.h", "gdn.h")]
    deps += [os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def _compile(src):
    obj = os.path.join(OBJ, src.replace(".cu", ".o"))
    subprocess.run(["nvcc", *FLAGS, *ARCH, "-c", os.path.join(CSRC, src), "-o", obj], check=True)
    return obj


def build(force=False):
    if not force and not _stale():
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    subprocess.run(["nvcc", "-shared", *ARCH, "-cudart", "static", "-o", LIB + ".tmp", *objs],
                   check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
