"""Builds sparse_moe_02_gb300/libmoe.so in-tree: every .cu in csrc/ compiled for sm_103a in
parallel, then linked into one shared library with the CUDA runtime linked statically.  Also
links libmoe_debug.so: the same objects with api.cu compiled under MOE_DEBUG (a routing
consistency check inside every moe_route and tensor-core forward, see moe_check_routing)."""
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe.so")
LIB_DEBUG = os.path.join(HERE, "libmoe_debug.so")
SOURCES = ["api.cu", "route.cu", "experts.cu", "decode.cu", "decode_q4.cu", "noalloc.cu", "probe.cu",
           "hostio.cu", "gdn.cu", "check.cu"]
HEADERS = ["layer.cuh", "plan.cuh", "ptx.cuh", "select.cuh", "q4.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + CSRC,
         "-I" + os.path.join(ROOT, "include")]


def _stale():
    if not os.path.exists(LIB) or not os.path.exists(LIB_DEBUG):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(LIB_DEBUG))
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps += [os.path.join(ROOT, "include", h) for h in ("moe.h", "gdn.h")]
    deps += [os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def _compile(src, debug=False):
    obj = os.path.join(OBJ, src.replace(".cu", "_debug.o" if debug else ".o"))
    defs = ["-DMOE_DEBUG"] if debug else []
    subprocess.run(["nvcc", *FLAGS, *defs, *ARCH, "-c", os.path.join(CSRC, src), "-o", obj],
                   check=True)
    return obj


def build(force=False):
    if not force and not _stale():
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES) + 1) as ex:
        futs = [ex.submit(_compile, src) for src in SOURCES]
        dbg = ex.submit(_compile, "api.cu", True)
        objs = [f.result() for f in futs]
        api_dbg = dbg.result()
    for out, objects in ((LIB, objs), (LIB_DEBUG, [api_dbg if o.endswith("/api.o") else o
                                                   for o in objs])):
        subprocess.run(["nvcc", "-shared", *ARCH, "-cudart", "static", "-o", out + ".tmp",
                        *objects], check=True)
        os.replace(out + ".tmp", out)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
