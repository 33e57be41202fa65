"""Builds libsynth.so (host generator + device fill) in this directory with nvcc."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libsynth.so")
SOURCES = ["synth_host.c", "synth_dev.cu"]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(os.path.join(HERE, s)) > t
               for s in SOURCES + ["synth.h", "build.py"])


def build(force=False):
    if not force and not _stale():
        return LIB
    cmd = ["nvcc", "-O2", "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
           "-gencode", "arch=compute_103a,code=sm_103a", "-o", LIB + ".tmp"]
    cmd += [os.path.join(HERE, s) for s in SOURCES] + ["-lpthread"]
    subprocess.run(cmd, check=True, cwd=HERE)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
