"""Builds liboracle.so (the CPU oracles of the MoE layer and of the Gated DeltaNet scan, test
infrastructure) in this directory with g++."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "liboracle.so")
SOURCES = ["moe_oracle.cpp", "gdn_oracle.cpp"]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(os.path.join(HERE, s)) > t
               for s in SOURCES + ["moe_oracle.h", "gdn_oracle.h", "build.py"])


def build(force=False):
    if not force and not _stale():
        return LIB
    # no fast-math and no FMA contraction: the same bits on every host
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-pthread", "-o", LIB + ".tmp"] + [os.path.join(HERE, s) for s in SOURCES]
    subprocess.run(cmd, check=True, cwd=HERE)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
