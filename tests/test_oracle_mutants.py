"""Each plausible mistake planted in a copy of the CPU oracle must fail at least one pin.

The mutant is built from a textually edited copy of oracle/moe_oracle.cpp in a temporary
directory, loaded through ORACLE_LIB, and the pin suite (tests/test_oracle_pins.py) is run
against it in a subprocess; the suite must fail.  Nothing here touches a GPU.
"""
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.cpp")

# (name, text to replace, replacement)
MUTANTS = [
    ("silu_sign", "(g / (1.0f + std::exp(-g)))", "(g / (1.0f + std::exp(g)))"),
    ("gate_up_swapped", "return (g / (1.0f + std::exp(-g))) * u;", "return (u / (1.0f + std::exp(-u))) * g;"),
    ("softmax_sign", "ex[j] = std::exp(l[kept[j]] - m);", "ex[j] = std::exp(m - l[kept[j]]);"),
    ("ties_to_higher_id", "order[e] = {-l[e], e};", "order[e] = {-l[e], -e};"),
    ("bias_dropped", "out[e] = acc + (bias ? bias[e] : 0.0f);", "out[e] = acc;"),
    ("router_transposed", "const uint16_t* wr = w_r + (int64_t)e * d;\n    float acc = 0.0f;\n    for (int i = 0; i < d; ++i) acc += widen(xr[i]) * widen(wr[i]);",
     "float acc = 0.0f;\n    for (int i = 0; i < d; ++i) acc += widen(xr[i]) * widen(w_r[(int64_t)i * E + e]);"),
    ("down_transposed", "for (int c = 0; c < f; ++c) acc += h[c] * wd(n, c);",
     "for (int c = 0; c < f; ++c) acc += h[c] * wd(c, n);"),
    # 4-bit weights: nibble order, group index, the bias term
    ("q4_nibbles_swapped", "const int q = (i & 1) ? (b >> 4) : (b & 15);",
     "const int q = (i & 1) ? (b & 15) : (b >> 4);"),
    ("q4_group_of_32", "const int64_t g = r * (K / 64) + i / 64;",
     "const int64_t g = r * (K / 64) + (i / 32) % (K / 64);"),
    ("q4_bias_dropped", "return widen(m.scales[g]) * (float)q + widen(m.biases[g]);",
     "return widen(m.scales[g]) * (float)q;"),
    ("shared_dropped", "for (int n = 0; n < d; ++n) acc[n] += o[n];", "for (int n = 0; n < d; ++n) acc[n] += 0.0f * o[n];"),
    ("weight_misaligned", "acc[n] += w[j] * o[n];", "acc[n] += w[(j + 1) % k] * o[n];"),
    ("round_truncates", "u += 0x7FFFu + lsb;", "(void)lsb;"),
    ("round_half_up", "u += 0x7FFFu + lsb;", "u += 0x8000u + 0 * lsb;"),
    ("tokens_descending", "for (int64_t t = 0; t < T; ++t)\n      for (int j = 0; j < k; ++j)\n        if (topk_idx[t * k + j] == e) {",
     "for (int64_t t = T - 1; t >= 0; --t)\n      for (int j = 0; j < k; ++j)\n        if (topk_idx[t * k + j] == e) {"),
    ("offsets_inclusive", "offsets[e + 1] = offsets[e] + counts[e];", "offsets[e + 1] = offsets[e] + counts[e] + (e == 0);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        shutil.copy(os.path.join(ROOT, "oracle", "moe_oracle.h"), tmp)
        with open(os.path.join(tmp, "moe_oracle.cpp"), "w") as fh:
            fh.write(src.replace(old, new))
        lib = os.path.join(tmp, "liboracle_mutant.so")
        subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
                        "-pthread", "-o", lib, os.path.join(tmp, "moe_oracle.cpp")], check=True)
        env = dict(os.environ, ORACLE_LIB=lib)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_unmutated_copy_passes_every_pin():
    # control: the same build-and-load route with no mutation must pass, so that the
    # failures above come from the planted mistakes
    tmp = tempfile.mkdtemp(prefix="oracle_copy_")
    try:
        shutil.copy(os.path.join(ROOT, "oracle", "moe_oracle.h"), tmp)
        shutil.copy(SRC, tmp)
        lib = os.path.join(tmp, "liboracle_copy.so")
        subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
                        "-pthread", "-o", lib, os.path.join(tmp, "moe_oracle.cpp")], check=True)
        env = dict(os.environ, ORACLE_LIB=lib)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stdout[-2000:]
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
