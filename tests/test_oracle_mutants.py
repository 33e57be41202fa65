"""Each plausible mistake planted in a copy of the CPU oracles must fail at least one pin.

The mutant is built from a textually edited copy of the oracle's sources (oracle/moe_oracle.cpp
for the MoE layer, oracle/gdn_oracle.cpp for the Gated DeltaNet scan) in a temporary
directory, loaded through ORACLE_LIB, and the pin suite of that oracle (tests/test_oracle_pins.py
or tests/test_gdn_oracle_pins.py) is run against it in a subprocess; the suite must fail.
Nothing here touches a GPU.
"""
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_DIR = os.path.join(ROOT, "oracle")
SOURCES = ("moe_oracle.cpp", "gdn_oracle.cpp")
HEADERS = ("moe_oracle.h", "gdn_oracle.h")

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


# Gated DeltaNet scan oracle: (name, text to replace, replacement)
GDN_MUTANTS = [
    ("gdn_delta_sign", "u[j] = b * (vt[j] - r[j]);", "u[j] = b * (vt[j] + r[j]);"),
    ("gdn_beta_dropped", "u[j] = b * (vt[j] - r[j]);", "u[j] = (vt[j] - r[j]);"),
    ("gdn_retrieve_before_decay",
     "    // decay\n    for (int i = 0; i < dk; ++i)\n      for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] *= a;\n    // retrieve: r = S^T k\n    for (int j = 0; j < dv; ++j) {\n      double acc = 0.0;\n      for (int i = 0; i < dk; ++i) acc += S[(int64_t)i * dv + j] * kt[i];\n      r[j] = acc;\n    }",
     "    // retrieve: r = S^T k\n    for (int j = 0; j < dv; ++j) {\n      double acc = 0.0;\n      for (int i = 0; i < dk; ++i) acc += S[(int64_t)i * dv + j] * kt[i];\n      r[j] = acc;\n    }\n    // decay\n    for (int i = 0; i < dk; ++i)\n      for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] *= a;"),
    ("gdn_retrieve_with_query", "acc += S[(int64_t)i * dv + j] * kt[i];\n      r[j] = acc;",
     "acc += S[(int64_t)i * dv + j] * qt[i];\n      r[j] = acc;"),
    ("gdn_read_with_key", "acc += S[(int64_t)i * dv + j] * qt[i];\n      o[row * dv + j] = acc;",
     "acc += S[(int64_t)i * dv + j] * kt[i];\n      o[row * dv + j] = acc;"),
    ("gdn_write_transposed", "S[(int64_t)i * dv + j] += kt[i] * u[j];",
     "S[(int64_t)i * dv + j] += kt[j % dk] * u[i % dv];"),
    ("gdn_decay_squared", "S[(int64_t)i * dv + j] *= a;", "S[(int64_t)i * dv + j] *= a * a;"),
    ("gdn_q_k_swapped_on_load", "kt[i] = widen_bf16(k[row * dk + i]);\n      qt[i] = widen_bf16(q[row * dk + i]);",
     "kt[i] = widen_bf16(q[row * dk + i]);\n      qt[i] = widen_bf16(k[row * dk + i]);"),
    ("gdn_state_not_carried", "for (int64_t e = 0; e < (int64_t)H * per; ++e) s_out[e] = s0 ? (double)s0[e] : 0.0;",
     "for (int64_t e = 0; e < (int64_t)H * per; ++e) s_out[e] = 0.0;"),
]


def _run_pins_against(target, old, new, pins):
    """Builds the oracle with `old` replaced by `new` in source `target` (no replacement when
    target is None) and returns the pin suite's exit code and output."""
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        for h in HEADERS:
            shutil.copy(os.path.join(ORACLE_DIR, h), tmp)
        for src in SOURCES:
            text = open(os.path.join(ORACLE_DIR, src)).read()
            if src == target:
                assert text.count(old) == 1, f"mutation anchor not found exactly once in {src}"
                text = text.replace(old, new)
            with open(os.path.join(tmp, src), "w") as fh:
                fh.write(text)
        lib = os.path.join(tmp, "liboracle_mutant.so")
        subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
                        "-pthread", "-o", lib] + [os.path.join(tmp, s) for s in SOURCES],
                       check=True)
        env = dict(os.environ, ORACLE_LIB=lib)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", pins)],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        return r.returncode, r.stdout
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, old, new):
    rc, out = _run_pins_against("moe_oracle.cpp", old, new, "test_oracle_pins.py")
    assert rc != 0, f"mutant {name} passed every pin:\n{out[-2000:]}"


@pytest.mark.parametrize("name,old,new", GDN_MUTANTS, ids=[m[0] for m in GDN_MUTANTS])
def test_planted_scan_mistake_fails_a_pin(name, old, new):
    rc, out = _run_pins_against("gdn_oracle.cpp", old, new, "test_gdn_oracle_pins.py")
    assert rc != 0, f"mutant {name} passed every pin:\n{out[-2000:]}"


@pytest.mark.parametrize("pins", ["test_oracle_pins.py", "test_gdn_oracle_pins.py"])
def test_unmutated_copy_passes_every_pin(pins):
    # control: the same build-and-load route with no mutation must pass, so that the
    # failures above come from the planted mistakes
    rc, out = _run_pins_against(None, None, None, pins)
    assert rc == 0, out[-2000:]
