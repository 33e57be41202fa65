"""Pins of the CPU oracle to facts fixed by the mathematics and by hand computation.

Source of the method: "Optimizing on-device inference for Apple Silicon" -- the router keeps
the top eight of 256 experts plus a shared expert (section "three distinct workload shapes");
histogram, prefix scan and scatter into expert groups (section "Keep expert routing on the
GPU"); gated activation and weighted output projection plus the shared expert's result
(section "Reduce intermediate and state traffic").

Each test pins one part against something other than the oracle's own formula: a brute force
(full sort, subset enumeration, stable argsort), a closed form (full softmax renormalised,
silu constants), a special case that reduces to a textbook dense SwiGLU FFN computed by
numpy in float64, an exact hand-computed case, and exact scaling laws.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def bf16(a):
    """float values -> bf16 bits, asserting the values are exactly representable."""
    a = np.asarray(a, dtype=np.float32)
    b = synth.f32_to_bf16(a)
    assert np.array_equal(synth.bf16_to_f32(b), a), "fixture value is not a bf16 number"
    return b


def rand_bf16(shape, sigma):
    return synth.f32_to_bf16(rng.normal(0.0, sigma, size=shape).astype(np.float32))


def f32(b):
    return synth.bf16_to_f32(b).astype(np.float64)


def dense_swiglu(x, wg, wu, wd):
    """Textbook dense SwiGLU FFN in float64 (numpy matmuls): (silu(x Wg^T) * (x Wu^T)) Wd^T."""
    g = f32(x) @ f32(wg).T
    u = f32(x) @ f32(wu).T
    h = g / (1.0 + np.exp(-g)) * u
    return h @ f32(wd).T


# ---------------------------------------------------------------- selection and weights

def _top_k_by_sort(l, k):
    order = sorted(range(len(l)), key=lambda e: (-float(l[e]), e))
    return sorted(order[:k])


def test_select_matches_full_sort_random_and_ties():
    for logits in (rng.normal(0, 2.26, size=(200, 256)).astype(np.float32),
                   rng.integers(0, 4, size=(200, 256)).astype(np.float32),  # many ties
                   np.zeros((3, 256), dtype=np.float32)):
        idx, _ = oracle.select(logits, 8)
        for t in range(logits.shape[0]):
            assert list(idx[t]) == _top_k_by_sort(logits[t], 8)


def test_select_is_max_sum_subset_by_enumeration():
    # E=16, k=8: the kept set is the unique subset of 8 with the largest logit sum
    for _ in range(10):
        l = rng.permutation(np.arange(16, dtype=np.float32) * 0.37 - 2.0)
        best = max(itertools.combinations(range(16), 8), key=lambda s: sum(float(l[e]) for e in s))
        idx, _ = oracle.select(l[None, :], 8)
        assert tuple(idx[0]) == tuple(sorted(best))


def test_weights_equal_full_softmax_renormalised():
    logits = rng.normal(0, 2.26, size=(300, 256)).astype(np.float32)
    idx, w = oracle.select(logits, 8)
    l64 = logits.astype(np.float64)
    full = np.exp(l64 - l64.max(axis=1, keepdims=True))
    full /= full.sum(axis=1, keepdims=True)
    kept = np.take_along_axis(full, idx.astype(np.int64), axis=1)
    ref = kept / kept.sum(axis=1, keepdims=True)
    assert np.max(np.abs(w - ref)) <= 1e-6
    assert np.max(np.abs(w.astype(np.float64).sum(axis=1) - 1.0)) <= 1e-6
    assert np.all(w > 0) and np.all(w <= 1)
    assert np.all(np.diff(idx, axis=1) > 0)  # ascending expert id


# ---------------------------------------------------------------- router logits

def test_router_logits_match_float64_matmul():
    x = rand_bf16((37, 128), 1.0)
    w_r = rand_bf16((256, 128), 0.05)
    bias = rng.normal(0, 1, size=256).astype(np.float32)
    ref = f32(x) @ f32(w_r).T + bias.astype(np.float64)
    l64 = oracle.router_logits_f64(x, w_r, bias)
    l32 = oracle.router_logits_f32(x, w_r, bias)
    assert np.max(np.abs(l64 - ref)) <= 1e-9
    assert np.max(np.abs(l32 - ref)) <= 1e-4


def test_route_selection_matches_numpy_when_gap_holds():
    x = rand_bf16((64, 512), 1.0)
    w_r = rand_bf16((256, 512), 0.05)
    ref = f32(x) @ f32(w_r).T
    gap = oracle.kth_gap(ref, 8)
    r = oracle.route(x, w_r, 8)
    for t in np.nonzero(gap >= 1e-3)[0]:
        assert list(r["topk_idx"][t]) == _top_k_by_sort(ref[t], 8)


# ---------------------------------------------------------------- routing structure

def test_route_structure_invariants_and_stable_sort():
    T, E, k = 300, 256, 8
    x = rand_bf16((T, 64), 1.0)
    w_r = rand_bf16((E, 64), 0.3)
    r = oracle.route(x, w_r, k)
    idx, counts, offsets, perm, inv = (r["topk_idx"], r["counts"], r["offsets"], r["perm"],
                                       r["inv_perm"])
    assert counts.sum() == T * k
    assert offsets[0] == 0 and offsets[E] == T * k and np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(perm), np.arange(T * k))
    assert np.array_equal(perm[inv], np.arange(T * k))  # inv_perm o perm = id
    flat = idx.reshape(-1)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg // k) > 0)  # tokens strictly ascending in a group
    # the stable sort of the assignments by expert id is the same permutation
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))


def test_route_structure_empty_input():
    counts, offsets, perm, inv = oracle.route_structure(np.zeros((0, 8), dtype=np.int32), 256)
    assert counts.sum() == 0 and offsets[-1] == 0 and perm.size == 0


# ---------------------------------------------------------------- expert FFN and combine

def test_silu_closed_form():
    cases = json.load(open(os.path.join(GOLDEN, "silu_closed_form.json")))["cases"]
    for c in cases:
        h, o = oracle.expert_ffn(bf16([1.0]), bf16([[c["g"]]]), bf16([[c["u"]]]), bf16([[1.0]]))
        assert abs(h[0] - c["h"]) <= 1e-6 * max(1.0, abs(c["h"])), c
        assert o[0] == h[0]


def _random_layer(d=64, E=16, f=32, fs=48):
    return dict(w_gate=rand_bf16((E, f, d), 0.1), w_up=rand_bf16((E, f, d), 0.1),
                w_down=rand_bf16((E, d, f), 0.1), ws_gate=rand_bf16((fs, d), 0.1),
                ws_up=rand_bf16((fs, d), 0.1), ws_down=rand_bf16((d, fs), 0.1))


def _forward(L, x, w_r, bias, k):
    return oracle.forward(x, w_r, bias, (L["w_gate"], L["w_up"], L["w_down"]),
                          (L["ws_gate"], L["ws_up"], L["ws_down"]), k)


def _assert_bf16_close(y_bits, ref):
    y = f32(y_bits)
    # one bf16 rounding of an fp32 sum: |err| <= 2^-8 |ref| plus fp32 accumulation slack
    assert np.all(np.abs(y - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * (1 + np.abs(ref).max()))


def test_one_hot_router_reduces_to_dense_swiglu():
    d, E, k = 64, 16, 4
    L = _random_layer(d, E)
    x = rand_bf16((9, d), 1.0)
    w_r = np.zeros((E, d), dtype=np.uint16)
    for j in (0, 5, 15):
        bias = np.zeros(E, dtype=np.float32)
        bias[j] = 100.0
        y, idx, w = _forward(L, x, w_r, bias, k)
        assert np.all(np.any(idx == j, axis=1))
        ref = dense_swiglu(x, L["w_gate"][j], L["w_up"][j], L["w_down"][j]) + \
            dense_swiglu(x, L["ws_gate"], L["ws_up"], L["ws_down"])
        _assert_bf16_close(y, ref)
    # shared expert zeroed: the layer is one dense SwiGLU FFN
    L0 = dict(L, ws_gate=np.zeros_like(L["ws_gate"]), ws_up=np.zeros_like(L["ws_up"]),
              ws_down=np.zeros_like(L["ws_down"]))
    bias = np.zeros(E, dtype=np.float32)
    bias[7] = 100.0
    y, _, _ = _forward(L0, x, w_r, bias, k)
    _assert_bf16_close(y, dense_swiglu(x, L["w_gate"][7], L["w_up"][7], L["w_down"][7]))


def test_two_hot_router_weights_each_expert_by_its_score():
    # logits 100 and 100 + ln 3 dominate: weights 1/4 and 3/4 on the right experts
    d, E, k = 64, 16, 4
    L = _random_layer(d, E)
    x = rand_bf16((5, d), 1.0)
    w_r = np.zeros((E, d), dtype=np.uint16)
    bias = np.zeros(E, dtype=np.float32)
    bias[2], bias[11] = 100.0, np.float32(100.0 + math.log(3.0))
    y, idx, w = _forward(L, x, w_r, bias, k)
    wm = {int(e): float(v) for e, v in zip(idx[0], w[0])}
    assert abs(wm[2] - 0.25) < 2e-6 and abs(wm[11] - 0.75) < 2e-6
    ref = 0.25 * dense_swiglu(x, L["w_gate"][2], L["w_up"][2], L["w_down"][2]) + \
        0.75 * dense_swiglu(x, L["w_gate"][11], L["w_up"][11], L["w_down"][11]) + \
        dense_swiglu(x, L["ws_gate"], L["ws_up"], L["ws_down"])
    _assert_bf16_close(y, ref)


def test_exact_small_case_bit_exact():
    G = json.load(open(os.path.join(GOLDEN, "exact_small_case.json")))
    D = G["dims"]
    E, d, f = D["E"], D["d"], D["f"]
    wg = np.zeros((E, f, d), dtype=np.float32)
    wu = np.zeros((E, f, d), dtype=np.float32)
    wd = np.zeros((E, d, f), dtype=np.float32)
    for e in range(E):
        wg[e] = wu[e] = (e + 1) / 8.0
        wd[e] = (e + 1) / 8.0
    for e, m in G["experts"].items():
        wg[int(e)], wu[int(e)], wd[int(e)] = m["w_gate"], m["w_up"], m["w_down"]
    S = G["shared"]
    y, idx, w = oracle.forward(bf16(G["x"]), bf16(G["w_r"]), None,
                               (bf16(wg), bf16(wu), bf16(wd)),
                               (bf16(S["w_gate"]), bf16(S["w_up"]), bf16(S["w_down"])), D["k"])
    assert idx.tolist() == G["expected"]["topk_idx"]
    assert w.tolist() == G["expected"]["topk_w"]
    assert np.array_equal(y, bf16(G["expected"]["y"]))


def test_scaling_down_projections_by_two_doubles_output_exactly():
    d, E, k = 64, 16, 4
    L = _random_layer(d, E)
    x = rand_bf16((11, d), 1.0)
    w_r = rand_bf16((E, d), 0.3)
    y1, _, _ = _forward(L, x, w_r, None, k)
    dbl = lambda b: bf16(2.0 * synth.bf16_to_f32(b))
    L2 = dict(L, w_down=dbl(L["w_down"]), ws_down=dbl(L["ws_down"]))
    y2, _, _ = _forward(L2, x, w_r, None, k)
    assert np.array_equal(synth.bf16_to_f32(y2), 2.0 * synth.bf16_to_f32(y1))


def test_relabelling_experts_leaves_output_unchanged():
    d, E, k = 64, 16, 4
    L = _random_layer(d, E)
    x = rand_bf16((11, d), 1.0)
    w_r = rand_bf16((E, d), 0.3)
    y1, idx1, w1 = _forward(L, x, w_r, None, k)
    pi = rng.permutation(E)  # new id of old expert e is pi[e]
    inv = np.argsort(pi)
    Lp = dict(L, w_gate=L["w_gate"][inv], w_up=L["w_up"][inv], w_down=L["w_down"][inv])
    y2, idx2, w2 = _forward(Lp, x, w_r[inv], None, k)
    for t in range(x.shape[0]):
        assert sorted(pi[idx1[t]].tolist()) == idx2[t].tolist()
        a = dict(zip(pi[idx1[t]].tolist(), w1[t].tolist()))
        b = dict(zip(idx2[t].tolist(), w2[t].tolist()))
        assert all(abs(a[e] - b[e]) < 1e-6 for e in a)
    # only the fp32 summation order of the routed terms changes
    assert np.all(np.abs(f32(y1) - f32(y2)) <= 2.0 ** -7 * np.abs(f32(y1)) + 1e-4)


def test_forward_sample_and_threads_are_invariant():
    d, E, k = 64, 16, 4
    L = _random_layer(d, E)
    x = rand_bf16((40, d), 1.0)
    w_r = rand_bf16((E, d), 0.3)
    y_all, idx_all, _ = oracle.forward(x, w_r, None, (L["w_gate"], L["w_up"], L["w_down"]),
                                       (L["ws_gate"], L["ws_up"], L["ws_down"]), k, nthreads=1)
    y_thr, _, _ = oracle.forward(x, w_r, None, (L["w_gate"], L["w_up"], L["w_down"]),
                                 (L["ws_gate"], L["ws_up"], L["ws_down"]), k, nthreads=5)
    assert np.array_equal(y_all, y_thr)
    toks = np.array([39, 0, 17])
    experts = {int(e): (L["w_gate"][e], L["w_up"][e], L["w_down"][e])
               for e in np.unique(idx_all[toks])}
    y_s, idx_s, _ = oracle.forward(x, w_r, None, experts, (L["ws_gate"], L["ws_up"],
                                                           L["ws_down"]), k, tokens=toks)
    assert np.array_equal(y_s, y_all[toks]) and np.array_equal(idx_s, idx_all[toks])
    with pytest.raises(ValueError):  # an expert the tokens need is missing
        oracle.forward(x, w_r, None, {}, (L["ws_gate"], L["ws_up"], L["ws_down"]), k,
                       tokens=toks)


def test_route_matches_forward_selection():
    d, E, k = 64, 16, 4
    L = _random_layer(d, E)
    x = rand_bf16((20, d), 1.0)
    w_r = rand_bf16((E, d), 0.3)
    _, idx, w = _forward(L, x, w_r, None, k)
    r = oracle.route(x, w_r, k)
    assert np.array_equal(idx, r["topk_idx"]) and np.array_equal(w, r["topk_w"])


# ---------------------------------------------------------------- input drawing rule

def test_gap_rule_redraws_and_is_reproducible():
    d, E, k = 512, 256, 8
    w_r = synth.host_weight(0, 0, "w_r", synth.Dims(d=d, f=128, fs=128))
    x, rounds, redraws = oracle.draw_x_with_gap(0, 0, 64, d, [(w_r, None)], k)
    assert np.all(oracle.kth_gap(oracle.router_logits_f64(x, w_r), k) >= 1e-3)
    assert redraws == int(rounds.sum())
    assert np.array_equal(x, synth.x_rows(0, 0, 64, d, rounds))


# ---------------------------------------------------------------- 4-bit group-affine weights
# Pinned through the encoding direction: integer weights v in [-8, 7] and per-group scales
# are packed here into codes (v + 8, two per byte, the lower nibble first) and bf16 scales and
# biases (bias = -8 * scale); dequantizing must give v * scale back, and with power-of-two
# scales (v * scale exact in bf16) the whole 4-bit layer must equal, bit for bit, the bf16
# layer on those weights -- whose own pins are above.

def _encode_q4(v, scales_f32, biases_f32=None):
    """v int [rows][K] in [-8, 7]; scales [rows][K/64] -> (codes, scale bits, bias bits)."""
    q = (np.asarray(v, dtype=np.int64) + 8).astype(np.uint8)
    codes = (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    s = synth.f32_to_bf16(np.asarray(scales_f32, dtype=np.float32))
    if biases_f32 is None:
        b = synth.f32_to_bf16(-8.0 * synth.bf16_to_f32(s))
    else:
        b = synth.f32_to_bf16(np.asarray(biases_f32, dtype=np.float32))
    return codes, s, b


def _pow2_scales(rng, shape):
    return np.ldexp(1.0, -rng.integers(6, 10, size=shape)).astype(np.float32)


def test_q4_dequant_roundtrip():
    rng = np.random.default_rng(11)
    v = rng.integers(-8, 8, size=(5, 256))
    s = _pow2_scales(rng, (5, 4))
    got = oracle.dequant_q4(*_encode_q4(v, s))
    assert np.array_equal(got, (v * np.repeat(s, 64, axis=1)).astype(np.float32))
    # general biases: scale*q + bias within one fp32 rounding of the exact value
    sc = rng.uniform(0.003, 0.006, size=(5, 4)).astype(np.float32)
    bi = rng.uniform(-0.05, 0.05, size=(5, 4)).astype(np.float32)
    codes, sb, bb = _encode_q4(v, sc, bi)
    exact = (np.repeat(synth.bf16_to_f32(sb), 64, 1).astype(np.float64) * (v + 8) +
             np.repeat(synth.bf16_to_f32(bb), 64, 1).astype(np.float64))
    got = oracle.dequant_q4(codes, sb, bb).astype(np.float64)
    assert np.max(np.abs(got - exact)) <= 2.0 ** -22 * np.max(np.abs(exact))


def test_q4_layer_equals_bf16_layer_on_its_weights():
    rng = np.random.default_rng(12)
    d, E, f, fs, k, T = 128, 16, 64, 128, 4, 7
    x = synth.f32_to_bf16(rng.standard_normal((T, d)).astype(np.float32))
    w_r = synth.f32_to_bf16((0.2 * rng.standard_normal((E, d))).astype(np.float32))

    def mat(rows, K):
        v = rng.integers(-8, 8, size=(rows, K))
        s = _pow2_scales(rng, (rows, K // 64))
        w = synth.f32_to_bf16((v * np.repeat(s, 64, axis=1)).astype(np.float32))
        return _encode_q4(v, s), w

    experts_q4, experts_bf = {}, ([], [], [])
    for e in range(E):
        g, u, dn = mat(f, d), mat(f, d), mat(d, f)
        experts_q4[e] = (g[0], u[0], dn[0])
        for i, m in enumerate((g, u, dn)):
            experts_bf[i].append(m[1])
    sg, su, sd = mat(fs, d), mat(fs, d), mat(d, fs)
    yq, iq, wq = oracle.forward_q4(x, w_r, None, experts_q4, (sg[0], su[0], sd[0]), k)
    yb, ib, wb = oracle.forward(x, w_r, None, tuple(np.stack(a) for a in experts_bf),
                                (sg[1], su[1], sd[1]), k)
    assert np.array_equal(iq, ib) and np.array_equal(wq, wb)
    assert np.array_equal(yq, yb)
