"""Pins of the input-side helpers that shape the synthetic workloads.

- oracle.kth_gap: the gap between the k-th and (k+1)-th largest logit of a row, checked on
  hand-built rows whose sorted order and gaps are written out below.
- oracle.draw_x_with_gap: every row it returns passes the 1e-3 gap rule when the gap is
  recomputed independently (fp64 dot products in a plain Python loop, Python's sorted()),
  and every redrawn row equals the generator's row of its redraw round.
- synth.skew_bias: the skewed-routing bias b_e = 2 ln(1 / rank_e^1.2) of the prefill
  configuration, checked at ranks 1, 2 and 256 against the closed form (the rank of expert
  perm[i] is i + 1 for the seeded permutation perm), and as a whole against math.log.
"""
import math

import numpy as np

import oracle
import synth


def test_kth_gap_hand_built_rows():
    # sorted: 3, 3, 2, 1.25, 0.5, -1  -> gaps k=1: 0, k=2: 1, k=3: 0.75, k=5: 1.5
    r0 = np.array([[0.5, 3.0, 1.25, 3.0, -1.0, 2.0]], dtype=np.float64)
    assert oracle.kth_gap(r0, 1)[0] == 0.0
    assert oracle.kth_gap(r0, 2)[0] == 1.0
    assert oracle.kth_gap(r0, 3)[0] == 0.75
    assert oracle.kth_gap(r0, 5)[0] == 1.5
    # sorted: 9, 7, 6, 4, 4, 1, 0, -2 -> gaps k=1: 2, k=2: 1, k=3: 2, k=4: 0, k=5: 3
    r1 = np.array([[4.0, -2.0, 9.0, 0.0, 6.0, 1.0, 7.0, 4.0]], dtype=np.float64)
    assert oracle.kth_gap(r1, 1)[0] == 2.0
    assert oracle.kth_gap(r1, 2)[0] == 1.0
    assert oracle.kth_gap(r1, 3)[0] == 2.0
    assert oracle.kth_gap(r1, 4)[0] == 0.0   # the two 4s
    assert oracle.kth_gap(r1, 5)[0] == 3.0
    # rows are independent and the result has one entry per row
    both = np.concatenate([np.pad(r0, ((0, 0), (0, 2)), constant_values=-5.0), r1])
    assert np.array_equal(oracle.kth_gap(both, 2), np.array([1.0, 1.0]))


def _gap_plain(x_bits_row, w_r_bits, bias, k):
    """k-th minus (k+1)-th largest fp64 logit of one token, by plain loops."""
    x = synth.bf16_to_f32(x_bits_row).astype(np.float64).tolist()
    logits = []
    for e in range(w_r_bits.shape[0]):
        w = synth.bf16_to_f32(w_r_bits[e]).astype(np.float64).tolist()
        s = 0.0
        for a, b in zip(x, w):
            s += a * b
        logits.append(s + (float(bias[e]) if bias is not None else 0.0))
    srt = sorted(logits, reverse=True)
    return srt[k - 1] - srt[k]


def test_draw_x_with_gap_meets_the_rule_and_redraws_from_the_generator():
    dims = synth.Dims(d=128, E=16, k=8, f=128, fs=128)
    w_r = synth.host_weight(3, 0, "w_r", dims)
    bias = synth.skew_bias(3, 0, dims.E)
    T = 24
    # a large minimum gap forces redraws on this small router
    x, rounds, redraws = oracle.draw_x_with_gap(3, 0, T, dims.d, [(w_r, bias)], dims.k,
                                                min_gap=0.05)
    assert redraws > 0 and redraws == int(rounds.sum())
    for t in range(T):
        assert _gap_plain(x[t], w_r, bias, dims.k) >= 0.05 - 1e-12
        # the row is the generator's row t of its redraw round
        want = synth.normal_bf16(3, synth.stream_id(synth.X, 0, int(rounds[t])), t * dims.d,
                                 dims.d, synth.SIGMA_X)
        assert np.array_equal(x[t], want)
    # rows never redrawn are the plain first-round rows
    first = synth.x_rows(3, 0, T, dims.d)
    for t in np.flatnonzero(rounds == 0):
        assert np.array_equal(x[t], first[t])


def test_skew_bias_closed_form_at_ranks_1_2_256():
    E = 256
    for seed, layer in ((0, 0), (7, 3)):
        b = synth.skew_bias(seed, layer, E)
        perm = synth.permutation(seed, synth.stream_id(synth.RANKS, layer), E)
        assert sorted(perm.tolist()) == list(range(E))          # a permutation of the experts
        # rank of expert perm[i] is i + 1; b = 2 ln(1 / rank^1.2)
        assert b[perm[0]] == 0.0                                 # rank 1
        assert abs(b[perm[1]] - 2.0 * math.log(1.0 / 2 ** 1.2)) <= 1e-6   # rank 2: -1.6636
        assert abs(b[perm[1]] + 1.6635532333438687) <= 1e-6
        assert abs(b[perm[255]] - 2.0 * math.log(1.0 / 256 ** 1.2)) <= 1e-5  # rank 256
        assert abs(b[perm[255]] + 13.308425866750948) <= 1e-5
        for i in range(E):
            assert abs(float(b[perm[i]]) - 2.0 * math.log((i + 1) ** -1.2)) <= 1e-5
        # larger rank, smaller bias
        assert np.all(np.diff(b[perm]) < 0)
