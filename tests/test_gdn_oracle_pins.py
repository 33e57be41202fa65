"""Pins of the Gated DeltaNet scan oracle (oracle.gdn_scan) to results fixed by the mathematics
of the gated delta rule, not by the oracle's own loops.  No GPU.

The rule (gdn_oracle.h; Yang, Kautz & Hatamizadeh, "Gated Delta Networks", with the state
stored key-major): S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T and
o_t = S_t^T q_t.  Each pin below checks one consequence of it:

- no writes (beta = 0): pure decay, S_t = (prod alpha) S_0, o_t = (prod alpha) S_0^T q_t;
- a full write (beta = 1) under a unit key stores the value exactly: S_t^T k_t = v_t;
- orthonormal keys, no decay, full writes: the memory is the sum of outer products k_t v_t^T
  and recalls every stored value;
- random inputs against the dense transition-matrix form computed by numpy matrix products
  (a different computation from the oracle's per-step loops);
- a scan split in two, the second half starting from the first half's state (rounded to fp32,
  the type the state has at the boundary), gives the whole scan's result;
- the state and outputs are jointly linear in (S_0, v): doubling both doubles them exactly.
dk != dv in every pin, so a transposed state or output fails.
"""
import numpy as np

import oracle
import synth


def _bf16(a):
    """bf16 bits of values that bf16 holds exactly."""
    a = np.asarray(a, dtype=np.float32)
    bits = synth.f32_to_bf16(a)
    assert np.array_equal(synth.bf16_to_f32(bits), a), "pin values must be exact in bf16"
    return bits


def _f(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


def _rand_inputs(seed, T, H, dk, dv, zero_state=False):
    return synth.gdn_inputs(seed, T, H, dk, dv, layer=7, zero_state=zero_state)


def test_no_write_is_pure_decay():
    T, H, dk, dv = 12, 2, 16, 8
    q, k, v, alpha, _, s0 = _rand_inputs(1, T, H, dk, dv)
    beta = np.zeros((T, H), dtype=np.float32)
    o, s = oracle.gdn_scan(q, k, v, alpha, beta, s0)
    decay = np.cumprod(alpha.astype(np.float64), axis=0)          # [T][H]
    S0 = s0.astype(np.float64)
    for h in range(H):
        want_o = decay[:, h:h + 1] * (_f(q[:, h, :]) @ S0[h])     # o_t = c_t S0^T q_t
        np.testing.assert_allclose(o[:, h, :], want_o, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(s[h], decay[-1, h] * S0[h], rtol=1e-12, atol=1e-14)


def test_full_write_under_a_unit_key_stores_the_value():
    # k_t: +-1/2 in four coordinates (|k|^2 = 1 exactly), beta = 1, q_t = k_t: after the write,
    # reading with the key returns v_t, whatever alpha and the previous state
    T, H, dk, dv = 10, 3, 16, 8
    rng = np.random.default_rng(5)
    kf = np.zeros((T, H, dk), dtype=np.float32)
    for t in range(T):
        for h in range(H):
            idx = rng.choice(dk, 4, replace=False)
            kf[t, h, idx] = rng.choice([-0.5, 0.5], 4)
    k = _bf16(kf)
    _, _, v, alpha, _, s0 = _rand_inputs(2, T, H, dk, dv)
    beta = np.ones((T, H), dtype=np.float32)
    o, _ = oracle.gdn_scan(k, k, v, alpha, beta, s0)
    np.testing.assert_allclose(o, _f(v), rtol=0, atol=1e-12)


def test_orthonormal_keys_build_an_outer_product_memory():
    # S_0 = 0, alpha = 1, beta = 1, k_t = e_{p(t)} with distinct p(t): S_T = sum_t e_{p(t)} v_t^T,
    # so row p(t) of S_T is v_t and every other row is zero; q_t = e_{p(s)} recalls v_s for
    # s <= t and 0 for a key not yet written
    T, H, dk, dv = 6, 2, 8, 5
    perm = [3, 0, 6, 1, 7, 4]
    kf = np.zeros((T, H, dk), dtype=np.float32)
    qf = np.zeros((T, H, dk), dtype=np.float32)
    recall = [2, 0, 1, 5, 4, 5]          # token t reads key p(recall[t])
    for t in range(T):
        kf[t, :, perm[t]] = 1.0
        qf[t, :, perm[recall[t]]] = 1.0
    _, _, v, _, _, _ = _rand_inputs(3, T, H, dk, dv)
    ones = np.ones((T, H), dtype=np.float32)
    o, s = oracle.gdn_scan(_bf16(qf), _bf16(kf), v, ones, ones, None)
    vf = _f(v)
    for h in range(H):
        want = np.zeros((dk, dv))
        for t in range(T):
            want[perm[t]] = vf[t, h]
        assert np.array_equal(s[h], want)
        for t in range(T):
            exp = vf[recall[t], h] if recall[t] <= t else np.zeros(dv)
            assert np.array_equal(o[t, h], exp)


def test_matches_the_dense_transition_form():
    T, H, dk, dv = 9, 2, 12, 7
    q, k, v, alpha, beta, s0 = _rand_inputs(4, T, H, dk, dv)
    o, s = oracle.gdn_scan(q, k, v, alpha, beta, s0)
    for h in range(H):
        S = s0[h].astype(np.float64)
        for t in range(T):
            kt = _f(k[t, h]).reshape(dk, 1)
            a, b = float(alpha[t, h]), float(beta[t, h])
            A = a * (np.eye(dk) - b * (kt @ kt.T))
            S = A @ S + b * (kt @ _f(v[t, h]).reshape(1, dv))
            np.testing.assert_allclose(o[t, h], S.T @ _f(q[t, h]), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(s[h], S, rtol=1e-10, atol=1e-12)


def test_split_scan_continues():
    T, H, dk, dv = 14, 2, 16, 8
    q, k, v, alpha, beta, s0 = _rand_inputs(5, T, H, dk, dv)
    o, s = oracle.gdn_scan(q, k, v, alpha, beta, s0)
    c = 5
    o1, s1 = oracle.gdn_scan(q[:c], k[:c], v[:c], alpha[:c], beta[:c], s0)
    # the state goes back in as fp32 (the entry point's type): equal up to that rounding
    o2, s2 = oracle.gdn_scan(q[c:], k[c:], v[c:], alpha[c:], beta[c:], s1.astype(np.float32))
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(s2, s, rtol=1e-6, atol=1e-7)
    assert np.array_equal(o1, o[:c])


def test_joint_linearity_in_state_and_values():
    T, H, dk, dv = 11, 2, 16, 8
    q, k, v, alpha, beta, s0 = _rand_inputs(6, T, H, dk, dv)
    o, s = oracle.gdn_scan(q, k, v, alpha, beta, s0)
    v2 = synth.f32_to_bf16(2.0 * synth.bf16_to_f32(v))              # exact: power of two
    o2, s2 = oracle.gdn_scan(q, k, v2, alpha, beta, 2.0 * s0)
    assert np.array_equal(o2, 2.0 * o) and np.array_equal(s2, 2.0 * s)


def test_zero_length_returns_the_initial_state():
    H, dk, dv = 2, 16, 8
    q, k, v, alpha, beta, s0 = _rand_inputs(7, 0, H, dk, dv)
    o, s = oracle.gdn_scan(q, k, v, alpha, beta, s0)
    assert o.shape == (0, H, dv) and np.array_equal(s, s0.astype(np.float64))
