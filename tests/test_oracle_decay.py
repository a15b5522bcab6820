"""Pins for the exponentially decayed masked operator in the fp64 oracle.

Reading (HLA summary, section 4 names decayed operators without their form):
one scalar gamma decays every prefix moment per token, so that
    o_t = sum_{i<=j<=t} gamma^{2t-i-j} (q_t.k_i)(k_i.q_j) v_j,
normalised by the same sum without v.  gamma = 1 is the masked operator.
"""
import numpy as np
import pytest

import oracle


def rel(a, b):
    return float(np.abs(np.asarray(a) - np.asarray(b)).max() / max(np.abs(np.asarray(b)).max(), 1e-300))


def rand_inputs(rng, BH, T, d, dv, positive=False):
    f = rng.random if positive else rng.standard_normal
    return f((BH, T, d)) / np.sqrt(d), f((BH, T, d)) / np.sqrt(d), rng.standard_normal((BH, T, dv))


@pytest.mark.parametrize("gamma", [0.97, 0.8, 0.3])
@pytest.mark.parametrize("BH,T,d,dv", [(1, 40, 6, 6), (2, 7, 1, 3), (1, 1, 4, 4), (3, 20, 5, 2)])
def test_serial_equals_bruteforce(BH, T, d, dv, gamma):
    rng = np.random.default_rng(400 + T)
    Q, K, V = rand_inputs(rng, BH, T, d, dv)
    assert rel(oracle.decay_serial(Q, K, V, gamma), oracle.decay_bruteforce(Q, K, V, gamma)) < 1e-12
    Q, K, V = rand_inputs(rng, BH, T, d, dv, positive=True)
    assert rel(oracle.decay_serial(Q, K, V, gamma, True), oracle.decay_bruteforce(Q, K, V, gamma, True)) < 1e-12


def test_gamma_one_is_the_masked_operator():
    rng = np.random.default_rng(51)
    Q, K, V = rand_inputs(rng, 2, 50, 6, 4)
    np.testing.assert_array_equal(oracle.decay_serial(Q, K, V, 1.0), oracle.serial(Q, K, V))


def test_gamma_zero_keeps_only_the_current_token():
    """gamma = 0: only i = j = t survives, o_t = (q_t.k_t)^2 v_t."""
    rng = np.random.default_rng(52)
    Q, K, V = rand_inputs(rng, 2, 12, 5, 3)
    qk = (Q * K).sum(-1, keepdims=True)
    np.testing.assert_allclose(oracle.decay_serial(Q, K, V, 0.0), qk ** 2 * V, rtol=1e-13, atol=1e-15)


def test_closed_form_unit_vectors():
    """q_t = k_t = e: o_t = sum_j v_j gamma^{2(t-j)} (1 - gamma^{j+1}) / (1 - gamma)."""
    T, d, g = 30, 4, 0.9
    rng = np.random.default_rng(53)
    e = np.zeros(d); e[0] = 1.0
    Qe = np.tile(e, (1, T, 1))
    V = rng.standard_normal((1, T, 3))
    expect = np.zeros((T, 3))
    for t in range(T):
        j = np.arange(t + 1)
        wgt = g ** (2 * (t - j)) * (1 - g ** (j + 1)) / (1 - g)
        expect[t] = (wgt[:, None] * V[0, :t + 1]).sum(0)
    np.testing.assert_allclose(oracle.decay_serial(Qe, Qe, V, g)[0], expect, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("L", [1, 3, 16, 33])
def test_chunked_equals_serial(L):
    """Chunk summaries joined by the decayed combine (factor gamma^{n_B}) and a
    restart per chunk reproduce the recurrence."""
    rng = np.random.default_rng(54)
    Q, K, V = rand_inputs(rng, 2, 70, 6, 5)
    assert rel(oracle.decay_chunked(Q, K, V, L, 0.9), oracle.decay_serial(Q, K, V, 0.9)) < 1e-12
    Q, K, V = rand_inputs(rng, 1, 70, 6, 5, positive=True)
    assert rel(oracle.decay_chunked(Q, K, V, L, 0.7, True), oracle.decay_serial(Q, K, V, 0.7, True)) < 1e-12


def test_combine_equals_concatenation():
    rng = np.random.default_rng(55)
    d, dv, g = 5, 4, 0.85
    Q, K, V = rand_inputs(rng, 1, 25, d, dv)
    whole = oracle.decay_chunk_summaries(Q, K, V, 25, g)[0, 0]
    for cut in (1, 9, 24):
        a = oracle.decay_chunk_summaries(Q[:, :cut], K[:, :cut], V[:, :cut], cut, g)[0, 0]
        b = oracle.decay_chunk_summaries(Q[:, cut:], K[:, cut:], V[:, cut:], 25 - cut, g)[0, 0]
        assert rel(oracle.decay_combine(a, b, d, dv, 25 - cut, g), whole) < 1e-13


def test_pform_step_equals_serial_and_final_state():
    """The compact decode step (S|P|p) reproduces the G-form outputs; its final
    state is P = S C - G, p = S m - h of the whole-sequence summary."""
    rng = np.random.default_rng(56)
    d, dv, T, n, g = 6, 5, 25, 3, 0.9
    for norm in (False, True):
        Q, K, V = rand_inputs(rng, n, T, d, dv, positive=norm)
        st = np.zeros((n, d * d + d * dv + d))
        outs = []
        for t in range(T):
            st, o = oracle.decay_step_pform(st, Q[:, t], K[:, t], V[:, t], g, norm)
            outs.append(o)
        np.testing.assert_allclose(np.stack(outs, 1), oracle.decay_serial(Q, K, V, g, norm), rtol=1e-11, atol=1e-12)
        whole = oracle.decay_chunk_summaries(Q, K, V, T, g)[:, 0]
        np.testing.assert_allclose(st, oracle.summary_to_pform_state(whole, d, dv), rtol=1e-11, atol=1e-12)


def test_causality():
    rng = np.random.default_rng(57)
    Q, K, V = rand_inputs(rng, 1, 30, 5, 4)
    base = oracle.decay_serial(Q, K, V, 0.8)
    K2, V2 = K.copy(), V.copy()
    K2[:, 13:] *= -1; V2[:, 13:] += 2
    np.testing.assert_array_equal(oracle.decay_serial(Q, K2, V2, 0.8)[:, :13], base[:, :13])
