"""Pins for the AHLA part of the fp64 oracle (HLA summary, section 2 "AHLA").

Reading pinned here: the operator Q (K^T Q)(K^T V) under the causal mask is
    o_t = sum_{j<=i<=t} (q_t.k_i)(q_i.k_j) v_j      (A A V, A = tril(Q K^T)),
with summaries P = sum k v^T, m = sum k, E = sum_i k_i q_i^T P_i,
n = sum_i k_i (q_i . m_i) and, for joining segments, M = sum k q^T.
What fixes each expected value is named in the test: brute force, library
matrix products, closed forms, the unmasked operator, invariants.
"""
import numpy as np
import pytest

import oracle


def rel(a, b):
    return float(np.abs(np.asarray(a) - np.asarray(b)).max() / max(np.abs(np.asarray(b)).max(), 1e-300))


def rand_inputs(rng, BH, T, d, dv, positive=False):
    if positive:
        Q = rng.random((BH, T, d)) / np.sqrt(d)
        K = rng.random((BH, T, d)) / np.sqrt(d)
    else:
        Q = rng.standard_normal((BH, T, d)) / np.sqrt(d)
        K = rng.standard_normal((BH, T, d)) / np.sqrt(d)
    V = rng.standard_normal((BH, T, dv))
    return Q, K, V


@pytest.mark.parametrize("BH,T,d,dv", [(1, 48, 16, 16), (2, 7, 1, 3), (3, 20, 5, 2), (1, 1, 4, 4), (1, 2, 3, 5)])
def test_serial_equals_bruteforce(BH, T, d, dv):
    rng = np.random.default_rng(200 + T)
    Q, K, V = rand_inputs(rng, BH, T, d, dv)
    assert rel(oracle.ahla_serial(Q, K, V), oracle.ahla_bruteforce(Q, K, V)) < 1e-12
    Qp, Kp, Vp = rand_inputs(rng, BH, T, d, dv, positive=True)
    assert rel(oracle.ahla_serial(Qp, Kp, Vp, normalized=True),
               oracle.ahla_bruteforce(Qp, Kp, Vp, normalized=True)) < 1e-12


def test_dense_library_form():
    """(A A) V with A = tril(Q K^T) through numpy matmul."""
    rng = np.random.default_rng(21)
    Q, K, V = rand_inputs(rng, 3, 96, 8, 6)
    assert rel(oracle.ahla_serial(Q, K, V), oracle.dense_causal_aav(Q, K, V)) < 1e-12
    Q, K, V = rand_inputs(rng, 2, 80, 8, 6, positive=True)
    assert rel(oracle.ahla_serial(Q, K, V, normalized=True), oracle.dense_causal_aav(Q, K, V, normalized=True)) < 1e-12


def test_differs_from_hla():
    """AHLA (j <= i) and HLA (i <= j) are different operators on generic inputs."""
    rng = np.random.default_rng(22)
    Q, K, V = rand_inputs(rng, 1, 20, 4, 3)
    assert rel(oracle.ahla_serial(Q, K, V), oracle.serial(Q, K, V)) > 1e-3


def test_closed_form_single_token():
    """T=1: o_0 = (q.k)^2 v_0; normalised o_0 = v_0."""
    rng = np.random.default_rng(23)
    Q, K, V = rand_inputs(rng, 4, 1, 6, 3)
    qk = (Q * K).sum(-1, keepdims=True)
    np.testing.assert_allclose(oracle.ahla_serial(Q, K, V), qk ** 2 * V, rtol=1e-13, atol=1e-15)
    Qp, Kp, Vp = rand_inputs(rng, 4, 1, 6, 3, positive=True)
    np.testing.assert_allclose(oracle.ahla_serial(Qp, Kp, Vp, normalized=True), Vp, rtol=1e-13)


def test_closed_form_unit_vectors():
    """q_t = k_t = e: o_t = sum_{j<=t} (t-j+1) v_j (HLA gives (j+1) here),
    den_t = (t+1)(t+2)/2."""
    T, d, dv = 40, 5, 3
    rng = np.random.default_rng(24)
    e = np.zeros(d); e[1] = 1.0
    Q = np.tile(e, (1, T, 1)); K = Q.copy()
    V = rng.standard_normal((1, T, dv))
    t = np.arange(T)
    expect = np.stack([((tt - t[:tt + 1] + 1)[:, None] * V[0, :tt + 1]).sum(0) for tt in range(T)])
    np.testing.assert_allclose(oracle.ahla_serial(Q, K, V)[0], expect, rtol=1e-13, atol=1e-12)
    den = ((t + 1) * (t + 2) / 2.0)[:, None]
    np.testing.assert_allclose(oracle.ahla_serial(Q, K, V, normalized=True)[0], expect / den, rtol=1e-13, atol=1e-13)


def test_scalar_case_by_hand_loops():
    """d = dv = 1: o_t = q_t * sum_{j<=i<=t} k_i q_i k_j v_j, as plain loops."""
    rng = np.random.default_rng(25)
    T = 12
    q, k, v = rng.standard_normal(T), rng.standard_normal(T), rng.standard_normal(T)
    expect = np.zeros(T)
    for t in range(T):
        s = 0.0
        for i in range(t + 1):
            for j in range(i + 1):
                s += k[i] * q[i] * k[j] * v[j]
        expect[t] = q[t] * s
    got = oracle.ahla_serial(q[None, :, None], k[None, :, None], v[None, :, None])[0, :, 0]
    np.testing.assert_allclose(got, expect, rtol=1e-12, atol=1e-14)


def test_unmasked_operator_from_final_summaries():
    """The whole-sequence M and P are K^T Q and K^T V, so Q M P is the unmasked
    operator Q (K^T Q)(K^T V) of section 2 (library products)."""
    rng = np.random.default_rng(26)
    d, dv, T = 6, 4, 25
    Q, K, V = rand_inputs(rng, 1, T, d, dv)
    rec = oracle.ahla_chunk_summaries(Q, K, V, L=T)[0, 0]
    M = rec[:d * d].reshape(d, d)
    P = rec[d * d:d * d + d * dv].reshape(d, dv)
    q, k, v = Q[0], K[0], V[0]
    assert rel(q @ M @ P, q @ (k.T @ q) @ (k.T @ v)) < 1e-13


def test_causality_bit_exact():
    rng = np.random.default_rng(27)
    Q, K, V = rand_inputs(rng, 2, 50, 8, 4)
    base = oracle.ahla_serial(Q, K, V)
    for cut in (0, 17, 49):
        Q2, K2, V2 = Q.copy(), K.copy(), V.copy()
        Q2[:, cut + 1:] = rng.standard_normal(Q2[:, cut + 1:].shape)
        K2[:, cut + 1:] *= -3.0
        V2[:, cut + 1:] += 1.0
        np.testing.assert_array_equal(oracle.ahla_serial(Q2, K2, V2)[:, :cut + 1], base[:, :cut + 1])


@pytest.mark.parametrize("L", [1, 3, 16, 64, 100, 105])
def test_scan_equals_serial(L):
    """Exclusive Blelloch scan over AHLA chunk summaries (the shared
    semidirect combine with S->M, C->P, G->E) reproduces the recurrence."""
    rng = np.random.default_rng(28)
    Q, K, V = rand_inputs(rng, 2, 100, 8, 7)
    assert rel(oracle.ahla_chunked(Q, K, V, L=L), oracle.ahla_serial(Q, K, V)) < 1e-12
    Qp, Kp, Vp = rand_inputs(rng, 1, 100, 8, 7, positive=True)
    assert rel(oracle.ahla_chunked(Qp, Kp, Vp, L=L, normalized=True),
               oracle.ahla_serial(Qp, Kp, Vp, normalized=True)) < 1e-12


def test_combine_equals_concatenation():
    """combine(summary(A), summary(B)) == summary(A ++ B): pins E = E_A + E_B
    + M_B P_A with the non-symmetric M (a transposed operand fails here)."""
    rng = np.random.default_rng(29)
    d, dv = 6, 4
    Q, K, V = rand_inputs(rng, 1, 30, d, dv)
    whole = oracle.ahla_chunk_summaries(Q, K, V, L=30)[0, 0]
    for cut in (1, 13, 29):
        a = oracle.ahla_chunk_summaries(Q[:, :cut], K[:, :cut], V[:, :cut], L=cut)[0, 0]
        b = oracle.ahla_chunk_summaries(Q[:, cut:], K[:, cut:], V[:, cut:], L=30 - cut)[0, 0]
        assert rel(oracle.combine(a, b, d, dv), whole) < 1e-13


def test_chunk_summary_definition():
    """M = K^T Q, P = K^T V, m = sum k (library); E, n by explicit double loops."""
    rng = np.random.default_rng(30)
    d, dv, T = 5, 3, 9
    Q, K, V = rand_inputs(rng, 1, T, d, dv)
    rec = oracle.ahla_chunk_summaries(Q, K, V, L=T)[0, 0]
    q, k, v = Q[0], K[0], V[0]
    E = np.zeros((d, dv)); n = np.zeros(d)
    for i in range(T):
        for j in range(i + 1):
            E += np.outer(k[i] * (q[i] @ k[j]), v[j])
            n += k[i] * (q[i] @ k[j])
    expect = np.concatenate([(k.T @ q).ravel(), (k.T @ v).ravel(), k.sum(0), E.ravel(), n])
    assert rel(rec, expect) < 1e-13


def test_step_equals_serial_and_final_state():
    rng = np.random.default_rng(31)
    d, dv, T, n = 6, 5, 25, 3
    Q, K, V = rand_inputs(rng, n, T, d, dv)
    state = np.zeros((n, oracle.ahla_state_len(d, dv)))
    outs = []
    for t in range(T):
        state, o = oracle.ahla_step(state, Q[:, t], K[:, t], V[:, t])
        outs.append(o)
    np.testing.assert_allclose(np.stack(outs, axis=1), oracle.ahla_serial(Q, K, V), rtol=1e-13, atol=1e-13)
    whole = oracle.ahla_chunk_summaries(Q, K, V, L=T)[:, 0]
    np.testing.assert_allclose(state, oracle.ahla_summary_to_state(whole, d, dv), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("mutant", [5, 6])
def test_planted_mistakes_fail_a_pin(mutant):
    """E reading P_{t-1} (strict j < i) fails brute force; a transposed M
    fails the concatenation pin."""
    rng = np.random.default_rng(32)
    d, dv = 4, 3
    Q, K, V = rand_inputs(rng, 1, 12, d, dv)
    bad_serial = rel(oracle.ahla_serial(Q, K, V, mutant=mutant), oracle.ahla_bruteforce(Q, K, V)) > 1e-6
    whole = oracle.ahla_chunk_summaries(Q, K, V, L=12)[0, 0]
    a = oracle.ahla_chunk_summaries(Q[:, :5], K[:, :5], V[:, :5], L=5, mutant=mutant)[0, 0]
    b = oracle.ahla_chunk_summaries(Q[:, 5:], K[:, 5:], V[:, 5:], L=7, mutant=mutant)[0, 0]
    bad_combine = rel(oracle.combine(a, b, d, dv, mutant=mutant), whole) > 1e-6
    assert bad_serial or bad_combine
