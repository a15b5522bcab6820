"""Pins for the unmasked second-order operator in the fp64 oracle.

HLA summary, section 1: S_t C_t is the naive product whose "future" terms the
cross summary G_t removes; "Results and claims" lists the unmasked operator
as a variant.  Reading: o_t = q_t^T S_t C_t = sum_{i<=t, j<=t} (q_t.k_i)(k_i.q_j) v_j,
normalised by q_t^T S_t m_t.
"""
import numpy as np
import pytest

import oracle


def rel(a, b):
    return float(np.abs(np.asarray(a) - np.asarray(b)).max() / max(np.abs(np.asarray(b)).max(), 1e-300))


def rand_inputs(rng, BH, T, d, dv, positive=False):
    f = rng.random if positive else rng.standard_normal
    Q = f((BH, T, d)) / np.sqrt(d)
    K = f((BH, T, d)) / np.sqrt(d)
    return Q, K, rng.standard_normal((BH, T, dv))


@pytest.mark.parametrize("BH,T,d,dv", [(1, 40, 8, 8), (2, 7, 1, 3), (3, 20, 5, 2), (1, 1, 4, 4)])
def test_serial_equals_bruteforce(BH, T, d, dv):
    rng = np.random.default_rng(300 + T)
    Q, K, V = rand_inputs(rng, BH, T, d, dv)
    assert rel(oracle.unmasked_serial(Q, K, V), oracle.unmasked_bruteforce(Q, K, V)) < 1e-12
    Q, K, V = rand_inputs(rng, BH, T, d, dv, positive=True)
    assert rel(oracle.unmasked_serial(Q, K, V, True), oracle.unmasked_bruteforce(Q, K, V, True)) < 1e-12


def test_library_running_sums():
    rng = np.random.default_rng(41)
    Q, K, V = rand_inputs(rng, 2, 60, 6, 5)
    assert rel(oracle.unmasked_serial(Q, K, V), oracle.dense_unmasked(Q, K, V)) < 1e-12
    Q, K, V = rand_inputs(rng, 2, 60, 6, 5, positive=True)
    assert rel(oracle.unmasked_serial(Q, K, V, True), oracle.dense_unmasked(Q, K, V, True)) < 1e-12


def test_last_token_is_the_full_product():
    """At t = T-1 the moments are the whole sequence's: o = q^T (K^T K)(Q^T V)."""
    rng = np.random.default_rng(42)
    Q, K, V = rand_inputs(rng, 1, 30, 6, 4)
    q, k, v = Q[0], K[0], V[0]
    assert rel(oracle.unmasked_serial(Q, K, V)[0, -1], q[-1] @ (k.T @ k) @ (q.T @ v)) < 1e-13


def test_masked_plus_correction():
    """Unmasked minus masked output is q_t^T G_t (section 1: G removes the
    future terms), G_t taken from the masked oracle's whole-prefix summary."""
    rng = np.random.default_rng(43)
    d, dv, T = 5, 3, 25
    Q, K, V = rand_inputs(rng, 1, T, d, dv)
    un = oracle.unmasked_serial(Q, K, V)[0]
    ma = oracle.serial(Q, K, V)[0]
    off = d * d + d * dv + d
    for t in (0, 7, 24):
        rec = oracle.chunk_summaries(Q[:, :t + 1], K[:, :t + 1], V[:, :t + 1], L=t + 1)[0, 0]
        G = rec[off:off + d * dv].reshape(d, dv)
        np.testing.assert_allclose(un[t] - ma[t], Q[0, t] @ G, rtol=1e-11, atol=1e-12)


def test_closed_forms():
    """T=1: (q.k)^2 v.  q_t = k_t = e: o_t = (t+1) sum_{j<=t} v_j, den_t = (t+1)^2."""
    rng = np.random.default_rng(44)
    Q, K, V = rand_inputs(rng, 3, 1, 4, 2)
    qk = (Q * K).sum(-1, keepdims=True)
    np.testing.assert_allclose(oracle.unmasked_serial(Q, K, V), qk ** 2 * V, rtol=1e-13, atol=1e-15)
    T, d = 30, 4
    e = np.zeros(d); e[3] = 1.0
    Qe = np.tile(e, (1, T, 1))
    V = rng.standard_normal((1, T, 3))
    t = np.arange(T)[:, None]
    expect = (t + 1) * np.cumsum(V[0], axis=0)
    np.testing.assert_allclose(oracle.unmasked_serial(Qe, Qe, V)[0], expect, rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(oracle.unmasked_serial(Qe, Qe, V, True)[0], expect / (t + 1) ** 2, rtol=1e-13)


def test_causality_and_step():
    rng = np.random.default_rng(45)
    Q, K, V = rand_inputs(rng, 2, 30, 6, 4)
    base = oracle.unmasked_serial(Q, K, V)
    Q2, K2, V2 = Q.copy(), K.copy(), V.copy()
    K2[:, 11:] *= -2; V2[:, 11:] += 1
    np.testing.assert_array_equal(oracle.unmasked_serial(Q2, K2, V2)[:, :11], base[:, :11])
    st = np.zeros((2, oracle.unmasked_state_len(6, 4)))
    outs = []
    for t in range(30):
        st, o = oracle.unmasked_step(st, Q[:, t], K[:, t], V[:, t])
        outs.append(o)
    np.testing.assert_allclose(np.stack(outs, 1), base, rtol=1e-13, atol=1e-13)
    k, q, v = K[1], Q[1], V[1]
    np.testing.assert_allclose(st[1], np.concatenate([(k.T @ k).ravel(), (q.T @ v).ravel(), q.sum(0)]), rtol=1e-13,
                               atol=1e-13)
