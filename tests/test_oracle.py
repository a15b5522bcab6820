"""Pins for the fp64 oracle, against things other than the oracle itself.

Each test names what fixes the expected value:
  * a hand-worked example (tests/golden/hla2_hand_worked.json),
  * closed forms and special cases of the definition
    o_t = sum_{i<=j<=t} (q_t.k_i)(k_i.q_j) v_j   (HLA summary, section 1),
  * library matrix products (A = tril(Q K^T), O = tril(A A^T) V),
  * invariants the pages claim: strict causality ("Results and claims"),
    scan == serial ("Parallel training via associative scans"),
  * brute force on tiny inputs.
Planted mistakes (oracle compiled with HLA2_ORACLE_MUTANT) must fail a pin.
"""
import json
import os

import numpy as np
import pytest

import oracle
from higher_order_linear_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hla2_hand_worked.json")


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


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        g = json.load(f)
    return {k: (np.array(v, dtype=np.float64) if isinstance(v, list) and k not in ("derivation",) else v)
            for k, v in g.items()}


# ---------------------------------------------------------------- golden ----
def test_golden_outputs(golden):
    Q, K, V = golden["Q"][None], golden["K"][None], golden["V"][None]
    for fn in (oracle.serial, oracle.bruteforce, oracle.dense_causal_aatv,
               lambda *a, **k: oracle.chunked(*a, L=2, **k)):
        np.testing.assert_allclose(fn(Q, K, V)[0], golden["O"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(fn(Q, K, V, normalized=True)[0], golden["O_normalized"], rtol=1e-14, atol=1e-14)


def test_golden_summaries_and_combine(golden):
    Q, K, V = golden["Q"][None], golden["K"][None], golden["V"][None]
    s = oracle.chunk_summaries(Q, K, V, L=2)[0]
    np.testing.assert_array_equal(s, golden["chunk_summaries"])
    c = oracle.combine(s[0], s[1], 2, 2)
    np.testing.assert_array_equal(c, golden["combined"])
    # the whole sequence as one chunk is the same state
    whole = oracle.chunk_summaries(Q, K, V, L=3)[0, 0]
    np.testing.assert_array_equal(whole, golden["combined"])


# ------------------------------------------------------- definition pins ----
@pytest.mark.parametrize("BH,T,d,dv", [(1, 64, 16, 16), (2, 7, 1, 3), (3, 20, 5, 2), (1, 1, 4, 4), (1, 2, 3, 5)])
def test_serial_equals_bruteforce(BH, T, d, dv):
    rng = np.random.default_rng(100 + T)
    Q, K, V = rand_inputs(rng, BH, T, d, dv)
    ref = oracle.bruteforce(Q, K, V)
    assert rel(oracle.serial(Q, K, V), ref) < 1e-12
    Qp, Kp, Vp = rand_inputs(rng, BH, T, d, dv, positive=True)
    refn = oracle.bruteforce(Qp, Kp, Vp, normalized=True)
    assert rel(oracle.serial(Qp, Kp, Vp, normalized=True), refn) < 1e-12


def test_workload0_three_ways():
    """Workload 0 (B1 H1 T64 d16 fp32): serial == O(T^3) brute force == chunk-16 scan."""
    w = W.WORKLOADS[0]
    q, k, v = W.make_inputs(w)
    Q, K, V = (x.double().numpy() for x in (q, k, v))
    ref = oracle.bruteforce(Q, K, V)
    assert rel(oracle.serial(Q, K, V), ref) < 1e-12
    assert rel(oracle.chunked(Q, K, V, L=16), ref) < 1e-12
    assert rel(oracle.dense_causal_aatv(Q, K, V), ref) < 1e-12


def test_dense_library_form():
    """tril(A A^T) V with A = tril(Q K^T) through numpy matmul (a library routine)."""
    rng = np.random.default_rng(7)
    Q, K, V = rand_inputs(rng, 3, 96, 8, 6)
    assert rel(oracle.serial(Q, K, V), oracle.dense_causal_aatv(Q, K, V)) < 1e-12
    Q, K, V = rand_inputs(rng, 2, 80, 8, 6, positive=True)
    assert rel(oracle.serial(Q, K, V, normalized=True), oracle.dense_causal_aatv(Q, K, V, normalized=True)) < 1e-12


def test_closed_form_single_token():
    """T=1: o_0 = (q.k)^2 v_0; normalised o_0 = v_0."""
    rng = np.random.default_rng(3)
    Q, K, V = rand_inputs(rng, 4, 1, 6, 3)
    qk = (Q * K).sum(-1, keepdims=True)
    np.testing.assert_allclose(oracle.serial(Q, K, V), qk ** 2 * V, rtol=1e-13, atol=1e-15)
    Qp, Kp, Vp = rand_inputs(rng, 4, 1, 6, 3, positive=True)
    np.testing.assert_allclose(oracle.serial(Qp, Kp, Vp, normalized=True), Vp, rtol=1e-13)


def test_closed_form_unit_vectors():
    """q_t = k_t = e for all t: o_t = sum_{j<=t} (j+1) v_j, den_t = (t+1)(t+2)/2."""
    T, d, dv = 40, 5, 3
    rng = np.random.default_rng(4)
    e = np.zeros(d); e[2] = 1.0
    Q = np.tile(e, (1, T, 1)); K = Q.copy()
    V = rng.standard_normal((1, T, dv))
    j = np.arange(T)[:, None]
    expect = np.cumsum((j + 1) * V[0], axis=0)
    np.testing.assert_allclose(oracle.serial(Q, K, V)[0], expect, rtol=1e-13, atol=1e-12)
    den = ((j + 1) * (j + 2) / 2.0)
    np.testing.assert_allclose(oracle.serial(Q, K, V, normalized=True)[0], expect / den, rtol=1e-13, atol=1e-13)


def test_scalar_case_by_hand_loops():
    """d = dv = 1: o_t = q_t * sum_{i<=j<=t} k_i^2 q_j v_j, written as plain loops."""
    rng = np.random.default_rng(5)
    T = 12
    q, k, v = rng.standard_normal(T), rng.standard_normal(T), rng.standard_normal(T)
    expect = np.zeros(T)
    for t in range(T):
        s = 0.0
        for j in range(t + 1):
            for i in range(j + 1):
                s += k[i] * k[i] * q[j] * v[j]
        expect[t] = q[t] * s
    got = oracle.serial(q[None, :, None], k[None, :, None], v[None, :, None])[0, :, 0]
    np.testing.assert_allclose(got, expect, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ invariants ----
def test_causality_bit_exact():
    """Outputs at t depend only on tokens j <= t ("Results and claims")."""
    rng = np.random.default_rng(6)
    Q, K, V = rand_inputs(rng, 2, 50, 8, 4)
    base = oracle.serial(Q, K, V)
    for cut in (0, 17, 49):
        Q2, K2, V2 = Q.copy(), K.copy(), V.copy()
        Q2[:, cut + 1:] = rng.standard_normal(Q2[:, cut + 1:].shape)
        K2[:, cut + 1:] *= -3.0
        V2[:, cut + 1:] += 1.0
        out = oracle.serial(Q2, K2, V2)
        np.testing.assert_array_equal(out[:, :cut + 1], base[:, :cut + 1])


def test_zero_padding_invariance():
    rng = np.random.default_rng(8)
    Q, K, V = rand_inputs(rng, 2, 37, 6, 5)
    pad = lambda x: np.concatenate([x, np.zeros((x.shape[0], 27, x.shape[2]))], axis=1)
    base = oracle.serial(Q, K, V)
    np.testing.assert_array_equal(oracle.serial(pad(Q), pad(K), pad(V))[:, :37], base)
    # chunked with a ragged tail equals the padded chunked run
    np.testing.assert_allclose(oracle.chunked(Q, K, V, L=16), oracle.chunked(pad(Q), pad(K), pad(V), L=16)[:, :37],
                               rtol=0, atol=1e-13)


@pytest.mark.parametrize("L", [1, 3, 16, 64, 100, 105])
def test_scan_equals_serial(L):
    """Exclusive Blelloch scan over chunk summaries reproduces the serial recurrence."""
    rng = np.random.default_rng(9)
    Q, K, V = rand_inputs(rng, 2, 100, 8, 7)
    ref = oracle.serial(Q, K, V)
    assert rel(oracle.chunked(Q, K, V, L=L), ref) < 1e-12
    Qp, Kp, Vp = rand_inputs(rng, 1, 100, 8, 7, positive=True)
    assert rel(oracle.chunked(Qp, Kp, Vp, L=L, normalized=True), oracle.serial(Qp, Kp, Vp, normalized=True)) < 1e-12


def test_combine_equals_concatenation():
    """combine(summary(A), summary(B)) == summary(A ++ B): pins the cross terms S_B C_A, S_B m_A."""
    rng = np.random.default_rng(10)
    d, dv = 6, 4
    Q, K, V = rand_inputs(rng, 1, 30, d, dv)
    whole = oracle.chunk_summaries(Q, K, V, L=30)[0, 0]
    for cut in (1, 13, 29):
        a = oracle.chunk_summaries(Q[:, :cut], K[:, :cut], V[:, :cut], L=cut)[0, 0]
        b = oracle.chunk_summaries(Q[:, cut:], K[:, cut:], V[:, cut:], L=30 - cut)[0, 0]
        assert rel(oracle.combine(a, b, d, dv), whole) < 1e-13


def test_chunk_summary_definition():
    """S = K^T K, C = Q^T V, m = sum q (library products); G, h by explicit double loops."""
    rng = np.random.default_rng(11)
    d, dv, T = 5, 3, 9
    Q, K, V = rand_inputs(rng, 1, T, d, dv)
    rec = oracle.chunk_summaries(Q, K, V, L=T)[0, 0]
    q, k, v = Q[0], K[0], V[0]
    G = np.zeros((d, dv)); h = np.zeros(d)
    for i in range(T):
        for j in range(i):
            G += np.outer(k[i] * (k[i] @ q[j]), v[j])
            h += k[i] * (k[i] @ q[j])
    expect = np.concatenate([(k.T @ k).ravel(), (q.T @ v).ravel(), q.sum(0), G.ravel(), h])
    assert rel(rec, expect) < 1e-13


def test_scan_bracketings():
    """Left fold == Blelloch tree == random bracketings (associativity of the combine)."""
    rng = np.random.default_rng(12)
    d, dv, N = 4, 3, 11
    summ = rng.standard_normal((2, N, oracle.record_len(d, dv)))
    fold = oracle.scan_fold(summ, d, dv)
    tree = oracle.scan_blelloch(summ, d, dv)
    assert rel(tree, fold) < 1e-12
    np.testing.assert_array_equal(fold[:, 0], 0.0)
    for trial in range(5):
        items = [summ[0, i] for i in range(N)]
        while len(items) > 1:
            i = int(rng.integers(0, len(items) - 1))
            items[i:i + 2] = [oracle.combine(items[i], items[i + 1], d, dv)]
        inclusive = oracle.combine(fold[0, N - 1], summ[0, N - 1], d, dv)
        assert rel(items[0], inclusive) < 1e-12


def test_step_equals_serial_and_final_state():
    rng = np.random.default_rng(13)
    d, dv, T, n = 6, 5, 25, 3
    Q, K, V = rand_inputs(rng, n, T, d, dv)
    state = np.zeros((n, oracle.record_len(d, dv)))
    outs = []
    for t in range(T):
        state, o = oracle.step(state, Q[:, t], K[:, t], V[:, t])
        outs.append(o)
    outs = np.stack(outs, axis=1)
    np.testing.assert_allclose(outs, oracle.serial(Q, K, V), rtol=1e-13, atol=1e-13)
    whole = oracle.chunk_summaries(Q, K, V, L=T)[:, 0]
    np.testing.assert_allclose(state, oracle.summary_to_decode_state(whole, d, dv), rtol=1e-13, atol=1e-13)


# --------------------------------------------------------- planted bugs ----
@pytest.mark.parametrize("mutant", [1, 2, 3, 4])
def test_planted_mistakes_fail_a_pin(mutant):
    """Each deliberate oracle mistake (dropped G, wrong sign, C_t for C_{t-1},
    swapped cross term) is caught by brute force or by the concatenation pin."""
    rng = np.random.default_rng(14)
    d, dv = 4, 3
    Q, K, V = rand_inputs(rng, 1, 12, d, dv)
    bad_serial = rel(oracle.serial(Q, K, V, mutant=mutant), oracle.bruteforce(Q, K, V)) > 1e-6
    whole = oracle.chunk_summaries(Q, K, V, L=12)[0, 0]
    a = oracle.chunk_summaries(Q[:, :5], K[:, :5], V[:, :5], L=5, mutant=mutant)[0, 0]
    b = oracle.chunk_summaries(Q[:, 5:], K[:, 5:], V[:, 5:], L=7, mutant=mutant)[0, 0]
    bad_combine = rel(oracle.combine(a, b, d, dv, mutant=mutant), whole) > 1e-6
    assert bad_serial or bad_combine


def test_pform_state_is_the_masked_product():
    """P = S C - G and p = S m - h equal the masked sums
    sum_{i<=j} k_i k_i^T q_j v_j^T and sum_{i<=j} k_i (k_i . q_j) (explicit loops)."""
    rng = np.random.default_rng(15)
    d, dv, T = 4, 3, 11
    Q, K, V = rand_inputs(rng, 1, T, d, dv)
    rec = oracle.chunk_summaries(Q, K, V, L=T)[0, 0]
    pst = oracle.summary_to_pform_state(rec, d, dv)
    q, k, v = Q[0], K[0], V[0]
    P = np.zeros((d, dv)); p = np.zeros(d)
    for j in range(T):
        for i in range(j + 1):
            P += np.outer(k[i] * (k[i] @ q[j]), v[j])
            p += k[i] * (k[i] @ q[j])
    expect = np.concatenate([(k.T @ k).ravel(), P.ravel(), p])
    assert rel(pst, expect) < 1e-13
