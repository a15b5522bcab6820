"""The chunk algebra each tensor-core walk computes, written out in fp64 with
numpy and checked against the oracle (CPU only).  The walks evaluate these
products with bf16 operands on the tensor cores; here every step is exact,
so chunked and serial results agree to rounding (1e-12).  Small heads and
short chunks keep the checks fast; the algebra does not depend on the chunk
length, and the sequences span several chunks with a ragged tail.

Formulas (per head, chunk of L tokens with local index t, state at the
chunk start; HLA summary, arXiv 2510.27258):
- masked HLA (section 1, P = S C - G): A = tril(Q K^T), X = Q S0 + A K,
  W = tril(A A^T + (Q S0) Q^T), O = Q P0 + W V, P += X^T V, S += K^T K;
- unmasked (section 1's naive product S_t C_t): X = Q S0 + A K,
  W = tril(X Q^T), O = X C0 + W V, S += K^T K, C += Q^T V;
- AHLA (section 2): Y = Q P0 + A V, O = Q E0 + A Y, E += K^T Y, P += K^T V;
- decayed (section 4's decayed operators, one factor g per token): the
  operands carry the factors the way the walk places them (A~ with a column
  factor g^{-(i+1)}, sX = g^{2L-1-t} X', W~ = g^{-2L} tril(Q sX^T), output
  row factor g^{2(t+1)}, S updated with sqrt(b) K on both sides), and the
  segment summary keeps C and P in the frame of the segment's last token.
"""
import numpy as np
import pytest

import oracle

TOL = 1e-12


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def draw(T, d, dv, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, d)) / np.sqrt(d), rng.standard_normal((T, d)) / np.sqrt(d),
            rng.standard_normal((T, dv)) / np.sqrt(d))


def chunks(T, L):
    for c0 in range(0, T, L):
        yield c0, min(T, c0 + L)


def hla_walk(Q, K, V, L):
    d, dv = Q.shape[1], V.shape[1]
    S, P = np.zeros((d, d)), np.zeros((d, dv))
    O = np.zeros((Q.shape[0], dv))
    for c0, c1 in chunks(Q.shape[0], L):
        q, k, v = Q[c0:c1], K[c0:c1], V[c0:c1]
        A = np.tril(q @ k.T)
        X0 = q @ S
        X = X0 + A @ k
        W = np.tril(A @ A.T + X0 @ q.T)
        O[c0:c1] = q @ P + W @ v
        P = P + X.T @ v
        S = S + k.T @ k
    return O


def unmasked_walk(Q, K, V, L):
    d, dv = Q.shape[1], V.shape[1]
    S, C = np.zeros((d, d)), np.zeros((d, dv))
    O = np.zeros((Q.shape[0], dv))
    for c0, c1 in chunks(Q.shape[0], L):
        q, k, v = Q[c0:c1], K[c0:c1], V[c0:c1]
        A = np.tril(q @ k.T)
        X = q @ S + A @ k
        W = np.tril(X @ q.T)
        O[c0:c1] = X @ C + W @ v
        S = S + k.T @ k
        C = C + q.T @ v
    return O


def ahla_walk(Q, K, V, L):
    d, dv = Q.shape[1], V.shape[1]
    P, E = np.zeros((d, dv)), np.zeros((d, dv))
    O = np.zeros((Q.shape[0], dv))
    for c0, c1 in chunks(Q.shape[0], L):
        q, k, v = Q[c0:c1], K[c0:c1], V[c0:c1]
        A = np.tril(q @ k.T)
        Y = q @ P + A @ v
        O[c0:c1] = q @ E + A @ Y
        E = E + k.T @ Y
        P = P + k.T @ v
    return O


def decay_out_walk(Q, K, V, g, L, S0=None, P0=None, c_begin=0, c_end=None):
    """Output walk of chunks [c_begin, c_end) from the state (S0, P0) at
    c_begin's start, with the factors where the tensor-core walk puts them."""
    d, dv = Q.shape[1], V.shape[1]
    T = Q.shape[0]
    S = np.zeros((d, d)) if S0 is None else S0.copy()
    P = np.zeros((d, dv)) if P0 is None else P0.copy()
    O = np.zeros((T, dv))
    n = (T + L - 1) // L if c_end is None else c_end
    t = np.arange(L, dtype=np.float64)
    for c in range(c_begin, n):
        c0, c1 = c * L, min(T, (c + 1) * L)
        Lc = c1 - c0
        q, k, v = (np.zeros((L, X.shape[1])) for X in (Q, K, V))
        q[:Lc], k[:Lc], v[:Lc] = Q[c0:c1], K[c0:c1], V[c0:c1]
        At = np.tril(q @ k.T) * (g ** -(t + 1))[None, :]          # column factor
        Xp = q @ S + At @ k                                          # X^g_t / a_t
        sX = (g ** (2 * Lc - 1 - t))[:, None] * Xp                   # b_t^2 X^g_t
        Wt = g ** (-2.0 * Lc) * np.tril(q @ sX.T)                    # constant factor
        Op = q @ P + Wt @ v
        O[c0:c1] = ((g ** (2 * (t + 1)))[:, None] * Op)[:Lc]         # row factor
        Kp = (g ** (0.5 * (Lc - 1 - t)))[:, None] * k                # sqrt(b) K
        S = g ** Lc * S + Kp.T @ Kp
        P = g ** (2 * Lc) * P + sX.T @ v
    return O, S, P


def decay_summary_walk(Q, K, V, g, L, c_begin, c_end):
    """Segment summary S (running), C and P in the frame of the segment's last token."""
    d, dv = Q.shape[1], V.shape[1]
    T = Q.shape[0]
    S, C, P = np.zeros((d, d)), np.zeros((d, dv)), np.zeros((d, dv))
    seg_end = min(T, c_end * L)
    t = np.arange(L, dtype=np.float64)
    for c in range(c_begin, c_end):
        c0, c1 = c * L, min(T, (c + 1) * L)
        Lc = c1 - c0
        F = g ** (seg_end - c1)
        q, k, v = (np.zeros((L, X.shape[1])) for X in (Q, K, V))
        q[:Lc], k[:Lc], v[:Lc] = Q[c0:c1], K[c0:c1], V[c0:c1]
        At = np.tril(q @ k.T) * (g ** -(t + 1))[None, :]
        Xp = q @ S + At @ k
        P = P + ((F * F * g ** (2 * Lc - 1 - t))[:, None] * Xp).T @ v
        C = C + ((F * g ** (Lc - 1 - t))[:, None] * q).T @ v
        Kp = (g ** (0.5 * (Lc - 1 - t)))[:, None] * k
        S = g ** Lc * S + Kp.T @ Kp
    return S, C, P


@pytest.mark.parametrize("T,L", [(1, 8), (37, 8), (100, 16), (64, 16)])
def test_hla_chunk_walk_equals_serial(T, L):
    Q, K, V = draw(T, 8, 6, seed=T + L)
    assert rel(hla_walk(Q, K, V, L), oracle.serial(Q, K, V)) < TOL


@pytest.mark.parametrize("T,L", [(1, 8), (37, 8), (100, 16)])
def test_unmasked_chunk_walk_equals_serial(T, L):
    Q, K, V = draw(T, 8, 6, seed=2 * T + L)
    assert rel(unmasked_walk(Q, K, V, L), oracle.unmasked_serial(Q, K, V)) < TOL


@pytest.mark.parametrize("T,L", [(1, 8), (37, 8), (100, 16)])
def test_ahla_chunk_walk_equals_serial(T, L):
    Q, K, V = draw(T, 8, 6, seed=3 * T + L)
    assert rel(ahla_walk(Q, K, V, L), oracle.ahla_serial(Q, K, V)) < TOL


@pytest.mark.parametrize("g", [1.0, 0.99, 0.9, 0.8])
@pytest.mark.parametrize("T,L", [(1, 8), (37, 8), (100, 16)])
def test_decay_output_walk_with_kernel_factors_equals_serial(T, L, g):
    Q, K, V = draw(T, 8, 6, seed=5 * T + L)
    O, _, _ = decay_out_walk(Q, K, V, g, L)
    assert rel(O, oracle.decay_serial(Q, K, V, g)) < TOL


@pytest.mark.parametrize("g", [1.0, 0.95, 0.8])
def test_decay_segments_summary_prefix_then_outputs(g):
    """Two segments: the first's end-frame summary (S, C, P) is the decayed
    state the second segment starts from, and its outputs then equal the
    serial recurrence's (the oracle's summary and combine agree with it)."""
    T, L, d, dv = 90, 8, 8, 6
    Q, K, V = draw(T, d, dv, seed=int(g * 1000))
    split = 5  # chunks in the first segment
    S1, C1, P1 = decay_summary_walk(Q, K, V, g, L, 0, split)
    rec = oracle.decay_chunk_summaries(Q[None], K[None], V[None], split * L, g)[0][0]
    Sr = rec[:d * d].reshape(d, d)
    Cr = rec[d * d:d * d + d * dv].reshape(d, dv)
    Gr = rec[d * d + d * dv + d:d * d + 2 * d * dv + d].reshape(d, dv)
    assert rel(S1, Sr) < TOL and rel(C1, Cr) < TOL and rel(P1, Sr @ Cr - Gr) < TOL
    O1, _, _ = decay_out_walk(Q, K, V, g, L, c_end=split)
    O2, _, _ = decay_out_walk(Q, K, V, g, L, S0=S1, P0=P1, c_begin=split)
    ref = oracle.decay_serial(Q, K, V, g)
    assert rel(O1[:split * L], ref[:split * L]) < TOL
    assert rel(O2[split * L:], ref[split * L:]) < TOL
