"""fp64 CPU oracle for masked second-order HLA -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA library never links,
loads or calls it, and it imports nothing from the CUDA side.

The arithmetic lives in ``hla2_oracle.c`` (plain C, fp64); this module builds
it with gcc and marshals numpy arrays through ctypes.  ``dense_causal_aatv``
is a second, independent statement of the same definition through library
matrix products, used only to pin the C code.

Citations ("HLA summary"): technical summary pages of "Higher-order Linear
Attention" (arXiv 2510.27258), Japanese and French editions on gist.science;
section 1 "Second-order HLA", section 4 "Parallel training via associative
scans", section "Results and claims".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hla2_oracle.c")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}


def lib_path(mutant: int = 0) -> str:
    name = "libhla2_oracle.so" if mutant == 0 else f"libhla2_oracle_mutant{mutant}.so"
    return os.path.join(_HERE, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU, no CUDA).  ``mutant`` plants one of
    the deliberate mistakes in the C source (used only by the pin tests)."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lpthread"]
    if mutant:
        cmd.insert(1, f"-DHLA2_ORACLE_MUTANT={int(mutant)}")
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib(mutant: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if mutant not in _LIBS:
            lib = ctypes.CDLL(build(mutant))
            dp = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            lib.hla2_oracle_serial.argtypes = [dp, dp, dp, dp, i, i, i, i, i, i]
            lib.hla2_oracle_bruteforce.argtypes = [dp, dp, dp, dp, i, i, i, i, i]
            lib.hla2_oracle_chunk_summaries.argtypes = [dp, dp, dp, dp, i, i, i, i, i]
            lib.hla2_oracle_combine.argtypes = [dp, dp, dp, i, i]
            lib.hla2_oracle_combine.restype = None
            lib.hla2_oracle_scan_fold.argtypes = [dp, dp, i, i, i, i]
            lib.hla2_oracle_scan_blelloch.argtypes = [dp, dp, i, i, i, i]
            lib.hla2_oracle_chunked.argtypes = [dp, dp, dp, dp, i, i, i, i, i, i]
            lib.hla2_oracle_step.argtypes = [dp, dp, dp, dp, dp, i, i, i, i]
            lib.hla2_oracle_record_len.argtypes = [i, i]
            lib.hla2_oracle_record_len.restype = ctypes.c_longlong
            _LIBS[mutant] = lib
        return _LIBS[mutant]


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _heads(Q, K, V):
    """Accept [..., T, d] arrays; flatten the leading axes into heads."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    lead = Q.shape[:-2]
    T, d = Q.shape[-2:]
    dv = V.shape[-1]
    if K.shape != Q.shape or V.shape[:-1] != Q.shape[:-1]:
        raise ValueError("Q, K, V shapes disagree")
    BH = int(np.prod(lead)) if lead else 1
    return Q.reshape(BH, T, d), K.reshape(BH, T, d), V.reshape(BH, T, dv), lead, BH, T, d, dv


def record_len(d: int, dv: int) -> int:
    return d * d + 2 * d * dv + 2 * d


def serial(Q, K, V, normalized: bool = False, nthreads: int = 1, mutant: int = 0) -> np.ndarray:
    """o_t by the serial recurrence (HLA summary, section 1)."""
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    rc = _lib(mutant).hla2_oracle_serial(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized), int(nthreads))
    if rc:
        raise RuntimeError("oracle serial failed")
    return O.reshape(*lead, T, dv)


def bruteforce(Q, K, V, normalized: bool = False, mutant: int = 0) -> np.ndarray:
    """o_t = sum_{i<=j<=t} (q_t.k_i)(k_i.q_j) v_j, O(T^3 d)."""
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    if _lib(mutant).hla2_oracle_bruteforce(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized)):
        raise RuntimeError("oracle bruteforce failed")
    return O.reshape(*lead, T, dv)


def chunked(Q, K, V, L: int, normalized: bool = False, mutant: int = 0) -> np.ndarray:
    """Chunk summaries + exclusive Blelloch scan + per-chunk restart (section 4)."""
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    if _lib(mutant).hla2_oracle_chunked(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized), int(L)):
        raise RuntimeError("oracle chunked failed")
    return O.reshape(*lead, T, dv)


def chunk_summaries(Q, K, V, L: int, mutant: int = 0) -> np.ndarray:
    """[..., N, record] with record S|C|m|G|h of each L-token chunk."""
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    N = (T + L - 1) // L
    out = np.zeros((BH, N, record_len(d, dv)))
    if _lib(mutant).hla2_oracle_chunk_summaries(_p(Q), _p(K), _p(V), _p(out), BH, T, d, dv, int(L)):
        raise RuntimeError("oracle chunk_summaries failed")
    return out.reshape(*lead, N, record_len(d, dv))


def combine(a, b, d: int, dv: int, mutant: int = 0) -> np.ndarray:
    """Semidirect combine, a earlier, b later (section 4)."""
    a, b = _f64(a), _f64(b)
    out = np.zeros(record_len(d, dv))
    _lib(mutant).hla2_oracle_combine(_p(a), _p(b), _p(out), d, dv)
    return out


def _scan(fn, summ, d, dv):
    summ = _f64(summ)
    lead = summ.shape[:-2]
    N, R = summ.shape[-2:]
    if R != record_len(d, dv):
        raise ValueError("record length mismatch")
    BH = int(np.prod(lead)) if lead else 1
    out = np.zeros((BH, N, R))
    if fn(_p(summ.reshape(BH, N, R)), _p(out), BH, N, d, dv):
        raise RuntimeError("oracle scan failed")
    return out.reshape(*lead, N, R)


def scan_fold(summ, d: int, dv: int, mutant: int = 0) -> np.ndarray:
    """Exclusive scan as a left fold of combines."""
    return _scan(_lib(mutant).hla2_oracle_scan_fold, summ, d, dv)


def scan_blelloch(summ, d: int, dv: int, mutant: int = 0) -> np.ndarray:
    """Exclusive Blelloch (up-sweep / down-sweep) scan."""
    return _scan(_lib(mutant).hla2_oracle_scan_blelloch, summ, d, dv)


def step(state, q, k, v, normalized: bool = False, mutant: int = 0):
    """One decode step on n heads; returns (new_state, o).  State order S|C|G|m|h."""
    state = _f64(state).copy()
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, d = q.shape
    dv = v.shape[1]
    o = np.zeros((n, dv))
    if _lib(mutant).hla2_oracle_step(_p(state), _p(q), _p(k), _p(v), _p(o), n, d, dv, int(normalized)):
        raise RuntimeError("oracle step failed")
    return state, o


def summary_to_decode_state(rec, d: int, dv: int) -> np.ndarray:
    """Reorder a summary record S|C|m|G|h into the decode order S|C|G|m|h."""
    rec = _f64(rec)
    nS, nC = d * d, d * dv
    S = rec[..., :nS]
    C = rec[..., nS:nS + nC]
    m = rec[..., nS + nC:nS + nC + d]
    G = rec[..., nS + nC + d:nS + 2 * nC + d]
    h = rec[..., nS + 2 * nC + d:]
    return np.concatenate([S, C, G, m, h], axis=-1)


def summary_to_pform_state(rec, d: int, dv: int) -> np.ndarray:
    """Summary record S|C|m|G|h -> P-form decode state S|P|p with
    P = S C - G and p = S m - h (HLA summary, section 1: G and h remove the
    future terms of the naive product, so P and p are the masked products)."""
    rec = _f64(rec)
    nS, nC = d * d, d * dv
    S = rec[..., :nS].reshape(*rec.shape[:-1], d, d)
    C = rec[..., nS:nS + nC].reshape(*rec.shape[:-1], d, dv)
    m = rec[..., nS + nC:nS + nC + d]
    G = rec[..., nS + nC + d:nS + 2 * nC + d].reshape(*rec.shape[:-1], d, dv)
    h = rec[..., nS + 2 * nC + d:]
    P = S @ C - G
    p = np.einsum("...ab,...b->...a", S, m) - h
    lead = rec.shape[:-1]
    return np.concatenate([S.reshape(*lead, nS), P.reshape(*lead, nC), p], axis=-1)


def dense_causal_aatv(Q, K, V, normalized: bool = False) -> np.ndarray:
    """Independent statement through library matmuls: A = tril(Q K^T),
    O = tril(A A^T) V (HLA summary, section 2 names the A A^T V structure;
    the outer tril keeps j <= t, the causality claim of "Results and claims").
    Normalised: divide by the row sums of tril(A A^T)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    A = np.tril(Q @ np.swapaxes(K, -1, -2))
    W = np.tril(A @ np.swapaxes(A, -1, -2))
    O = W @ V
    if normalized:
        O = O / W.sum(axis=-1, keepdims=True)
    return O


# ------------------------------------------------------------------ AHLA ----
# HLA summary, section 2 "AHLA": operator Q (K^T Q)(K^T V); masked reading
#   o_t = sum_{j<=i<=t} (q_t.k_i)(q_i.k_j) v_j   (causal A A V, A = tril(Q K^T)).
# Summary record M|P|m|E|n (M = sum k q^T, P = sum k v^T, m = sum k,
# E = sum_i k_i q_i^T P_i, n = sum_i k_i (q_i . m_i)); decode state P|E|m|n.

def _ahla_lib(mutant: int = 0) -> ctypes.CDLL:
    lib = _lib(mutant)
    if not getattr(lib, "_ahla_typed", False):
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.hla2_oracle_ahla_serial.argtypes = [dp, dp, dp, dp, i, i, i, i, i]
        lib.hla2_oracle_ahla_bruteforce.argtypes = [dp, dp, dp, dp, i, i, i, i, i]
        lib.hla2_oracle_ahla_chunk_summaries.argtypes = [dp, dp, dp, dp, i, i, i, i, i]
        lib.hla2_oracle_ahla_chunked.argtypes = [dp, dp, dp, dp, i, i, i, i, i, i]
        lib.hla2_oracle_ahla_step.argtypes = [dp, dp, dp, dp, dp, i, i, i, i]
        lib._ahla_typed = True
    return lib


def ahla_state_len(d: int, dv: int) -> int:
    """Decode state P|E|m|n per head."""
    return 2 * d * dv + 2 * d


def ahla_serial(Q, K, V, normalized: bool = False, mutant: int = 0) -> np.ndarray:
    """AHLA outputs by the serial recurrence."""
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    if _ahla_lib(mutant).hla2_oracle_ahla_serial(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized)):
        raise RuntimeError("oracle ahla_serial failed")
    return O.reshape(*lead, T, dv)


def ahla_bruteforce(Q, K, V, normalized: bool = False, mutant: int = 0) -> np.ndarray:
    """AHLA by its definition, O(T^3 d)."""
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    if _ahla_lib(mutant).hla2_oracle_ahla_bruteforce(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized)):
        raise RuntimeError("oracle ahla_bruteforce failed")
    return O.reshape(*lead, T, dv)


def ahla_chunk_summaries(Q, K, V, L: int, mutant: int = 0) -> np.ndarray:
    """[..., N, record] with record M|P|m|E|n of each L-token chunk."""
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    N = (T + L - 1) // L
    out = np.zeros((BH, N, record_len(d, dv)))
    if _ahla_lib(mutant).hla2_oracle_ahla_chunk_summaries(_p(Q), _p(K), _p(V), _p(out), BH, T, d, dv, int(L)):
        raise RuntimeError("oracle ahla_chunk_summaries failed")
    return out.reshape(*lead, N, record_len(d, dv))


def ahla_chunked(Q, K, V, L: int, normalized: bool = False, mutant: int = 0) -> np.ndarray:
    """AHLA chunk summaries + exclusive Blelloch scan + per-chunk restart."""
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    if _ahla_lib(mutant).hla2_oracle_ahla_chunked(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized),
                                                  int(L)):
        raise RuntimeError("oracle ahla_chunked failed")
    return O.reshape(*lead, T, dv)


def ahla_step(state, q, k, v, normalized: bool = False, mutant: int = 0):
    """One AHLA decode step on n heads; returns (new_state, o).  State P|E|m|n."""
    state = _f64(state).copy()
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, d = q.shape
    dv = v.shape[1]
    o = np.zeros((n, dv))
    if _ahla_lib(mutant).hla2_oracle_ahla_step(_p(state), _p(q), _p(k), _p(v), _p(o), n, d, dv, int(normalized)):
        raise RuntimeError("oracle ahla_step failed")
    return state, o


def ahla_summary_to_state(rec, d: int, dv: int) -> np.ndarray:
    """Summary record M|P|m|E|n -> decode state P|E|m|n (M is only needed to
    combine segments, not to continue a sequence)."""
    rec = _f64(rec)
    nS, nC = d * d, d * dv
    P = rec[..., nS:nS + nC]
    m = rec[..., nS + nC:nS + nC + d]
    E = rec[..., nS + nC + d:nS + 2 * nC + d]
    n = rec[..., nS + 2 * nC + d:]
    return np.concatenate([P, E, m, n], axis=-1)


def dense_causal_aav(Q, K, V, normalized: bool = False) -> np.ndarray:
    """Independent statement through library matmuls: A = tril(Q K^T),
    O = (A A) V (HLA summary, section 2: A A V where HLA has A A^T V; A A is
    lower triangular already).  Normalised: divide by the row sums of A A."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    A = np.tril(Q @ np.swapaxes(K, -1, -2))
    W = A @ A
    O = W @ V
    if normalized:
        O = O / W.sum(axis=-1, keepdims=True)
    return O


# -------------------------------------------------------------- unmasked ----
# o_t = q_t^T S_t C_t = sum_{i<=t, j<=t} (q_t.k_i)(k_i.q_j) v_j (no G correction);
# normalised by q_t^T S_t m_t.  Decode state S|C|m.

def _unmasked_lib(mutant: int = 0) -> ctypes.CDLL:
    lib = _lib(mutant)
    if not getattr(lib, "_unmasked_typed", False):
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.hla2_oracle_unmasked_serial.argtypes = [dp, dp, dp, dp, i, i, i, i, i]
        lib.hla2_oracle_unmasked_bruteforce.argtypes = [dp, dp, dp, dp, i, i, i, i, i]
        lib.hla2_oracle_unmasked_step.argtypes = [dp, dp, dp, dp, dp, i, i, i, i]
        lib._unmasked_typed = True
    return lib


def unmasked_state_len(d: int, dv: int) -> int:
    return d * d + d * dv + d


def unmasked_serial(Q, K, V, normalized: bool = False) -> np.ndarray:
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    if _unmasked_lib().hla2_oracle_unmasked_serial(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized)):
        raise RuntimeError("oracle unmasked_serial failed")
    return O.reshape(*lead, T, dv)


def unmasked_bruteforce(Q, K, V, normalized: bool = False) -> np.ndarray:
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    if _unmasked_lib().hla2_oracle_unmasked_bruteforce(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized)):
        raise RuntimeError("oracle unmasked_bruteforce failed")
    return O.reshape(*lead, T, dv)


def unmasked_step(state, q, k, v, normalized: bool = False):
    """One unmasked decode step on n heads; returns (new_state, o).  State S|C|m."""
    state = _f64(state).copy()
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, d = q.shape
    dv = v.shape[1]
    o = np.zeros((n, dv))
    if _unmasked_lib().hla2_oracle_unmasked_step(_p(state), _p(q), _p(k), _p(v), _p(o), n, d, dv, int(normalized)):
        raise RuntimeError("oracle unmasked_step failed")
    return state, o


def dense_unmasked(Q, K, V, normalized: bool = False) -> np.ndarray:
    """Independent statement through library routines: running sums
    S_t = cumsum k k^T, C_t = cumsum q v^T, m_t = cumsum q, then q_t^T S_t C_t."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    S = np.cumsum(np.einsum("...ta,...tb->...tab", K, K), axis=-3)
    C = np.cumsum(np.einsum("...ta,...te->...tae", Q, V), axis=-3)
    u = np.einsum("...tab,...tb->...ta", S, Q)
    O = np.einsum("...ta,...tae->...te", u, C)
    if normalized:
        m = np.cumsum(Q, axis=-2)
        O = O / np.einsum("...ta,...ta->...t", u, m)[..., None]
    return O


# ----------------------------------------------------------------- decay ----
# o_t = sum_{i<=j<=t} gamma^{2t-i-j} (q_t.k_i)(k_i.q_j) v_j: every prefix moment
# decays by gamma per token.  Decode state in P-form: S|P|p.

def _decay_lib() -> ctypes.CDLL:
    lib = _lib(0)
    if not getattr(lib, "_decay_typed", False):
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        d_ = ctypes.c_double
        lib.hla2_oracle_decay_serial.argtypes = [dp, dp, dp, dp, i, i, i, i, i, d_]
        lib.hla2_oracle_decay_bruteforce.argtypes = [dp, dp, dp, dp, i, i, i, i, i, d_]
        lib.hla2_oracle_decay_chunk_summaries.argtypes = [dp, dp, dp, dp, i, i, i, i, i, d_]
        lib.hla2_oracle_decay_combine.argtypes = [dp, dp, dp, i, i, i, d_]
        lib.hla2_oracle_decay_combine.restype = None
        lib.hla2_oracle_decay_chunked.argtypes = [dp, dp, dp, dp, i, i, i, i, i, i, d_]
        lib.hla2_oracle_decay_step_pform.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, d_]
        lib._decay_typed = True
    return lib


def decay_serial(Q, K, V, gamma: float, normalized: bool = False) -> np.ndarray:
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    if _decay_lib().hla2_oracle_decay_serial(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized), float(gamma)):
        raise RuntimeError("oracle decay_serial failed")
    return O.reshape(*lead, T, dv)


def decay_bruteforce(Q, K, V, gamma: float, normalized: bool = False) -> np.ndarray:
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    if _decay_lib().hla2_oracle_decay_bruteforce(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized),
                                                 float(gamma)):
        raise RuntimeError("oracle decay_bruteforce failed")
    return O.reshape(*lead, T, dv)


def decay_chunk_summaries(Q, K, V, L: int, gamma: float) -> np.ndarray:
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    N = (T + L - 1) // L
    out = np.zeros((BH, N, record_len(d, dv)))
    if _decay_lib().hla2_oracle_decay_chunk_summaries(_p(Q), _p(K), _p(V), _p(out), BH, T, d, dv, int(L),
                                                      float(gamma)):
        raise RuntimeError("oracle decay_chunk_summaries failed")
    return out.reshape(*lead, N, record_len(d, dv))


def decay_combine(a, b, d: int, dv: int, nB: int, gamma: float) -> np.ndarray:
    a, b = _f64(a), _f64(b)
    out = np.zeros(record_len(d, dv))
    _decay_lib().hla2_oracle_decay_combine(_p(a), _p(b), _p(out), d, dv, int(nB), float(gamma))
    return out


def decay_chunked(Q, K, V, L: int, gamma: float, normalized: bool = False) -> np.ndarray:
    Q, K, V, lead, BH, T, d, dv = _heads(Q, K, V)
    O = np.zeros((BH, T, dv))
    if _decay_lib().hla2_oracle_decay_chunked(_p(Q), _p(K), _p(V), _p(O), BH, T, d, dv, int(normalized), int(L),
                                              float(gamma)):
        raise RuntimeError("oracle decay_chunked failed")
    return O.reshape(*lead, T, dv)


def decay_step_pform(state, q, k, v, gamma: float, normalized: bool = False):
    """One decayed decode step on the P-form state S|P|p; returns (new_state, o)."""
    state = _f64(state).copy()
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, d = q.shape
    dv = v.shape[1]
    o = np.zeros((n, dv))
    if _decay_lib().hla2_oracle_decay_step_pform(_p(state), _p(q), _p(k), _p(v), _p(o), n, d, dv, int(normalized),
                                                 float(gamma)):
        raise RuntimeError("oracle decay_step_pform failed")
    return state, o
