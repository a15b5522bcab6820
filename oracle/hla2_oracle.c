/*
 * hla2_oracle.c -- plain fp64 CPU oracle for masked second-order HLA.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only through the seeded inputs.
 *
 * Source of every formula ("HLA summary" below): the technical summary pages
 * of "Higher-order Linear Attention" (arXiv 2510.27258) on gist.science, in
 * their Japanese and French editions, which agree section by section.
 *
 *   [§1]  section "1. Second-order HLA": the prefix moments
 *           S_t = sum_{i<=t} k_i k_i^T,  C_t = sum_{i<=t} q_i v_i^T,
 *           m_t = sum_{i<=t} q_i,
 *         the cross summaries G_t, h_t that remove the "future" terms of the
 *         naive product S_t C_t, the unnormalised output
 *           o_t = q_t^T (S_t C_t - G_t),
 *         and a ratio-normalised variant that divides by a masked
 *         denominator built from the analogous summaries.
 *   [§2]  section "2. AHLA": the asymmetric variant, operator
 *         Q (K^T Q)(K^T V), i.e. an A A V structure where HLA has A A^T V,
 *         with streaming summaries P^KV_t, m^K_t, E_t, n_t (the AHLA block
 *         at the end of this file states the reading taken).
 *   [§4]  section "4. Parallel training via associative scans": segment
 *         summaries joined by a semidirect-product operator whose cross term
 *         is S_B C_A; an exclusive Blelloch scan over them reproduces the
 *         serial recurrence exactly.
 *   [R]   section "Results and claims": O(d^2 + d dv) per token, outputs at
 *         time t depend only on tokens j <= t.
 *
 * Readings where the pages are silent (each is pinned by a test):
 *   - The pages name G_t and h_t but print no recurrence for them.  We take
 *       G_t = G_{t-1} + k_t k_t^T C_{t-1},   h_t = h_{t-1} + k_t k_t^T m_{t-1},
 *     the unique choice that makes o_t equal the causal sum
 *       o_t = sum_{0<=i<=j<=t} (q_t.k_i)(k_i.q_j) v_j,
 *     i.e. causal A A^T V with A = tril(Q K^T) and the (t,j) entries of
 *     A A^T kept only for j <= t.  Pinned by the brute-force triple sum.
 *   - Denominator of the normalised variant: den_t = q_t^T (S_t m_t - h_t)
 *     = sum_{i<=j<=t} (q_t.k_i)(k_i.q_j); plain IEEE division, no epsilon.
 *   - Combine (A earlier, B later): S,C,m add; G = G_A + G_B + S_B C_A;
 *     h = h_A + h_B + S_B m_A.  Pinned against the summary of the
 *     concatenated segment.
 *   - State starts at zero; tokens are 0-based.
 *
 * Layouts: Q,K [BH][T][d], V,O [BH][T][dv], row-major fp64.
 * Summary / decode-state record (per head), fp64 row-major, in this order:
 *   S (d*d) | C (d*dv) | m (d) | G (d*dv) | h (d)          ("summary")
 *   S (d*d) | C (d*dv) | G (d*dv) | m (d) | h (d)          ("decode state")
 * The two orders are the ones the CUDA library's interface uses.
 *
 * Build:  gcc -O2 -std=c11 -shared -fPIC -o libhla2_oracle.so hla2_oracle.c -lpthread
 * Defining HLA2_ORACLE_MUTANT=<n> plants one deliberate mistake (tests use
 * this to show that the pins catch it); never defined otherwise.  1-4 are in
 * the HLA functions, 5-6 in the AHLA ones.
 */
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

#ifndef HLA2_ORACLE_MUTANT
#define HLA2_ORACLE_MUTANT 0
#endif

/* ---------------------------------------------------------------------- */
/* One head's running state, G-form, as in [§1].                          */
/* ---------------------------------------------------------------------- */
typedef struct {
    int d, dv;
    double *S, *C, *m, *G, *h; /* d*d, d*dv, d, d*dv, d */
} state_t;

static int state_alloc(state_t* s, int d, int dv) {
    size_t n = (size_t)d * d + 2 * (size_t)d * dv + 2 * (size_t)d;
    double* p = (double*)calloc(n, sizeof(double));
    if (!p) return -1;
    s->d = d; s->dv = dv;
    s->S = p;
    s->C = s->S + (size_t)d * d;
    s->m = s->C + (size_t)d * dv;
    s->G = s->m + d;
    s->h = s->G + (size_t)d * dv;
    return 0;
}
static void state_free(state_t* s) { free(s->S); s->S = 0; }
static void state_zero(state_t* s) {
    size_t n = (size_t)s->d * s->d + 2 * (size_t)s->d * s->dv + 2 * (size_t)s->d;
    memset(s->S, 0, n * sizeof(double));
}

/*
 * Absorb one token (q, k, v) into the state: the online update of [§1].
 * Order matters: G and h use C_{t-1} and m_{t-1}, i.e. before C and m grow.
 * w  = C_{t-1}^T k            (dv)
 * G += k w^T                  (= k k^T C_{t-1})
 * h += k (k . m_{t-1})
 * S += k k^T ;  C += q v^T ;  m += q
 */
static void absorb(state_t* s, const double* q, const double* k, const double* v,
                   double* w /* scratch dv */) {
    const int d = s->d, dv = s->dv;
    for (int e = 0; e < dv; ++e) {
        double acc = 0.0;
        for (int a = 0; a < d; ++a) acc += s->C[(size_t)a * dv + e] * k[a];
        w[e] = acc;
    }
#if HLA2_ORACLE_MUTANT == 3
    /* mistake: uses C_t (after adding q v^T) instead of C_{t-1} */
    {
        double kq = 0.0;
        for (int a = 0; a < d; ++a) kq += k[a] * q[a];
        for (int e = 0; e < dv; ++e) w[e] += kq * v[e];
    }
#endif
    double km = 0.0;
    for (int a = 0; a < d; ++a) km += k[a] * s->m[a];
    for (int a = 0; a < d; ++a) {
        for (int e = 0; e < dv; ++e) s->G[(size_t)a * dv + e] += k[a] * w[e];
        s->h[a] += k[a] * km;
    }
    for (int a = 0; a < d; ++a)
        for (int b = 0; b < d; ++b) s->S[(size_t)a * d + b] += k[a] * k[b];
    for (int a = 0; a < d; ++a)
        for (int e = 0; e < dv; ++e) s->C[(size_t)a * dv + e] += q[a] * v[e];
    for (int a = 0; a < d; ++a) s->m[a] += q[a];
}

/*
 * Output for the current token from the current state, [§1]:
 *   u = S_t q_t ;  o_t = u^T C_t - q_t^T G_t     (never forms S_t C_t: O(d^2 + d dv))
 *   normalised: den_t = u . m_t - q_t . h_t ;  o_t /= den_t
 */
static void emit(const state_t* s, const double* q, double* o, int normalized,
                 double* u /* scratch d */) {
    const int d = s->d, dv = s->dv;
    for (int a = 0; a < d; ++a) {
        double acc = 0.0;
        for (int b = 0; b < d; ++b) acc += s->S[(size_t)a * d + b] * q[b];
        u[a] = acc;
    }
    for (int e = 0; e < dv; ++e) {
        double acc = 0.0;
        for (int a = 0; a < d; ++a) {
#if HLA2_ORACLE_MUTANT == 1
            /* mistake: drops the cross-summary correction G */
            acc += u[a] * s->C[(size_t)a * dv + e];
#elif HLA2_ORACLE_MUTANT == 2
            /* mistake: wrong sign on the correction */
            acc += u[a] * s->C[(size_t)a * dv + e] + q[a] * s->G[(size_t)a * dv + e];
#else
            acc += u[a] * s->C[(size_t)a * dv + e] - q[a] * s->G[(size_t)a * dv + e];
#endif
        }
        o[e] = acc;
    }
    if (normalized) {
        double den = 0.0;
        for (int a = 0; a < d; ++a) den += u[a] * s->m[a] - q[a] * s->h[a];
        for (int e = 0; e < dv; ++e) o[e] /= den;
    }
}

/* ---------------------------------------------------------------------- */
/* Serial recurrence over whole sequences (the oracle proper).            */
/* ---------------------------------------------------------------------- */
typedef struct {
    const double *Q, *K, *V;
    double* O;
    int BH, T, d, dv, normalized;
    int head_begin, head_end;
    int status;
} serial_job_t;

static void* serial_worker(void* arg) {
    serial_job_t* j = (serial_job_t*)arg;
    state_t s;
    if (state_alloc(&s, j->d, j->dv)) { j->status = -1; return 0; }
    double* scratch = (double*)malloc(sizeof(double) * (size_t)(j->d + j->dv));
    if (!scratch) { state_free(&s); j->status = -1; return 0; }
    for (int bh = j->head_begin; bh < j->head_end; ++bh) {
        state_zero(&s);
        const double* Qh = j->Q + (size_t)bh * j->T * j->d;
        const double* Kh = j->K + (size_t)bh * j->T * j->d;
        const double* Vh = j->V + (size_t)bh * j->T * j->dv;
        double* Oh = j->O + (size_t)bh * j->T * j->dv;
        for (int t = 0; t < j->T; ++t) {
            const double* q = Qh + (size_t)t * j->d;
            const double* k = Kh + (size_t)t * j->d;
            const double* v = Vh + (size_t)t * j->dv;
            absorb(&s, q, k, v, scratch);
            emit(&s, q, Oh + (size_t)t * j->dv, j->normalized, scratch);
        }
    }
    free(scratch);
    state_free(&s);
    j->status = 0;
    return 0;
}

/*
 * o_t for every head and token by the serial recurrence of [§1].
 * Heads are independent and split over `nthreads` POSIX threads.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int hla2_oracle_serial(const double* Q, const double* K, const double* V, double* O,
                       int BH, int T, int d, int dv, int normalized, int nthreads) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > BH) nthreads = BH > 0 ? BH : 1;
    serial_job_t* jobs = (serial_job_t*)calloc((size_t)nthreads, sizeof(serial_job_t));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -1; }
    for (int i = 0; i < nthreads; ++i) {
        serial_job_t* j = &jobs[i];
        j->Q = Q; j->K = K; j->V = V; j->O = O;
        j->BH = BH; j->T = T; j->d = d; j->dv = dv; j->normalized = normalized;
        j->head_begin = (int)((long long)BH * i / nthreads);
        j->head_end = (int)((long long)BH * (i + 1) / nthreads);
    }
    int rc = 0;
    if (nthreads == 1) {
        serial_worker(&jobs[0]);
        rc = jobs[0].status;
    } else {
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], 0, serial_worker, &jobs[i]);
        for (int i = 0; i < nthreads; ++i) {
            pthread_join(th[i], 0);
            if (jobs[i].status) rc = -1;
        }
    }
    free(jobs); free(th);
    return rc;
}

/*
 * The plain definition, O(T^3 d): o_t = sum_{i<=j<=t} (q_t.k_i)(k_i.q_j) v_j,
 * den_t = sum_{i<=j<=t} (q_t.k_i)(k_i.q_j).  Only for tiny inputs.
 */
int hla2_oracle_bruteforce(const double* Q, const double* K, const double* V, double* O,
                           int BH, int T, int d, int dv, int normalized) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0) return -1;
    for (int bh = 0; bh < BH; ++bh) {
        const double* Qh = Q + (size_t)bh * T * d;
        const double* Kh = K + (size_t)bh * T * d;
        const double* Vh = V + (size_t)bh * T * dv;
        double* Oh = O + (size_t)bh * T * dv;
        for (int t = 0; t < T; ++t) {
            double* o = Oh + (size_t)t * dv;
            for (int e = 0; e < dv; ++e) o[e] = 0.0;
            double den = 0.0;
            for (int j = 0; j <= t; ++j) {
                for (int i = 0; i <= j; ++i) {
                    double qk = 0.0, kq = 0.0;
                    for (int a = 0; a < d; ++a) {
                        qk += Qh[(size_t)t * d + a] * Kh[(size_t)i * d + a];
                        kq += Kh[(size_t)i * d + a] * Qh[(size_t)j * d + a];
                    }
                    double w = qk * kq;
                    den += w;
                    for (int e = 0; e < dv; ++e) o[e] += w * Vh[(size_t)j * dv + e];
                }
            }
            if (normalized)
                for (int e = 0; e < dv; ++e) o[e] /= den;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Segment summaries, combine and scans, [§4].                            */
/* ---------------------------------------------------------------------- */
static size_t summary_len(int d, int dv) {
    return (size_t)d * d + 2 * (size_t)d * dv + 2 * (size_t)d;
}

/* copy a G-form state into a summary record S|C|m|G|h */
static void state_to_summary(const state_t* s, double* r) {
    const int d = s->d, dv = s->dv;
    size_t o = 0;
    memcpy(r + o, s->S, sizeof(double) * (size_t)d * d); o += (size_t)d * d;
    memcpy(r + o, s->C, sizeof(double) * (size_t)d * dv); o += (size_t)d * dv;
    memcpy(r + o, s->m, sizeof(double) * (size_t)d); o += d;
    memcpy(r + o, s->G, sizeof(double) * (size_t)d * dv); o += (size_t)d * dv;
    memcpy(r + o, s->h, sizeof(double) * (size_t)d);
}
static void summary_to_state(const double* r, state_t* s) {
    const int d = s->d, dv = s->dv;
    size_t o = 0;
    memcpy(s->S, r + o, sizeof(double) * (size_t)d * d); o += (size_t)d * d;
    memcpy(s->C, r + o, sizeof(double) * (size_t)d * dv); o += (size_t)d * dv;
    memcpy(s->m, r + o, sizeof(double) * (size_t)d); o += d;
    memcpy(s->G, r + o, sizeof(double) * (size_t)d * dv); o += (size_t)d * dv;
    memcpy(s->h, r + o, sizeof(double) * (size_t)d);
}

/*
 * Summary of every chunk of L tokens (the last one may be shorter): the state
 * the recurrence of [§1] reaches from zero on that chunk alone.  Output
 * [BH][N][record], N = ceil(T/L), record S|C|m|G|h.
 */
int hla2_oracle_chunk_summaries(const double* Q, const double* K, const double* V,
                                double* summ, int BH, int T, int d, int dv, int L) {
    if (!Q || !K || !V || !summ || BH < 0 || T < 0 || d <= 0 || dv <= 0 || L <= 0) return -1;
    const int N = (T + L - 1) / L;
    const size_t R = summary_len(d, dv);
    state_t s;
    if (state_alloc(&s, d, dv)) return -1;
    double* w = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!w) { state_free(&s); return -1; }
    for (int bh = 0; bh < BH; ++bh) {
        for (int c = 0; c < N; ++c) {
            state_zero(&s);
            int t1 = (c + 1) * L < T ? (c + 1) * L : T;
            for (int t = c * L; t < t1; ++t)
                absorb(&s, Q + ((size_t)bh * T + t) * d, K + ((size_t)bh * T + t) * d,
                       V + ((size_t)bh * T + t) * dv, w);
            state_to_summary(&s, summ + ((size_t)bh * N + c) * R);
        }
    }
    free(w);
    state_free(&s);
    return 0;
}

/*
 * The semidirect-product combine of [§4]; A is the earlier segment:
 *   S = S_A + S_B, C = C_A + C_B, m = m_A + m_B,
 *   G = G_A + G_B + S_B C_A,  h = h_A + h_B + S_B m_A.
 * `out` may alias neither input.
 */
void hla2_oracle_combine(const double* A, const double* B, double* out, int d, int dv) {
    const size_t nS = (size_t)d * d, nC = (size_t)d * dv;
    const double *SA = A, *CA = A + nS, *mA = CA + nC, *GA = mA + d, *hA = GA + nC;
    const double *SB = B, *CB = B + nS, *mB = CB + nC, *GB = mB + d, *hB = GB + nC;
    double *S = out, *C = out + nS, *m = C + nC, *G = m + d, *h = G + nC;
    for (size_t i = 0; i < nS; ++i) S[i] = SA[i] + SB[i];
    for (size_t i = 0; i < nC; ++i) C[i] = CA[i] + CB[i];
    for (int i = 0; i < d; ++i) m[i] = mA[i] + mB[i];
    for (int a = 0; a < d; ++a) {
        for (int e = 0; e < dv; ++e) {
            double acc = 0.0;
            for (int b = 0; b < d; ++b) acc += SB[(size_t)a * d + b] * CA[(size_t)b * dv + e];
#if HLA2_ORACLE_MUTANT == 4
            /* mistake: cross term with the operands swapped (S_A C_B) */
            acc = 0.0;
            for (int b = 0; b < d; ++b) acc += SA[(size_t)a * d + b] * CB[(size_t)b * dv + e];
#endif
            G[(size_t)a * dv + e] = GA[(size_t)a * dv + e] + GB[(size_t)a * dv + e] + acc;
        }
        double acc = 0.0;
        for (int b = 0; b < d; ++b) acc += SB[(size_t)a * d + b] * mA[b];
        h[a] = hA[a] + hB[a] + acc;
    }
}

/*
 * Exclusive scan by a left fold: prefix[0] = identity (all zeros),
 * prefix[n] = combine(prefix[n-1], summ[n-1]).  [BH][N][record] in and out.
 */
int hla2_oracle_scan_fold(const double* summ, double* prefix, int BH, int N, int d, int dv) {
    if (!summ || !prefix || BH < 0 || N < 0 || d <= 0 || dv <= 0) return -1;
    const size_t R = summary_len(d, dv);
    for (int bh = 0; bh < BH; ++bh) {
        const double* in = summ + (size_t)bh * N * R;
        double* out = prefix + (size_t)bh * N * R;
        if (N == 0) continue;
        memset(out, 0, sizeof(double) * R);
        for (int n = 1; n < N; ++n) hla2_oracle_combine(out + (n - 1) * R, in + (n - 1) * R, out + n * R, d, dv);
    }
    return 0;
}

/*
 * Exclusive Blelloch scan (work-efficient up-sweep then down-sweep) with the
 * non-commutative combine of [§4].  The array is padded with identities to a
 * power of two.  In the down-sweep a left child receives its parent's prefix
 * and a right child receives combine(parent prefix, left child's total), so
 * every prefix composes in time order (earlier then later).
 */
int hla2_oracle_scan_blelloch(const double* summ, double* prefix, int BH, int N, int d, int dv) {
    if (!summ || !prefix || BH < 0 || N < 0 || d <= 0 || dv <= 0) return -1;
    const size_t R = summary_len(d, dv);
    int P = 1;
    while (P < N) P <<= 1;
    double* x = (double*)malloc(sizeof(double) * R * (size_t)P);
    double* tmp = (double*)malloc(sizeof(double) * R);
    if (!x || !tmp) { free(x); free(tmp); return -1; }
    for (int bh = 0; bh < BH; ++bh) {
        if (N == 0) continue;
        memset(x, 0, sizeof(double) * R * (size_t)P);
        memcpy(x, summ + (size_t)bh * N * R, sizeof(double) * R * (size_t)N);
        /* up-sweep: x[right] <- combine(x[left], x[right]) */
        for (int stride = 1; stride < P; stride <<= 1) {
            for (int i = 2 * stride - 1; i < P; i += 2 * stride) {
                hla2_oracle_combine(x + (size_t)(i - stride) * R, x + (size_t)i * R, tmp, d, dv);
                memcpy(x + (size_t)i * R, tmp, sizeof(double) * R);
            }
        }
        /* down-sweep */
        memset(x + (size_t)(P - 1) * R, 0, sizeof(double) * R);
        for (int stride = P >> 1; stride >= 1; stride >>= 1) {
            for (int i = 2 * stride - 1; i < P; i += 2 * stride) {
                double* left = x + (size_t)(i - stride) * R;
                double* right = x + (size_t)i * R;
                /* new right = combine(parent prefix (in right), left total) */
                hla2_oracle_combine(right, left, tmp, d, dv);
                memcpy(left, right, sizeof(double) * R); /* left <- parent prefix */
                memcpy(right, tmp, sizeof(double) * R);
            }
        }
        memcpy(prefix + (size_t)bh * N * R, x, sizeof(double) * R * (size_t)N);
    }
    free(x); free(tmp);
    return 0;
}

/*
 * The chunk-parallel method of [§4] in fp64: chunk summaries, exclusive
 * Blelloch scan, then every chunk restarts the serial recurrence from its
 * exclusive prefix state and emits its outputs.  [§4] states that this is
 * exactly the serial recurrence.
 */
int hla2_oracle_chunked(const double* Q, const double* K, const double* V, double* O,
                        int BH, int T, int d, int dv, int normalized, int L) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0 || L <= 0) return -1;
    const int N = (T + L - 1) / L;
    const size_t R = summary_len(d, dv);
    double* summ = (double*)malloc(sizeof(double) * R * (size_t)(N > 0 ? N : 1) * (size_t)(BH > 0 ? BH : 1));
    double* pre = (double*)malloc(sizeof(double) * R * (size_t)(N > 0 ? N : 1) * (size_t)(BH > 0 ? BH : 1));
    double* scratch = (double*)malloc(sizeof(double) * (size_t)(d + dv));
    state_t s;
    int rc = -1;
    if (!summ || !pre || !scratch || state_alloc(&s, d, dv)) goto done;
    if (hla2_oracle_chunk_summaries(Q, K, V, summ, BH, T, d, dv, L)) goto done_s;
    if (hla2_oracle_scan_blelloch(summ, pre, BH, N, d, dv)) goto done_s;
    for (int bh = 0; bh < BH; ++bh) {
        for (int c = 0; c < N; ++c) {
            summary_to_state(pre + ((size_t)bh * N + c) * R, &s);
            int t1 = (c + 1) * L < T ? (c + 1) * L : T;
            for (int t = c * L; t < t1; ++t) {
                const double* q = Q + ((size_t)bh * T + t) * d;
                absorb(&s, q, K + ((size_t)bh * T + t) * d, V + ((size_t)bh * T + t) * dv, scratch);
                emit(&s, q, O + ((size_t)bh * T + t) * dv, normalized, scratch);
            }
        }
    }
    rc = 0;
done_s:
    state_free(&s);
done:
    free(summ); free(pre); free(scratch);
    return rc;
}

/*
 * One streaming decode step for n independent heads, [§1] online update:
 * absorb (q,k,v) into each head's state, then emit o.  State record per head
 * (decode order) S|C|G|m|h, updated in place.  q,k [n][d], v,o [n][dv].
 */
int hla2_oracle_step(double* state, const double* q, const double* k, const double* v,
                     double* o, int n, int d, int dv, int normalized) {
    if (!state || !q || !k || !v || !o || n < 0 || d <= 0 || dv <= 0) return -1;
    const size_t R = summary_len(d, dv);
    state_t s;
    if (state_alloc(&s, d, dv)) return -1;
    double* scratch = (double*)malloc(sizeof(double) * (size_t)(d + dv));
    if (!scratch) { state_free(&s); return -1; }
    const size_t nS = (size_t)d * d, nC = (size_t)d * dv;
    for (int i = 0; i < n; ++i) {
        double* r = state + (size_t)i * R;
        /* decode order S|C|G|m|h -> working state */
        memcpy(s.S, r, sizeof(double) * nS);
        memcpy(s.C, r + nS, sizeof(double) * nC);
        memcpy(s.G, r + nS + nC, sizeof(double) * nC);
        memcpy(s.m, r + nS + 2 * nC, sizeof(double) * (size_t)d);
        memcpy(s.h, r + nS + 2 * nC + d, sizeof(double) * (size_t)d);
        absorb(&s, q + (size_t)i * d, k + (size_t)i * d, v + (size_t)i * dv, scratch);
        emit(&s, q + (size_t)i * d, o + (size_t)i * dv, normalized, scratch);
        memcpy(r, s.S, sizeof(double) * nS);
        memcpy(r + nS, s.C, sizeof(double) * nC);
        memcpy(r + nS + nC, s.G, sizeof(double) * nC);
        memcpy(r + nS + 2 * nC, s.m, sizeof(double) * (size_t)d);
        memcpy(r + nS + 2 * nC + d, s.h, sizeof(double) * (size_t)d);
    }
    free(scratch);
    state_free(&s);
    return 0;
}

/* Record length in doubles (same for summary and decode order). */
long long hla2_oracle_record_len(int d, int dv) { return (long long)summary_len(d, dv); }

/* ====================================================================== */
/* AHLA: asymmetric second-order variant, HLA summary section 2.          */
/*                                                                        */
/* The pages give the operator Q (K^T Q)(K^T V) and name its streaming    */
/* summaries P^KV_t, m^K_t, E_t, n_t, without printing their updates.     */
/* Reading (pinned by brute force): causal A A V with A = tril(Q K^T),    */
/*   o_t = sum_{j<=i<=t} (q_t.k_i)(q_i.k_j) v_j,                         */
/* i.e. query t reaches key i, whose query i reaches key j <= i:          */
/*   P_t = P_{t-1} + k_t v_t^T       m_t = m_{t-1} + k_t                  */
/*   E_t = E_{t-1} + k_t (q_t^T P_t) n_t = n_{t-1} + k_t (q_t . m_t)      */
/*   o_t = q_t^T E_t ;  normalised: o_t / (q_t^T n_t).                    */
/* Segment summary record (same length as HLA's):                         */
/*   M (d*d, = sum k q^T) | P (d*dv) | m (d) | E (d*dv) | n (d)            */
/* and the combine (A earlier, B later) is HLA's with S->M, C->P, G->E:   */
/*   M, P, m add;  E = E_A + E_B + M_B P_A;  n = n_A + n_B + M_B m_A.    */
/* ====================================================================== */
typedef struct {
    int d, dv;
    double *M, *P, *m, *E, *n; /* d*d, d*dv, d, d*dv, d */
} astate_t;

static int astate_alloc(astate_t* s, int d, int dv) {
    double* p = (double*)calloc(summary_len(d, dv), sizeof(double));
    if (!p) return -1;
    s->d = d; s->dv = dv;
    s->M = p;
    s->P = s->M + (size_t)d * d;
    s->m = s->P + (size_t)d * dv;
    s->E = s->m + d;
    s->n = s->E + (size_t)d * dv;
    return 0;
}
static void astate_zero(astate_t* s) { memset(s->M, 0, sizeof(double) * summary_len(s->d, s->dv)); }

/* absorb token t (P and m grow first: E and n use P_t and m_t) */
static void ahla_absorb(astate_t* s, const double* q, const double* k, const double* v, double* w) {
    const int d = s->d, dv = s->dv;
#if HLA2_ORACLE_MUTANT == 5
    /* mistake: E and n read P_{t-1}, m_{t-1} (drops the j = i terms) */
    for (int e = 0; e < dv; ++e) {
        double acc = 0.0;
        for (int a = 0; a < d; ++a) acc += q[a] * s->P[(size_t)a * dv + e];
        w[e] = acc;
    }
    double qm = 0.0;
    for (int a = 0; a < d; ++a) qm += q[a] * s->m[a];
#endif
    for (int a = 0; a < d; ++a) {
        for (int e = 0; e < dv; ++e) s->P[(size_t)a * dv + e] += k[a] * v[e];
        s->m[a] += k[a];
#if HLA2_ORACLE_MUTANT == 6
        /* mistake: cross operand transposed (sum q k^T instead of k q^T) */
        for (int b = 0; b < d; ++b) s->M[(size_t)a * d + b] += q[a] * k[b];
#else
        for (int b = 0; b < d; ++b) s->M[(size_t)a * d + b] += k[a] * q[b];
#endif
    }
#if HLA2_ORACLE_MUTANT != 5
    for (int e = 0; e < dv; ++e) {
        double acc = 0.0;
        for (int a = 0; a < d; ++a) acc += q[a] * s->P[(size_t)a * dv + e];
        w[e] = acc;
    }
    double qm = 0.0;
    for (int a = 0; a < d; ++a) qm += q[a] * s->m[a];
#endif
    for (int a = 0; a < d; ++a) {
        for (int e = 0; e < dv; ++e) s->E[(size_t)a * dv + e] += k[a] * w[e];
        s->n[a] += k[a] * qm;
    }
}
static void ahla_emit(const astate_t* s, const double* q, double* o, int normalized) {
    const int d = s->d, dv = s->dv;
    for (int e = 0; e < dv; ++e) {
        double acc = 0.0;
        for (int a = 0; a < d; ++a) acc += q[a] * s->E[(size_t)a * dv + e];
        o[e] = acc;
    }
    if (normalized) {
        double den = 0.0;
        for (int a = 0; a < d; ++a) den += q[a] * s->n[a];
        for (int e = 0; e < dv; ++e) o[e] /= den;
    }
}

/* AHLA outputs by the serial recurrence. */
int hla2_oracle_ahla_serial(const double* Q, const double* K, const double* V, double* O,
                            int BH, int T, int d, int dv, int normalized) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0) return -1;
    astate_t s;
    if (astate_alloc(&s, d, dv)) return -1;
    double* w = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!w) { free(s.M); return -1; }
    for (int bh = 0; bh < BH; ++bh) {
        astate_zero(&s);
        for (int t = 0; t < T; ++t) {
            const double* q = Q + ((size_t)bh * T + t) * d;
            ahla_absorb(&s, q, K + ((size_t)bh * T + t) * d, V + ((size_t)bh * T + t) * dv, w);
            ahla_emit(&s, q, O + ((size_t)bh * T + t) * dv, normalized);
        }
    }
    free(w);
    free(s.M);
    return 0;
}

/* The definition, O(T^3 d): o_t = sum_{j<=i<=t} (q_t.k_i)(q_i.k_j) v_j. */
int hla2_oracle_ahla_bruteforce(const double* Q, const double* K, const double* V, double* O,
                                int BH, int T, int d, int dv, int normalized) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0) return -1;
    for (int bh = 0; bh < BH; ++bh) {
        const double* Qh = Q + (size_t)bh * T * d;
        const double* Kh = K + (size_t)bh * T * d;
        const double* Vh = V + (size_t)bh * T * dv;
        for (int t = 0; t < T; ++t) {
            double* o = O + ((size_t)bh * T + t) * dv;
            for (int e = 0; e < dv; ++e) o[e] = 0.0;
            double den = 0.0;
            for (int i = 0; i <= t; ++i) {
                double qk_ti = 0.0;
                for (int a = 0; a < d; ++a) qk_ti += Qh[(size_t)t * d + a] * Kh[(size_t)i * d + a];
                for (int j = 0; j <= i; ++j) {
                    double qk_ij = 0.0;
                    for (int a = 0; a < d; ++a) qk_ij += Qh[(size_t)i * d + a] * Kh[(size_t)j * d + a];
                    const double wgt = qk_ti * qk_ij;
                    den += wgt;
                    for (int e = 0; e < dv; ++e) o[e] += wgt * Vh[(size_t)j * dv + e];
                }
            }
            if (normalized)
                for (int e = 0; e < dv; ++e) o[e] /= den;
        }
    }
    return 0;
}

/* AHLA chunk summaries M|P|m|E|n of every L-token chunk (state from zero). */
int hla2_oracle_ahla_chunk_summaries(const double* Q, const double* K, const double* V,
                                     double* summ, int BH, int T, int d, int dv, int L) {
    if (!Q || !K || !V || !summ || BH < 0 || T < 0 || d <= 0 || dv <= 0 || L <= 0) return -1;
    const int N = (T + L - 1) / L;
    const size_t R = summary_len(d, dv);
    astate_t s;
    if (astate_alloc(&s, d, dv)) return -1;
    double* w = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!w) { free(s.M); return -1; }
    for (int bh = 0; bh < BH; ++bh)
        for (int c = 0; c < N; ++c) {
            astate_zero(&s);
            const int t1 = (c + 1) * L < T ? (c + 1) * L : T;
            for (int t = c * L; t < t1; ++t)
                ahla_absorb(&s, Q + ((size_t)bh * T + t) * d, K + ((size_t)bh * T + t) * d,
                            V + ((size_t)bh * T + t) * dv, w);
            memcpy(summ + ((size_t)bh * N + c) * R, s.M, sizeof(double) * R);
        }
    free(w);
    free(s.M);
    return 0;
}

/* AHLA chunked forward: chunk summaries, exclusive Blelloch scan with the
 * combine above (the HLA combine routine, whose algebra is the same), then
 * every chunk restarts the recurrence from its prefix. */
int hla2_oracle_ahla_chunked(const double* Q, const double* K, const double* V, double* O,
                             int BH, int T, int d, int dv, int normalized, int L) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0 || L <= 0) return -1;
    const int N = (T + L - 1) / L;
    const size_t R = summary_len(d, dv);
    double* summ = (double*)malloc(sizeof(double) * R * (size_t)(N > 0 ? N : 1) * (size_t)(BH > 0 ? BH : 1));
    double* pre = (double*)malloc(sizeof(double) * R * (size_t)(N > 0 ? N : 1) * (size_t)(BH > 0 ? BH : 1));
    double* w = (double*)malloc(sizeof(double) * (size_t)dv);
    astate_t s;
    int rc = -1;
    if (!summ || !pre || !w || astate_alloc(&s, d, dv)) goto out;
    if (hla2_oracle_ahla_chunk_summaries(Q, K, V, summ, BH, T, d, dv, L) ||
        hla2_oracle_scan_blelloch(summ, pre, BH, N, d, dv)) {
        free(s.M);
        goto out;
    }
    for (int bh = 0; bh < BH; ++bh)
        for (int c = 0; c < N; ++c) {
            memcpy(s.M, pre + ((size_t)bh * N + c) * R, sizeof(double) * R);
            const int t1 = (c + 1) * L < T ? (c + 1) * L : T;
            for (int t = c * L; t < t1; ++t) {
                const double* q = Q + ((size_t)bh * T + t) * d;
                ahla_absorb(&s, q, K + ((size_t)bh * T + t) * d, V + ((size_t)bh * T + t) * dv, w);
                ahla_emit(&s, q, O + ((size_t)bh * T + t) * dv, normalized);
            }
        }
    free(s.M);
    rc = 0;
out:
    free(summ); free(pre); free(w);
    return rc;
}

/* One AHLA decode step for n heads; state per head P|E|m|n (2 d dv + 2 d). */
int hla2_oracle_ahla_step(double* state, const double* q, const double* k, const double* v,
                          double* o, int n, int d, int dv, int normalized) {
    if (!state || !q || !k || !v || !o || n < 0 || d <= 0 || dv <= 0) return -1;
    astate_t s;
    if (astate_alloc(&s, d, dv)) return -1;
    double* w = (double*)malloc(sizeof(double) * (size_t)dv);
    if (!w) { free(s.M); return -1; }
    const size_t nC = (size_t)d * dv, R = 2 * nC + 2 * (size_t)d;
    for (int i = 0; i < n; ++i) {
        double* r = state + (size_t)i * R;
        memcpy(s.P, r, sizeof(double) * nC);
        memcpy(s.E, r + nC, sizeof(double) * nC);
        memcpy(s.m, r + 2 * nC, sizeof(double) * (size_t)d);
        memcpy(s.n, r + 2 * nC + d, sizeof(double) * (size_t)d);
        ahla_absorb(&s, q + (size_t)i * d, k + (size_t)i * d, v + (size_t)i * dv, w);
        ahla_emit(&s, q + (size_t)i * d, o + (size_t)i * dv, normalized);
        memcpy(r, s.P, sizeof(double) * nC);
        memcpy(r + nC, s.E, sizeof(double) * nC);
        memcpy(r + 2 * nC, s.m, sizeof(double) * (size_t)d);
        memcpy(r + 2 * nC + d, s.n, sizeof(double) * (size_t)d);
    }
    free(w);
    free(s.M);
    return 0;
}

/* ====================================================================== */
/* Unmasked second-order HLA: o_t = q_t^T S_t C_t (HLA summary, section 1 */
/* names the naive product S_t C_t that G_t corrects; the "Results and    */
/* claims" section lists the unmasked operator among the variants).       */
/*   o_t = sum_{i<=t} sum_{j<=t} (q_t.k_i)(k_i.q_j) v_j                   */
/* normalised: o_t / (q_t^T S_t m_t).  State S, C, m only; segments join  */
/* by plain addition (no cross term), so a scan is a running sum.         */
/* Decode state per head: S (d*d) | C (d*dv) | m (d).                     */
/* ====================================================================== */
static void unmasked_absorb(double* S, double* C, double* m, const double* q, const double* k, const double* v,
                            int d, int dv) {
    for (int a = 0; a < d; ++a) {
        for (int b = 0; b < d; ++b) S[(size_t)a * d + b] += k[a] * k[b];
        for (int e = 0; e < dv; ++e) C[(size_t)a * dv + e] += q[a] * v[e];
        m[a] += q[a];
    }
}
static void unmasked_emit(const double* S, const double* C, const double* m, const double* q, double* o,
                          double* u, int d, int dv, int normalized) {
    for (int a = 0; a < d; ++a) {
        double acc = 0.0;
        for (int b = 0; b < d; ++b) acc += S[(size_t)a * d + b] * q[b];
        u[a] = acc;
    }
    for (int e = 0; e < dv; ++e) {
        double acc = 0.0;
        for (int a = 0; a < d; ++a) acc += u[a] * C[(size_t)a * dv + e];
        o[e] = acc;
    }
    if (normalized) {
        double den = 0.0;
        for (int a = 0; a < d; ++a) den += u[a] * m[a];
        for (int e = 0; e < dv; ++e) o[e] /= den;
    }
}

/* Unmasked outputs by the serial recurrence. */
int hla2_oracle_unmasked_serial(const double* Q, const double* K, const double* V, double* O,
                                int BH, int T, int d, int dv, int normalized) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0) return -1;
    const size_t n = (size_t)d * d + (size_t)d * dv + (size_t)d + (size_t)d;
    double* buf = (double*)malloc(sizeof(double) * n);
    if (!buf) return -1;
    double *S = buf, *C = S + (size_t)d * d, *m = C + (size_t)d * dv, *u = m + d;
    for (int bh = 0; bh < BH; ++bh) {
        memset(buf, 0, sizeof(double) * n);
        for (int t = 0; t < T; ++t) {
            const double* q = Q + ((size_t)bh * T + t) * d;
            unmasked_absorb(S, C, m, q, K + ((size_t)bh * T + t) * d, V + ((size_t)bh * T + t) * dv, d, dv);
            unmasked_emit(S, C, m, q, O + ((size_t)bh * T + t) * dv, u, d, dv, normalized);
        }
    }
    free(buf);
    return 0;
}

/* The definition, O(T^3 d): every pair i <= t, j <= t. */
int hla2_oracle_unmasked_bruteforce(const double* Q, const double* K, const double* V, double* O,
                                    int BH, int T, int d, int dv, int normalized) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0) return -1;
    for (int bh = 0; bh < BH; ++bh) {
        const double* Qh = Q + (size_t)bh * T * d;
        const double* Kh = K + (size_t)bh * T * d;
        const double* Vh = V + (size_t)bh * T * dv;
        for (int t = 0; t < T; ++t) {
            double* o = O + ((size_t)bh * T + t) * dv;
            for (int e = 0; e < dv; ++e) o[e] = 0.0;
            double den = 0.0;
            for (int i = 0; i <= t; ++i) {
                double qk = 0.0;
                for (int a = 0; a < d; ++a) qk += Qh[(size_t)t * d + a] * Kh[(size_t)i * d + a];
                for (int j = 0; j <= t; ++j) {
                    double kq = 0.0;
                    for (int a = 0; a < d; ++a) kq += Kh[(size_t)i * d + a] * Qh[(size_t)j * d + a];
                    den += qk * kq;
                    for (int e = 0; e < dv; ++e) o[e] += qk * kq * Vh[(size_t)j * dv + e];
                }
            }
            if (normalized)
                for (int e = 0; e < dv; ++e) o[e] /= den;
        }
    }
    return 0;
}

/* One unmasked decode step for n heads; state per head S|C|m. */
int hla2_oracle_unmasked_step(double* state, const double* q, const double* k, const double* v,
                              double* o, int n, int d, int dv, int normalized) {
    if (!state || !q || !k || !v || !o || n < 0 || d <= 0 || dv <= 0) return -1;
    double* u = (double*)malloc(sizeof(double) * (size_t)d);
    if (!u) return -1;
    const size_t R = (size_t)d * d + (size_t)d * dv + (size_t)d;
    for (int i = 0; i < n; ++i) {
        double* S = state + (size_t)i * R;
        double* C = S + (size_t)d * d;
        double* m = C + (size_t)d * dv;
        unmasked_absorb(S, C, m, q + (size_t)i * d, k + (size_t)i * d, v + (size_t)i * dv, d, dv);
        unmasked_emit(S, C, m, q + (size_t)i * d, o + (size_t)i * dv, u, d, dv, normalized);
    }
    free(u);
    return 0;
}

/* ====================================================================== */
/* Exponentially decayed masked operator (HLA summary, section 4 lists     */
/* decayed variants among the operators the scan covers; the decay form is */
/* not printed).  Reading: one scalar gamma in (0, 1] decays every prefix  */
/* moment per token,                                                       */
/*   S_t = g S + k k^T,  C_t = g C + q v^T,  m_t = g m + q,                */
/*   G_t = g^2 G + g k k^T C_{t-1},  h_t = g^2 h + g k k^T m_{t-1},        */
/*   o_t = q_t^T (S_t C_t - G_t)                                           */
/*       = sum_{i<=j<=t} g^{2t-i-j} (q_t.k_i)(k_i.q_j) v_j,                 */
/* normalised by q_t^T (S_t m_t - h_t).  gamma = 1 is the masked operator. */
/* Compact (P-form) decode state S | P | p with P = S C - G, p = S m - h:  */
/*   S_t = g S + k k^T, u = S_t q, P_t = g^2 P + u v^T, p_t = g^2 p + u.   */
/* Segment combine (A earlier, B later, B spanning n_B tokens, f = g^n_B): */
/*   S = f S_A + S_B, C = f C_A + C_B, m = f m_A + m_B,                    */
/*   G = f^2 G_A + G_B + f S_B C_A,  h = f^2 h_A + h_B + f S_B m_A.        */
/* ====================================================================== */
static void decay_absorb(state_t* s, const double* q, const double* k, const double* v, double g, double* w) {
    const int d = s->d, dv = s->dv;
    for (int e = 0; e < dv; ++e) {
        double acc = 0.0;
        for (int a = 0; a < d; ++a) acc += s->C[(size_t)a * dv + e] * k[a];
        w[e] = acc;
    }
    double km = 0.0;
    for (int a = 0; a < d; ++a) km += k[a] * s->m[a];
    for (int a = 0; a < d; ++a) {
        for (int e = 0; e < dv; ++e)
            s->G[(size_t)a * dv + e] = g * g * s->G[(size_t)a * dv + e] + g * k[a] * w[e];
        s->h[a] = g * g * s->h[a] + g * k[a] * km;
    }
    for (int a = 0; a < d; ++a)
        for (int b = 0; b < d; ++b) s->S[(size_t)a * d + b] = g * s->S[(size_t)a * d + b] + k[a] * k[b];
    for (int a = 0; a < d; ++a)
        for (int e = 0; e < dv; ++e) s->C[(size_t)a * dv + e] = g * s->C[(size_t)a * dv + e] + q[a] * v[e];
    for (int a = 0; a < d; ++a) s->m[a] = g * s->m[a] + q[a];
}

/* Decayed outputs by the serial recurrence (G-form). */
int hla2_oracle_decay_serial(const double* Q, const double* K, const double* V, double* O,
                             int BH, int T, int d, int dv, int normalized, double gamma) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0) return -1;
    state_t s;
    if (state_alloc(&s, d, dv)) return -1;
    double* scratch = (double*)malloc(sizeof(double) * (size_t)(d + dv));
    if (!scratch) { state_free(&s); return -1; }
    for (int bh = 0; bh < BH; ++bh) {
        state_zero(&s);
        for (int t = 0; t < T; ++t) {
            const double* q = Q + ((size_t)bh * T + t) * d;
            decay_absorb(&s, q, K + ((size_t)bh * T + t) * d, V + ((size_t)bh * T + t) * dv, gamma, scratch);
            emit(&s, q, O + ((size_t)bh * T + t) * dv, normalized, scratch);
        }
    }
    free(scratch);
    state_free(&s);
    return 0;
}

/* The definition, O(T^3 d): weights gamma^{2t-i-j} over i <= j <= t. */
int hla2_oracle_decay_bruteforce(const double* Q, const double* K, const double* V, double* O,
                                 int BH, int T, int d, int dv, int normalized, double gamma) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0) return -1;
    for (int bh = 0; bh < BH; ++bh) {
        const double* Qh = Q + (size_t)bh * T * d;
        const double* Kh = K + (size_t)bh * T * d;
        const double* Vh = V + (size_t)bh * T * dv;
        for (int t = 0; t < T; ++t) {
            double* o = O + ((size_t)bh * T + t) * dv;
            for (int e = 0; e < dv; ++e) o[e] = 0.0;
            double den = 0.0;
            for (int i = 0; i <= t; ++i) {
                double qk = 0.0;
                for (int a = 0; a < d; ++a) qk += Qh[(size_t)t * d + a] * Kh[(size_t)i * d + a];
                for (int j = i; j <= t; ++j) {
                    double kq = 0.0;
                    for (int a = 0; a < d; ++a) kq += Kh[(size_t)i * d + a] * Qh[(size_t)j * d + a];
                    double wgt = qk * kq;
                    for (int r = 0; r < 2 * t - i - j; ++r) wgt *= gamma;
                    den += wgt;
                    for (int e = 0; e < dv; ++e) o[e] += wgt * Vh[(size_t)j * dv + e];
                }
            }
            if (normalized)
                for (int e = 0; e < dv; ++e) o[e] /= den;
        }
    }
    return 0;
}

/* Decayed chunk summaries S|C|m|G|h of every L-token chunk (state from zero). */
int hla2_oracle_decay_chunk_summaries(const double* Q, const double* K, const double* V, double* summ,
                                      int BH, int T, int d, int dv, int L, double gamma) {
    if (!Q || !K || !V || !summ || BH < 0 || T < 0 || d <= 0 || dv <= 0 || L <= 0) return -1;
    const int N = (T + L - 1) / L;
    const size_t R = summary_len(d, dv);
    state_t s;
    if (state_alloc(&s, d, dv)) return -1;
    double* w = (double*)malloc(sizeof(double) * (size_t)(d + dv));
    if (!w) { state_free(&s); return -1; }
    for (int bh = 0; bh < BH; ++bh)
        for (int c = 0; c < N; ++c) {
            state_zero(&s);
            const int t1 = (c + 1) * L < T ? (c + 1) * L : T;
            for (int t = c * L; t < t1; ++t)
                decay_absorb(&s, Q + ((size_t)bh * T + t) * d, K + ((size_t)bh * T + t) * d,
                             V + ((size_t)bh * T + t) * dv, gamma, w);
            memcpy(summ + ((size_t)bh * N + c) * R, s.S, sizeof(double) * R);
        }
    free(w);
    state_free(&s);
    return 0;
}

/* Decayed combine: A earlier, B later spanning nB tokens. */
void hla2_oracle_decay_combine(const double* A, const double* B, double* out, int d, int dv, int nB, double gamma) {
    const size_t nS = (size_t)d * d, nC = (size_t)d * dv;
    const double *SA = A, *CA = A + nS, *mA = CA + nC, *GA = mA + d, *hA = GA + nC;
    const double *SB = B, *CB = B + nS, *mB = CB + nC, *GB = mB + d, *hB = GB + nC;
    double *S = out, *C = out + nS, *m = C + nC, *G = m + d, *h = G + nC;
    double f = 1.0;
    for (int r = 0; r < nB; ++r) f *= gamma;
    for (int a = 0; a < d; ++a) {
        for (int e = 0; e < dv; ++e) {
            double acc = 0.0;
            for (int b = 0; b < d; ++b) acc += SB[(size_t)a * d + b] * CA[(size_t)b * dv + e];
            G[(size_t)a * dv + e] = f * f * GA[(size_t)a * dv + e] + GB[(size_t)a * dv + e] + f * acc;
        }
        double acc = 0.0;
        for (int b = 0; b < d; ++b) acc += SB[(size_t)a * d + b] * mA[b];
        h[a] = f * f * hA[a] + hB[a] + f * acc;
    }
    for (size_t i = 0; i < nS; ++i) S[i] = f * SA[i] + SB[i];
    for (size_t i = 0; i < nC; ++i) C[i] = f * CA[i] + CB[i];
    for (int i = 0; i < d; ++i) m[i] = f * mA[i] + mB[i];
}

/* Decayed chunked forward: chunk summaries, an exclusive left fold with the
 * decayed combine, then every chunk restarts the recurrence from its prefix. */
int hla2_oracle_decay_chunked(const double* Q, const double* K, const double* V, double* O,
                              int BH, int T, int d, int dv, int normalized, int L, double gamma) {
    if (!Q || !K || !V || !O || BH < 0 || T < 0 || d <= 0 || dv <= 0 || L <= 0) return -1;
    const int N = (T + L - 1) / L;
    const size_t R = summary_len(d, dv);
    const size_t NB = (size_t)(N > 0 ? N : 1) * (size_t)(BH > 0 ? BH : 1);
    double* summ = (double*)malloc(sizeof(double) * R * NB);
    double* pre = (double*)calloc(R * NB, sizeof(double));
    double* w = (double*)malloc(sizeof(double) * (size_t)(d + dv));
    state_t s;
    int rc = -1;
    if (!summ || !pre || !w || state_alloc(&s, d, dv)) goto out;
    if (hla2_oracle_decay_chunk_summaries(Q, K, V, summ, BH, T, d, dv, L, gamma)) { state_free(&s); goto out; }
    for (int bh = 0; bh < BH; ++bh)
        for (int c = 1; c < N; ++c) {
            const int nB = L;  /* chunk c-1 is never the last chunk, so it spans L tokens */
            hla2_oracle_decay_combine(pre + ((size_t)bh * N + c - 1) * R, summ + ((size_t)bh * N + c - 1) * R,
                                      pre + ((size_t)bh * N + c) * R, d, dv, nB, gamma);
        }
    for (int bh = 0; bh < BH; ++bh)
        for (int c = 0; c < N; ++c) {
            memcpy(s.S, pre + ((size_t)bh * N + c) * R, sizeof(double) * R);
            const int t1 = (c + 1) * L < T ? (c + 1) * L : T;
            for (int t = c * L; t < t1; ++t) {
                const double* q = Q + ((size_t)bh * T + t) * d;
                decay_absorb(&s, q, K + ((size_t)bh * T + t) * d, V + ((size_t)bh * T + t) * dv, gamma, w);
                emit(&s, q, O + ((size_t)bh * T + t) * dv, normalized, w);
            }
        }
    state_free(&s);
    rc = 0;
out:
    free(summ); free(pre); free(w);
    return rc;
}

/* One decayed decode step on the P-form state S|P|p for n heads. */
int hla2_oracle_decay_step_pform(double* state, const double* q, const double* k, const double* v, double* o,
                                 int n, int d, int dv, int normalized, double gamma) {
    if (!state || !q || !k || !v || !o || n < 0 || d <= 0 || dv <= 0) return -1;
    double* u = (double*)malloc(sizeof(double) * (size_t)d);
    if (!u) return -1;
    const size_t R = (size_t)d * d + (size_t)d * dv + (size_t)d;
    const double g = gamma;
    for (int i = 0; i < n; ++i) {
        double* S = state + (size_t)i * R;
        double* P = S + (size_t)d * d;
        double* p = P + (size_t)d * dv;
        const double* qi = q + (size_t)i * d;
        const double* ki = k + (size_t)i * d;
        const double* vi = v + (size_t)i * dv;
        for (int a = 0; a < d; ++a)
            for (int b = 0; b < d; ++b) S[(size_t)a * d + b] = g * S[(size_t)a * d + b] + ki[a] * ki[b];
        for (int a = 0; a < d; ++a) {
            double acc = 0.0;
            for (int b = 0; b < d; ++b) acc += S[(size_t)a * d + b] * qi[b];
            u[a] = acc;
        }
        for (int a = 0; a < d; ++a) {
            for (int e = 0; e < dv; ++e) P[(size_t)a * dv + e] = g * g * P[(size_t)a * dv + e] + u[a] * vi[e];
            p[a] = g * g * p[a] + u[a];
        }
        double den = 0.0;
        for (int a = 0; a < d; ++a) den += qi[a] * p[a];
        for (int e = 0; e < dv; ++e) {
            double acc = 0.0;
            for (int a = 0; a < d; ++a) acc += qi[a] * P[(size_t)a * dv + e];
            o[(size_t)i * dv + e] = normalized ? acc / den : acc;
        }
    }
    free(u);
    return 0;
}
