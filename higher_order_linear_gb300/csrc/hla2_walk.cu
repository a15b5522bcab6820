// hla2_walk.cu -- segment walks of masked second-order HLA on CUDA cores.
//
// HLA summary (arXiv 2510.27258): section 1 "Second-order HLA" (prefix
// moments S, C, m; cross summaries G, h; o_t = q_t^T (S_t C_t - G_t); ratio
// normalisation) and section 4 "Parallel training via associative scans"
// (segment summaries joined by an exclusive scan reproduce the serial
// recurrence).
//
// A CTA owns one contiguous segment of one head and walks its tokens with the
// state held in shared memory (fp32).  Three modes:
//   mode 0  P-form segment summary from a zero state:
//             S, C, m as usual, P = S C - G, p = S m - h.
//           In P-form the per-token update needs no d x d x dv product:
//             S_t = S_{t-1} + k k^T,  u = S_t q,  P_t = P_{t-1} + u v^T,
//             p_t = p_{t-1} + u   (P_t - P_{t-1} = sum_{i<=t} k_i k_i^T q_t v_t^T).
//   mode 1  outputs: start from the segment's exclusive prefix (S0, P0, p0)
//           and emit o_t = q_t^T P_t (divided by q_t^T p_t when normalised).
//   mode 2  G-form chunk summary from a zero state (S|C|m|G|h), by the
//           recurrence G += k (C_{t-1}^T k), h += k (k . m_{t-1}).
// `gamma` (modes 0 and 1, P-form) decays every prefix moment per token:
// S = gamma S + k k^T, C = gamma C + q v^T, m = gamma m + q, and in P-form
// P = gamma^2 P + u v^T, p = gamma^2 p + u (gamma = 1: the masked operator,
// bit for bit, since the products by 1 are exact).
// With `unmasked` set, modes 0 and 1 compute the unmasked operator
// o_t = q_t^T S_t C_t (section 1's naive product, no G correction): mode 0
// keeps only the plain sums S, C, m, and mode 1 starts from the prefix
// (S0, C0, m0) and takes, per token, S += k k^T, u = S q, C += q v^T,
// o = u^T C (divided by u . m when normalised).
// S is symmetric (a sum of outer products formed elementwise), so S q is
// taken as a column reduction, which matches the thread layout of the walk.
#include "hla2_internal.h"

namespace hla2 {
namespace {

constexpr int kWalkThreads = 512;
constexpr int kTokBlock = 16;   // tokens staged per refill

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

struct WalkSmem {
    float *S, *X, *C, *m, *x, *tq, *tk, *tv, *u, *part, *misc;
};

__host__ __device__ inline size_t walk_smem_floats(int mode, int d, int dv) {
    const int mx = d > dv ? d : dv;
    const int nrg = kWalkThreads / (d < dv ? d : dv);  // upper bound of row groups
    size_t n = 0;
    n += (size_t)d * d;                 // S
    n += (size_t)d * dv;                // X (P or G)
    if (mode != 1) n += (size_t)d * dv; // C
    n += 2 * (size_t)d;                 // m, x
    n += (size_t)kTokBlock * (2 * d + dv);
    n += mx;                            // u / w
    n += (size_t)nrg * mx;              // partial column sums
    n += 8;                             // misc scalars
    return n;
}

template <typename Tin, int MODE>
__global__ void __launch_bounds__(kWalkThreads)
walk_kernel(const Tin* __restrict__ Q, const Tin* __restrict__ K, const Tin* __restrict__ V,
            float* __restrict__ O, const float* __restrict__ prefix, float* __restrict__ summ,
            int T, int d, int dv, int normalized, int unmasked, float gamma, SegPlan plan) {
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    const int mx = d > dv ? d : dv;
    const int mn = d < dv ? d : dv;
    WalkSmem s;
    s.S = sm;
    s.X = s.S + (size_t)d * d;
    s.C = s.X + (size_t)d * dv;
    s.m = s.C + (MODE != 1 ? (size_t)d * dv : 0);
    s.x = s.m + d;
    s.tq = s.x + d;
    s.tk = s.tq + kTokBlock * d;
    s.tv = s.tk + kTokBlock * d;
    s.u = s.tv + kTokBlock * dv;
    s.part = s.u + mx;
    s.misc = s.part + (size_t)(kWalkThreads / mn) * mx;

    const int tid = threadIdx.x;
    int head, seg;
    block_segment(plan, gridDim.y, (long long)blockIdx.y * gridDim.x + blockIdx.x, head, seg);
    const long long c0 = seg_chunk_begin(plan, seg);
    const long long c1 = seg_chunk_begin(plan, seg + 1);
    const int t0 = (int)(c0 * plan.granule);
    const int t1 = (int)min((long long)T, c1 * plan.granule);
    const size_t R = record_len(d, dv);
    const RecOff ro = summary_offsets(d, dv);

    // thread layouts: (row group, column) over d x dv and over d x d
    const int ev = tid % dv, rgv = tid / dv, nrgv = kWalkThreads / dv;
    const int es = tid % d, rgs = tid / d, nrgs = kWalkThreads / d;
    const bool act_v = rgv < nrgv;
    const bool act_s = rgs < nrgs;
    const float g = gamma, g2 = gamma * gamma;

    // ---- initial state ----
    if (MODE == 1) {
        const float* pre = prefix + ((size_t)head * plan.nseg + seg) * R;
        // P-form: X = P, x = p;  unmasked: X = C, x = m
        const size_t oX = unmasked ? ro.C : ro.X, ox = unmasked ? ro.m : ro.x;
        for (int i = tid; i < d * d; i += kWalkThreads) s.S[i] = pre[ro.S + i];
        for (int i = tid; i < d * dv; i += kWalkThreads) s.X[i] = pre[oX + i];
        for (int i = tid; i < d; i += kWalkThreads) s.x[i] = pre[ox + i];
    } else {
        for (int i = tid; i < d * d; i += kWalkThreads) s.S[i] = 0.f;
        for (int i = tid; i < d * dv; i += kWalkThreads) { s.X[i] = 0.f; s.C[i] = 0.f; }
        for (int i = tid; i < d; i += kWalkThreads) { s.m[i] = 0.f; s.x[i] = 0.f; }
    }
    __syncthreads();

    const size_t qbase = (size_t)head * T * d;
    const size_t vbase = (size_t)head * T * dv;
    for (int tb = t0; tb < t1; tb += kTokBlock) {
        const int nt = min(kTokBlock, t1 - tb);
        for (int i = tid; i < nt * d; i += kWalkThreads) {
            s.tq[i] = to_f(Q[qbase + (size_t)tb * d + i]);
            s.tk[i] = to_f(K[qbase + (size_t)tb * d + i]);
        }
        for (int i = tid; i < nt * dv; i += kWalkThreads) s.tv[i] = to_f(V[vbase + (size_t)tb * dv + i]);
        __syncthreads();

        for (int j = 0; j < nt; ++j) {
            const float* q = s.tq + j * d;
            const float* k = s.tk + j * d;
            const float* v = s.tv + j * dv;
            if (MODE == 2) {
                // w partial = sum_a k_a C[a][e] (C_{t-1}); k . m_{t-1}
                if (act_v) {
                    float acc = 0.f;
                    for (int a = rgv; a < d; a += nrgv) acc = fmaf(k[a], s.C[a * dv + ev], acc);
                    s.part[rgv * mx + ev] = acc;
                }
                if (tid < 32) {
                    float km = 0.f;
                    for (int a = tid; a < d; a += 32) km = fmaf(k[a], s.m[a], km);
                    for (int o = 16; o > 0; o >>= 1) km += __shfl_xor_sync(0xffffffffu, km, o);
                    if (tid == 0) s.misc[0] = km;
                }
                __syncthreads();
                if (tid < dv) {
                    float w = 0.f;
                    for (int r = 0; r < nrgv; ++r) w += s.part[r * mx + tid];
                    s.u[tid] = w;
                }
                __syncthreads();
                const float km = s.misc[0];
                if (act_v)
                    for (int a = rgv; a < d; a += nrgv) {
                        const int i = a * dv + ev;
                        s.X[i] = fmaf(k[a], s.u[ev], s.X[i]);
                        s.C[i] = fmaf(q[a], v[ev], s.C[i]);
                    }
                if (act_s)
                    for (int a = rgs; a < d; a += nrgs) s.S[a * d + es] = fmaf(k[a], k[es], s.S[a * d + es]);
                if (tid < d) {
                    s.x[tid] = fmaf(k[tid], km, s.x[tid]);
                    s.m[tid] += q[tid];
                }
                __syncthreads();
            } else {
                // S_t = gamma S_{t-1} + k k^T
                if (act_s)
                    for (int a = rgs; a < d; a += nrgs) s.S[a * d + es] = fmaf(k[a], k[es], g * s.S[a * d + es]);
                __syncthreads();
                // u = S_t q (column reduction; S symmetric)
                if (act_s) {
                    float acc = 0.f;
                    for (int a = rgs; a < d; a += nrgs) acc = fmaf(q[a], s.S[a * d + es], acc);
                    s.part[rgs * mx + es] = acc;
                }
                __syncthreads();
                if (tid < d) {
                    float u = 0.f;
                    for (int r = 0; r < nrgs; ++r) u += s.part[r * mx + tid];
                    s.u[tid] = u;
                    if (unmasked) {
                        if (MODE == 1) s.x[tid] += q[tid];  // m_t = m_{t-1} + q
                    } else {
                        s.x[tid] = fmaf(g2, s.x[tid], u);    // p_t = gamma^2 p_{t-1} + u
                    }
                    if (MODE == 0) s.m[tid] = fmaf(g, s.m[tid], q[tid]);
                }
                __syncthreads();
                // P_t = P_{t-1} + u v^T ; outputs o_e = sum_a q_a P_t[a][e]
                if (act_v) {
                    float acc = 0.f;
                    if (unmasked) {
                        // mode 1: C_t = C_{t-1} + q v^T and o_e = sum_a u_a C_t[a][e]; mode 0: C only
                        for (int a = rgv; a < d; a += nrgv) {
                            const int i = a * dv + ev;
                            if (MODE == 1) {
                                const float cn = fmaf(q[a], v[ev], s.X[i]);
                                s.X[i] = cn;
                                acc = fmaf(s.u[a], cn, acc);
                            } else {
                                s.C[i] = fmaf(q[a], v[ev], s.C[i]);
                            }
                        }
                    } else {
                        for (int a = rgv; a < d; a += nrgv) {
                            const int i = a * dv + ev;
                            const float pn = fmaf(s.u[a], v[ev], g2 * s.X[i]);
                            s.X[i] = pn;
                            if (MODE == 0) s.C[i] = fmaf(q[a], v[ev], g * s.C[i]);
                            acc = fmaf(q[a], pn, acc);
                        }
                    }
                    if (MODE == 1) s.part[rgv * mx + ev] = acc;
                }
                if (MODE == 1 && normalized && tid >= kWalkThreads - 32) {
                    const int l = tid - (kWalkThreads - 32);
                    const float* dv_ = unmasked ? s.u : q;  // den = u . m_t  (P-form: q . p_t)
                    float den = 0.f;
                    for (int a = l; a < d; a += 32) den = fmaf(dv_[a], s.x[a], den);
                    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
                    if (l == 0) s.misc[1] = den;
                }
                __syncthreads();
                if (MODE == 1 && tid < dv) {
                    float o = 0.f;
                    for (int r = 0; r < nrgv; ++r) o += s.part[r * mx + tid];
                    if (normalized) o = o / s.misc[1];
                    O[vbase + (size_t)(tb + j) * dv + tid] = o;
                }
                // the next token's S update writes S only; part is re-written
                // only after the S-update barrier, so no extra barrier here.
            }
        }
        __syncthreads();  // token staging buffers are refilled next
    }

    if (MODE != 1) {
        float* out = summ + ((size_t)head * plan.nseg + seg) * R;
        for (int i = tid; i < d * d; i += kWalkThreads) out[ro.S + i] = s.S[i];
        for (int i = tid; i < d * dv; i += kWalkThreads) { out[ro.C + i] = s.C[i]; out[ro.X + i] = s.X[i]; }
        for (int i = tid; i < d; i += kWalkThreads) { out[ro.m + i] = s.m[i]; out[ro.x + i] = s.x[i]; }
    }
}

template <typename Tin, int MODE>
cudaError_t launch_walk_t(const void* Q, const void* K, const void* V, float* O, const float* prefix,
                          float* summ, int BH, int T, int d, int dv, int normalized, int unmasked, float gamma,
                          SegPlan plan, cudaStream_t s) {
    const size_t bytes = walk_smem_floats(MODE, d, dv) * sizeof(float);
    auto kern = walk_kernel<Tin, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.nseg, BH);
    kern<<<grid, kWalkThreads, bytes, s>>>(static_cast<const Tin*>(Q), static_cast<const Tin*>(K),
                                           static_cast<const Tin*>(V), O, prefix, summ, T, d, dv, normalized,
                                           unmasked, gamma, plan);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_walk(int mode, const void* Q, const void* K, const void* V, int dtype, float* O,
                        const float* prefix, float* summ, int BH, int T, int d, int dv, int normalized,
                        int unmasked, float gamma, SegPlan plan, cudaStream_t s) {
    if (BH == 0 || plan.nseg == 0) return cudaSuccess;
    if (dtype == 1) {
        switch (mode) {
            case 0: return launch_walk_t<__nv_bfloat16, 0>(Q, K, V, O, prefix, summ, BH, T, d, dv, normalized, unmasked, gamma, plan, s);
            case 1: return launch_walk_t<__nv_bfloat16, 1>(Q, K, V, O, prefix, summ, BH, T, d, dv, normalized, unmasked, gamma, plan, s);
            default: return launch_walk_t<__nv_bfloat16, 2>(Q, K, V, O, prefix, summ, BH, T, d, dv, normalized, unmasked, gamma, plan, s);
        }
    }
    switch (mode) {
        case 0: return launch_walk_t<float, 0>(Q, K, V, O, prefix, summ, BH, T, d, dv, normalized, unmasked, gamma, plan, s);
        case 1: return launch_walk_t<float, 1>(Q, K, V, O, prefix, summ, BH, T, d, dv, normalized, unmasked, gamma, plan, s);
        default: return launch_walk_t<float, 2>(Q, K, V, O, prefix, summ, BH, T, d, dv, normalized, unmasked, gamma, plan, s);
    }
}

size_t walk_smem_bytes(int mode, int d, int dv) { return walk_smem_floats(mode, d, dv) * sizeof(float); }

}  // namespace hla2
