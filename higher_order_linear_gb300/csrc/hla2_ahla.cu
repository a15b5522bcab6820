// hla2_ahla.cu -- AHLA, the asymmetric second-order variant, on CUDA cores.
//
// HLA summary (arXiv 2510.27258), section 2 "AHLA": the operator
// Q (K^T Q)(K^T V), an A A V structure (HLA's is A A^T V), kept as streaming
// summaries P^KV_t, m^K_t, E_t, n_t.  Under the causal mask
//   o_t = sum_{j<=i<=t} (q_t.k_i)(q_i.k_j) v_j
// and, per token,
//   P_t = P_{t-1} + k_t v_t^T            m_t = m_{t-1} + k_t
//   E_t = E_{t-1} + k_t (P_t^T q_t)^T    n_t = n_{t-1} + k_t (q_t . m_t)
//   o_t = E_t^T q_t,  normalised  o_t / (q_t . n_t).
// Segments join with section 4's semidirect combine under S -> M = sum k q^T,
// C -> P, G -> E, h -> n: E_AB = E_A + E_B + M_B P_A, n_AB = n_A + n_B + M_B m_A.
//
// Every read of a just-updated quantity is expanded so that one pass over a
// matrix both reads its old value and writes its new one:
//   w   = P_t^T q = P_{t-1}^T q + (q.k) v        qm = q.m_{t-1} + q.k
//   o_t = E_{t-1}^T q + (q.k) w                   den = q.n_{t-1} + (q.k) qm
//
// Segment walks: a CTA owns one contiguous segment of one head, state in
// shared memory (fp32).  mode 0 builds the summary M|P|m|E|n from a zero
// state; mode 1 starts from the segment's exclusive prefix (P, m, E, n) and
// writes outputs.  Decode step: one CTA per head streams P then E once.
#include "hla2_internal.h"

namespace hla2 {
namespace {

constexpr int kWalkThreads = 512;
constexpr int kTokBlock = 16;  // tokens staged per refill (= warps per CTA)

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

struct AhlaSmem {
    float *M, *P, *E, *m, *n, *tq, *tk, *tv, *qk, *w, *partA, *partB, *misc;
};

__host__ __device__ inline size_t ahla_smem_floats(int mode, int d, int dv) {
    size_t f = 0;
    if (mode == 0) f += (size_t)d * d;                     // M
    f += 2 * (size_t)d * dv;                               // P, E
    f += 2 * (size_t)d;                                    // m, n
    f += (size_t)kTokBlock * (2 * d + dv) + kTokBlock;     // staged tokens, q.k per token
    f += (size_t)dv;                                       // w
    f += 2 * (size_t)kWalkThreads;                         // column partials (two buffers)
    f += 8;                                                // misc scalars
    return f;
}

template <typename Tin, int MODE>
__global__ void __launch_bounds__(kWalkThreads)
ahla_walk_kernel(const Tin* __restrict__ Q, const Tin* __restrict__ K, const Tin* __restrict__ V,
                 float* __restrict__ O, const float* __restrict__ prefix, float* __restrict__ summ,
                 int T, int d, int dv, int normalized, SegPlan plan) {
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    AhlaSmem s;
    s.M = sm;
    s.P = s.M + (MODE == 0 ? (size_t)d * d : 0);
    s.E = s.P + (size_t)d * dv;
    s.m = s.E + (size_t)d * dv;
    s.n = s.m + d;
    s.tq = s.n + d;
    s.tk = s.tq + kTokBlock * d;
    s.tv = s.tk + kTokBlock * d;
    s.qk = s.tv + kTokBlock * dv;
    s.w = s.qk + kTokBlock;
    s.partA = s.w + dv;
    s.partB = s.partA + kWalkThreads;
    s.misc = s.partB + kWalkThreads;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int head, seg;
    block_segment(plan, gridDim.y, (long long)blockIdx.y * gridDim.x + blockIdx.x, head, seg);
    const long long c0 = seg_chunk_begin(plan, seg);
    const long long c1 = seg_chunk_begin(plan, seg + 1);
    const int t0 = (int)(c0 * plan.granule);
    const int t1 = (int)min((long long)T, c1 * plan.granule);
    const RecOff ro = summary_offsets(d, dv);  // M|P|m|E|n at the S|C|m|X|x offsets
    const bool norm = MODE == 0 || normalized;  // m and n are carried

    // thread layouts: (row group, column) over d x dv and d x d
    const int ev = tid % dv, rgv = tid / dv, nrgv = kWalkThreads / dv;
    const int es = tid % d, rgs = tid / d, nrgs = kWalkThreads / d;
    const bool act_v = rgv < nrgv;
    const bool act_s = rgs < nrgs;

    if (MODE == 1) {
        const float* pre = prefix + ((size_t)head * plan.nseg + seg) * ro.R;
        for (int i = tid; i < d * dv; i += kWalkThreads) {
            s.P[i] = pre[ro.C + i];
            s.E[i] = pre[ro.X + i];
        }
        for (int i = tid; i < d; i += kWalkThreads) {
            s.m[i] = normalized ? pre[ro.m + i] : 0.f;
            s.n[i] = normalized ? pre[ro.x + i] : 0.f;
        }
    } else {
        for (int i = tid; i < d * d; i += kWalkThreads) s.M[i] = 0.f;
        for (int i = tid; i < d * dv; i += kWalkThreads) { s.P[i] = 0.f; s.E[i] = 0.f; }
        for (int i = tid; i < d; i += kWalkThreads) { s.m[i] = 0.f; s.n[i] = 0.f; }
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
        if (warp < nt) {  // q.k of token `warp` of the block
            float acc = 0.f;
            for (int a = lane; a < d; a += 32) acc = fmaf(s.tq[warp * d + a], s.tk[warp * d + a], acc);
            acc = warp_sum(acc);
            if (lane == 0) s.qk[warp] = acc;
        }
        __syncthreads();

        for (int j = 0; j < nt; ++j) {
            const float* q = s.tq + j * d;
            const float* k = s.tk + j * d;
            const float* v = s.tv + j * dv;
            const float qk = s.qk[j];
            // pass P: y = P_{t-1}^T q (column partials), P += k v^T; M += k q^T
            if (act_v) {
                const float ve = v[ev];
                float acc = 0.f;
                for (int a = rgv; a < d; a += nrgv) {
                    const int i = a * dv + ev;
                    const float p = s.P[i];
                    acc = fmaf(q[a], p, acc);
                    s.P[i] = fmaf(k[a], ve, p);
                }
                s.partA[rgv * dv + ev] = acc;
            }
            if (MODE == 0 && act_s)
                for (int a = rgs; a < d; a += nrgs) s.M[a * d + es] = fmaf(k[a], q[es], s.M[a * d + es]);
            if (norm && warp == kTokBlock - 1) {  // q.m_{t-1}, q.n_{t-1}; m += k
                float qm = 0.f, qn = 0.f;
                for (int a = lane; a < d; a += 32) {
                    qm = fmaf(q[a], s.m[a], qm);
                    qn = fmaf(q[a], s.n[a], qn);
                    s.m[a] += k[a];
                }
                qm = warp_sum(qm); qn = warp_sum(qn);
                if (lane == 0) { s.misc[2 * (j & 1)] = qm + qk; s.misc[2 * (j & 1) + 1] = qn; }
            }
            __syncthreads();
            if (tid < dv) {
                float y = 0.f;
                for (int r = 0; r < nrgv; ++r) y += s.partA[r * dv + tid];
                s.w[tid] = fmaf(qk, v[tid], y);
            }
            __syncthreads();
            // pass E: z = E_{t-1}^T q (column partials), E += k w^T; n += k qm
            if (act_v) {
                const float we = s.w[ev];
                float acc = 0.f;
                for (int a = rgv; a < d; a += nrgv) {
                    const int i = a * dv + ev;
                    const float e = s.E[i];
                    if (MODE == 1) acc = fmaf(q[a], e, acc);
                    s.E[i] = fmaf(k[a], we, e);
                }
                if (MODE == 1) s.partB[rgv * dv + ev] = acc;
            }
            if (norm && tid >= kWalkThreads - 32) {
                const float qm = s.misc[2 * (j & 1)];
                for (int a = lane; a < d; a += 32) s.n[a] = fmaf(k[a], qm, s.n[a]);
            }
            if (MODE == 1) {
                __syncthreads();
                if (tid < dv) {
                    float z = 0.f;
                    for (int r = 0; r < nrgv; ++r) z += s.partB[r * dv + tid];
                    float o = fmaf(qk, s.w[tid], z);
                    if (normalized) o = o / fmaf(qk, s.misc[2 * (j & 1)], s.misc[2 * (j & 1) + 1]);
                    O[vbase + (size_t)(tb + j) * dv + tid] = o;
                }
            }
            // The next token writes partA and P, read only before the second
            // barrier above, and w only after its own first barrier, which
            // every reader here precedes.  Its scalars go to the other half
            // of misc (token parity), since the last warp writes them before
            // that barrier while the output threads may still read these.
        }
        __syncthreads();  // staging buffers are refilled next
    }

    if (MODE == 0) {
        float* out = summ + ((size_t)head * plan.nseg + seg) * ro.R;
        for (int i = tid; i < d * d; i += kWalkThreads) out[ro.S + i] = s.M[i];
        for (int i = tid; i < d * dv; i += kWalkThreads) { out[ro.C + i] = s.P[i]; out[ro.X + i] = s.E[i]; }
        for (int i = tid; i < d; i += kWalkThreads) { out[ro.m + i] = s.m[i]; out[ro.x + i] = s.n[i]; }
    }
}

template <typename Tin, int MODE>
cudaError_t launch_ahla_walk_t(const void* Q, const void* K, const void* V, float* O, const float* prefix,
                               float* summ, int BH, int T, int d, int dv, int normalized, SegPlan plan,
                               cudaStream_t s) {
    const size_t bytes = ahla_smem_floats(MODE, d, dv) * sizeof(float);
    auto kern = ahla_walk_kernel<Tin, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.nseg, BH);
    kern<<<grid, kWalkThreads, bytes, s>>>(static_cast<const Tin*>(Q), static_cast<const Tin*>(K),
                                           static_cast<const Tin*>(V), O, prefix, summ, T, d, dv, normalized,
                                           plan);
    note_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------- decode step ----
constexpr int kStepThreads = 256;
constexpr int kUnroll = 8;

__device__ __forceinline__ float4 ld_stream(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_stream(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

// One streamed pass over a d x dv matrix X: z = X^T q (old X) and X += k u^T.
// Column partials land in part[tid][0..3].  d, dv powers of two in [4, 128].
__device__ __forceinline__ void stream_pass(float* X, const float* sq, const float* sk, const float* su,
                                            float (*part)[4], int d, int dv) {
    const int tid = threadIdx.x;
    const int gc = dv >> 2;
    const int rows_per = kStepThreads / gc;
    const int c4 = tid % gc;
    const int rg = tid / gc;
    float z[4] = {0.f, 0.f, 0.f, 0.f};
    const float4 u4 = *reinterpret_cast<const float4*>(&su[4 * c4]);
    for (int a0 = 0; a0 < d; a0 += rows_per * kUnroll) {
        float4 r[kUnroll];
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            const int a = a0 + i * rows_per + rg;
            if (a < d) r[i] = ld_stream(X + (size_t)a * dv + 4 * c4);
        }
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            const int a = a0 + i * rows_per + rg;
            if (a < d) {
                const float qa = sq[a], ka = sk[a];
                float4 x = r[i];
                z[0] = fmaf(qa, x.x, z[0]); z[1] = fmaf(qa, x.y, z[1]);
                z[2] = fmaf(qa, x.z, z[2]); z[3] = fmaf(qa, x.w, z[3]);
                x.x = fmaf(ka, u4.x, x.x); x.y = fmaf(ka, u4.y, x.y);
                x.z = fmaf(ka, u4.z, x.z); x.w = fmaf(ka, u4.w, x.w);
                st_stream(X + (size_t)a * dv + 4 * c4, x);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) part[tid][j] = z[j];
}

// Column e of the partials: sum over the row groups.
__device__ __forceinline__ float column_sum(float (*part)[4], int e, int d, int dv) {
    const int gc = dv >> 2;
    const int rows_per = kStepThreads / gc;
    const int cc = e >> 2, j = e & 3;
    const int nr = rows_per < d ? rows_per : d;
    float y = 0.f;
    for (int r = 0; r < nr; ++r) y += part[r * gc + cc][j];
    return y;
}

// State per head P|E|m|n (2 d dv + 2 d floats, fp32, row-major).
__global__ void __launch_bounds__(kStepThreads)
ahla_step_kernel(float* __restrict__ state, const float* __restrict__ q, const float* __restrict__ k,
                 const float* __restrict__ v, float* __restrict__ o, int d, int dv, int normalized) {
    __shared__ __align__(16) float sq[128], sk[128], sv[128], sw[128];
    __shared__ __align__(16) float part[kStepThreads][4];
    __shared__ float sdots[3];

    const int head = blockIdx.x;
    const int tid = threadIdx.x;
    const size_t R = 2 * (size_t)d * dv + 2 * (size_t)d;
    float* P = state + (size_t)head * R;
    float* E = P + (size_t)d * dv;
    float* m = E + (size_t)d * dv;
    float* n = m + d;

    if (tid < d) {
        sq[tid] = q[(size_t)head * d + tid];
        sk[tid] = k[(size_t)head * d + tid];
    }
    if (tid < dv) sv[tid] = v[(size_t)head * dv + tid];
    __syncthreads();
    if (tid < 32) {  // q.k, q.m_{t-1}, q.n_{t-1}; m += k (m and n are kept for either variant)
        float qk = 0.f, qm = 0.f, qn = 0.f;
        for (int a = tid; a < d; a += 32) {
            qk = fmaf(sq[a], sk[a], qk);
            const float ma = m[a];
            qm = fmaf(sq[a], ma, qm);
            qn = fmaf(sq[a], n[a], qn);
            m[a] = ma + sk[a];
        }
        qk = warp_sum(qk); qm = warp_sum(qm); qn = warp_sum(qn);
        if (tid == 0) { sdots[0] = qk; sdots[1] = qm + qk; sdots[2] = qn; }
    }
    // pass P: y = P^T q, P += k v^T
    stream_pass(P, sq, sk, sv, part, d, dv);
    __syncthreads();
    const float qk = sdots[0];
    if (tid < dv) sw[tid] = fmaf(qk, sv[tid], column_sum(part, tid, d, dv));  // w = P_t^T q
    __syncthreads();
    // pass E: z = E^T q, E += k w^T; n += k (q.m_t)
    stream_pass(E, sq, sk, sw, part, d, dv);
    if (tid >= kStepThreads - 32) {
        const float qm = sdots[1];
        for (int a = tid - (kStepThreads - 32); a < d; a += 32) n[a] = fmaf(sk[a], qm, n[a]);
    }
    __syncthreads();
    if (tid < dv) {
        float out = fmaf(qk, sw[tid], column_sum(part, tid, d, dv));
        if (normalized) out = out / fmaf(qk, sdots[1], sdots[2]);
        o[(size_t)head * dv + tid] = out;
    }
}

}  // namespace

cudaError_t launch_ahla_walk(int mode, const void* Q, const void* K, const void* V, int dtype, float* O,
                             const float* prefix, float* summ, int BH, int T, int d, int dv, int normalized,
                             SegPlan plan, cudaStream_t s) {
    if (BH == 0 || plan.nseg == 0) return cudaSuccess;
    if (dtype == 1)
        return mode == 0 ? launch_ahla_walk_t<__nv_bfloat16, 0>(Q, K, V, O, prefix, summ, BH, T, d, dv, normalized, plan, s)
                         : launch_ahla_walk_t<__nv_bfloat16, 1>(Q, K, V, O, prefix, summ, BH, T, d, dv, normalized, plan, s);
    return mode == 0 ? launch_ahla_walk_t<float, 0>(Q, K, V, O, prefix, summ, BH, T, d, dv, normalized, plan, s)
                     : launch_ahla_walk_t<float, 1>(Q, K, V, O, prefix, summ, BH, T, d, dv, normalized, plan, s);
}

cudaError_t launch_ahla_step(float* state, const float* q, const float* k, const float* v, float* o, int n, int d,
                             int dv, int normalized, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    ahla_step_kernel<<<n, kStepThreads, 0, s>>>(state, q, k, v, o, d, dv, normalized);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace hla2
