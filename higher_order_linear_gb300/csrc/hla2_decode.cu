// hla2_decode.cu -- streaming decode step of masked second-order HLA.
//
// HLA summary (arXiv 2510.27258), section 1 "Second-order HLA": the online
// update of the prefix summaries and the output o_t = q_t^T (S_t C_t - G_t)
// at O(d^2 + d dv) per token; "Results and claims": that cost does not depend
// on the prefix length.
//
// One CTA per head.  The state S|C|G|m|h (fp32, row-major) is streamed from
// HBM once and written back once, with 16-byte coalesced accesses, in three
// passes whose reductions feed the next pass:
//   pass S : S' = S + k k^T, and u = S' q          (row reductions)
//   pass C : w = C^T k, y = C^T u (columns), C' = C + q v^T
//   pass G : z = G^T q (columns), G' = G + k w^T
// then  o = y + (u.q) v - z - (q.k) w,  m' = m + q,  h' = h + k (k.m),
// and, normalised, o /= u.m' - q.h'.
// Every state byte crosses HBM exactly twice (read + write): the step is
// bandwidth-bound, 8*(d^2 + 2 d dv + 2 d) + 4*(2d + 2dv) bytes per head.
#include "hla2_internal.h"

namespace hla2 {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;  // float4 loads in flight per thread per batch

__device__ __forceinline__ float4 ld_stream(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_stream(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// d and dv are powers of two in [4, 128].  Four CTAs per SM (64 registers).
__global__ void __launch_bounds__(kThreads, 4)
step_kernel(float* __restrict__ state, const float* __restrict__ q, const float* __restrict__ k,
            const float* __restrict__ v, float* __restrict__ o, int d, int dv, int normalized) {
    __shared__ __align__(16) float sq[128], sk[128], sv[128], su[128], sw[128], sy[128], sz[128];
    __shared__ __align__(16) float part[3][kThreads][4];  // per-thread column partials (w, y or z)
    __shared__ float sdots[5];

    const int head = blockIdx.x;
    const int tid = threadIdx.x;
    const size_t R = (size_t)d * d + 2 * (size_t)d * dv + 2 * (size_t)d;
    float* S = state + (size_t)head * R;
    float* C = S + (size_t)d * d;
    float* G = C + (size_t)d * dv;
    float* m = G + (size_t)d * dv;
    float* h = m + d;

    if (tid < d) {
        sq[tid] = q[(size_t)head * d + tid];
        sk[tid] = k[(size_t)head * d + tid];
        su[tid] = 0.f;
    }
    if (tid < dv) sv[tid] = v[(size_t)head * dv + tid];
    __syncthreads();

    // ---- pass S: S' = S + k k^T ; u = S' q --------------------------------
    {
        const int g = d >> 2;                 // float4s per row (power of two <= 32)
        const int nf = (d * d) >> 2;
        for (int base = 0; base < nf; base += kThreads * kUnroll) {
            float4 r[kUnroll];
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) {
                const int f = base + i * kThreads + tid;
                if (f < nf) r[i] = ld_stream(S + 4 * (size_t)f);
            }
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) {
                const int f = base + i * kThreads + tid;
                float part_u = 0.f;
                int a = 0;
                if (f < nf) {
                    a = f / g;
                    const int b = (f - a * g) * 4;
                    const float ka = sk[a];
                    float4 x = r[i];
                    x.x = fmaf(ka, sk[b + 0], x.x);
                    x.y = fmaf(ka, sk[b + 1], x.y);
                    x.z = fmaf(ka, sk[b + 2], x.z);
                    x.w = fmaf(ka, sk[b + 3], x.w);
                    st_stream(S + 4 * (size_t)f, x);
                    part_u = x.x * sq[b] + x.y * sq[b + 1] + x.z * sq[b + 2] + x.w * sq[b + 3];
                }
                // reduce across the g lanes that share row a (aligned lane groups)
                for (int off = g >> 1; off > 0; off >>= 1) part_u += __shfl_xor_sync(0xffffffffu, part_u, off);
                if (f < nf && (tid & (g - 1)) == 0) su[a] += part_u;  // one writer per row per batch step
            }
        }
    }
    const int gc = dv >> 2;        // float4 columns per row
    const int rows_per = kThreads / gc;  // rows covered per sweep (gc divides 256)
    const int c4 = tid % gc;
    const int rg = tid / gc;
    // The first batch of C is loaded before the barrier that ends pass S (its
    // loads need nothing from that pass), so the stream does not pause there.
    float4 r[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
        const int a = i * rows_per + rg;
        if (a < d) r[i] = ld_stream(C + (size_t)a * dv + 4 * c4);
    }
    __syncthreads();

    // ---- pass C: w = C^T k, y = C^T u (old C), C' = C + q v^T -------------
    {
        float pw[4] = {0.f, 0.f, 0.f, 0.f}, py[4] = {0.f, 0.f, 0.f, 0.f};
        const float4 v4 = *reinterpret_cast<const float4*>(&sv[4 * c4]);
        for (int a0 = 0; a0 < d; a0 += rows_per * kUnroll) {
            if (a0 > 0) {
#pragma unroll
                for (int i = 0; i < kUnroll; ++i) {
                    const int a = a0 + i * rows_per + rg;
                    if (a < d) r[i] = ld_stream(C + (size_t)a * dv + 4 * c4);
                }
            }
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) {
                const int a = a0 + i * rows_per + rg;
                if (a < d) {
                    const float ka = sk[a], ua = su[a], qa = sq[a];
                    float4 x = r[i];
                    pw[0] = fmaf(ka, x.x, pw[0]); pw[1] = fmaf(ka, x.y, pw[1]);
                    pw[2] = fmaf(ka, x.z, pw[2]); pw[3] = fmaf(ka, x.w, pw[3]);
                    py[0] = fmaf(ua, x.x, py[0]); py[1] = fmaf(ua, x.y, py[1]);
                    py[2] = fmaf(ua, x.z, py[2]); py[3] = fmaf(ua, x.w, py[3]);
                    x.x = fmaf(qa, v4.x, x.x); x.y = fmaf(qa, v4.y, x.y);
                    x.z = fmaf(qa, v4.z, x.z); x.w = fmaf(qa, v4.w, x.w);
                    st_stream(C + (size_t)a * dv + 4 * c4, x);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) { part[0][tid][j] = pw[j]; part[1][tid][j] = py[j]; }
    }
    // likewise the first batch of G before the barrier that ends pass C
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
        const int a = i * rows_per + rg;
        if (a < d) r[i] = ld_stream(G + (size_t)a * dv + 4 * c4);
    }
    __syncthreads();
    if (tid < dv) {
        const int cc = tid >> 2, j = tid & 3;
        float w = 0.f, y = 0.f;
        for (int r = 0; r < rows_per; ++r) { w += part[0][r * gc + cc][j]; y += part[1][r * gc + cc][j]; }
        sw[tid] = w;
        sy[tid] = y;
    }
    __syncthreads();

    // ---- pass G: z = G^T q (old G), G' = G + k w^T --------------------------
    {
        float pz[4] = {0.f, 0.f, 0.f, 0.f};
        const float4 w4 = *reinterpret_cast<const float4*>(&sw[4 * c4]);
        for (int a0 = 0; a0 < d; a0 += rows_per * kUnroll) {
            if (a0 > 0) {
#pragma unroll
                for (int i = 0; i < kUnroll; ++i) {
                    const int a = a0 + i * rows_per + rg;
                    if (a < d) r[i] = ld_stream(G + (size_t)a * dv + 4 * c4);
                }
            }
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) {
                const int a = a0 + i * rows_per + rg;
                if (a < d) {
                    const float ka = sk[a], qa = sq[a];
                    float4 x = r[i];
                    pz[0] = fmaf(qa, x.x, pz[0]); pz[1] = fmaf(qa, x.y, pz[1]);
                    pz[2] = fmaf(qa, x.z, pz[2]); pz[3] = fmaf(qa, x.w, pz[3]);
                    x.x = fmaf(ka, w4.x, x.x); x.y = fmaf(ka, w4.y, x.y);
                    x.z = fmaf(ka, w4.z, x.z); x.w = fmaf(ka, w4.w, x.w);
                    st_stream(G + (size_t)a * dv + 4 * c4, x);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) part[2][tid][j] = pz[j];
    }
    // ---- small dot products (warp 0): u.q, q.k, k.m_old --------------------
    if (tid < 32) {
        float uq = 0.f, qk = 0.f, km = 0.f;
        for (int a = tid; a < d; a += 32) {
            uq += su[a] * sq[a];
            qk += sq[a] * sk[a];
            km += sk[a] * m[a];
        }
        uq = warp_sum(uq); qk = warp_sum(qk); km = warp_sum(km);
        if (tid == 0) { sdots[0] = uq; sdots[1] = qk; sdots[2] = km; }
    }
    __syncthreads();
    if (tid < dv) {
        const int cc = tid >> 2, j = tid & 3;
        float z = 0.f;
        for (int r = 0; r < rows_per; ++r) z += part[2][r * gc + cc][j];
        sz[tid] = z;
    }
    // m' = m + q, h' = h + k (k.m_old), den = u.m' - q.h'
    if (tid < 32) {
        float um = 0.f, qh = 0.f;
        const float km = sdots[2];
        for (int a = tid; a < d; a += 32) {
            const float mn = m[a] + sq[a];
            const float hn = fmaf(sk[a], km, h[a]);
            um += su[a] * mn;
            qh += sq[a] * hn;
            m[a] = mn;
            h[a] = hn;
        }
        um = warp_sum(um); qh = warp_sum(qh);
        if (tid == 0) sdots[3] = um - qh;
    }
    __syncthreads();
    if (tid < dv) {
        float out = sy[tid] + sdots[0] * sv[tid] - sz[tid] - sdots[1] * sw[tid];
        if (normalized) out = out / sdots[3];
        o[(size_t)head * dv + tid] = out;
    }
}

}  // namespace

cudaError_t launch_step(float* state, const float* q, const float* k, const float* v, float* o,
                        int n, int d, int dv, int normalized, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    step_kernel<<<n, kThreads, 0, s>>>(state, q, k, v, o, d, dv, normalized);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace hla2

// ---------------------------------------------------------------------------
// Compact P-form decode state: S (d x d) | P = S C - G (d x dv) | p = S m - h (d).
// The same outputs with a third fewer state bytes at d = dv, because
//   S_t = S + k k^T,  u = S_t q,  o = q^T P_{t-1} + (q . u) v,
//   P_t = P + u v^T,  p_t = p + u,  den = q . p_t
// (P_t - P_{t-1} = S_t q_t v_t^T).  Two passes: S (row reductions give u),
// then P (column reductions give q^T P_{t-1} while P is updated).
//
// With a per-token decay gamma of every prefix moment (the decayed masked
// operator), S_t = gamma S + k k^T, P_t = gamma^2 P + u v^T, p_t = gamma^2 p + u
// and o = gamma^2 q^T P_{t-1} + (q . u) v; gamma = 1 gives the lines above.
//
// The unmasked operator o_t = q_t^T S_t C_t (no G correction) has the same
// two-pass shape on the state S | C | m, with the roles of q and u swapped in
// the second pass:
//   S_t = S + k k^T,  u = S_t q,  o = u^T C_{t-1} + (u . q) v,
//   C_t = C + q v^T,  m_t = m + q,  den = u . m_t.
// ---------------------------------------------------------------------------
namespace hla2 {
namespace {

template <bool UNMASKED>
__global__ void __launch_bounds__(kThreads)
step_pform_kernel(float* __restrict__ state, const float* __restrict__ q, const float* __restrict__ k,
                  const float* __restrict__ v, float* __restrict__ o, int d, int dv, int normalized, float gamma) {
    const float gm = gamma, gm2 = gamma * gamma;  // per-token decay (1: none)
    __shared__ __align__(16) float sq[128], sk[128], sv[128], su[128];
    __shared__ __align__(16) float part[kThreads][4];
    __shared__ float sdots[2];

    const int head = blockIdx.x;
    const int tid = threadIdx.x;
    const size_t R = (size_t)d * d + (size_t)d * dv + (size_t)d;
    float* S = state + (size_t)head * R;
    float* P = S + (size_t)d * d;
    float* p = P + (size_t)d * dv;

    if (tid < d) {
        sq[tid] = q[(size_t)head * d + tid];
        sk[tid] = k[(size_t)head * d + tid];
        su[tid] = 0.f;
    }
    if (tid < dv) sv[tid] = v[(size_t)head * dv + tid];
    __syncthreads();

    // ---- pass S: S' = S + k k^T ; u = S' q ---------------------------------
    {
        const int g = d >> 2;
        const int nf = (d * d) >> 2;
        for (int base = 0; base < nf; base += kThreads * kUnroll) {
            float4 r[kUnroll];
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) {
                const int f = base + i * kThreads + tid;
                if (f < nf) r[i] = ld_stream(S + 4 * (size_t)f);
            }
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) {
                const int f = base + i * kThreads + tid;
                float part_u = 0.f;
                int a = 0;
                if (f < nf) {
                    a = f / g;
                    const int b = (f - a * g) * 4;
                    const float ka = sk[a];
                    float4 x = r[i];
                    x.x = fmaf(ka, sk[b + 0], gm * x.x);
                    x.y = fmaf(ka, sk[b + 1], gm * x.y);
                    x.z = fmaf(ka, sk[b + 2], gm * x.z);
                    x.w = fmaf(ka, sk[b + 3], gm * x.w);
                    st_stream(S + 4 * (size_t)f, x);
                    part_u = x.x * sq[b] + x.y * sq[b + 1] + x.z * sq[b + 2] + x.w * sq[b + 3];
                }
                for (int off = g >> 1; off > 0; off >>= 1) part_u += __shfl_xor_sync(0xffffffffu, part_u, off);
                if (f < nf && (tid & (g - 1)) == 0) su[a] += part_u;
            }
        }
    }
    const int gc = dv >> 2;
    const int rows_per = kThreads / gc;
    const int c4 = tid % gc;
    const int rg = tid / gc;
    // the first batch of P is loaded before the barrier that ends pass S
    float4 r[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
        const int a = i * rows_per + rg;
        if (a < d) r[i] = ld_stream(P + (size_t)a * dv + 4 * c4);
    }
    __syncthreads();

    // ---- pass P: y = P^T q (old P), P' = P + u v^T -------------------------
    {
        float py[4] = {0.f, 0.f, 0.f, 0.f};
        const float4 v4 = *reinterpret_cast<const float4*>(&sv[4 * c4]);
        for (int a0 = 0; a0 < d; a0 += rows_per * kUnroll) {
            if (a0 > 0) {
#pragma unroll
                for (int i = 0; i < kUnroll; ++i) {
                    const int a = a0 + i * rows_per + rg;
                    if (a < d) r[i] = ld_stream(P + (size_t)a * dv + 4 * c4);
                }
            }
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) {
                const int a = a0 + i * rows_per + rg;
                if (a < d) {
                    // P-form: reduce with q, update with u;  unmasked: reduce with u, update with q
                    const float qa = UNMASKED ? su[a] : sq[a], ua = UNMASKED ? sq[a] : su[a];
                    float4 x = r[i];
                    py[0] = fmaf(qa, x.x, py[0]); py[1] = fmaf(qa, x.y, py[1]);
                    py[2] = fmaf(qa, x.z, py[2]); py[3] = fmaf(qa, x.w, py[3]);
                    x.x = fmaf(ua, v4.x, gm2 * x.x); x.y = fmaf(ua, v4.y, gm2 * x.y);
                    x.z = fmaf(ua, v4.z, gm2 * x.z); x.w = fmaf(ua, v4.w, gm2 * x.w);
                    st_stream(P + (size_t)a * dv + 4 * c4, x);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) part[tid][j] = py[j];
    }
    // q . u and, normalised, p' = p + u and q . p'
    if (tid < 32) {
        float qu = 0.f, qp = 0.f;
        for (int a = tid; a < d; a += 32) {
            const float pn = fmaf(gm2, p[a], UNMASKED ? sq[a] : su[a]);  // gamma^2 p + u  |  m + q
            qu += sq[a] * su[a];
            qp += (UNMASKED ? su[a] : sq[a]) * pn;               // q . p_t  |  u . m_t
            p[a] = pn;
        }
        qu = warp_sum(qu); qp = warp_sum(qp);
        if (tid == 0) { sdots[0] = qu; sdots[1] = qp; }
    }
    __syncthreads();
    if (tid < dv) {
        const int cc = tid >> 2, j = tid & 3;
        float y = 0.f;
        for (int r = 0; r < rows_per; ++r) y += part[r * gc + cc][j];
        float out = fmaf(gm2, y, sdots[0] * sv[tid]);
        if (normalized) out = out / sdots[1];
        o[(size_t)head * dv + tid] = out;
    }
}

}  // namespace

cudaError_t launch_step_pform(float* state, const float* q, const float* k, const float* v, float* o, int n, int d,
                              int dv, int normalized, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    step_pform_kernel<false><<<n, kThreads, 0, s>>>(state, q, k, v, o, d, dv, normalized, 1.0f);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_step_unmasked(float* state, const float* q, const float* k, const float* v, float* o, int n,
                                 int d, int dv, int normalized, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    step_pform_kernel<true><<<n, kThreads, 0, s>>>(state, q, k, v, o, d, dv, normalized, 1.0f);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_step_pform_decay(float* state, const float* q, const float* k, const float* v, float* o, int n,
                                    int d, int dv, int normalized, float gamma, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    step_pform_kernel<false><<<n, kThreads, 0, s>>>(state, q, k, v, o, d, dv, normalized, gamma);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace hla2
