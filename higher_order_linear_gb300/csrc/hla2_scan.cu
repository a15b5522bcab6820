// hla2_scan.cu -- exclusive scan of HLA segment summaries.
//
// HLA summary (arXiv 2510.27258), section 4 "Parallel training via
// associative scans": segment summaries are joined by a semidirect-product
// operator whose cross term is S_B C_A, and an exclusive scan over them gives
// every segment the exact state of the serial recurrence at its start.
//
// The combine adds S, C and m, so the exclusive prefix of the corrected part
// unrolls to a plain sum of per-record terms:
//   G-form:  G_<n = sum_{r<n} (G_r + S_r C_<r),   h_<n = sum_{r<n} (h_r + S_r m_<r)
//   P-form:  P_<n = sum_{r<n} (P_r + S_<r C_r),   p_<n = sum_{r<n} (p_r + S_<r m_r)
// (P = S C - G, p = S m - h.)  The scan therefore runs as
//   1. exclusive running sums of (S, C, m) along the record axis,
//   2. one d x d by d x (dv+1) product per record (batched, fp32),
//   3. exclusive running sums of the corrected part.
// Steps 1 and 3 are element-parallel: one thread per state element walks the
// record axis, so consecutive threads touch consecutive floats.
#include "hla2_internal.h"

namespace hla2 {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanUnroll = 8;

template <bool WRITE>
__global__ void __launch_bounds__(kScanThreads)
exscan_kernel(const float* in, float* out, int N, size_t R, size_t off, size_t len, float* total,
              size_t total_stride) {
    const size_t i = (size_t)blockIdx.x * kScanThreads + threadIdx.x;
    const int bh = blockIdx.y;
    if (i >= len) return;
    const float* pin = in + (size_t)bh * N * R + off + i;
    float* pout = out + (size_t)bh * N * R + off + i;
    float run = 0.f;
    int r = 0;
    for (; r + kScanUnroll <= N; r += kScanUnroll) {
        float x[kScanUnroll];
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) x[j] = pin[(size_t)(r + j) * R];
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) {
            if (WRITE) pout[(size_t)(r + j) * R] = run;
            run += x[j];
        }
    }
    for (; r < N; ++r) {
        const float x = pin[(size_t)r * R];
        if (WRITE) pout[(size_t)r * R] = run;
        run += x;
    }
    if (total) total[(size_t)bh * total_stride + i] = run;
}

// Same scan, four consecutive elements per thread (16-byte accesses); used
// when the element range, the record length and the pointers allow it.  U
// records are loaded at a time (more in flight for long record axes).
template <bool WRITE, int U>
__global__ void __launch_bounds__(kScanThreads)
exscan4_kernel(const float* in, float* out, int N, size_t R, size_t off, size_t len, float* total,
               size_t total_stride) {
    const size_t i = ((size_t)blockIdx.x * kScanThreads + threadIdx.x) * 4;
    const int bh = blockIdx.y;
    if (i >= len) return;
    const float* pin = in + (size_t)bh * N * R + off + i;
    float* pout = out + (size_t)bh * N * R + off + i;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    // U records per round, every load of a round issued before its sums (the
    // last round predicated, so that a short axis is one round of loads)
    for (int r = 0; r < N; r += U) {
        float4 x[U];
#pragma unroll
        for (int j = 0; j < U; ++j)
            if (r + j < N) x[j] = *reinterpret_cast<const float4*>(pin + (size_t)(r + j) * R);
#pragma unroll
        for (int j = 0; j < U; ++j) {
            if (r + j >= N) break;
            if (WRITE) *reinterpret_cast<float4*>(pout + (size_t)(r + j) * R) = run;
            run.x += x[j].x; run.y += x[j].y; run.z += x[j].z; run.w += x[j].w;
        }
    }
    if (total) *reinterpret_cast<float4*>(total + (size_t)bh * total_stride + i) = run;
}

// out = alpha*base + A [B | bx], 64 x 64 output tile per CTA, 4 x 4 per thread.
constexpr int kTile = 64, kKs = 16;

__global__ void __launch_bounds__(256)
cross_kernel(CrossArgs a) {
    __shared__ float As[kKs][kTile + 4];
    __shared__ float Bs[kKs][kTile + 4];
    const int nb = blockIdx.z;
    const int row0 = blockIdx.y * kTile;
    const int col0 = blockIdx.x * kTile;
    const int d = a.d, dv = a.dv;
    const int ncol = dv + (a.bx ? 1 : 0);
    const float* A = a.A + (long long)nb * a.sA;
    const float* B = a.B + (long long)nb * a.sB;
    const float* bx = a.bx ? a.bx + (long long)nb * a.sbx : nullptr;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < d; k0 += kKs) {
        for (int i = threadIdx.x; i < kKs * kTile; i += 256) {
            const int kk = i / kTile, rr = i % kTile;
            const int arow = row0 + rr, kcol = k0 + kk;
            As[kk][rr] = (arow < d && kcol < d) ? A[(size_t)arow * d + kcol] : 0.f;
            const int ccol = col0 + rr;
            float bv = 0.f;
            if (kcol < d) {
                if (ccol < dv) bv = B[(size_t)kcol * dv + ccol];
                else if (ccol == dv && bx) bv = bx[kcol];
            }
            Bs[kk][rr] = bv;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kKs; ++kk) {
            float ar[4], br[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { ar[i] = As[kk][ty * 4 + i]; br[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
        }
        __syncthreads();
    }
    const float* base = a.base ? a.base + (long long)nb * a.sbase : nullptr;
    const float* basex = a.basex ? a.basex + (long long)nb * a.sbasex : nullptr;
    float* out = a.out + (long long)nb * a.sout;
    float* outx = a.outx ? a.outx + (long long)nb * a.soutx : nullptr;
    if (a.pscale) {
        const float sc = a.pscale[(a.pscale_off + nb) % a.pscale_mod];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] *= sc;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = row0 + ty * 4 + i;
        if (r >= d) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = col0 + tx * 4 + j;
            if (c < dv) {
                const float b0 = base ? base[(size_t)r * dv + c] : 0.f;
                out[(size_t)r * dv + c] = fmaf(a.alpha, b0, acc[i][j]);
            } else if (c == dv && c < ncol && outx) {
                const float b0 = basex ? basex[r] : 0.f;
                outx[r] = fmaf(a.alpha, b0, acc[i][j]);
            }
        }
    }
}

// Decayed scans (the decayed operator's segment combine): per-record factors
// and an exclusive running sum that decays the running value by the factor of
// the record it passes.
__global__ void decay_factors_kernel(float* fac, int T, float gamma, SegPlan plan) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= plan.nseg) return;
    const long long c0 = seg_chunk_begin(plan, r);
    const long long c1 = seg_chunk_begin(plan, r + 1);
    const long long t1 = min((long long)T, c1 * plan.granule);
    // gamma^n by repeated squaring in double precision (fp32 products over
    // thousands of tokens would drift)
    double f = 1.0, base = (double)gamma;
    for (long long e = t1 - c0 * plan.granule; e > 0; e >>= 1) {
        if (e & 1) f *= base;
        base *= base;
    }
    fac[r] = (float)f;
    fac[plan.nseg + r] = (float)(f * f);
}

__global__ void __launch_bounds__(kScanThreads)
decay_exscan_kernel(const float* in, float* out, int N, size_t R, size_t off, size_t len, float* total,
                    size_t total_stride, const float* __restrict__ fac) {
    const size_t i = (size_t)blockIdx.x * kScanThreads + threadIdx.x;
    const int bh = blockIdx.y;
    if (i >= len) return;
    const float* pin = in + (size_t)bh * N * R + off + i;
    float* pout = out + (size_t)bh * N * R + off + i;
    float run = 0.f;
    int r = 0;
    for (; r + kScanUnroll <= N; r += kScanUnroll) {
        float x[kScanUnroll];
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) x[j] = pin[(size_t)(r + j) * R];
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) {
            pout[(size_t)(r + j) * R] = run;
            run = fmaf(fac[r + j], run, x[j]);
        }
    }
    for (; r < N; ++r) {
        const float x = pin[(size_t)r * R];
        pout[(size_t)r * R] = run;
        run = fmaf(fac[r], run, x);
    }
    if (total) total[(size_t)bh * total_stride + i] = run;
}

// Same decayed scan, four consecutive elements per thread (16-byte accesses).
__global__ void __launch_bounds__(kScanThreads)
decay_exscan4_kernel(const float* in, float* out, int N, size_t R, size_t off, size_t len, float* total,
                     size_t total_stride, const float* __restrict__ fac) {
    const size_t i = ((size_t)blockIdx.x * kScanThreads + threadIdx.x) * 4;
    const int bh = blockIdx.y;
    if (i >= len) return;
    const float* pin = in + (size_t)bh * N * R + off + i;
    float* pout = out + (size_t)bh * N * R + off + i;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    int r = 0;
    for (; r + kScanUnroll <= N; r += kScanUnroll) {
        float4 x[kScanUnroll];
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) x[j] = *reinterpret_cast<const float4*>(pin + (size_t)(r + j) * R);
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) {
            *reinterpret_cast<float4*>(pout + (size_t)(r + j) * R) = run;
            const float f = fac[r + j];
            run = make_float4(fmaf(f, run.x, x[j].x), fmaf(f, run.y, x[j].y), fmaf(f, run.z, x[j].z),
                              fmaf(f, run.w, x[j].w));
        }
    }
    for (; r < N; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(pin + (size_t)r * R);
        *reinterpret_cast<float4*>(pout + (size_t)r * R) = run;
        const float f = fac[r];
        run = make_float4(fmaf(f, run.x, x.x), fmaf(f, run.y, x.y), fmaf(f, run.z, x.z), fmaf(f, run.w, x.w));
    }
    if (total) *reinterpret_cast<float4*>(total + (size_t)bh * total_stride + i) = run;
}

// Final state in decode order from the P-form totals of a head (one record
// S|C|m|P|p): S, C, m copied, G = S C - P (fp32, summed in k order) and
// h = S m - p.  CTA (row block, column block, head) owns the 16 x 32 block of
// G at rows 16 blk_r.., columns 32 blk_c..: it stages its S rows and C
// columns in shared memory (every load issued before the first store), then
// thread t forms row t / 8 of the block at the four columns 4 (t % 8) .. + 3.
// Column block 0 also copies its S rows and forms h for them; every CTA
// copies its part of C.
constexpr int kTailRows = 16, kTailCols = 32, kTailThreads = 128;

__global__ void __launch_bounds__(kTailThreads)
state_tail_kernel(const float* tot, float* state, int d, int dv, RecOff so, RecOff dof) {
    __shared__ __align__(16) float sC[128][kTailCols];   // C[k][c0 + j]
    __shared__ float sS[kTailRows][128 + 1];              // S[i0 + r][k], padded rows
    __shared__ float sm[128];
    __shared__ float sp[kTailRows];                       // p[i0 + r]
    const int head = blockIdx.z, i0 = blockIdx.x * kTailRows, c0 = blockIdx.y * kTailCols;
    const int nr = d - i0 < kTailRows ? d - i0 : kTailRows;
    const int nc = dv - c0 < kTailCols ? dv - c0 : kTailCols;
    const float* t = tot + (size_t)head * so.R;
    float* o = state + (size_t)head * dof.R;
    const int tid = threadIdx.x;
    float vp[4];  // P at this thread's G entries (row tid / 8, columns 4 (tid % 8) .. + 3 of the block)
    {
        // every load is issued before the first shared-memory store, so that
        // they overlap (fixed trip counts, predicated on the sizes)
        constexpr int kNC = 128 * kTailCols / kTailThreads, kNS = kTailRows * 128 / kTailThreads;
        float vc[kNC], vs[kNS];
#pragma unroll
        for (int q = 0; q < kNC; ++q) {
            const int i = tid + q * kTailThreads, k = i / kTailCols, j = i % kTailCols;
            vc[q] = (k < d && j < nc) ? t[so.C + (size_t)k * dv + c0 + j] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kNS; ++q) {
            const int i = tid + q * kTailThreads, r = i / 128, k = i % 128;
            vs[q] = (r < nr && k < d) ? t[so.S + (size_t)(i0 + r) * d + k] : 0.f;
        }
        const float vm = tid < d ? t[so.m + tid] : 0.f;
        const float vps = (blockIdx.y == 0 && tid < nr) ? t[so.x + i0 + tid] : 0.f;
        {
            const int r = tid >> 3, j0 = 4 * (tid & 7);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                vp[q] = (r < nr && j0 + q < nc) ? t[so.X + (size_t)(i0 + r) * dv + c0 + j0 + q] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kNC; ++q) {
            const int i = tid + q * kTailThreads;
            sC[i / kTailCols][i % kTailCols] = vc[q];
        }
#pragma unroll
        for (int q = 0; q < kNS; ++q) {
            const int i = tid + q * kTailThreads;
            sS[i / 128][i % 128] = vs[q];
        }
        sm[tid] = vm;
        if (tid < kTailRows) sp[tid] = vps;
    }
    __syncthreads();
    for (int i = tid; i < nr * nc; i += kTailThreads) {
        const int r = i / nc, j = i % nc;
        o[dof.C + (size_t)(i0 + r) * dv + c0 + j] = sC[i0 + r][j];
    }
    if (blockIdx.y == 0) {
        for (int i = tid; i < nr * d; i += kTailThreads) o[dof.S + (size_t)i0 * d + i] = sS[i / d][i % d];
        if (blockIdx.x == 0)
            for (int i = tid; i < d; i += kTailThreads) o[dof.m + i] = sm[i];
        // h: warp w takes rows w, w + 4, ... (lanes split k, then a fixed-order reduction)
        const int lane = tid & 31;
        for (int r = tid >> 5; r < nr; r += kTailThreads / 32) {
            float h = 0.f;
            for (int k = lane; k < d; k += 32) h = fmaf(sS[r][k], sm[k], h);
#pragma unroll
            for (int w = 16; w >= 1; w >>= 1) h += __shfl_xor_sync(0xffffffffu, h, w);
            if (lane == 0) o[dof.x + i0 + r] = h - sp[r];
        }
    }
    const int r = tid >> 3, j0 = 4 * (tid & 7);
    if (r >= nr || j0 >= nc) return;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
    for (int k = 0; k < d; ++k) {
        const float4 c = *reinterpret_cast<const float4*>(&sC[k][j0]);
        const float x = sS[r][k];
        a0 = fmaf(x, c.x, a0); a1 = fmaf(x, c.y, a1); a2 = fmaf(x, c.z, a2); a3 = fmaf(x, c.w, a3);
    }
    const float acc[4] = {a0, a1, a2, a3};
    const size_t g = (size_t)(i0 + r) * dv + c0 + j0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (j0 + q < nc) o[dof.X + g + q] = acc[q] - vp[q];
}

__global__ void copy_strided_kernel(const float* src, long long s_src, float* dst, long long s_dst, size_t len) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int b = blockIdx.y;
    if (i < len) dst[(long long)b * s_dst + i] = src[(long long)b * s_src + i];
}

}  // namespace

cudaError_t launch_exscan(const float* in, float* out, int BH, int N, size_t R, size_t off, size_t len,
                          float* total, size_t total_stride, cudaStream_t s) {
    if (BH == 0 || len == 0) return cudaSuccess;
    const bool vec = ((off | len | R | total_stride) % 4 == 0) && ((reinterpret_cast<uintptr_t>(in) |
                     reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(total)) % 16 == 0);
    if (!out && !total) return cudaErrorInvalidValue;
    if (vec) {
        dim3 grid((unsigned)((len / 4 + kScanThreads - 1) / kScanThreads), BH);
        // axes longer than 8 records keep 16 records per thread in flight (the
        // element range alone gives too few threads to cover the latency)
        if (N > kScanUnroll) {
            if (out) exscan4_kernel<true, 16><<<grid, kScanThreads, 0, s>>>(in, out, N, R, off, len, total, total_stride);
            else exscan4_kernel<false, 16><<<grid, kScanThreads, 0, s>>>(in, out, N, R, off, len, total, total_stride);
        } else {
            if (out) exscan4_kernel<true, kScanUnroll><<<grid, kScanThreads, 0, s>>>(in, out, N, R, off, len, total,
                                                                                       total_stride);
            else exscan4_kernel<false, kScanUnroll><<<grid, kScanThreads, 0, s>>>(in, out, N, R, off, len, total,
                                                                                    total_stride);
        }
    } else {
        dim3 grid((unsigned)((len + kScanThreads - 1) / kScanThreads), BH);
        if (out) exscan_kernel<true><<<grid, kScanThreads, 0, s>>>(in, out, N, R, off, len, total, total_stride);
        else exscan_kernel<false><<<grid, kScanThreads, 0, s>>>(in, out, N, R, off, len, total, total_stride);
    }
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_cross(const CrossArgs& a, cudaStream_t s) {
    if (a.nb == 0) return cudaSuccess;
    const int ncol = a.dv + (a.bx ? 1 : 0);
    dim3 grid((ncol + kTile - 1) / kTile, (a.d + kTile - 1) / kTile, a.nb);
    cross_kernel<<<grid, 256, 0, s>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_decay_factors(float* fac, int T, float gamma, SegPlan plan, cudaStream_t s) {
    if (plan.nseg == 0) return cudaSuccess;
    decay_factors_kernel<<<(plan.nseg + 255) / 256, 256, 0, s>>>(fac, T, gamma, plan);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_decay_exscan(const float* in, float* out, int BH, int N, size_t R, size_t off, size_t len,
                                float* total, size_t total_stride, const float* fac, cudaStream_t s) {
    if (BH == 0 || len == 0) return cudaSuccess;
    const bool vec = ((off | len | R | total_stride) % 4 == 0) && ((reinterpret_cast<uintptr_t>(in) |
                     reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(total)) % 16 == 0);
    if (vec) {
        dim3 grid((unsigned)((len / 4 + kScanThreads - 1) / kScanThreads), BH);
        decay_exscan4_kernel<<<grid, kScanThreads, 0, s>>>(in, out, N, R, off, len, total, total_stride, fac);
    } else {
        dim3 grid((unsigned)((len + kScanThreads - 1) / kScanThreads), BH);
        decay_exscan_kernel<<<grid, kScanThreads, 0, s>>>(in, out, N, R, off, len, total, total_stride, fac);
    }
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_state_tail(const float* tot, float* state, int BH, int d, int dv, cudaStream_t s) {
    if (BH == 0) return cudaSuccess;
    if (d <= 0 || dv <= 0 || d > 128 || dv > 128 || BH > 65535) return cudaErrorInvalidValue;
    dim3 grid((d + kTailRows - 1) / kTailRows, (dv + kTailCols - 1) / kTailCols, BH);
    state_tail_kernel<<<grid, kTailThreads, 0, s>>>(tot, state, d, dv, summary_offsets(d, dv), decode_offsets(d, dv));
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_copy_strided(const float* src, long long s_src, float* dst, long long s_dst, size_t len,
                                int nb, cudaStream_t s) {
    if (nb == 0 || len == 0) return cudaSuccess;
    dim3 grid((unsigned)((len + 255) / 256), nb);
    copy_strided_kernel<<<grid, 256, 0, s>>>(src, s_src, dst, s_dst, len);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace hla2
