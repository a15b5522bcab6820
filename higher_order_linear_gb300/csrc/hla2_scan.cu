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
            pout[(size_t)(r + j) * R] = run;
            run += x[j];
        }
    }
    for (; r < N; ++r) {
        const float x = pin[(size_t)r * R];
        pout[(size_t)r * R] = run;
        run += x;
    }
    if (total) total[(size_t)bh * total_stride + i] = run;
}

// Same scan, four consecutive elements per thread (16-byte accesses); used
// when the element range, the record length and the pointers allow it.
__global__ void __launch_bounds__(kScanThreads)
exscan4_kernel(const float* in, float* out, int N, size_t R, size_t off, size_t len, float* total,
               size_t total_stride) {
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
            run.x += x[j].x; run.y += x[j].y; run.z += x[j].z; run.w += x[j].w;
        }
    }
    for (; r < N; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(pin + (size_t)r * R);
        *reinterpret_cast<float4*>(pout + (size_t)r * R) = run;
        run.x += x.x; run.y += x.y; run.z += x.z; run.w += x.w;
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
    if (vec) {
        dim3 grid((unsigned)((len / 4 + kScanThreads - 1) / kScanThreads), BH);
        exscan4_kernel<<<grid, kScanThreads, 0, s>>>(in, out, N, R, off, len, total, total_stride);
    } else {
        dim3 grid((unsigned)((len + kScanThreads - 1) / kScanThreads), BH);
        exscan_kernel<<<grid, kScanThreads, 0, s>>>(in, out, N, R, off, len, total, total_stride);
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

cudaError_t launch_copy_strided(const float* src, long long s_src, float* dst, long long s_dst, size_t len,
                                int nb, cudaStream_t s) {
    if (nb == 0 || len == 0) return cudaSuccess;
    dim3 grid((unsigned)((len + 255) / 256), nb);
    copy_strided_kernel<<<grid, 256, 0, s>>>(src, s_src, dst, s_dst, len);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace hla2
