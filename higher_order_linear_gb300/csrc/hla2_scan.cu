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

// Decayed exclusive scan of P-form records, sequential over the records of
// one head.  A CTA owns kRows consecutive state rows (of S, C, P and of the
// vectors m, p) of one head and carries their running prefix in shared
// memory; the cross terms S C_r and S m_r need the CTA's S rows against all
// of C_r, read from global memory (coalesced along the value axis).
constexpr int kRows = 16;

__global__ void __launch_bounds__(256)
decay_scan_kernel(const float* __restrict__ summ, float* __restrict__ prefix, float* __restrict__ tot,
                  int T, int d, int dv, float gamma, SegPlan plan) {
    extern __shared__ float dsm[];
    const int head = blockIdx.y;
    const int r0 = blockIdx.x * kRows;
    const int nr = min(kRows, d - r0);
    const RecOff ro = summary_offsets(d, dv);
    float* sS = dsm;                      // kRows x d   running S rows
    float* sC = sS + kRows * d;           // kRows x dv  running C rows
    float* sP = sC + kRows * dv;          // kRows x dv  running P rows
    float* sm = sP + kRows * dv;          // kRows       running m
    float* sp = sm + kRows;               // kRows       running p
    float* sX = sp + kRows;               // kRows x (dv + 1)  cross terms S C_r | S m_r
    const int tid = threadIdx.x;
    for (int i = tid; i < kRows * d; i += 256) sS[i] = 0.f;
    for (int i = tid; i < kRows * dv; i += 256) { sC[i] = 0.f; sP[i] = 0.f; }
    if (tid < kRows) { sm[tid] = 0.f; sp[tid] = 0.f; }
    __syncthreads();
    const int w = dv + 1;
    for (int r = 0; r < plan.nseg; ++r) {
        const long long c0 = (long long)r * plan.nchunk / plan.nseg;
        const long long c1 = (long long)(r + 1) * plan.nchunk / plan.nseg;
        const long long t1 = min((long long)T, c1 * plan.granule);
        const int nb = (int)(t1 - c0 * plan.granule);  // tokens of segment r
        // f = gamma^nb by repeated squaring in double precision (fp32 products
        // over thousands of tokens would drift)
        double fd = 1.0, base = (double)gamma;
        for (int e = nb; e > 0; e >>= 1) {
            if (e & 1) fd *= base;
            base *= base;
        }
        const float f = (float)fd;
        const float* rec = summ + ((size_t)head * plan.nseg + r) * ro.R;
        float* pre = prefix + ((size_t)head * plan.nseg + r) * ro.R;
        // the exclusive prefix of record r is the running state
        for (int i = tid; i < nr * d; i += 256) pre[ro.S + (size_t)r0 * d + i] = sS[i];
        for (int i = tid; i < nr * dv; i += 256) pre[ro.X + (size_t)r0 * dv + i] = sP[i];
        if (tid < nr) pre[ro.x + r0 + tid] = sp[tid];
        if (tot) {
            for (int i = tid; i < nr * dv; i += 256) pre[ro.C + (size_t)r0 * dv + i] = sC[i];
            if (tid < nr) pre[ro.m + r0 + tid] = sm[tid];
        }
        // cross terms with the running S (before it absorbs record r)
        for (int i = tid; i < nr * w; i += 256) {
            const int a = i / w, e = i % w;
            const float* srow = sS + a * d;
            float acc = 0.f;
            if (e < dv)
                for (int b = 0; b < d; ++b) acc = fmaf(srow[b], rec[ro.C + (size_t)b * dv + e], acc);
            else
                for (int b = 0; b < d; ++b) acc = fmaf(srow[b], rec[ro.m + b], acc);
            sX[i] = acc;
        }
        __syncthreads();
        const float f2 = f * f;
        for (int i = tid; i < nr * dv; i += 256) {
            const int a = i / dv, e = i % dv;
            const size_t gi = (size_t)(r0 + a) * dv + e;
            sP[i] = fmaf(f2, sP[i], fmaf(f, sX[a * w + e], rec[ro.X + gi]));
            sC[i] = fmaf(f, sC[i], rec[ro.C + gi]);
        }
        if (tid < nr) {
            sp[tid] = fmaf(f2, sp[tid], fmaf(f, sX[tid * w + dv], rec[ro.x + r0 + tid]));
            sm[tid] = fmaf(f, sm[tid], rec[ro.m + r0 + tid]);
        }
        for (int i = tid; i < nr * d; i += 256) sS[i] = fmaf(f, sS[i], rec[ro.S + (size_t)r0 * d + i]);
        __syncthreads();
    }
    if (tot) {
        float* out = tot + (size_t)head * ro.R;
        for (int i = tid; i < nr * d; i += 256) out[ro.S + (size_t)r0 * d + i] = sS[i];
        for (int i = tid; i < nr * dv; i += 256) {
            out[ro.C + (size_t)r0 * dv + i] = sC[i];
            out[ro.X + (size_t)r0 * dv + i] = sP[i];
        }
        if (tid < nr) {
            out[ro.m + r0 + tid] = sm[tid];
            out[ro.x + r0 + tid] = sp[tid];
        }
    }
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

cudaError_t launch_decay_scan(const float* summ, float* prefix, float* tot, int BH, int T, int d, int dv,
                              float gamma, SegPlan plan, cudaStream_t s) {
    if (BH == 0 || plan.nseg == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * ((size_t)kRows * d + 2 * (size_t)kRows * dv + 2 * kRows +
                                         (size_t)kRows * (dv + 1));
    dim3 grid((d + kRows - 1) / kRows, BH);
    decay_scan_kernel<<<grid, 256, smem, s>>>(summ, prefix, tot, T, d, dv, gamma, plan);
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
