// hla2_tc_scan.cu -- the forward's exclusive scan over segment summaries in
// one launch, with the cross products on tensor cores.
//
// HLA summary (arXiv 2510.27258), section 4 "Parallel training via
// associative scans": segment summaries are joined by a semidirect-product
// combine whose cross term is a d x d by d x dv product, and an exclusive
// scan gives every segment the state of the serial recurrence at its start.
//
// The forward cuts each head into a few segments (about ten on the long
// workloads), so the scan is short and latency-bound: the element-serial
// sums and the batched products it used to run as three launches cost more in
// launch and pass latency than in work.  Here one CTA computes one segment's
// prefix by folding the records before it, in order:
//   HLA (P-form):  S_<r = sum_{j<r} S_j,        P_<r = sum_{j<r} (P_j + S_<j C_j)
//                  (normalised: p_<r = sum_{j<r} (p_j + S_<j m_j))
//   decayed:       S_<j+1 = f_j S_<j + S_j,     P_<j+1 = f_j^2 P_<j + P_j + f_j S_<j C_j
//                  (f_j = gamma^{tokens of segment j}, the decayed combine)
//   AHLA:          P_<r = sum_{j<r} P_j,        E_<r = sum_{j<r} (E_j + M_j P_<j)
// The running sums stay in fp32 registers; each product is taken on the
// tensor cores with both operands split into bf16 hi + lo parts
// (hi*hi + hi*lo + lo*hi, fp32 accumulation in tensor memory), which keeps
// about 16 significant bits of every operand, as the batched cross kernel did.
// CTA r does r - 1 products (the first prefix factor is zero), so the last
// segment's CTA bounds the launch; with about ten segments that is far below
// the three launches it replaces.
#include "hla2_tc_common.cuh"

namespace hla2 {
namespace {

constexpr int kScanWarps = 16;  // four per 32-lane quarter of tensor memory
constexpr int kScanThreadsTC = kScanWarps * 32;

template <int D>
struct ScanTileLayout {
    static constexpr uint32_t kA = 128u * D * 2u;  // A operand keeps 128 rows (MMA M = 128); rows >= D are zero
    static constexpr uint32_t kB = (uint32_t)D * D * 2u;
    static constexpr uint32_t Ahi = 0, Alo = kA, Bhi = 2 * kA, Blo = 2 * kA + kB;
    static constexpr uint32_t kBytes = 2 * kA + 2 * kB;
};

template <int NC>
__device__ __forceinline__ void tmem_ld_nc(uint32_t taddr, float (&v)[NC]) {
    static_assert(NC == 16 || NC == 32, "16 or 32 columns");
    uint32_t r[32];
    if (NC == 32) {
        tmem_ld32(taddr, r);
    } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    }
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < NC; ++i) v[i] = __uint_as_float(r[i]);
}

// Loads NC consecutive floats (16-byte aligned) into v.
template <int NC>
__device__ __forceinline__ void ld_row(const float* p, float (&v)[NC]) {
#pragma unroll
    for (int i = 0; i < NC; i += 4) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(p + i));
        v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
    }
}
template <int NC>
__device__ __forceinline__ void st_row(float* p, const float (&v)[NC]) {
#pragma unroll
    for (int i = 0; i < NC; i += 4) *reinterpret_cast<float4*>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}
template <int NC>
__device__ __forceinline__ void put_split_row(const Tile& hi, const Tile& lo, int r, int c0, const float (&v)[NC]) {
#pragma unroll
    for (int i = 0; i < NC; i += 4) put4_split(hi, lo, r, c0 + i, make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
}

template <int D, int OP, bool EXTRA>
__global__ void __launch_bounds__(kScanThreadsTC, 1) tc_scan_kernel(ScanArgs a) {
    using TL = ScanTileLayout<D>;
    constexpr int NC = D / 4;  // columns per thread: four warps share a lane quarter
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    __shared__ __align__(8) unsigned long long bar_mma;
    __shared__ uint32_t tmem_slot;
    __shared__ float px_part[4][128];  // normalised walk: partial S_<j m_j per column part
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, part = warp >> 2;
    const int row = quarter * 32 + lane;
    const int c0 = part * NC;
    const bool state_row = row < D;
    const int r = blockIdx.x, head = blockIdx.y;
    const size_t R = a.R;
    const float* rec0 = a.summ + (size_t)head * a.nseg * R;
    float* out = a.prefix + ((size_t)head * a.nseg + r) * R;
    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tAh{dsm + TL::Ahi, 128}, tAl{dsm + TL::Alo, 128}, tBh{dsm + TL::Bhi, D}, tBl{dsm + TL::Blo, D};
    constexpr uint32_t kCols = D < 32 ? 32 : D;

    // field offsets: the running pair (acc1, acc2) and the record fields feeding them
    //   HLA / decayed: acc1 = S (S), acc2 = P (X); product S_<j C_j, C at C
    //   AHLA:          acc1 = P (C), acc2 = E (X); product M_j P_<j, M at S
    const size_t off1 = (OP == kScanAHLA) ? a.ro.C : a.ro.S;
    const size_t off2 = a.ro.X;
    const size_t offR = (OP == kScanAHLA) ? a.ro.S : a.ro.C;  // the record's own product factor

    if (tid == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&bar_mma), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // A rows >= D never change: zero them once (both parts)
    if (D < 128)
        for (int i = tid; i < (128 - D) * D / 4; i += kScanThreadsTC)
            put4_split(tAh, tAl, D + i / (D / 4), (i % (D / 4)) * 4, make_float4(0.f, 0.f, 0.f, 0.f));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    constexpr uint32_t idesc = idesc_bf16(128, D, false, true);

    float acc1[NC], acc2[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) acc1[i] = acc2[i] = 0.f;
    float px = 0.f, ax = 0.f;  // normalised: this part's sum of S_<j m_j, and sum of p_j (part 0)
    bool ok = true;
    uint32_t phase = 0;

    for (int j = 0; j < r; ++j) {
        const float* rec = rec0 + (size_t)j * R;
        // the product has a zero factor for j = 0 (S_<0 = 0, P_<0 = 0)
        const bool prod = j > 0;
        if (prod) {
            // operands of this record's product: A (M = output rows, K-major),
            // B (rows = contraction index, read MN-major)
            if (state_row) {
                float x[NC];
                ld_row<NC>(rec + offR + (size_t)row * D + c0, x);
                if (OP == kScanAHLA) {
                    put_split_row<NC>(tAh, tAl, row, c0, x);      // A = M_j
                    put_split_row<NC>(tBh, tBl, row, c0, acc1);   // B = P_<j
                } else {
                    put_split_row<NC>(tAh, tAl, row, c0, acc1);   // A = S_<j
                    put_split_row<NC>(tBh, tBl, row, c0, x);      // B = C_j
                }
            }
            fence_proxy_async();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (tid == 0) {
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tmem, tAh.kmaj(ks), tBh.mnmaj(ks), idesc, ks > 0);
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tmem, tAh.kmaj(ks), tBl.mnmaj(ks), idesc, 1);
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tmem, tAl.kmaj(ks), tBh.mnmaj(ks), idesc, 1);
                mma_commit(smem_u32(&bar_mma));
            }
            __syncwarp();
        }
        // while the products run: this record's summands (S_<j, P_<j, or
        // P_<j, E_<j for AHLA, already fed the tiles and the p term above)
        float f = 1.f, f2 = 1.f;
        if (OP == kScanDecay) {
            f = __ldg(a.fac + j);
            f2 = __ldg(a.fac + a.nseg + j);
        }
        if (EXTRA && state_row) {
            // p_<r gathers p_j + S_<j m_j: this thread's columns of S_<j times m_j
            float m[NC];
            ld_row<NC>(rec + a.ro.m + c0, m);
#pragma unroll
            for (int i = 0; i < NC; ++i) px = fmaf(acc1[i], m[i], px);
            if (part == 0) ax += __ldg(rec + a.ro.x + row);
        }
        if (state_row) {
            float x[NC];
            ld_row<NC>(rec + off1 + (size_t)row * D + c0, x);
#pragma unroll
            for (int i = 0; i < NC; ++i) acc1[i] = fmaf(f, acc1[i], x[i]);
            ld_row<NC>(rec + off2 + (size_t)row * D + c0, x);
#pragma unroll
            for (int i = 0; i < NC; ++i) acc2[i] = fmaf(f2, acc2[i], x[i]);
        }
        if (prod) {
            // bounded wait for the products, then this thread's lane and columns
            bool done = mbar_try(smem_u32(&bar_mma), phase);
            if (!done) {
                const unsigned long long t0 = globaltimer();
                while (!(done = mbar_try(smem_u32(&bar_mma), phase)))
                    if (globaltimer() - t0 > kWaitNs) break;
            }
            phase ^= 1u;
            tc_fence_after();
            if (!done) {
                if (lane == 0) atomicExch(a.status, (int)kDevWaitTimeout);
                s_abort = 1;
            }
            __syncwarp();
            // the load is warp-collective: a warp loads only once every lane saw
            // the products complete; rows >= D are loaded and ignored
            if (__all_sync(0xffffffffu, done)) {
                float pr[NC];
                tmem_ld_nc<NC>(tmem + lane_off + (uint32_t)c0, pr);
#pragma unroll
                for (int i = 0; i < NC; ++i) acc2[i] = fmaf(f, pr[i], acc2[i]);
            }
            tc_fence_before();
            __syncthreads();  // tensor memory and the operand tiles are reused by the next product
            if (s_abort) {  // block-uniform: read after the barrier
                ok = false;
                break;
            }
        }
    }
    if (EXTRA) {
        px_part[part][row] = px;
        __syncthreads();
    }
    if (ok && state_row) {
        st_row<NC>(out + off1 + (size_t)row * D + c0, acc1);
        st_row<NC>(out + off2 + (size_t)row * D + c0, acc2);
        if (EXTRA && part == 0) out[a.ro.x + row] = ax + px_part[0][row] + px_part[1][row] + px_part[2][row] +
                                                    px_part[3][row];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
}

template <int D, int OP, bool EXTRA>
cudaError_t launch_scan_t(const ScanArgs& a, int BH, cudaStream_t s) {
    const size_t smem = ScanTileLayout<D>::kBytes + 1024;
    auto kern = tc_scan_kernel<D, OP, EXTRA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.nseg, BH);
    kern<<<grid, kScanThreadsTC, smem, s>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_scan(int op, const ScanArgs& a, int BH, int d, int dv, cudaStream_t s) {
    if (BH == 0 || a.nseg == 0) return cudaSuccess;
    if (d != dv || (d != 64 && d != 128) || BH > 65535 || a.nseg > 65535) return cudaErrorInvalidValue;
    if (a.extra && op != kScanHLA) return cudaErrorInvalidValue;
    if (op == kScanHLA) {
        if (a.extra) return d == 128 ? launch_scan_t<128, kScanHLA, true>(a, BH, s) : launch_scan_t<64, kScanHLA, true>(a, BH, s);
        return d == 128 ? launch_scan_t<128, kScanHLA, false>(a, BH, s) : launch_scan_t<64, kScanHLA, false>(a, BH, s);
    }
    if (op == kScanDecay)
        return d == 128 ? launch_scan_t<128, kScanDecay, false>(a, BH, s) : launch_scan_t<64, kScanDecay, false>(a, BH, s);
    if (op == kScanAHLA)
        return d == 128 ? launch_scan_t<128, kScanAHLA, false>(a, BH, s) : launch_scan_t<64, kScanAHLA, false>(a, BH, s);
    return cudaErrorInvalidValue;
}

}  // namespace hla2
