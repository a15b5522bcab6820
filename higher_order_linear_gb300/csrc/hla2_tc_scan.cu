// hla2_tc_scan.cu -- the forward's exclusive scan over segment summaries in
// one launch, with the cross products on tensor cores.
//
// HLA summary (arXiv 2510.27258), section 4 "Parallel training via
// associative scans": segment summaries are joined by a semidirect-product
// combine whose cross term is a d x d by d x dv product, and an exclusive
// scan gives every segment the state of the serial recurrence at its start.
//
// The forward cuts each head into a few segments (about ten on the long
// workloads), so the scan is short and latency-bound.  It runs as one launch
// of a CTA per (head, record r):
//   1. fold the product factor over the earlier records: S_<r (HLA, with the
//      decay factors for the decayed operator) or P_<r (AHLA), which is also
//      the prefix's own final value;
//   2. take record r's cross product on tensor cores: the term
//      X_r = P_r + S_<r C_r (HLA), P_r + f_r S_<r C_r (decayed, f_r =
//      gamma^{tokens of segment r}), E_r + M_r P_<r (AHLA); normalised HLA
//      also x_r = p_r + S_<r m_r;
//   3. a second launch (the element-parallel running sums of hla2_scan.cu)
//      turns the terms into exclusive prefix sums in place:
//      P_<n = sum_{r<n} X_r (decayed: P_<n+1 = f_n^2 P_<n + X_n).
// Every product has both operands split into bf16 hi + lo parts
// (hi*hi + hi*lo + lo*hi, fp32 accumulation in tensor memory), which keeps
// about 16 significant bits of every operand.  Running sums are fp32, laid out
// so that a warp reads and writes whole rows of a record.
#include "hla2_tc_common.cuh"

namespace hla2 {
namespace {

constexpr int kScanWarps = 16;  // four per 32-lane quarter of tensor memory
// Scans of up to this many segments run in one launch (each CTA sums its
// whole prefix); longer ones take one product per CTA and a running-sum pass.
// On GB300 the single launch took 8.6 us at 3 segments (against 18.6 us for
// the two launches) and 43 us at 10 (against 27 us).
constexpr int kScanFullMaxSegments = 4;
constexpr int kScanThreadsTC = kScanWarps * 32;
constexpr int kTotParts = 8;  // CTAs per head that form the plain totals (ScanArgs::tot)

template <int D>
struct ScanTileLayout {
    static constexpr uint32_t kA = 128u * D * 2u;  // A operand keeps 128 rows (MMA M = 128); rows >= D are zero
    static constexpr uint32_t kB = (uint32_t)D * D * 2u;
    static constexpr uint32_t Ahi = 0, Alo = kA, Bhi = 2 * kA, Blo = 2 * kA + kB;
    static constexpr int kStageLd = D + 4;  // fp32 row stride of the product staging (padded against bank conflicts)
    static constexpr uint32_t Stage = 2 * kA + 2 * kB;
    static constexpr uint32_t kBytes = Stage + (uint32_t)D * kStageLd * 4u;
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

// Element layout of the running sums: thread t holds the float4 pieces
// f = t + kScanThreadsTC * i of a D x D matrix (row 4f / D, column 4f % D),
// so that a warp reads and writes whole rows (coalesced).  Only the product
// drain uses the tensor-memory layout (lane = row), through a staging buffer.
template <int D>
struct Piece {
    static constexpr int N = D * D / 4 / kScanThreadsTC;  // float4 pieces per thread
    __device__ static int row(int tid, int i) { return (4 * (tid + kScanThreadsTC * i)) / D; }
    __device__ static int col(int tid, int i) { return (4 * (tid + kScanThreadsTC * i)) % D; }
};

template <int D>
__device__ __forceinline__ void ld_mat(const float* m, int tid, float4 (&v)[Piece<D>::N]) {
#pragma unroll
    for (int i = 0; i < Piece<D>::N; ++i) v[i] = __ldg(reinterpret_cast<const float4*>(m) + tid + kScanThreadsTC * i);
}

// FULL: CTA r computes its whole prefix (every term X_j, j < r, summed in
// registers): one launch, r - 1 products in a row; for short scans.
// Otherwise CTA r computes only its own term X_r, and an exclusive running
// sum over the records (a second, element-parallel launch) completes the
// prefixes: one product per CTA; for longer scans.
template <int D, int OP, bool EXTRA, bool FULL>
__global__ void __launch_bounds__(kScanThreadsTC, 1) tc_scan_kernel(ScanArgs a) {
    using TL = ScanTileLayout<D>;
    using PC = Piece<D>;
    constexpr int NV = PC::N;
    constexpr int NC = D / 4;  // drain: columns per warp (four warps share a lane quarter)
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    __shared__ __align__(8) unsigned long long bar_mma;
    __shared__ __align__(8) unsigned long long ring_bar[3];  // the fold's record ring (one barrier per buffer)
    __shared__ uint32_t tmem_slot;
    __shared__ int s_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, part = warp >> 2;
    const int drow = quarter * 32 + lane;  // tensor-memory lane this thread drains
    const int dc0 = part * NC;
    // grid (BH, nseg [+ kTotParts]): the records with the longest folds
    // (largest r) go first, the plain totals last
    const int head = blockIdx.x, r = a.nseg - 1 - (int)blockIdx.y;
    const size_t R = a.R;
    if ((int)blockIdx.y >= a.nseg) {
        // plain totals over the records, part z of the float4 range, records
        // added in order
        const int z = (int)blockIdx.y - a.nseg;
        const size_t n4 = a.tot_len / 4, per = (n4 + kTotParts - 1) / kTotParts;
        const size_t i_end = n4 < (z + 1) * per ? n4 : (z + 1) * per;
        const float4* src = reinterpret_cast<const float4*>(a.summ + (size_t)head * a.nseg * R);
        float4* dst = reinterpret_cast<float4*>(a.tot + (size_t)head * R);
        const size_t R4 = R / 4;
        for (size_t i = z * per + tid; i < i_end; i += kScanThreadsTC) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            int j = 0;
            for (; j + 4 <= a.nseg; j += 4) {
                float4 x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) x[u] = __ldg(src + (size_t)(j + u) * R4 + i);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc.x += x[u].x; acc.y += x[u].y; acc.z += x[u].z; acc.w += x[u].w;
                }
            }
            for (; j < a.nseg; ++j) {
                const float4 x = __ldg(src + (size_t)j * R4 + i);
                acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
            }
            dst[i] = acc;
        }
        return;
    }
    const float* rec0 = a.summ + (size_t)head * a.nseg * R;
    float* out = a.prefix + ((size_t)head * a.nseg + r) * R;
    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tAh{dsm + TL::Ahi, 128}, tAl{dsm + TL::Alo, 128}, tBh{dsm + TL::Bhi, D}, tBl{dsm + TL::Blo, D};
    float* stage = reinterpret_cast<float*>(dsm_raw + (dsm - smem_u32(dsm_raw)) + TL::Stage);
    constexpr uint32_t kCols = D < 32 ? 32 : D;

    // fields: F1 is folded over the earlier records into the prefix factor
    // (S_<j, or P_<j for AHLA), which is also the prefix's own final value;
    // record j's term is X_j = F2_j + f_j * (product), F2 and the product:
    //   HLA / decayed: F1 = S, F2 = P (at X), product S_<j C_j  (C at C)
    //   AHLA:          F1 = P (at C), F2 = E (at X), product M_j P_<j  (M at S)
    const size_t off1 = (OP == kScanAHLA) ? a.ro.C : a.ro.S;
    const size_t off2 = a.ro.X;
    const size_t offR = (OP == kScanAHLA) ? a.ro.S : a.ro.C;

    if (tid == 0) {
        s_flag = 0;
        mbar_init(smem_u32(&bar_mma), 1);
        for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&ring_bar[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (D < 128)  // A rows >= D stay zero
        for (int i = tid; i < (128 - D) * D / 4; i += kScanThreadsTC)
            put4_split(tAh, tAl, D + i / (D / 4), (i % (D / 4)) * 4, make_float4(0.f, 0.f, 0.f, 0.f));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    constexpr uint32_t idesc = idesc_bf16(128, D, false, true);
    uint32_t phase = 0;

    // acc += f * (the product of record j's factor xop with the running factor
    // acc1), on tensor cores; false when a bounded wait ran out (block-uniform)
    auto add_product = [&](const float4 (&acc1)[NV], const float4 (&xop)[NV], float f, float4 (&acc)[NV]) -> bool {
        // A (output rows, K-major), B (rows = contraction index, MN-major)
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int rr = PC::row(tid, i), cc = PC::col(tid, i);
            if (OP == kScanAHLA) {
                put4_split(tAh, tAl, rr, cc, xop[i]);   // A = M_j
                put4_split(tBh, tBl, rr, cc, acc1[i]);  // B = P_<j
            } else {
                put4_split(tAh, tAl, rr, cc, acc1[i]);  // A = S_<j
                put4_split(tBh, tBl, rr, cc, xop[i]);   // B = C_j
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();  // tiles written; the previous staged product read
        tc_fence_after();
        if (tid == 0) {
            for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tmem, tAh.kmaj(ks), tBh.mnmaj(ks), idesc, ks > 0);
            for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tmem, tAh.kmaj(ks), tBl.mnmaj(ks), idesc, 1);
            for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tmem, tAl.kmaj(ks), tBh.mnmaj(ks), idesc, 1);
            mma_commit(smem_u32(&bar_mma));
        }
        __syncwarp();
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
            s_flag = 1;
        }
        __syncwarp();
        // drain (warp-collective, lane = row) into the staging buffer, only
        // once every lane saw the products complete; rows >= D are dropped
        if (__all_sync(0xffffffffu, done)) {
            float pr[NC];
            tmem_ld_nc<NC>(tmem + lane_off + (uint32_t)dc0, pr);
            if (drow < D)
#pragma unroll
                for (int i = 0; i < NC; i += 4)
                    *reinterpret_cast<float4*>(stage + drow * TL::kStageLd + dc0 + i) =
                        make_float4(pr[i], pr[i + 1], pr[i + 2], pr[i + 3]);
        }
        tc_fence_before();
        __syncthreads();  // staged; tensor memory free for the next product
        if (s_flag) return false;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const float4 y = *reinterpret_cast<const float4*>(stage + PC::row(tid, i) * TL::kStageLd + PC::col(tid, i));
            acc[i] = make_float4(fmaf(f, y.x, acc[i].x), fmaf(f, y.y, acc[i].y), fmaf(f, y.z, acc[i].z),
                                 fmaf(f, y.w, acc[i].w));
        }
        return true;
    };
    auto fold = [&](float4 (&acc)[NV], const float* m, float f) {  // acc = f * acc + m
        float4 x[NV];
        ld_mat<D>(m, tid, x);
#pragma unroll
        for (int i = 0; i < NV; ++i)
            acc[i] = make_float4(fmaf(f, acc[i].x, x[i].x), fmaf(f, acc[i].y, x[i].y), fmaf(f, acc[i].z, x[i].z),
                                 fmaf(f, acc[i].w, x[i].w));
    };
    // normalised: x_j = p_j + S_<j m_j, per row (threads sharing a row reduce over it)
    constexpr int kLanesPerRow = D / 4;
    auto add_pterm = [&](const float4 (&acc1)[NV], const float* rec, float (&px)[NV]) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const float4 m = __ldg(reinterpret_cast<const float4*>(rec + a.ro.m + PC::col(tid, i)));
            px[i] += acc1[i].x * m.x + acc1[i].y * m.y + acc1[i].z * m.z + acc1[i].w * m.w;
        }
    };

    float4 acc1[NV], acc2[NV];  // F1 folded; the prefix's corrected part (FULL) or this record's term
    float px[NV];
    float ax = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        acc1[i] = acc2[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        px[i] = 0.f;
    }
    if (FULL) {
        // the whole prefix: X_<j+1 = f_j^2 X_<j + F2_j + f_j (product of record j)
        for (int j = 0; j < r; ++j) {
            const float* rec = rec0 + (size_t)j * R;
            const float f = (OP == kScanDecay) ? __ldg(a.fac + j) : 1.f;
            const float f2 = (OP == kScanDecay) ? __ldg(a.fac + a.nseg + j) : 1.f;
            fold(acc2, rec + off2, f2);
            if (EXTRA) {
                add_pterm(acc1, rec, px);
                if (tid < D) ax += __ldg(rec + a.ro.x + tid);
            }
            if (j > 0) {
                float4 xop[NV];
                ld_mat<D>(rec + offR, tid, xop);
                if (!add_product(acc1, xop, f, acc2)) break;
            }
            fold(acc1, rec + off1, f);
        }
    } else {
        // this record's term X_r; the running sum over records follows in a second launch.
        // The fold's records arrive by bulk copies into a ring of kRing
        // shared-memory buffers (the operand tiles and the staging are free
        // until the product; at D < 128 the ring starts past A, whose rows
        // >= D hold zeros), kRing records in flight, folded in order.
        constexpr int kRing = (D == 128) ? 3 : 2;
        constexpr uint32_t kRecBytes = (uint32_t)D * D * 4u, kRingOff = (D < 128) ? TL::Bhi : 0u;
        static_assert(kRingOff + kRing * kRecBytes <= TL::kBytes, "the ring fits the kernel's shared memory");
        LoadLedger<kRing> ring(smem_u32(&ring_bar[0]));
        auto issue_rec = [&](int j) {  // thread 0
            const int b = j % kRing;
            ring.note(b);
            mbar_expect_tx(smem_u32(&ring_bar[b]), kRecBytes);
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(dsm + kRingOff + (uint32_t)b * kRecBytes), "l"(rec0 + (size_t)j * R + off1),
                         "r"(kRecBytes), "r"(smem_u32(&ring_bar[b]))
                         : "memory");
        };
        if (tid == 0)
            for (int j = 0; j < kRing && j < r; ++j) issue_rec(j);
        for (int i0 = 0; i0 < r; ++i0) {
            const uint32_t rb = smem_u32(&ring_bar[i0 % kRing]), par = (uint32_t)((i0 / kRing) & 1);
            bool ok = mbar_try(rb, par);
            if (!ok) {
                const unsigned long long t0 = globaltimer();
                while (!(ok = mbar_try(rb, par)))
                    if (globaltimer() - t0 > kWaitNs) break;
            }
            if (!ok) {
                atomicExch(a.status, (int)kDevWaitTimeout);
                s_flag = 1;
            }
            const float* buf = reinterpret_cast<const float*>(dsm_raw + (dsm - smem_u32(dsm_raw)) + kRingOff +
                                                              (uint32_t)(i0 % kRing) * kRecBytes);
            const float f = (OP == kScanDecay) ? __ldg(a.fac + i0) : 1.f;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const float4 x = reinterpret_cast<const float4*>(buf)[tid + kScanThreadsTC * i];
                acc1[i] = make_float4(fmaf(f, acc1[i].x, x.x), fmaf(f, acc1[i].y, x.y), fmaf(f, acc1[i].z, x.z),
                                      fmaf(f, acc1[i].w, x.w));
            }
            __syncthreads();  // every thread has read the buffer (and seen any timeout)
            if (s_flag) break;
            if (tid == 0 && i0 + kRing < r) issue_rec(i0 + kRing);
        }
        // no copy may still be landing when the buffers become operand tiles
        if (tid == 0 && !ring.settle()) atomicExch(a.status, (int)kDevWaitTimeout);
        __syncthreads();
        const float* rec = rec0 + (size_t)r * R;
        fold(acc2, rec + off2, 1.f);
        if (EXTRA) {
            add_pterm(acc1, rec, px);
            if (tid < D) ax = __ldg(rec + a.ro.x + tid);
        }
        if (r > 0) {
            float4 xop[NV];
            ld_mat<D>(rec + offR, tid, xop);
            add_product(acc1, xop, (OP == kScanDecay) ? __ldg(a.fac + r) : 1.f, acc2);
        }
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        reinterpret_cast<float4*>(out + off1)[tid + kScanThreadsTC * i] = acc1[i];
        reinterpret_cast<float4*>(out + off2)[tid + kScanThreadsTC * i] = acc2[i];
    }
    if (EXTRA) {
        float* rowdot = stage;
        __syncthreads();  // every thread has read the staged products
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float v = px[i];
#pragma unroll
            for (int o = kLanesPerRow / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if ((tid % kLanesPerRow) == 0) rowdot[PC::row(tid, i)] = v;
        }
        __syncthreads();
        if (tid < D) out[a.ro.x + tid] = ax + rowdot[tid];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
}

template <int D, int OP, bool EXTRA, bool FULL>
cudaError_t launch_scan_t(const ScanArgs& a, int BH, cudaStream_t s) {
    const size_t smem = ScanTileLayout<D>::kBytes + 1024;
    auto kern = tc_scan_kernel<D, OP, EXTRA, FULL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(BH, a.nseg + (a.tot ? kTotParts : 0));
    kern<<<grid, kScanThreadsTC, smem, s>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

template <int D, bool FULL>
cudaError_t launch_scan_d(int op, const ScanArgs& a, int BH, cudaStream_t s) {
    if (op == kScanHLA)
        return a.extra ? launch_scan_t<D, kScanHLA, true, FULL>(a, BH, s) : launch_scan_t<D, kScanHLA, false, FULL>(a, BH, s);
    if (op == kScanDecay) return launch_scan_t<D, kScanDecay, false, FULL>(a, BH, s);
    return launch_scan_t<D, kScanAHLA, false, FULL>(a, BH, s);
}

}  // namespace

int tc_scan_full_max_segments() { return kScanFullMaxSegments; }

cudaError_t launch_tc_scan(int op, const ScanArgs& a, int BH, int d, int dv, cudaStream_t s) {
    if (BH == 0 || a.nseg == 0) return cudaSuccess;
    if (d != dv || (d != 64 && d != 128) || BH > 65535 || a.nseg > 65535) return cudaErrorInvalidValue;
    if ((a.extra && op != kScanHLA) || (op != kScanHLA && op != kScanDecay && op != kScanAHLA))
        return cudaErrorInvalidValue;
    if (a.tot && (a.tot_len % 4 != 0 || a.tot_len > a.R || a.R % 4 != 0 || a.nseg + kTotParts > 65535))
        return cudaErrorInvalidValue;
    const bool full = !a.terms_only && a.nseg <= kScanFullMaxSegments;
    if (d == 128) return full ? launch_scan_d<128, true>(op, a, BH, s) : launch_scan_d<128, false>(op, a, BH, s);
    return full ? launch_scan_d<64, true>(op, a, BH, s) : launch_scan_d<64, false>(op, a, BH, s);
}

}  // namespace hla2
