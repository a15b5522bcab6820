// hla2_tc_chunk.cu -- chunk summaries (hla2_chunk_summaries) of masked
// second-order HLA on GB300 tensor cores, for bf16 inputs, d = dv in
// {64, 128} and chunk lengths L in {64, 128}.
//
// HLA summary (arXiv 2510.27258), section 4 "Parallel training via
// associative scans": every chunk of L tokens is summarised by the moments
// S = K^T K, C = Q^T V, m = Q^T 1 and the cross summaries
//   G = K^T stril(K Q^T) V,   h = K^T stril(K Q^T) 1
// (stril: strictly below the diagonal, i.e. key i > query j inside the chunk),
// which the exclusive scan then joins.
//
// One CTA takes one 128-token tile of one head: two chunks at L = 64, one at
// L = 128.  Products over tokens are kept per chunk by splitting their
// K-steps (chunk a's 64 tokens, then chunk b's); B = K Q^T is formed for the
// whole tile and masked block-diagonally.  S, C and B are exact in fp32 (bf16
// inputs, fp32 accumulation).  G needs B and then Y = B V as operands, so
// both are split into bf16 hi + lo parts (Y = B_hi V + B_lo V,
// G = K^T Y_hi + K^T Y_lo), which keeps the fp32 summaries' accuracy
// (about 4e-6 of the largest entry in emulation).  m and h are sums over
// the chunk's rows on CUDA cores (h from fp32 row sums of B).
#include "hla2_tc_common.cuh"

namespace hla2 {
namespace {

struct ChunkParams {
    int T, N;       // tokens and chunks per head
    float* summ;    // [BH][N][R] records S|C|m|G|h
    int* status;
};

template <int D>
struct ChunkLayout {
    static constexpr uint32_t kTok = kL * D * 2;  // Q, K, V tiles
    static constexpr uint32_t kSq = kL * kL * 2;  // B (then Y) hi and lo tiles
    static constexpr uint32_t Q = 0, K = kTok, V = 2 * kTok, Bhi = 3 * kTok, Blo = Bhi + kSq;
    static constexpr uint32_t kBytes = Blo + kSq;
};

template <int D, int L>
__global__ void __launch_bounds__(kThreadsTC, 1)
tc_chunk_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                const __grid_constant__ CUtensorMap mV, ChunkParams p) {
    using LY = ChunkLayout<D>;
    constexpr int CPT = kL / L;  // chunks per 128-token tile
    constexpr int KS = L / 16;   // K-steps per chunk of a token contraction
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    enum { LD, C1, C2, C3, D1, D2, FIN, NBAR };
    __shared__ __align__(8) unsigned long long bars[NBAR];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    __shared__ float rowsum[2][kL];  // B row sums, per column half

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issuer = warp == kDrainWarps;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int row = quarter * 32 + lane;
    const int tile = blockIdx.x, head = blockIdx.y;
    const int chunk0 = tile * CPT;  // first chunk of this tile
    const bool state_rows = !issuer && ((D == 128) || quarter < D / 32);
    const size_t R = record_len(D, D);
    const RecOff ro = summary_offsets(D, D);

    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tQ{dsm + LY::Q, kL}, tK{dsm + LY::K, kL}, tV{dsm + LY::V, kL};
    const Tile tBh{dsm + LY::Bhi, kL}, tBl{dsm + LY::Blo, kL};
    auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };
    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), (i == D1 || i == D2) ? kDrainWarps : 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // tensor-memory regions: R0 = B then G of the tile's second chunk,
    // R1 = S of the first chunk then C of the second, R2 = S of the second
    // chunk then Y, R3 = C of the first chunk then G of the first
    const uint32_t tR0 = tmem, tR1 = tmem + 128, tR2 = tmem + 128 + D, tR3 = tmem + 128 + 2 * D;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int c128 = half * 64, cD = half * (D / 2);

    auto wait_bar = [&](int b, uint32_t parity) -> bool {
        const uint32_t a = bar(b);
        if (abort_flag) return false;
        if (mbar_try(a, parity)) return true;
        const unsigned long long t0 = globaltimer();
        while (!mbar_try(a, parity)) {
            if (abort_flag) return false;
            if (globaltimer() - t0 > kWaitNs) {
                abort_flag = 1;
                atomicExch(p.status, (int)kDevWaitTimeout);
                return false;
            }
        }
        return true;
    };
    auto drained = [&](int b) {
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(b)) : "memory");
    };
    // this warp's share (rows 32q.., D/2 columns) of a D x D fp32 region to
    // field `off` of chunk ch's record, unless the chunk lies past the head's end
    auto store_field = [&](uint32_t treg, int ch, size_t off) {
        uint32_t r[64];
        tmem_ld_cols<D / 2>(treg + lane_off + cD, r);
        if (chunk0 + ch >= p.N) return;
        float* dst = p.summ + ((size_t)head * p.N + chunk0 + ch) * R + off + (size_t)row * D + cD;
#pragma unroll
        for (int j = 0; j < D / 2; j += 4)
            *reinterpret_cast<float4*>(dst + j) = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                             __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
    };

    constexpr uint32_t iSq = idesc_bf16(128, 128, false, false);  // B = K Q^T
    constexpr uint32_t iMM = idesc_bf16(128, D, true, true);      // K^T K, Q^T V, K^T Y
    constexpr uint32_t iKM = idesc_bf16(128, D, false, true);     // B V

    if (issuer) {
        // lane 0 issues the tile loads and settles them before the CTA exits
        LoadLedger<1> loads(bar(LD));
        if (lane == 0) {
            loads.note(0);
            mbar_expect_tx(bar(LD), 3u * kL * D * 2u);
#pragma unroll
            for (int k = 0; k < D / 64; ++k) {
                tma_load_3d(tQ.base + k * tQ.block_bytes(), &mQ, k * 64, tile * kL, head, bar(LD));
                tma_load_3d(tK.base + k * tK.block_bytes(), &mK, k * 64, tile * kL, head, bar(LD));
                tma_load_3d(tV.base + k * tV.block_bytes(), &mV, k * 64, tile * kL, head, bar(LD));
            }
            if (wait_bar(LD, 0)) {
                tc_fence_after();
                // group 1: B = K Q^T (whole tile); S and C of the first chunk,
                // S of the second (each over its own K-steps)
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tR0, tK.kmaj(ks), tQ.kmaj(ks), iSq, ks > 0);
                for (int ks = 0; ks < KS; ++ks) mma_bf16(tR1, tK.mnmaj(ks), tK.mnmaj(ks), iMM, ks > 0);
                for (int ks = 0; ks < KS; ++ks) mma_bf16(tR3, tQ.mnmaj(ks), tV.mnmaj(ks), iMM, ks > 0);
                if (CPT == 2)
                    for (int ks = 0; ks < KS; ++ks) mma_bf16(tR2, tK.mnmaj(KS + ks), tK.mnmaj(KS + ks), iMM, ks > 0);
                mma_commit(bar(C1));
                if (wait_bar(D1, 0)) {
                    tc_fence_after();
                    // group 2: C of the second chunk; Y = B_hi V + B_lo V (the
                    // masked B keeps every chunk's products to itself)
                    if (CPT == 2)
                        for (int ks = 0; ks < KS; ++ks) mma_bf16(tR1, tQ.mnmaj(KS + ks), tV.mnmaj(KS + ks), iMM, ks > 0);
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tR2, tBh.kmaj(ks), tV.mnmaj(ks), iKM, ks > 0);
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tR2, tBl.kmaj(ks), tV.mnmaj(ks), iKM, 1);
                    mma_commit(bar(C2));
                    if (wait_bar(D2, 0)) {
                        tc_fence_after();
                        // group 3: G = K^T (Y_hi + Y_lo) per chunk (Y tiles in
                        // place of B, rows = tokens, read MN-major)
                        for (int ks = 0; ks < KS; ++ks) mma_bf16(tR3, tK.mnmaj(ks), tBh.mnmaj(ks), iMM, ks > 0);
                        for (int ks = 0; ks < KS; ++ks) mma_bf16(tR3, tK.mnmaj(ks), tBl.mnmaj(ks), iMM, 1);
                        if (CPT == 2) {
                            for (int ks = 0; ks < KS; ++ks)
                                mma_bf16(tR0, tK.mnmaj(KS + ks), tBh.mnmaj(KS + ks), iMM, ks > 0);
                            for (int ks = 0; ks < KS; ++ks) mma_bf16(tR0, tK.mnmaj(KS + ks), tBl.mnmaj(KS + ks), iMM, 1);
                        }
                        mma_commit(bar(C3));
                    }
                }
            }
            if (!mma_wait_all(bar(FIN))) atomicExch(p.status, (int)kDevWaitTimeout);
            if (!loads.settle()) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else {
        // ========================== drain warps ==========================
        if (wait_bar(LD, 0) && wait_bar(C1, 0)) {
            tc_fence_after();
            // S (and C) of the first chunk and S of the second to the records
            // first: group 2 reuses their regions once B has been drained
            if (state_rows) {
                store_field(tR1, 0, ro.S);
                store_field(tR3, 0, ro.C);
                if (CPT == 2) store_field(tR2, 1, ro.S);
            }
            // B -> bf16 hi + lo (strictly lower, same chunk), fp32 row sums
            {
                uint32_t r[64];
                tmem_ld_cols<64>(tR0 + lane_off + c128, r);
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const int col = c128 + j;
                    const bool keep = col < row && (col / L) == (row / L);
                    if (!keep) r[j] = 0u;
                    s += __uint_as_float(r[j]);
                }
                rowsum[half][row] = s;
                put_row32_split2(tBh, tBl, row, c128, r, false);
                put_row32_split2(tBh, tBl, row, c128 + 32, r + 32, false);
            }
            drained(D1);
        }
        // m (per chunk, column sums of Q) and h = K^T rowsum(B), on CUDA cores
        // over the tile's rows while the tensor cores continue
        asm volatile("bar.sync 1, %0;" ::"r"(kDrainWarps * 32) : "memory");  // row sums complete
        for (int i = tid; i < CPT * D * 2; i += kDrainWarps * 32) {
            const int which = i / (CPT * D);  // 0: m, 1: h
            const int ch = (i / D) % CPT, a = i % D;
            const Tile& t = which == 0 ? tQ : tK;
            float s = 0.f;
            for (int r = ch * L; r < (ch + 1) * L; ++r) {
                unsigned short u;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(u) : "r"(t.chunk(r, a >> 6, (a & 63) >> 3) + (uint32_t)(a & 7) * 2u));
                const float x = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(&u));
                s = (which == 0) ? s + x : fmaf(x, rowsum[0][r] + rowsum[1][r], s);  // Q, K tiles loaded (LD)
            }
            if (chunk0 + ch < p.N) p.summ[((size_t)head * p.N + chunk0 + ch) * R + (which == 0 ? ro.m : ro.x) + a] = s;
        }
        if (wait_bar(C2, 0)) {
            tc_fence_after();
            // Y -> bf16 hi + lo in place of B (B V has completed)
            {
                uint32_t r[64];
                tmem_ld_cols<D / 2>(tR2 + lane_off + cD, r);
                put_row32_split2(tBh, tBl, row, cD, r, false);
                if (D == 128) put_row32_split2(tBh, tBl, row, cD + 32, r + 32, false);
            }
            drained(D2);
            if (state_rows && CPT == 2) store_field(tR1, 1, ro.C);
            if (wait_bar(C3, 0)) {
                tc_fence_after();
                if (state_rows) {
                    store_field(tR3, 0, ro.X);
                    if (CPT == 2) store_field(tR0, 1, ro.X);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

template <int D, int L>
cudaError_t launch_chunk_t(const void* Q, const void* K, const void* V, float* summ, int BH, int T, int N,
                           int* status, cudaStream_t s) {
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mk, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mv, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64))
        return cudaErrorInvalidValue;
    ChunkParams prm{T, N, summ, status};
    const size_t smem = ChunkLayout<D>::kBytes + 1024;
    auto kern = tc_chunk_kernel<D, L>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((T + kL - 1) / kL, BH);
    kern<<<grid, kThreadsTC, smem, s>>>(mq, mk, mv, prm);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool tc_chunk_supported(int d, int dv, int L, int dtype, int device) {
    return d == dv && (d == 64 || d == 128) && (L == 64 || L == 128) && tc_supported(d, dv, dtype, 0, device);
}

cudaError_t launch_tc_chunk(const void* Q, const void* K, const void* V, float* summ, int BH, int T, int d, int L,
                            int* status, cudaStream_t s) {
    if (BH == 0) return cudaSuccess;
    if ((long long)(T + kL - 1) / kL > 2147483647LL || BH > 65535) return cudaErrorInvalidValue;
    const int N = (T + L - 1) / L;
    if (d == 128) return L == 64 ? launch_chunk_t<128, 64>(Q, K, V, summ, BH, T, N, status, s)
                                 : launch_chunk_t<128, 128>(Q, K, V, summ, BH, T, N, status, s);
    if (d == 64) return L == 64 ? launch_chunk_t<64, 64>(Q, K, V, summ, BH, T, N, status, s)
                                : launch_chunk_t<64, 128>(Q, K, V, summ, BH, T, N, status, s);
    return cudaErrorInvalidValue;
}

}  // namespace hla2
