// hla2_tc_out.cu -- the output walk of the masked second-order HLA forward
// on GB300 tensor cores, pipelined across chunks.
//
// HLA summary (arXiv 2510.27258), section 1 "Second-order HLA" (o_t =
// q_t^T (S_t C_t - G_t)) and section 4 "Parallel training via associative
// scans" (each segment restarts from its exact prefix state).
//
// One CTA walks one segment of one head in chunks of L = 128 tokens from the
// segment's prefix state (S0, P0), P = S C - G.  For a chunk's Q, K, V:
//   A = tril(Q K^T)              (i <= t, diagonal kept)
//   X = Q S0 + A K               (row t is S_t q_t, so that P grows by X^T V)
//   W = tril(Q X^T)              (W_tj = q_t^T S_j q_j for j <= t)
//   O = Q P0 + W V               (the chunk's outputs, o_t = q_t^T P_t)
//   P0 += X^T V,  S0 += K^T K
// W = tril(Q X^T) equals tril(A A^T + (Q S0) Q^T) and takes one product
// instead of two.
//
// Tensor memory holds two working regions besides the running S and P:
//   alpha: A, then W            beta: X (= Q S0 + A K), then O
// so that the next chunk's A = Q K^T can start in alpha as soon as W has been
// drained, while O of the current chunk is still being formed and drained in
// beta; Q is double-buffered for the same reason, and each chunk's V starts
// loading as soon as the previous O has completed.  In shared memory the bf16
// A and then W share one tile, X another (O leaves through both); the bf16
// operand copies of S0 and P0 share a third: S0 is read by Q S0 early in a
// chunk, P0 by Q P0 late in it.
//
// Precision: products take bf16 operands with fp32 accumulation; the running
// S and P stay fp32 in tensor memory.  On a head's first chunk, where an
// output can be a single product (t = 0 gives (q.k)^2 v) and roundings do not
// average out, X and W are split into bf16 hi + lo parts (W = Q X_hi^T +
// Q X_lo^T, O = W_hi V + W_lo V).
#include "hla2_tc_common.cuh"

namespace hla2 {
namespace {

struct OutParams {
    int T, nseg, nchunk, seglen;
    const float* prefix;  // segment prefix records (S and P read)
    int* status;
};

template <int D>
struct OutLayout {
    static constexpr uint32_t kTok = kL * D * 2;  // Q, K, V tiles
    static constexpr uint32_t kSq = kL * kL * 2;  // A / W tile; X tile (O staging)
    static constexpr uint32_t kSt = D * D * 2;    // S0 / P0 tile
    static constexpr uint32_t Q0 = 0, Q1 = kTok, K = 2 * kTok, V = 3 * kTok, A = 4 * kTok, X = A + kSq, SP = X + kSq;
    static constexpr uint32_t kBytes = SP + kSt;
};

// Warp roles as in the other walks: warps 0..7 drain tensor memory (warp w
// owns lane quarter w % 4 and column half w / 4 of every region), warp 8
// (lane 0) issues every TMA copy and MMA; they meet only on mbarriers.
template <int D>
__global__ void __launch_bounds__(kThreadsTC, 1)
tc_out_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
              const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mO,
              const __grid_constant__ CUtensorMap mR, OutParams p) {
    using LY = OutLayout<D>;
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    // loads | MMA commits | drains | final wait | drain warp w's prefix boxes
    enum { LQ0, LQ1, LK, LV, CA, CQS, CX, CW, CP, CO, DA, DP, DX, DW, DO, DS, FIN, PB, NBAR = PB + kDrainWarps };
    __shared__ __align__(8) unsigned long long bars[NBAR];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const bool issuer = warp == kDrainWarps;
    const int quarter = warp & 3;
    const int half = (warp >> 2) & 1;
    const int row = quarter * 32 + lane;  // TMEM lane / tile row owned by a drain thread
    int head, seg;
    const SegPlan plan{kL, p.nchunk, p.nseg, p.seglen};
    block_segment(plan, gridDim.y, (long long)blockIdx.y * gridDim.x + blockIdx.x, head, seg);
    const int c_begin = seg_chunk_begin(plan, seg);
    const int c_end = seg_chunk_begin(plan, seg + 1);
    const int nchunks = c_end - c_begin;
    const bool state_rows = !issuer && ((D == 128) || quarter < D / 32);  // drain warp holding rows < D
    constexpr int kStateWarps = (D == 128) ? kDrainWarps : 2 * (D / 32);

    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tQ0{dsm + LY::Q0, kL}, tQ1{dsm + LY::Q1, kL}, tK{dsm + LY::K, kL}, tV{dsm + LY::V, kL};
    const Tile tA{dsm + LY::A, kL}, tX{dsm + LY::X, kL}, tSP{dsm + LY::SP, D};
    auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == DA || i == DX || i == DW || i == DO) cnt = kDrainWarps;
            if (i == DS || i == DP) cnt = kStateWarps;
            mbar_init(bar(i), cnt);
        }
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
    const uint32_t tAl_ = tmem + 0;           // alpha: A, then W (and W_lo on a head's first chunk)
    const uint32_t tBe_ = tmem + 128;         // beta: Q S0 + A K = X, then O
    const uint32_t tS_ = tmem + 128 + D;      // running S
    const uint32_t tP_ = tmem + 128 + 2 * D;  // running P
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int c128 = half * 64;     // this drain warp's columns in a 128-wide region
    const int cD = half * (D / 2);  // ... and in a D-wide region

    constexpr uint32_t kTileBytes = kL * D * 2;
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
    auto issue_load = [&](int b, const CUtensorMap* map, const Tile& t, int chunk) {
        mbar_expect_tx(bar(b), kTileBytes);
#pragma unroll
        for (int k = 0; k < D / 64; ++k) tma_load_3d(t.base + k * t.block_bytes(), map, k * 64, chunk * kL, head, bar(b));
    };
    // a drain warp announces that its share of a region is done
    auto drained = [&](int b) {
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(b)) : "memory");
    };
    auto drain128 = [&](uint32_t treg, const Tile& t, bool mask) {
        uint32_t r[64];
        tmem_ld_cols<64>(treg + lane_off + c128, r);
        put_row32(t, row, c128, r, mask);
        put_row32(t, row, c128 + 32, r + 32, mask);
    };
    auto drainD = [&](uint32_t treg, const Tile& t) {
        uint32_t r[64];
        tmem_ld_cols<D / 2>(treg + lane_off + cD, r);
        put_row32(t, row, cD, r, false);
        if (D == 128) put_row32(t, row, cD + 32, r + 32, false);
    };
    // packed W_lo: drain warp h stores the bf16 pairs of its W columns
    // [64h, 64h+64) into the first 32 of those columns, which it has itself
    // just read, so no other warp's pending read is overwritten.  K-step ks
    // of W_lo V reads 8 packed columns.
    auto wlo_col = [](int ks) -> uint32_t { return (uint32_t)((ks >> 2) * 64 + 8 * (ks & 3)); };

    // ---- prologue: the first tiles start moving while the drain warps load
    // the segment prefix (S0, P0) into tensor memory and S0 into its tile ----
    if (issuer && lane == 0 && nchunks > 0) {
        issue_load(LQ0, &mQ, tQ0, c_begin);
        issue_load(LK, &mK, tK, c_begin);
        issue_load(LV, &mV, tV, c_begin);
        if (nchunks > 1) issue_load(LQ1, &mQ, tQ1, c_begin + 1);
    }
    if (state_rows && nchunks > 0) {
        // S0 (record row 0) and P0 (record row 2D + 1) arrive as this warp's
        // 32 x 32 fp32 boxes by bulk tensor loads (mR maps the records as
        // (3D + 2) rows of D floats) into a private staging area in the A / X
        // tiles, which nothing else touches before the first chunk
        const int rec = head * p.nseg + seg;
        const uint32_t stage = dsm + LY::A + (uint32_t)warp * (uint32_t)(D / 64) * 4096u;
#pragma unroll 1
        for (int m = 0; m < 2; ++m) {
            if (lane == 0) {
                fence_proxy_async();
                mbar_expect_tx(bar(PB + warp), (uint32_t)(D / 64) * 4096u);
#pragma unroll
                for (int g = 0; g < D / 64; ++g)
                    tma_load_3d(stage + (uint32_t)g * 4096u, &mR, cD + 32 * g, (m == 0 ? 0 : 2 * D + 1) + quarter * 32, rec,
                                bar(PB + warp));
            }
            __syncwarp();
            if (!wait_bar(PB + warp, (uint32_t)m)) break;
#pragma unroll
            for (int g = 0; g < D / 64; ++g) {
                const int cb = cD + 32 * g;
                uint32_t r[32];
                box32_read(stage + (uint32_t)g * 4096u, lane, r);
                tmem_st32((m == 0 ? tS_ : tP_) + lane_off + cb, r);
                if (m == 0) put_row32(tSP, row, cb, r, false);  // bf16 S0; P0 follows once Q S0 has read it
            }
            __syncwarp();  // every lane has read the boxes before the next load reuses them
        }
        tmem_st_wait();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    constexpr uint32_t iSq = idesc_bf16(128, 128, false, false);  // 128 x 128, both K-major
    constexpr uint32_t iSD = idesc_bf16(128, 128, false, false);  // W = Q X^T: N = 128 tokens
    constexpr uint32_t iKK = idesc_bf16(128, D, false, false);    // N = D, both K-major
    constexpr uint32_t iKM = idesc_bf16(128, D, false, true);     // A K-major, B MN-major
    constexpr uint32_t iMM = idesc_bf16(128, D, true, true);      // both MN-major

    if (issuer) {
        // ============================ issuer ============================
        if (lane == 0 && nchunks > 0) {
            for (int it = 0; it < nchunks; ++it) {
                const int c = c_begin + it;
                const uint32_t ph = it & 1, pph = (it + 1) & 1;
                const bool has_next = it + 1 < nchunks;
                const bool first = c == 0;            // S0 = P0 = 0; X, W split
                const bool prev_first = it > 0 && c == 1;
                const Tile& tQ = (it & 1) ? tQ1 : tQ0;
                if (!wait_bar((it & 1) ? LQ1 : LQ0, (uint32_t)((it >> 1) & 1)) || !wait_bar(LK, ph)) break;
                // alpha is free once the previous W was drained (and, after a
                // head's first chunk, once O has read W_lo from it)
                if (it > 0 && !wait_bar(prev_first ? DO : DW, pph)) break;
                tc_fence_after();
                // A = Q K^T
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tAl_, tQ.kmaj(ks), tK.kmaj(ks), iSq, ks > 0);
                mma_commit(bar(CA));
                if (it > 0) {
                    // the previous O complete: the V tile and the other Q buffer
                    // are no longer read, so this chunk's V and the next Q start
                    // moving; then beta free (O read out) and S0 in its tile
                    if (!wait_bar(CO, pph)) break;
                    issue_load(LV, &mV, tV, c);
                    if (has_next) issue_load((it + 1) & 1 ? LQ1 : LQ0, &mQ, (it + 1) & 1 ? tQ1 : tQ0, c + 1);
                    if (!wait_bar(DO, pph) || !wait_bar(DS, pph)) break;
                    tc_fence_after();
                }
                // X = Q S0 (S0 symmetric: its tile read K-major), then S += K^T K
                if (!first)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tBe_, tQ.kmaj(ks), tSP.kmaj(ks), iKK, ks > 0);
                mma_commit(bar(CQS));
                for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tS_, tK.mnmaj(ks), tK.mnmaj(ks), iMM, 1);
                if (!wait_bar(DA, ph)) break;  // sA = A
                tc_fence_after();
                // X += A K
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tBe_, tA.kmaj(ks), tK.mnmaj(ks), iKM, (!first || ks > 0) ? 1u : 0u);
                mma_commit(bar(CX));
                if (has_next) {
                    if (!wait_bar(CX, ph)) break;
                    issue_load(LK, &mK, tK, c + 1);  // K was last read by A K
                }
                if (!wait_bar(DX, ph)) break;  // sX = X (and X_lo in sA on a head's first chunk); beta free
                tc_fence_after();
                // W = Q X^T (+ Q X_lo^T)
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tAl_, tQ.kmaj(ks), tX.kmaj(ks), iSD, ks > 0);
                if (first)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tAl_, tQ.kmaj(ks), tA.kmaj(ks), iSD, 1);
                mma_commit(bar(CW));
                // P += X^T V once P0 of this chunk has left TMEM P
                if (!wait_bar(LV, ph) || !wait_bar(DP, ph)) break;
                tc_fence_after();
                for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tP_, tX.mnmaj(ks), tV.mnmaj(ks), iMM, 1);
                mma_commit(bar(CP));
                if (!wait_bar(DW, ph)) break;  // sA = W (hi; W_lo packed in alpha on a first chunk)
                tc_fence_after();
                // O = Q P0 + W V (+ W_lo V)
                if (!first)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tBe_, tQ.kmaj(ks), tSP.mnmaj(ks), iKM, ks > 0);
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tBe_, tA.kmaj(ks), tV.mnmaj(ks), iKM, (!first || ks > 0) ? 1u : 0u);
                if (first)
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16_tmem_a(tBe_, tAl_ + wlo_col(ks), tV.mnmaj(ks), iKM, 1);
                mma_commit(bar(CO));
            }
            if (!mma_wait_all(bar(FIN))) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else {
        // ========================== drain warps ==========================
        for (int it = 0; it < nchunks; ++it) {
            const uint32_t ph = it & 1;
            const int c = c_begin + it;
            const bool has_next = it + 1 < nchunks;
            const bool first = c == 0;
            // A -> sA (masked).  sA last held W of the previous chunk (read by
            // its O, complete) and then one of its O boxes: wait until the
            // bulk stores have read both O pieces out of sA and sX.
            if (!wait_bar(CA, ph)) break;
            tc_fence_after();
            if (lane == 0) tma_store_wait_read();
            __syncwarp();
            drain128(tAl_, tA, true);
            drained(DA);
            // P0 of this chunk -> the S0 / P0 tile, once Q S0 has read S0 (a
            // head's first chunk has P0 = 0 and skips Q P0)
            if (!wait_bar(CQS, ph)) break;
            tc_fence_after();
            if (state_rows) {
                if (!first) drainD(tP_, tSP);
                drained(DP);
            }
            // X -> sX (bf16; the previous O boxes left it before the A drain);
            // on a head's first chunk split into hi (sX) and lo (sA: A has been
            // read by A K, and W goes there only once W has read X_lo)
            if (!wait_bar(CX, ph)) break;
            tc_fence_after();
            {
                uint32_t x[64];
                tmem_ld_cols<D / 2>(tBe_ + lane_off + cD, x);
                if (first) {
                    put_row32_split2(tX, tA, row, cD, x, false);
                    if (D == 128) put_row32_split2(tX, tA, row, cD + 32, x + 32, false);
                } else {
                    put_row32(tX, row, cD, x, false);
                    if (D == 128) put_row32(tX, row, cD + 32, x + 32, false);
                }
            }
            drained(DX);
            // W -> sA (masked): A there was last read by A K, complete
            if (!wait_bar(CW, ph)) break;
            tc_fence_after();
            if (first) {
                uint32_t lo[32];
                {
                    uint32_t r[64];
                    tmem_ld_cols<64>(tAl_ + lane_off + c128, r);
                    put_row32_split(tA, row, c128, r, true, lo);  // W_hi -> sA (masked)
                    put_row32_split(tA, row, c128 + 32, r + 32, true, lo + 16);
                }
                tmem_st32(tAl_ + lane_off + (uint32_t)c128, lo);  // W_lo -> alpha (own columns, packed)
                tmem_st_wait();
            } else {
                drain128(tAl_, tA, true);
            }
            drained(DW);
            // O: out of beta into registers (beta then free), the next chunk's
            // S0 into its tile (Q P0 has read P0), then O leaves by bulk tensor
            // stores, staged in sX (X was last read by X^T V) and, at D = 128,
            // sA (W was last read by O), one 4 KB box per warp in each
            if (!wait_bar(CO, ph)) break;
            tc_fence_after();
            {
                uint32_t r[64];
                tmem_ld_cols<D / 2>(tBe_ + lane_off + cD, r);
                drained(DO);
                if (state_rows && has_next) {
                    drainD(tS_, tSP);
                    drained(DS);
                }
                const uint32_t wbox = (uint32_t)half * (kL * 128u) + (uint32_t)(quarter * 32) * 128u;
                const int t0 = c * kL + quarter * 32;  // first token of this warp's rows
#pragma unroll
                for (int g = 0; g < D / 64; ++g) {
                    const uint32_t scratch = (g == 0 ? tX.base : tA.base) + wbox;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st_shared_v4(scratch + (uint32_t)lane * 128u + (uint32_t)((q ^ (lane & 7)) << 4),
                                     r[32 * g + 4 * q], r[32 * g + 4 * q + 1], r[32 * g + 4 * q + 2],
                                     r[32 * g + 4 * q + 3]);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&mO, scratch, cD + 32 * g, t0, head);
                        tma_store_commit();
                    }
                }
            }
        }
        if (lane == 0) tma_store_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

template <int D>
cudaError_t launch_out_t(const void* Q, const void* K, const void* V, float* O, const float* prefix, int BH, int T,
                         SegPlan plan, int* status, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mo, mr;
    if (!make_map(&mq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mk, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mv, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64))
        return cudaErrorInvalidValue;
    // mR: the segment prefix records as (3D + 2) rows of D floats, 32 x 32 boxes
    if (!make_map(&mr, prefix, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, 3 * D + 2, BH * plan.nseg, 32, 32))
        return cudaErrorInvalidValue;
    // O: fp32 boxes of 32 rows x 32 columns (one drain warp's piece)
    if (!make_map(&mo, O, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, T, BH, 32, 32)) return cudaErrorInvalidValue;
    OutParams prm{T, plan.nseg, plan.nchunk, plan.seglen, prefix, status};
    const size_t smem = OutLayout<D>::kBytes + 1024;
    auto kern = tc_out_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.nseg, BH);
    kern<<<grid, kThreadsTC, smem, s>>>(mq, mk, mv, mo, mr, prm);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_out(const void* Q, const void* K, const void* V, float* O, const float* prefix, int BH, int T,
                          int d, int dv, SegPlan plan, int* status, cudaStream_t s) {
    if (BH == 0 || plan.nseg == 0) return cudaSuccess;
    if (plan.granule != kL || d != dv) return cudaErrorInvalidValue;
    if (d == 128) return launch_out_t<128>(Q, K, V, O, prefix, BH, T, plan, status, s);
    if (d == 64) return launch_out_t<64>(Q, K, V, O, prefix, BH, T, plan, status, s);
    return cudaErrorInvalidValue;
}

}  // namespace hla2
