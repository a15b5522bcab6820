// hla2_decay_tc.cu -- tensor-core segment summary walk of the exponentially
// decayed masked operator on GB300 (sm_103a): tcgen05.mma with TMEM
// accumulators, TMA tiles.  The outputs run on the pipelined output walk
// (hla2_tc_out.cu) with the chunk form below.
//
// Operator (HLA summary, arXiv 2510.27258, section 4 names decayed operators
// among those the scan covers): every prefix moment decays by gamma per token,
//   S_t = g S + k k^T,   P_t = g^2 P + S_t q_t v_t^T,   o_t = q_t^T P_t,
// i.e. o_t = sum_{i<=j<=t} g^{2t-i-j} (q_t.k_i)(k_i.q_j) v_j (P = S C - G).
//
// Chunk form.  For a chunk of L tokens (local index t, 128 rows, L real) with
// the state (S0, P0) at its start, a_t = g^{t+1}, b_t = g^{L-1-t}:
//   X^g_t = a_t S0 q_t + sum_{i<=t} g^{t-i} (q_t.k_i) k_i      (= S_t q_t)
//   o_t   = a_t^2 q_t^T P0 + sum_{j<=t} g^{2(t-j)} (q_t.X^g_j) v_j
//   S'    = g^L S0 + K^T diag(b) K,   P' = g^{2L} P0 + X^g^T diag(b^2) V.
// Every per-token factor is moved into an operand that is rounded to bf16
// anyway, or into a factor common to a whole accumulator row, so that Q, K, V
// enter the products exactly:
//   A~  = tril(Q K^T) * g^{-(i+1)}            (column factor)
//   X'  = Q S0 + A~ K                          (= X^g_t / a_t)
//   sX  = g^{2L-1-t} X'_t                      (= b_t^2 X^g_t: the P update's operand)
//   W~  = g^{-2L} tril(Q sX^T)                 (constant factor)
//   O'  = Q P0 + W~ V,  o_t = g^{2(t+1)} O'_t  (row factor)
//   S  += K'^T K' with K' = diag(sqrt(b)) K (K scaled in place once its
//         other products are done), after TMEM S was scaled by g^L (P by g^{2L}).
// The negative powers stay within g^{-2L}; with g >= 0.8 every intermediate is
// a finite fp32 / bf16 number (products too small to represent only drop terms
// that are negligible against the output).  W~ is split into bf16 hi + lo on
// every chunk (the lo part packed in tensor memory), and on a head's first
// chunk A~ and sX are split as well.
//
// Summary walk (mode 0): per segment S (running), and C, P accumulated in the
// frame of the segment's last token: chunk c contributes with the factor
// F_c = g^{(tokens of the segment after chunk c)}, C += (diag(F_c b) Q)^T V,
// P += (F_c^2 b^2 X^g)^T V, so neither needs rescaling from chunk to chunk.
//
// Roles as in the other walks: warp 8 (lane 0) issues every copy and MMA,
// warps 0..7 drain tensor memory; they meet only on mbarriers, every wait
// bounded in time.
#include <cmath>

#include "hla2_tc_common.cuh"

namespace hla2 {
namespace {

struct DParams {
    int T, nseg, nchunk, seglen;
    float lg;  // log2(gamma)
    int* status;
};

__device__ __forceinline__ float gpow(float lg, float n) { return exp2f(n * lg); }
__device__ __forceinline__ int chunk_len(int T, int c) { return min(kL, T - c * kL); }

// 32 fp32 values (columns col0.., row r, scaled in place) times a column
// factor cf[col] (and a scalar s), optionally masked to columns <= r, written
// as bf16 (hi) to `hi` and, when split is set, the rounding remainder to `lo`.
__device__ __forceinline__ void put_row32_cf(const Tile& hi, const Tile& lo, bool split, int r, int col0, uint32_t* v,
                                             const float* cf, float s, bool mask) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        float f = __uint_as_float(v[j]) * (cf ? cf[col0 + j] : 1.f) * s;
        if (mask && col0 + j > r) f = 0.f;
        v[j] = __float_as_uint(f);
    }
    if (split) put_row32_split2(hi, lo, r, col0, v, false);
    else put_row32(hi, r, col0, v, false);
}

// Row r, columns [col0, col0 + 8n) of bf16 tile `src`, times s, to the same
// place of tile `dst` (same geometry).
template <int N8>
__device__ __forceinline__ void scale_row(const Tile& src, const Tile& dst, int r, int col0, float s) {
#pragma unroll
    for (int q = 0; q < N8; ++q) {
        const int col = col0 + 8 * q;
        const uint32_t a = src.chunk(r, col >> 6, (col & 63) >> 3);
        uint32_t w[4];
        ld_shared_v4(a, w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&w[h]);
            w[h] = pack_bf16(__low2float(p) * s, __high2float(p) * s);
        }
        st_shared_v4(dst.chunk(r, col >> 6, (col & 63) >> 3), w[0], w[1], w[2], w[3]);
    }
}

// ----------------------------------------------------------- summaries ----
// Q is double-buffered (chunk it uses buffer it & 1); once a chunk's A and X'
// products have completed, the drains scale its K tile in place by sqrt(b)
// (for S += K'^T K') and its Q tile by F_c b (for C += Q'^T V), so the segment
// sums need no staged copies and V enters unscaled.
template <int D>
struct DSumLayout {
    static constexpr uint32_t kTok = kL * D * 2;
    static constexpr uint32_t kSq = kL * kL * 2;
    static constexpr uint32_t kSt = D * D * 2;
    static constexpr uint32_t Q = 0, Q2 = Q + kTok, K = Q2 + kTok, V = K + kTok, A = V + kTok, X = A + kSq;
    static constexpr uint32_t S = X + kTok;
    static constexpr uint32_t kEnd = S + kSt;
    static constexpr uint32_t kPad = (D < 128) ? 16384u : 0u;
    static constexpr uint32_t kBytes = kEnd + kPad;
    static_assert(kEnd >= 8u * 3u * (D / 64) * 4096u || D < 128, "record staging must fit the tiles");
};

template <int D>
__global__ void __launch_bounds__(kThreadsTC + 32, 1)
decay_tc_sum_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mR, DParams p) {
    using LY = DSumLayout<D>;
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    enum { LQ, LQ2, LK, LV, CA, CX, CS, CC, CP, DA, DX, DK, DQ, DS, FIN, NBAR };
    __shared__ __align__(8) unsigned long long bars[NBAR];
    __shared__ float colf[kL];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issuer = warp == kDrainWarps;
    const bool producer = warp == kDrainWarps + 1;  // issues every tile load
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int row = quarter * 32 + lane;
    int head, seg;
    const SegPlan plan{kL, p.nchunk, p.nseg, p.seglen};
    block_segment(plan, gridDim.y, (long long)blockIdx.y * gridDim.x + blockIdx.x, head, seg);
    const int c_begin = seg_chunk_begin(plan, seg), c_end = seg_chunk_begin(plan, seg + 1);
    const int nchunks = c_end - c_begin;
    const bool state_rows = warp < kDrainWarps && ((D == 128) || quarter < D / 32);
    constexpr int kStateWarps = (D == 128) ? kDrainWarps : 2 * (D / 32);
    const float lg = p.lg;
    const int seg_end_tok = min(p.T, c_end * kL);

    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tQa{dsm + LY::Q, kL}, tQb{dsm + LY::Q2, kL}, tK{dsm + LY::K, kL}, tV{dsm + LY::V, kL};
    const Tile tA{dsm + LY::A, kL}, tX{dsm + LY::X, kL}, tS{dsm + LY::S, D};
    auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };

    if (tid < kL) colf[tid] = gpow(lg, -(float)(tid + 1));
    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == DA || i == DX || i == DK || i == DQ) cnt = kDrainWarps;
            if (i == DS) cnt = kStateWarps;
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
    // tensor memory: A~, then X' | S (running) | C, P (segment-end frame)
    const uint32_t tA_ = tmem + 0, tS_ = tmem + 128, tC_ = tmem + 128 + D, tP_ = tmem + 128 + 2 * D;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int c128 = half * 64;
    const int cD = half * (D / 2);

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
    // every tile load is issued by the issuer's lane 0, which settles them
    // (waits for the last of each barrier) before the CTA exits
    LoadLedger<4> loads(bar(0));  // LQ, LQ2, LK, LV
    auto issue_load = [&](int b, const CUtensorMap* map, const Tile& t, int chunk) {
        loads.note(b);
        mbar_expect_tx(bar(b), kTileBytes);
#pragma unroll
        for (int k = 0; k < D / 64; ++k) tma_load_3d(t.base + k * t.block_bytes(), map, k * 64, chunk * kL, head, bar(b));
    };
    auto drained = [&](int b) {
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(b)) : "memory");
    };

    constexpr uint32_t iSq = idesc_bf16(128, 128, false, false);
    constexpr uint32_t iKK = idesc_bf16(128, D, false, false);
    constexpr uint32_t iKM = idesc_bf16(128, D, false, true);
    constexpr uint32_t iMM = idesc_bf16(128, D, true, true);

    if (producer && lane == 0 && nchunks > 0) {
        issue_load(LQ, &mQ, tQa, c_begin);
        issue_load(LK, &mK, tK, c_begin);
        issue_load(LV, &mV, tV, c_begin);
        if (nchunks > 1) issue_load(LQ2, &mQ, tQb, c_begin + 1);
    }
    if (issuer) {
        if (lane == 0 && nchunks > 0) {
            for (int it = 0; it < nchunks; ++it) {
                const uint32_t ph = it & 1, pph = (it + 1) & 1;
                const bool qodd = it & 1;  // Q buffer of this chunk
                const Tile& tQ = qodd ? tQb : tQa;
                if (!wait_bar(qodd ? LQ2 : LQ, (uint32_t)((it >> 1) & 1)) || !wait_bar(LK, ph)) break;
                if (it > 0 && !wait_bar(DX, pph)) break;  // TMEM A (X' of the previous chunk) read
                tc_fence_after();
                // A = Q K^T
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQ.kmaj(ks), tK.kmaj(ks), iSq, ks > 0);
                mma_commit(bar(CA));
                if (it > 0 && !wait_bar(DS, pph)) break;  // sS = S0; TMEM S decayed
                if (!wait_bar(DA, ph)) break;              // sA = A~
                tc_fence_after();
                // X' = Q S0 + A~ K   (S0 = 0 on the segment's first chunk)
                if (it > 0)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQ.kmaj(ks), tS.kmaj(ks), iKK, ks > 0);
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tA_, tA.kmaj(ks), tK.mnmaj(ks), iKM, (it > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bar(CX));
                // S += K'^T K' (K' = diag(sqrt(b)) K, scaled in place by the drains)
                if (!wait_bar(DK, ph)) break;
                tc_fence_after();
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tS_, tK.mnmaj(ks), tK.mnmaj(ks), iMM, (it > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bar(CS));
                // C += Q'^T V (Q' = diag(F b) Q, scaled in place by the drains)
                if (!wait_bar(DQ, ph) || !wait_bar(LV, ph)) break;
                tc_fence_after();
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tC_, tQ.mnmaj(ks), tV.mnmaj(ks), iMM, (it > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bar(CC));
                if (!wait_bar(DX, ph)) break;  // sX = F^2 g^{2L-1-t} X'
                tc_fence_after();
                // P += sX^T V
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tP_, tX.mnmaj(ks), tV.mnmaj(ks), iMM, (it > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bar(CP));
            }
            // FIN completes once every product has: the records can be read out
            if (!mma_wait_all(bar(FIN))) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else if (producer) {
        // the next tiles once their last reader completed: K after the S
        // update, the Q after next into this chunk's buffer after C (Q' read),
        // V after the P update
        if (lane == 0) {
            for (int it = 0; it + 1 < nchunks; ++it) {
                const int c = c_begin + it;
                const uint32_t ph = it & 1;
                if (!wait_bar(CS, ph)) break;
                issue_load(LK, &mK, tK, c + 1);
                if (it + 2 < nchunks) {
                    if (!wait_bar(CC, ph)) break;
                    issue_load((it & 1) ? LQ2 : LQ, &mQ, (it & 1) ? tQb : tQa, c + 2);
                }
                if (!wait_bar(CP, ph)) break;
                issue_load(LV, &mV, tV, c + 1);
            }
            if (!loads.settle()) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else if (nchunks > 0) {
        // ========================== drain warps ==========================
        for (int it = 0; it < nchunks; ++it) {
            const int c = c_begin + it;
            const uint32_t ph = it & 1, pph = (it + 1) & 1;
            const bool has_next = it + 1 < nchunks;
            const Tile& tQ = (it & 1) ? tQb : tQa;
            const float L = (float)chunk_len(p.T, c);
            const float F = gpow(lg, (float)(seg_end_tok - min(p.T, (c + 1) * kL)));
            if (!wait_bar(CA, ph)) break;
            tc_fence_after();
            {
                uint32_t r[64];
                tmem_ld_cols<64>(tA_ + lane_off + c128, r);
                put_row32_cf(tA, tA, false, row, c128, r, colf, 1.f, true);
                put_row32_cf(tA, tA, false, row, c128 + 32, r + 32, colf, 1.f, true);
            }
            drained(DA);
            if (!wait_bar(CX, ph)) break;  // A and X' have read Q and K
            tc_fence_after();
            // K' = diag(sqrt(b)) K in place (row = token; b = g^{L-1-t})
            scale_row<D / 16>(tK, tK, row, cD, gpow(lg, 0.5f * (L - 1.f - (float)row)));
            drained(DK);
            if (it > 0 && !wait_bar(CP, pph)) break;  // the previous P update has read sX
            tc_fence_after();
            {
                // sX = F^2 g^{2L-1-t} X'
                uint32_t r[64];
                tmem_ld_cols<D / 2>(tA_ + lane_off + cD, r);
                const float xs = F * F * gpow(lg, 2.f * L - 1.f - (float)row);
                put_row32_cf(tX, tX, false, row, cD, r, nullptr, xs, false);
                if (D == 128) put_row32_cf(tX, tX, false, row, cD + 32, r + 32, nullptr, xs, false);
            }
            drained(DX);
            // Q' = diag(F b) Q in place
            scale_row<D / 16>(tQ, tQ, row, cD, F * gpow(lg, L - 1.f - (float)row));
            drained(DQ);
            if (state_rows && has_next) {
                if (!wait_bar(CS, ph)) break;
                tc_fence_after();
                // S0 of the next chunk -> sS; TMEM S decayed over the next chunk
                uint32_t r[64];
                tmem_ld_cols<D / 2>(tS_ + lane_off + cD, r);
                put_row32(tS, row, cD, r, false);
                if (D == 128) put_row32(tS, row, cD + 32, r + 32, false);
                const float decay = gpow(lg, (float)chunk_len(p.T, c + 1));
#pragma unroll
                for (int j = 0; j < D / 2; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * decay);
                tmem_st32(tS_ + lane_off + cD, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                if (D == 128) tmem_st32(tS_ + lane_off + cD + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                tmem_st_wait();
                drained(DS);
            }
        }
        // records S (row 0), C (row D), P (row 2D+1) through the dead tiles once
        // every product has completed
        if (state_rows && !abort_flag && wait_bar(FIN, 0)) {
            tc_fence_after();
            const uint32_t src[3] = {tS_, tC_, tP_};
            const int rows0[3] = {0, D, 2 * D + 1};
            const uint32_t scratch = dsm + (uint32_t)warp * (3u * (D / 64) * 4096u);
            const int rec = head * p.nseg + seg;
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                uint32_t r[64];
                tmem_ld_cols<D / 2>(src[m] + lane_off + cD, r);
#pragma unroll
                for (int g = 0; g < D / 64; ++g)
                    box32_store(&mR, scratch + (uint32_t)(m * (D / 64) + g) * 4096u, r + 32 * g, lane, cD + 32 * g,
                                rows0[m] + quarter * 32, rec);
            }
            if (lane == 0) tma_store_wait_all();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

template <int D>
cudaError_t launch_d(const void* Q, const void* K, const void* V, float* summ, int BH, int T, float gamma,
                     SegPlan plan, int* status, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mr;
    if (!make_map(&mq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mk, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mv, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64))
        return cudaErrorInvalidValue;
    if (!make_map(&mr, summ, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, 3 * D + 2, BH * plan.nseg, 32, 32))
        return cudaErrorInvalidValue;
    DParams prm{T, plan.nseg, plan.nchunk, plan.seglen, (float)std::log2((double)gamma), status};
    dim3 grid(plan.nseg, BH);
    const size_t smem = DSumLayout<D>::kBytes + 1024;
    auto kern = decay_tc_sum_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreadsTC + 32, smem, s>>>(mq, mk, mv, mr, prm);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool decay_tc_gamma_ok(float gamma) { return gamma >= kDecayTcMinGamma && gamma <= 1.f; }

cudaError_t launch_decay_tc_walk(int mode, const void* Q, const void* K, const void* V, float* O, const float* prefix,
                                 float* summ, int BH, int T, int d, int dv, float gamma, SegPlan plan, int* status,
                                 cudaStream_t s) {
    if (BH == 0 || plan.nseg == 0) return cudaSuccess;
    if (plan.granule != kL || d != dv || !decay_tc_gamma_ok(gamma)) return cudaErrorInvalidValue;
    // outputs: the walk pipelined across chunks (hla2_tc_out.cu)
    if (mode == 1)
        return launch_tc_out_decay(Q, K, V, O, prefix, BH, T, d, dv, (float)std::log2((double)gamma), plan, status, s);
    if (mode != 0) return cudaErrorInvalidValue;
    if (d == 128) return launch_d<128>(Q, K, V, summ, BH, T, gamma, plan, status, s);
    if (d == 64) return launch_d<64>(Q, K, V, summ, BH, T, gamma, plan, status, s);
    return cudaErrorInvalidValue;
}

}  // namespace hla2
