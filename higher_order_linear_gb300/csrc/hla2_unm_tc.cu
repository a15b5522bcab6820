// hla2_unm_tc.cu -- tensor-core segment walks of the unmasked second-order
// operator on GB300 (sm_103a): tcgen05.mma with TMEM accumulators, TMA tiles.
//
// HLA summary (arXiv 2510.27258), section 1: S_t C_t is the naive product
// whose "future" terms G_t removes; "Results and claims" lists the unmasked
// operator o_t = q_t^T S_t C_t = sum_{i<=t, j<=t} (q_t.k_i)(k_i.q_j) v_j.
// Its state (S, C) adds across segments (section 4's combine without a cross
// term), so the scan is a running sum.
//
// Summary walk (mode 0): per segment S = sum K^T K and C = sum Q^T V, two
// MMA groups per 128-token chunk with double-buffered Q, K, V tiles and no
// drain until the end.
//
// Output walk (mode 1), per chunk with the state (S0, C0) entering it:
//   A = tril(Q K^T)            (i <= t, diagonal kept)
//   X = Q S0 + A K             (row t is S_t q_t)
//   W = tril(X Q^T)            (j <= t)
//   O = X C0 + W V
//   S0 += K^T K,  C0 += Q^T V
// bf16 operands in shared memory, fp32 accumulators in tensor memory.  On a
// head's first chunk (where an output can be a single product) A, X and W are
// split into bf16 hi + lo parts and the lo parts enter the products too; that
// chunk has S0 = C0 = 0, so at d = 128 the S0 and C0 tiles hold the lo parts
// (the next chunk's S0 and C0 are written once that chunk's products are done).
//
// Roles as in the other walks: warp 8 (lane 0) issues every copy and MMA,
// warps 0..7 drain tensor memory (warp w: lane quarter w % 4, column half
// w / 4); they meet only on mbarriers, every wait bounded in time.
#include "hla2_tc_common.cuh"

namespace hla2 {
namespace {

struct UParams {
    int T, nseg, nchunk, seglen;
    int* status;
};

// ------------------------------------------------------------ summaries ----
template <int D>
struct USumLayout {
    static constexpr uint32_t kTok = kL * D * 2;  // Q, K or V tile
    static constexpr uint32_t kBuf = 3 * kTok;    // one chunk's Q | K | V
    static constexpr uint32_t kPad = (D < 128) ? 16384u : 0u;
    static constexpr uint32_t kBytes = 2 * kBuf + kPad;
};

template <int D>
__global__ void __launch_bounds__(kThreadsTC, 1)
unm_tc_sum_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                  const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mR, UParams p) {
    using LY = USumLayout<D>;
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    enum { L0, L1, F0, F1, FIN, NBAR };  // buffer b loaded / buffer b's products done / all products done
    __shared__ __align__(8) unsigned long long bars[NBAR];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issuer = warp == kDrainWarps;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    int head, seg;
    const SegPlan plan{kL, p.nchunk, p.nseg, p.seglen};
    block_segment(plan, gridDim.y, (long long)blockIdx.y * gridDim.x + blockIdx.x, head, seg);
    const int c_begin = seg_chunk_begin(plan, seg), c_end = seg_chunk_begin(plan, seg + 1);
    const int nchunks = c_end - c_begin;
    const bool state_rows = !issuer && ((D == 128) || quarter < D / 32);
    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };
    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), 1);
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
    const uint32_t tS_ = tmem, tC_ = tmem + D;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int cD = half * (D / 2);
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
    auto tileQ = [&](int b) { return Tile{dsm + (uint32_t)b * LY::kBuf, kL}; };
    auto tileK = [&](int b) { return Tile{dsm + (uint32_t)b * LY::kBuf + LY::kTok, kL}; };
    auto tileV = [&](int b) { return Tile{dsm + (uint32_t)b * LY::kBuf + 2 * LY::kTok, kL}; };
    // the issuer's lane 0 issues every tile load and settles them before the
    // CTA exits (waits for the last of each barrier)
    LoadLedger<2> loads(bar(L0));
    static_assert(L0 == 0 && L1 == 1, "load barriers first");
    auto load = [&](int b, int chunk) {
        loads.note(b);
        mbar_expect_tx(bar(L0 + b), 3u * LY::kTok);
#pragma unroll
        for (int k = 0; k < D / 64; ++k) {
            tma_load_3d(tileQ(b).base + k * tileQ(b).block_bytes(), &mQ, k * 64, chunk * kL, head, bar(L0 + b));
            tma_load_3d(tileK(b).base + k * tileK(b).block_bytes(), &mK, k * 64, chunk * kL, head, bar(L0 + b));
            tma_load_3d(tileV(b).base + k * tileV(b).block_bytes(), &mV, k * 64, chunk * kL, head, bar(L0 + b));
        }
    };
    constexpr uint32_t iMM = idesc_bf16(128, D, true, true);  // both MN-major

    if (issuer) {
        if (lane == 0 && nchunks > 0) {
            load(0, c_begin);
            if (nchunks > 1) load(1, c_begin + 1);
            for (int it = 0; it < nchunks; ++it) {
                const int b = it & 1;
                if (!wait_bar(L0 + b, (uint32_t)((it >> 1) & 1))) break;
                tc_fence_after();
                const uint32_t acc0 = it > 0 ? 1u : 0u;
                // S += K^T K,  C += Q^T V
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tS_, tileK(b).mnmaj(ks), tileK(b).mnmaj(ks), iMM, (acc0 || ks > 0) ? 1u : 0u);
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tC_, tileQ(b).mnmaj(ks), tileV(b).mnmaj(ks), iMM, (acc0 || ks > 0) ? 1u : 0u);
                mma_commit(bar(F0 + b));
                // the other buffer's products (the previous chunk) free it for chunk it + 1
                if (it >= 1 && it + 1 < nchunks) {
                    if (!wait_bar(F0 + (b ^ 1), (uint32_t)(((it - 1) >> 1) & 1))) break;
                    load(b ^ 1, c_begin + it + 1);
                }
            }
            // FIN completes once every product has: the records can be read out
            if (!mma_wait_all(bar(FIN))) atomicExch(p.status, (int)kDevWaitTimeout);
        }
        if (lane == 0 && !loads.settle()) atomicExch(p.status, (int)kDevWaitTimeout);
    } else if (state_rows && nchunks > 0) {
        // records S (row 0) and C (row D) leave as 32 x 32 boxes through the
        // dead tile area once the last chunk's products are done
        if (wait_bar(FIN, 0)) {
            tc_fence_after();
            const uint32_t src[2] = {tS_, tC_};
            const uint32_t scratch = dsm + (uint32_t)warp * (2u * (D / 64) * 4096u);
            const int rec = head * p.nseg + seg;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                uint32_t r[64];
                tmem_ld_cols<D / 2>(src[m] + lane_off + cD, r);
#pragma unroll
                for (int g = 0; g < D / 64; ++g)
                    box32_store(&mR, scratch + (uint32_t)(m * (D / 64) + g) * 4096u, r + 32 * g, lane, cD + 32 * g,
                                m * D + quarter * 32, rec);
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

// -------------------------------------------------------------- outputs ----
template <int D>
struct UOutLayout {
    static constexpr uint32_t kTok = kL * D * 2;  // Q, K, V, X tiles
    static constexpr uint32_t kSq = kL * kL * 2;  // A / W tile
    static constexpr uint32_t kSt = D * D * 2;    // S0 / C0 tiles
    static constexpr uint32_t Q = 0, K = Q + kTok, V = K + kTok, A = V + kTok, X = A + kSq;
    static constexpr uint32_t S = X + kTok, C = S + kSt;
    static constexpr uint32_t kEnd = C + kSt;
    // lo parts on a head's first chunk: at D = 128 in the S0 (A_lo, then W_lo)
    // and C0 (X_lo) tiles, which hold zeros there; own tiles at D = 64
    static constexpr uint32_t Alo = (D == 128) ? S : kEnd;
    static constexpr uint32_t Wlo = Alo;
    static constexpr uint32_t Xlo = (D == 128) ? C : kEnd + kSq;
    static constexpr uint32_t kEnd2 = (D == 128) ? kEnd : kEnd + kSq + kTok;
    static constexpr uint32_t kPad = (D < 128) ? 16384u : 0u;
    static constexpr uint32_t kBytes = kEnd2 + kPad;
};

template <int D>
__global__ void __launch_bounds__(kThreadsTC + 32, 1)
unm_tc_out_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                  const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mO,
                  const __grid_constant__ CUtensorMap mR, UParams p) {
    using LY = UOutLayout<D>;
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    // loads | MMA commits | drains | (PB + w: drain warp w's prefix boxes)
    enum { LQ, LK, LV, CA, CXS, CX2, CW, CO, CC, CSU, DA, DX, DW, DO, DS, DC, FIN, PB, NBAR = PB + kDrainWarps };
    __shared__ __align__(8) unsigned long long bars[NBAR];
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

    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tQ{dsm + LY::Q, kL}, tK{dsm + LY::K, kL}, tV{dsm + LY::V, kL};
    const Tile tA{dsm + LY::A, kL}, tX{dsm + LY::X, kL};
    const Tile tS{dsm + LY::S, D}, tC{dsm + LY::C, D};
    const Tile tAl{dsm + LY::Alo, kL}, tWl{dsm + LY::Wlo, kL}, tXl{dsm + LY::Xlo, kL};
    auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == DA || i == DX || i == DW || i == DO) cnt = kDrainWarps;
            if (i == DS || i == DC) cnt = kStateWarps;
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
    // tensor-memory regions: A then W then W V | X then X C0 | S | C
    const uint32_t tA_ = tmem + 0, tX_ = tmem + 128, tS_ = tmem + 256, tC_ = tmem + 256 + D;
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
    LoadLedger<3> loads(bar(0));  // LQ, LK, LV
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
    auto drain128 = [&](uint32_t treg, const Tile& t, bool mask) {
        uint32_t r[64];
        tmem_ld_cols<64>(treg + lane_off + c128, r);
        put_row32(t, row, c128, r, mask);
        put_row32(t, row, c128 + 32, r + 32, mask);
    };
    auto drain128s = [&](uint32_t treg, const Tile& hi, const Tile& lo, bool mask) {
        uint32_t r[64];
        tmem_ld_cols<64>(treg + lane_off + c128, r);
        put_row32_split2(hi, lo, row, c128, r, mask);
        put_row32_split2(hi, lo, row, c128 + 32, r + 32, mask);
    };
    auto drainD = [&](uint32_t treg, const Tile& t) {
        uint32_t r[64];
        tmem_ld_cols<D / 2>(treg + lane_off + cD, r);
        put_row32(t, row, cD, r, false);
        if (D == 128) put_row32(t, row, cD + 32, r + 32, false);
    };
    auto drainDs = [&](uint32_t treg, const Tile& hi, const Tile& lo) {
        uint32_t r[64];
        tmem_ld_cols<D / 2>(treg + lane_off + cD, r);
        put_row32_split2(hi, lo, row, cD, r, false);
        if (D == 128) put_row32_split2(hi, lo, row, cD + 32, r + 32, false);
    };

    // the first chunk's tiles start moving while the drain warps load the prefix
    if (producer && lane == 0 && nchunks > 0) {
        issue_load(LQ, &mQ, tQ, c_begin);
        issue_load(LK, &mK, tK, c_begin);
        issue_load(LV, &mV, tV, c_begin);
    }
    // ---- initial state: S0 (record row 0), C0 (record row D) by bulk tensor
    // loads into per-warp staging in the A / X tiles, then TMEM and bf16 tiles
    if (state_rows) {
        const int rec = head * p.nseg + seg;
        const uint32_t stage = dsm + LY::A + (uint32_t)warp * (uint32_t)(D / 64) * 4096u;
        LoadLedger<1> boxes(bar(PB + warp));
#pragma unroll 1
        for (int m = 0; m < 2; ++m) {
            if (lane == 0) {
                boxes.note(0);
                fence_proxy_async();
                mbar_expect_tx(bar(PB + warp), (uint32_t)(D / 64) * 4096u);
#pragma unroll
                for (int g = 0; g < D / 64; ++g)
                    tma_load_3d(stage + (uint32_t)g * 4096u, &mR, cD + 32 * g, m * D + quarter * 32, rec, bar(PB + warp));
            }
            __syncwarp();
            if (!wait_bar(PB + warp, (uint32_t)m)) break;
#pragma unroll
            for (int g = 0; g < D / 64; ++g) {
                const int cb = cD + 32 * g;
                uint32_t r[32];
                box32_read(stage + (uint32_t)g * 4096u, lane, r);
                tmem_st32((m == 0 ? tS_ : tC_) + lane_off + cb, r);
                put_row32(m == 0 ? tS : tC, row, cb, r, false);
            }
            __syncwarp();
        }
        if (lane == 0 && !boxes.settle()) atomicExch(p.status, (int)kDevWaitTimeout);
        tmem_st_wait();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    constexpr uint32_t iSq = idesc_bf16(128, 128, false, false);  // 128 x 128, both K-major
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
                const bool first = c == 0;  // S0 = C0 = 0; A, X, W split into hi + lo
                if (!wait_bar(LQ, ph) || !wait_bar(LK, ph)) break;
                if (it > 0 && !wait_bar(DO, pph)) break;  // O of the previous chunk read out of TMEM A
                tc_fence_after();
                // A = Q K^T
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQ.kmaj(ks), tK.kmaj(ks), iSq, ks > 0);
                mma_commit(bar(CA));
                if (it > 0 && !wait_bar(DS, pph)) break;  // sS = S0 of this chunk; TMEM S read
                tc_fence_after();
                // X = Q S0
                if (!first)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tX_, tQ.kmaj(ks), tS.kmaj(ks), iKK, ks > 0);
                mma_commit(bar(CXS));
                if (!wait_bar(DA, ph)) break;  // sA = A (and A_lo on the first chunk)
                tc_fence_after();
                // X += A K
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tX_, tA.kmaj(ks), tK.mnmaj(ks), iKM, (!first || ks > 0) ? 1u : 0u);
                if (first)
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tX_, tAl.kmaj(ks), tK.mnmaj(ks), iKM, 1);
                mma_commit(bar(CX2));
                if (has_next) {
                    // S += K^T K after A K, beside the X drain rather than the A
                    // drain (the state after the segment's last chunk is not needed)
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tS_, tK.mnmaj(ks), tK.mnmaj(ks), iMM, 1);
                    mma_commit(bar(CSU));
                }
                if (!wait_bar(DX, ph)) break;  // sX = X (and X_lo); TMEM X read
                tc_fence_after();
                // W = X Q^T
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tX.kmaj(ks), tQ.kmaj(ks), iSq, ks > 0);
                if (first)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tXl.kmaj(ks), tQ.kmaj(ks), iSq, 1);
                mma_commit(bar(CW));
                if (!first) {
                    // X C0 into TMEM X (read out at DX): it runs while W is drained, and
                    // the O drain adds it to W V
                    if (it > 0 && !wait_bar(DC, pph)) break;  // sC = C0 of this chunk; TMEM C read
                    tc_fence_after();
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tX_, tX.kmaj(ks), tC.mnmaj(ks), iKM, ks > 0);
                }
                if (!wait_bar(DW, ph)) break;  // sA = W (and W_lo); TMEM A read
                tc_fence_after();
                // O = W V  (+ X C0 from TMEM X)
                if (!wait_bar(LV, ph)) break;
                tc_fence_after();
                for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tA_, tA.kmaj(ks), tV.mnmaj(ks), iKM, ks > 0 ? 1u : 0u);
                if (first)
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tA_, tWl.kmaj(ks), tV.mnmaj(ks), iKM, 1);
                mma_commit(bar(CO));
                if (has_next) {
                    // C += Q^T V
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tC_, tQ.mnmaj(ks), tV.mnmaj(ks), iMM, 1);
                    mma_commit(bar(CC));
                }
            }
            if (!mma_wait_all(bar(FIN))) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else if (producer) {
        // the next chunk's tiles once their last reader completed: K after
        // A K, Q and V after Q^T V
        if (lane == 0) {
            for (int it = 0; it + 1 < nchunks; ++it) {
                const int c = c_begin + it;
                const uint32_t ph = it & 1;
                if (!wait_bar(CSU, ph)) break;  // S += K^T K, K's last reader
                issue_load(LK, &mK, tK, c + 1);
                if (!wait_bar(CC, ph)) break;
                issue_load(LQ, &mQ, tQ, c + 1);
                issue_load(LV, &mV, tV, c + 1);
            }
            if (!loads.settle()) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else {
        // ========================== drain warps ==========================
        for (int it = 0; it < nchunks; ++it) {
            const uint32_t ph = it & 1;
            const bool has_next = it + 1 < nchunks;
            const bool first = c_begin + it == 0;
            if (!wait_bar(CA, ph)) break;
            tc_fence_after();
            // this warp's first O piece has left its sA rows (the second, in sX, may not have)
            if (lane == 0) {
                if (D == 128) tma_store_wait_read_all_but_1();
                else tma_store_wait_read();
            }
            __syncwarp();
            if (first) drain128s(tA_, tA, tAl, true);  // A -> sA (hi), A_lo (masked)
            else drain128(tA_, tA, true);              // A -> sA (masked)
            drained(DA);
            if (!wait_bar(CX2, ph)) break;
            tc_fence_after();
            if (D == 128) {
                if (lane == 0) tma_store_wait_read();  // the second O piece has left its sX rows
                __syncwarp();
            }
            if (first) drainDs(tX_, tX, tXl);  // X -> sX (hi), X_lo
            else drainD(tX_, tX);              // X -> sX
            drained(DX);
            if (state_rows && has_next && !first) {
                if (!wait_bar(CSU, ph)) break;
                tc_fence_after();
                drainD(tS_, tS);  // S0 of the next chunk -> sS
                drained(DS);
            }
            if (!wait_bar(CW, ph)) break;
            tc_fence_after();
            if (first) drain128s(tA_, tA, tWl, true);  // W -> sA (hi), W_lo (masked)
            else drain128(tA_, tA, true);              // W -> sA (masked)
            drained(DW);
            if (!wait_bar(CO, ph)) break;
            tc_fence_after();
            {
                // O: piece 0 through this warp's 4 KB of sA, piece 1 (D = 128) through
                // the same rows of sX (both dead once the output products completed)
                uint32_t r[64];
                tmem_ld_cols<D / 2>(tA_ + lane_off + cD, r);
                if (!first) {
                    // + X C0 (TMEM X), 32 columns at a time
#pragma unroll
                    for (int g = 0; g < D / 64; ++g) {
                        uint32_t t[32];
                        tmem_ld32(tX_ + lane_off + cD + 32 * g, t);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            r[32 * g + j] = __float_as_uint(__uint_as_float(r[32 * g + j]) + __uint_as_float(t[j]));
                    }
                }
                drained(DO);
                const uint32_t wofs = (uint32_t)half * (kL * 128u) + (uint32_t)(quarter * 32) * 128u;
                const int t0 = (c_begin + it) * kL + quarter * 32;
                box32_store(&mO, tA.base + wofs, r, lane, cD, t0, head);
                if (D == 128) box32_store(&mO, tX.base + wofs, r + 32, lane, cD + 32, t0, head);
            }
            if (state_rows && has_next) {
                if (first) {
                    drainD(tS_, tS);  // S0 of the next chunk -> sS, once the lo parts there are dead
                    drained(DS);
                }
                if (!wait_bar(CC, ph)) break;
                tc_fence_after();
                drainD(tC_, tC);  // C0 of the next chunk -> sC
                drained(DC);
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
cudaError_t launch_u(int mode, const void* Q, const void* K, const void* V, float* O, const float* prefix, float* summ,
                     int BH, int T, SegPlan plan, int* status, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mo, mr;
    if (!make_map(&mq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mk, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mv, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64))
        return cudaErrorInvalidValue;
    // the segment records as (3D + 2) rows of D floats, 32 x 32 boxes
    if (!make_map(&mr, mode == 1 ? static_cast<const void*>(prefix) : static_cast<const void*>(summ),
                  CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, 3 * D + 2, BH * plan.nseg, 32, 32))
        return cudaErrorInvalidValue;
    UParams prm{T, plan.nseg, plan.nchunk, plan.seglen, status};
    dim3 grid(plan.nseg, BH);
    cudaError_t e;
    if (mode == 0) {
        const size_t smem = USumLayout<D>::kBytes + 1024;
        auto kern = unm_tc_sum_kernel<D>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreadsTC, smem, s>>>(mq, mk, mv, mr, prm);
    } else {
        if (!make_map(&mo, O, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, T, BH, 32, 32)) return cudaErrorInvalidValue;
        const size_t smem = UOutLayout<D>::kBytes + 1024;
        auto kern = unm_tc_out_kernel<D>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreadsTC + 32, smem, s>>>(mq, mk, mv, mo, mr, prm);
    }
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_unm_tc_walk(int mode, const void* Q, const void* K, const void* V, float* O, const float* prefix,
                               float* summ, int BH, int T, int d, int dv, SegPlan plan, int* status, cudaStream_t s) {
    if (BH == 0 || plan.nseg == 0) return cudaSuccess;
    if (plan.granule != kL || d != dv) return cudaErrorInvalidValue;
    if (d == 128) return launch_u<128>(mode, Q, K, V, O, prefix, summ, BH, T, plan, status, s);
    if (d == 64) return launch_u<64>(mode, Q, K, V, O, prefix, summ, BH, T, plan, status, s);
    return cudaErrorInvalidValue;
}

}  // namespace hla2
