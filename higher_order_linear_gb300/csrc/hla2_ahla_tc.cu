// hla2_ahla_tc.cu -- tensor-core segment walks of masked AHLA on GB300
// (sm_103a): tcgen05.mma with TMEM accumulators, TMA-staged tiles.
//
// HLA summary (arXiv 2510.27258), section 2 "AHLA": the operator
// Q (K^T Q)(K^T V) under the causal mask, o_t = sum_{j<=i<=t} (q_t.k_i)(q_i.k_j) v_j,
// kept as summaries P = sum k v^T, E = sum_i k_i q_i^T P_i (and, to join
// segments, M = sum k q^T); section 4 for the chunk-parallel form.
//
// One CTA walks one segment of one head in chunks of L = 128 tokens.  With
// the state (P0, E0) entering a chunk and the chunk's Q, K, V:
//   A = tril(Q K^T)            (i <= t, diagonal kept)
//   Y = Q P0 + A V             (row i is P_i^T q_i)
//   O = Q E0 + A Y             (the chunk's outputs)
//   E0 += K^T Y,   P0 += K^T V
// The summary walk starts from zero and also accumulates M += K^T Q.  Every
// product is a 128-row tcgen05.mma kind::f16 (bf16 operands in shared
// memory, fp32 accumulators in tensor memory).  A, Y, P0 and E0 are rounded
// to bf16 when written back as operands; P and E stay fp32 in tensor memory
// for the whole segment.  On a head's first chunk (where an output can be a
// single product: t = 0 gives (q.k)^2 v) A and Y are split into bf16 hi + lo
// parts: Y = Q P0 + A_hi V + A_lo V, O = A_hi Y_hi + A_lo Y_hi + A_hi Y_lo,
// E += K^T Y_hi + K^T Y_lo.  That chunk has P0 = E0 = 0, so at d = 128 the
// E0 and P0 tiles hold the lo parts of A and Y (P0 of the next chunk is then
// written only after every product of the first chunk has completed).
//
// Roles as in the HLA walk: warp 8 (lane 0) issues every TMA copy and MMA;
// warps 0..7 drain tensor memory (warp w: lane quarter w % 4, column half
// w / 4).  They meet only on mbarriers, every wait bounded in time.
#include "hla2_tc_common.cuh"

namespace hla2 {
namespace {

// Chunks ahead whose tiles a walk pulls into L2 before their TMA loads.  One:
// on the headline shape it beat none (11% faster forward), two and four.
constexpr int kAhead = 1;

struct AParams {
    int T, nseg, nchunk, seglen;
    float* summ;          // summary walk: output records M|P|m|E|n
    const float* prefix;  // output walk: input records (P, E read)
    int* status;
};

template <int D, int MODE>
struct ALayout {
    static constexpr uint32_t kTok = kL * D * 2;  // Q, K, V, Y tiles
    static constexpr uint32_t kSq = kL * kL * 2;  // A tile
    static constexpr uint32_t kSt = D * D * 2;    // P0 / E0 tiles
    static constexpr uint32_t Q = 0, K = Q + kTok, V = K + kTok, A = V + kTok, Y = A + kSq;
    static constexpr uint32_t P = Y + kTok;
    static constexpr uint32_t E = P + kSt;  // output walk only
    static constexpr uint32_t kEnd = (MODE == 1) ? E + kSt : E;
    // lo parts of A and Y on a head's first chunk (output walk): the E0 and
    // P0 tiles at D = 128 (same geometry, unused there), own tiles at D = 64
    static constexpr uint32_t Alo = (D == 128) ? E : kEnd;
    static constexpr uint32_t Ylo = (D == 128) ? P : kEnd + kSq;
    static constexpr uint32_t kEnd2 = (MODE == 1 && D < 128) ? kEnd + kSq + kTok : kEnd;
    // MN-major operands read with M = 128 > D see a second 64-column block
    // one block past the tile: keep valid memory there when D = 64.
    static constexpr uint32_t kPad = (D < 128) ? 16384u : 0u;
    static constexpr uint32_t kBytes = kEnd2 + kPad;
};

template <int D, int MODE>
__global__ void __launch_bounds__(kThreadsTC + 32, 1)
ahla_tc_walk_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mO,
                    const __grid_constant__ CUtensorMap mR, AParams p) {
    using LY = ALayout<D, MODE>;
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    // loads | MMA commits | drains
    // (PB + w: drain warp w's prefix boxes, output walk)
    enum { LQ, LK, LV, CA, CY, CQ, CO, CE, DA, DY, DO, DP, DE, FIN, PB, NBAR = PB + kDrainWarps };
    __shared__ __align__(8) unsigned long long bars[NBAR];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const bool issuer = warp == kDrainWarps;
    // a load warp issues every tile load as soon as its buffer is free, so
    // that the MMA issuer never blocks on a reload
    const bool producer = warp == kDrainWarps + 1;
    const int quarter = warp & 3;
    const int half = (warp >> 2) & 1;
    const int row = quarter * 32 + lane;
    int head, seg;
    const SegPlan plan{kL, p.nchunk, p.nseg, p.seglen};
    block_segment(plan, gridDim.y, (long long)blockIdx.y * gridDim.x + blockIdx.x, head, seg);
    const int c_begin = seg_chunk_begin(plan, seg);
    const int c_end = seg_chunk_begin(plan, seg + 1);
    const bool state_rows = warp < kDrainWarps && ((D == 128) || quarter < D / 32);
    constexpr int kStateWarps = (D == 128) ? kDrainWarps : 2 * (D / 32);

    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tQ{dsm + LY::Q, kL}, tK{dsm + LY::K, kL}, tV{dsm + LY::V, kL};
    const Tile tA{dsm + LY::A, kL}, tY{dsm + LY::Y, kL}, tAl{dsm + LY::Alo, kL}, tYl{dsm + LY::Ylo, kL};
    const Tile tP{dsm + LY::P, D}, tE{dsm + LY::E, D};
    auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == DA || i == DY || i == DO) cnt = kDrainWarps;
            if (i == DP || i == DE) cnt = kStateWarps;
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
    // tensor-memory regions (column offsets)
    //   output walk:  A then O | Y | P | E
    //   summary walk: A then Y | P | E | M
    const uint32_t tA_ = tmem + 0;
    const uint32_t tY_ = tmem + 128;  // output walk only
    const uint32_t tP_ = tmem + (MODE == 1 ? 256 : 128);
    const uint32_t tE_ = tP_ + D;
    const uint32_t tM_ = tE_ + D;     // summary walk only
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
    auto prefetch = [&](int chunk) {
#pragma unroll
        for (int k = 0; k < D / 64; ++k) {
            tma_prefetch_l2_3d(&mQ, k * 64, chunk * kL, head);
            tma_prefetch_l2_3d(&mK, k * 64, chunk * kL, head);
            tma_prefetch_l2_3d(&mV, k * 64, chunk * kL, head);
        }
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

    const int nchunks = c_end - c_begin;
    // The first chunk's tiles start moving now, while the drain warps load the
    // segment prefix below (the barriers were initialised before the first
    // __syncthreads, so the load warp may use them).
    if (producer && lane == 0 && nchunks > 0) {
        issue_load(LQ, &mQ, tQ, c_begin);
        issue_load(LK, &mK, tK, c_begin);
        issue_load(LV, &mV, tV, c_begin);
        for (int a = 1; a < kAhead && a < nchunks; ++a) prefetch(c_begin + a);
    }

    // ---- initial state (output walk): P0, E0 fp32 into TMEM, bf16 into smem ----
    if (MODE == 1 && state_rows) {
        const size_t R = (size_t)D * D + 2 * (size_t)D * D + 2 * (size_t)D;
        const float* pre = p.prefix + ((size_t)head * p.nseg + seg) * R;
        // P0 (record row D) and E0 (record row 2D + 1) arrive as this warp's
        // 32 x 32 fp32 boxes by bulk tensor loads (mR maps the records as
        // (3D + 2) rows of D floats) into a private staging area in the A / Y
        // tiles, which nothing else touches before the first chunk
        (void)pre;
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
                    tma_load_3d(stage + (uint32_t)g * 4096u, &mR, cD + 32 * g, (m == 0 ? D : 2 * D + 1) + quarter * 32, rec,
                                bar(PB + warp));
            }
            __syncwarp();
            if (!wait_bar(PB + warp, (uint32_t)m)) break;
#pragma unroll
            for (int g = 0; g < D / 64; ++g) {
                const int cb = cD + 32 * g;
                uint32_t r[32];
                box32_read(stage + (uint32_t)g * 4096u, lane, r);
                tmem_st32((m == 0 ? tP_ : tE_) + lane_off + cb, r);
                put_row32(m == 0 ? tP : tE, row, cb, r, false);
            }
            __syncwarp();  // every lane has read the boxes before the next load reuses them
        }
        if (lane == 0 && !boxes.settle()) atomicExch(p.status, (int)kDevWaitTimeout);
        tmem_st_wait();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    constexpr uint32_t iSq = idesc_bf16(128, 128, false, false);  // 128 x 128, both K-major
    constexpr uint32_t iKM = idesc_bf16(128, D, false, true);     // A K-major, B MN-major
    constexpr uint32_t iMM = idesc_bf16(128, D, true, true);      // both MN-major

    if (issuer) {
        // ============================ issuer ============================
        if (lane == 0 && nchunks > 0) {
            for (int it = 0; it < nchunks; ++it) {
                const int c = c_begin + it;
                const uint32_t ph = it & 1, pph = (it + 1) & 1;
                if (!wait_bar(LQ, ph) || !wait_bar(LK, ph)) break;
                if (MODE == 1) {
                    const bool first = c == 0;  // P0 = E0 = 0; A and Y split into hi + lo
                    if (it > 0 && !wait_bar(DO, pph)) break;  // O of the previous chunk read out of TMEM A
                    tc_fence_after();
                    // A = Q K^T
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQ.kmaj(ks), tK.kmaj(ks), iSq, ks > 0);
                    mma_commit(bar(CA));
                    if (it > 0 && !wait_bar(DP, pph)) break;  // sP = P0 of this chunk; TMEM P read
                    tc_fence_after();
                    // Y = Q P0
                    if (!first)
                        for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tY_, tQ.kmaj(ks), tP.mnmaj(ks), iKM, ks > 0);
                    if (!wait_bar(LV, ph)) break;
                    tc_fence_after();
                    // P += K^T V
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tP_, tK.mnmaj(ks), tV.mnmaj(ks), iMM, 1);
                    if (!wait_bar(DA, ph)) break;  // sA = A (and its lo part on the first chunk)
                    tc_fence_after();
                    // Y += A V
                    for (int ks = 0; ks < kL / 16; ++ks)
                        mma_bf16(tY_, tA.kmaj(ks), tV.mnmaj(ks), iKM, (!first || ks > 0) ? 1u : 0u);
                    if (first)
                        for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tY_, tAl.kmaj(ks), tV.mnmaj(ks), iKM, 1);
                    mma_commit(bar(CY));
                    if (it > 0 && !wait_bar(DE, pph)) break;  // sE = E0 of this chunk; TMEM E read
                    tc_fence_after();
                    // O = Q E0 (TMEM A is free once A was drained); this is Q's last read
                    if (!first)
                        for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQ.kmaj(ks), tE.mnmaj(ks), iKM, ks > 0);
                    mma_commit(bar(CQ));
                    if (!wait_bar(DY, ph)) break;  // sY = Y (and Y_lo on the first chunk); TMEM Y read
                    tc_fence_after();
                    // E += K^T Y first (K's last read), then O += A Y
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tE_, tK.mnmaj(ks), tY.mnmaj(ks), iMM, 1);
                    if (first)
                        for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tE_, tK.mnmaj(ks), tYl.mnmaj(ks), iMM, 1);
                    mma_commit(bar(CE));
                    for (int ks = 0; ks < kL / 16; ++ks)
                        mma_bf16(tA_, tA.kmaj(ks), tY.mnmaj(ks), iKM, (!first || ks > 0) ? 1u : 0u);
                    if (first) {
                        for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tA_, tAl.kmaj(ks), tY.mnmaj(ks), iKM, 1);
                        for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tA_, tA.kmaj(ks), tYl.mnmaj(ks), iKM, 1);
                    }
                    mma_commit(bar(CO));
                } else {
                    const uint32_t acc0 = it > 0 ? 1u : 0u;  // segment-local sums start at zero
                    tc_fence_after();
                    // A = Q K^T   (TMEM A is free: the previous Y was drained before its E product)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQ.kmaj(ks), tK.kmaj(ks), iSq, ks > 0);
                    mma_commit(bar(CA));
                    // M += K^T Q
                    for (int ks = 0; ks < kL / 16; ++ks)
                        mma_bf16(tM_, tK.mnmaj(ks), tQ.mnmaj(ks), iMM, (acc0 || ks > 0) ? 1u : 0u);
                    if (!wait_bar(LV, ph)) break;
                    if (it > 0 && !wait_bar(DP, pph)) break;  // sP = P_local of this chunk; TMEM P read
                    tc_fence_after();
                    // P += K^T V
                    for (int ks = 0; ks < kL / 16; ++ks)
                        mma_bf16(tP_, tK.mnmaj(ks), tV.mnmaj(ks), iMM, (acc0 || ks > 0) ? 1u : 0u);
                    if (!wait_bar(DA, ph)) break;  // sA = A; TMEM A read
                    tc_fence_after();
                    // Y = Q P_local + A V   (no P_local term on the segment's first chunk)
                    if (it > 0)
                        for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQ.kmaj(ks), tP.mnmaj(ks), iKM, ks > 0);
                    for (int ks = 0; ks < kL / 16; ++ks)
                        mma_bf16(tA_, tA.kmaj(ks), tV.mnmaj(ks), iKM, (acc0 || ks > 0) ? 1u : 0u);
                    mma_commit(bar(CY));
                    if (!wait_bar(DY, ph)) break;  // sY = Y; TMEM A read (Q and V no longer read)
                    tc_fence_after();
                    // E += K^T Y
                    for (int ks = 0; ks < kL / 16; ++ks)
                        mma_bf16(tE_, tK.mnmaj(ks), tY.mnmaj(ks), iMM, (acc0 || ks > 0) ? 1u : 0u);
                    mma_commit(bar(CE));
                }
            }
            if (!mma_wait_all(bar(FIN))) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else if (producer) {
        // ============================ loads ============================
        // the next chunk's tiles once their last reader completed: V after
        // A V (CY; in the summary walk also Q, whose last readers M and Y
        // precede it), Q after Q E0 (CQ, output walk), K after K^T Y (CE)
        if (lane == 0) {
            for (int it = 0; it + 1 < nchunks; ++it) {
                const int c = c_begin + it;
                const uint32_t ph = it & 1;
                if (kAhead > 0 && it + kAhead < nchunks) prefetch(c + kAhead);
                if (!wait_bar(CY, ph)) break;
                issue_load(LV, &mV, tV, c + 1);
                if (MODE == 0) issue_load(LQ, &mQ, tQ, c + 1);
                if (MODE == 1) {
                    if (!wait_bar(CQ, ph)) break;
                    issue_load(LQ, &mQ, tQ, c + 1);
                }
                if (!wait_bar(CE, ph)) break;
                issue_load(LK, &mK, tK, c + 1);
            }
            if (!loads.settle()) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else {
        // ========================== drain warps ==========================
        for (int it = 0; it < nchunks; ++it) {
            const uint32_t ph = it & 1;
            const bool has_next = it + 1 < nchunks;
            if (MODE == 1) {
                const bool first = c_begin + it == 0;
                if (!wait_bar(CA, ph)) break;
                tc_fence_after();
                // this warp's first O piece has left its sA rows (at D = 128 the
                // second piece, staged in sY, may still be in flight)
                if (lane == 0) {
                    if (D == 128) tma_store_wait_read_all_but_1();
                    else tma_store_wait_read();
                }
                __syncwarp();
                if (first) drain128s(tA_, tA, tAl, true);  // A -> sA (hi), A_lo (masked)
                else drain128(tA_, tA, true);              // A -> sA (masked)
                drained(DA);
                if (!wait_bar(CY, ph)) break;
                tc_fence_after();
                if (D == 128) {
                    if (lane == 0) tma_store_wait_read();  // the second O piece has left its sY rows
                    __syncwarp();
                }
                if (first) drainDs(tY_, tY, tYl);  // Y -> sY (hi), Y_lo
                else drainD(tY_, tY);              // Y -> sY
                drained(DY);
                if (state_rows && has_next && !first) {
                    drainD(tP_, tP);  // P0 of the next chunk -> sP (P += K^T V completed with Y)
                    drained(DP);
                }
                if (!wait_bar(CO, ph)) break;
                tc_fence_after();
                {
                    // O (fp32) leaves through the 4 KB of sA that hold this warp's own
                    // rows and column half (A there is dead once the output products
                    // completed), 32 rows x 32 columns per bulk tensor store.
                    uint32_t r[64];
                    tmem_ld_cols<D / 2>(tA_ + lane_off + cD, r);
                    drained(DO);  // TMEM A is free once O sits in registers
                    // piece 0 through this warp's 4 KB of sA, piece 1 (D = 128) through the
                    // same rows of sY: both dead once the output products (and K^T Y,
                    // committed before them) completed
                    const uint32_t wofs = (uint32_t)half * (kL * 128u) + (uint32_t)(quarter * 32) * 128u;
                    const int t0 = (c_begin + it) * kL + quarter * 32;
                    box32_store(&mO, tA.base + wofs, r, lane, cD, t0, head);
                    if (D == 128) box32_store(&mO, tY.base + wofs, r + 32, lane, cD + 32, t0, head);
                }
                if (state_rows && has_next) {
                    if (!wait_bar(CE, ph)) break;
                    tc_fence_after();
                    drainD(tE_, tE);  // E0 of the next chunk -> sE
                    drained(DE);
                    if (first) {
                        drainD(tP_, tP);  // P0 of the next chunk -> sP, once Y_lo there is dead
                        drained(DP);
                    }
                }
            } else {
                if (!wait_bar(CA, ph)) break;
                tc_fence_after();
                drain128(tA_, tA, true);  // A -> sA (masked)
                drained(DA);
                if (!wait_bar(CY, ph)) break;
                tc_fence_after();
                drainD(tA_, tY);  // Y -> sY
                drained(DY);
                if (state_rows && has_next) {
                    drainD(tP_, tP);  // P_local of the next chunk -> sP
                    drained(DP);
                }
            }
        }
        if (MODE == 1 && lane == 0) tma_store_wait_all();
        // ---- segment summary out (summary walk): M | P | . | E | . records, fp32 ----
        if (MODE == 0 && state_rows && nchunks > 0 && wait_bar(CE, (nchunks - 1) & 1)) {
            tc_fence_after();
            // M, P, E leave through 32 x 32 boxes and bulk tensor stores (mO maps
            // the records as (3D + 2) rows of D floats: M at row 0, P at row D,
            // E at row 2D + 1).  The last MMAs completed and no load is in
            // flight, so each warp stages its boxes in its own part of the tiles.
            const uint32_t src[3] = {tM_, tP_, tE_};
            const int row0[3] = {0, D, 2 * D + 1};
            const uint32_t scratch = dsm + (uint32_t)warp * (3u * (D / 64) * 4096u);
            const int rec = head * p.nseg + seg;
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                uint32_t r[64];
                tmem_ld_cols<D / 2>(src[m] + lane_off + cD, r);
#pragma unroll
                for (int g = 0; g < D / 64; ++g)
                    box32_store(&mR, scratch + (uint32_t)(m * (D / 64) + g) * 4096u, r + 32 * g, lane, cD + 32 * g,
                                row0[m] + quarter * 32, rec);
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

template <int D, int MODE>
cudaError_t launch_t(const void* Q, const void* K, const void* V, float* O, const float* prefix, float* summ, int BH,
                     int T, SegPlan plan, int* status, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mk, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mv, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64))
        return cudaErrorInvalidValue;
    // mR: the segment records (prefixes read by the output walk, summaries
    // written by the summary walk) as (3D + 2) rows of D floats, 32 x 32 boxes
    CUtensorMap mr;
    if (!make_map(&mr, MODE == 1 ? static_cast<const void*>(prefix) : static_cast<const void*>(summ),
                  CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, 3 * D + 2, BH * plan.nseg, 32, 32))
        return cudaErrorInvalidValue;
    if (MODE == 1) {
        if (!make_map(&mo, O, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, T, BH, 32, 32)) return cudaErrorInvalidValue;
    } else {
        mo = mr;  // unused
    }
    AParams prm{T, plan.nseg, plan.nchunk, plan.seglen, summ, prefix, status};
    const size_t smem = ALayout<D, MODE>::kBytes + 1024;
    auto kern = ahla_tc_walk_kernel<D, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.nseg, BH);
    kern<<<grid, kThreadsTC + 32, smem, s>>>(mq, mk, mv, mo, mr, prm);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ahla_tc_walk(int mode, const void* Q, const void* K, const void* V, float* O, const float* prefix,
                                float* summ, int BH, int T, int d, int dv, SegPlan plan, int* status, cudaStream_t s) {
    if (BH == 0 || plan.nseg == 0) return cudaSuccess;
    if (plan.granule != kL || d != dv) return cudaErrorInvalidValue;
    if (d == 128) return mode == 0 ? launch_t<128, 0>(Q, K, V, O, prefix, summ, BH, T, plan, status, s)
                                   : launch_t<128, 1>(Q, K, V, O, prefix, summ, BH, T, plan, status, s);
    if (d == 64) return mode == 0 ? launch_t<64, 0>(Q, K, V, O, prefix, summ, BH, T, plan, status, s)
                                  : launch_t<64, 1>(Q, K, V, O, prefix, summ, BH, T, plan, status, s);
    return cudaErrorInvalidValue;
}

}  // namespace hla2
