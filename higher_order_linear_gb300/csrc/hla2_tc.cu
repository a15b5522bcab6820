// hla2_tc.cu -- tensor-core segment summary walk of masked second-order HLA
// on GB300 (sm_103a): tcgen05.mma with TMEM accumulators, TMA-staged tiles.
// (The output walk, which restarts every segment from its prefix, is
// hla2_tc_out.cu.)
//
// HLA summary (arXiv 2510.27258): section 1 "Second-order HLA" (o_t =
// q_t^T (S_t C_t - G_t), the causal A A^T V structure of section 2) and
// section 4 "Parallel training via associative scans" (chunk-parallel form:
// segment summaries, exclusive scan, restart from the prefix).
//
// One CTA walks one segment of one head in chunks of L = 128 tokens, from a
// zero state.  With P = S C - G ("P-form"), the state entering a chunk is
// (S0, P0) and, for the chunk's Q, K, V (128 x d, 128 x d, 128 x dv):
//   A = tril(Q K^T)                     (i <= t, diagonal kept)
//   X = Q S0 + A K                      (so that P grows by X^T V)
//   P0 += X^T V,   S0 += K^T K,   C += Q^T V
// and the segment's S, C, P (with m and p when wanted) are its summary.
// Every product is a dense 128-row contraction issued as tcgen05.mma
// kind::f16 (bf16 operands from shared memory, fp32 accumulators in tensor
// memory).  fp32 results that feed a later product (A, X, S0) are rounded to
// bf16 when written back to shared memory; the running S, C and P stay fp32
// in tensor memory for the whole segment.
//
// Operand layout: every tile lives in shared memory as rows of 128 bytes
// (64 bf16) in the 128-byte-swizzled pattern TMA writes, split into 64-column
// blocks.  A tile whose rows are the product's M (or N) index is read as a
// K-major operand; a tile whose rows are the contraction index is read as an
// MN-major operand.  This lets every tensor-memory drain write whole rows.
#include "hla2_tc_common.cuh"

namespace hla2 {
namespace {

// Chunks ahead whose tiles the walk pulls into L2 before their TMA loads: on
// B1 H16 T65536 d128 one gains 3% (two: 0.5%, four: 12% slower).
constexpr int kAhead = 1;

// ------------------------------------------------------------- kernel ----
struct TCParams {
    int T, nseg, nchunk, seglen;
    float* summ;  // output records
    int* status;
};

template <int D, bool NORM = false>
struct Layout {
    // byte offsets of the tiles inside the 1024-aligned dynamic shared memory
    static constexpr uint32_t kTok = kL * D * 2;      // Q, K, V tiles
    static constexpr uint32_t kSq = kL * kL * 2;      // A tile, then X
    static constexpr uint32_t kSt = D * D * 2;        // S tile
    // NORM: the V tile's second 64-column block holds ones ([V | 1]).
    // At D = 128 X goes into the A tile (shared memory is full): A K, A's only
    // reader, has completed when X is drained, and the next A is drained only
    // after X^T V (issued before it) completed.  At D = 64 X has a tile of its
    // own, and X^T V of a chunk is issued after the next chunk's A = Q K^T
    // (kDeferP), off the chain A -> drain -> A K -> drain -> next A.
    static constexpr bool kSepX = D < 128;
    static constexpr uint32_t Q = 0, K = Q + kTok, V = K + kTok, A = V + (NORM ? 2 : 1) * kTok;
    static constexpr uint32_t X = kSepX ? A + kSq : A;
    static constexpr uint32_t Q2 = kSepX ? X + kTok : A + kSq;  // second Q buffer
    static constexpr uint32_t K2 = Q2 + kTok;                  // second K buffer
    static constexpr uint32_t S = K2 + kTok;
    static constexpr uint32_t kEnd = S + kSt;
    // ratio-normalised walk: bf16 lo halves of the split operands
    static constexpr uint32_t Alo = kEnd, Xlo = kSepX ? Alo + kSq : Alo;
    static constexpr uint32_t kNormEnd = kSepX ? Xlo + kTok : Alo + kSq;
    // MN-major operands read with M = 128 > D see a second 64-column block
    // one block past the tile: keep valid memory there when D = 64.
    static constexpr uint32_t kPad = (D < 128) ? 16384u : 0u;
    static constexpr uint32_t kBytes = (NORM ? kNormEnd : kEnd) + kPad;
    static_assert(!NORM || D == 64, "the normalised walk's split tiles fit at D = 64");
};

// Warp roles.  Warps 0..7 drain tensor memory: warp w owns TMEM lane quarter
// w % 4 (tile rows 32*(w%4)..+31) and column half w / 4 of every region.
// Warp 8 (lane 0) issues every TMA copy and every MMA.  The roles meet only
// on mbarriers: each group of MMAs is committed to its own barrier, and each
// drained region is announced on a barrier (one arrival per drain warp) that
// the issuer waits on before it overwrites the region or reads what the
// drain wrote.  Drains thus overlap the MMAs that do not depend on them.
//
// NORM (ratio-normalised variant, D = 64): A and X, which feed products,
// are split into bf16 hi + lo parts and the product is taken on both parts,
// which keeps about 16 significant bits.  S0 is rounded to bf16 as in the
// unnormalised walk (its rounding stays two orders below the 1e-4 bound on
// the normalised outputs, where A's or X's would exceed it).
// The extra value column of ones rides along: V is read as [V | 1] (the V
// tile's second 64-column block holds ones), so the N = D + 16 products
// C += Q^T [V | 1] and P += X^T [V | 1] also gather m = sum_t q_t and
// p = sum_t x_t in column D of C and P.
//
// XP (unnormalised summary walk whose final state is wanted): the segment's
// m = sum_t q_t and p = sum_t x_t are gathered on the CUDA cores.  For m, one
// more warp reads each chunk's Q tile by columns (lane l keeps running sums of
// the bf16 pairs l, l + 32, ... of every row, in row order) and the issuer
// refills a Q buffer only after that warp has read it (barriers DQ and DQ2,
// one per Q buffer like LQ and LQ2, so that a phase never completes twice
// before its waiter looks).  For p,
// each drain thread keeps a running sum of the X row it drains (fp32, before
// rounding); one transposing butterfly at the end sums a warp's rows and the
// four lane quarters are added in a fixed order.
// Threads: the drain warps, the issuer, a load warp and, with XP, the
// column-sum warp.
template <bool XP>
constexpr int walk_threads() { return kThreadsTC + 32 + (XP ? 32 : 0); }

template <int D, bool NORM, bool XP>
__global__ void __launch_bounds__(walk_threads<XP>(), 1)
tc_walk_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mR, TCParams p) {
    using LY = Layout<D, NORM>;
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    // loads | MMA commits | drains | final wait | XP: p exchange, Q column sums
    enum { LQ, LK, LV, LQ2, LK2, CA, CXS, CX2, CQ, CP, DA, DX, DS, FIN, PX, DQ, DQ2, NBAR };
    __shared__ __align__(8) unsigned long long bars[NBAR];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const bool issuer = warp == kDrainWarps;
    // a load warp issues every tile load as soon as its buffer is free, so
    // that neither a load nor an MMA waits behind the other's waits
    const bool producer = warp == kDrainWarps + 1;
    const bool msum = XP && warp == kDrainWarps + 2;  // XP: the Q column-sum warp
    const int quarter = warp & 3;
    const int half = (warp >> 2) & 1;
    const int row = quarter * 32 + lane;  // TMEM lane / tile row owned by a drain thread
    int head, seg;
    const SegPlan plan{kL, p.nchunk, p.nseg, p.seglen};
    block_segment(plan, gridDim.y, (long long)blockIdx.y * gridDim.x + blockIdx.x, head, seg);
    const int c_begin = seg_chunk_begin(plan, seg);
    const int c_end = seg_chunk_begin(plan, seg + 1);
    const bool state_rows = warp < kDrainWarps && ((D == 128) || quarter < D / 32);  // drain warp holding rows < D
    constexpr int kStateWarps = (D == 128) ? kDrainWarps : 2 * (D / 32);

    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tQ{dsm + LY::Q, kL}, tK0{dsm + LY::K, kL}, tV{dsm + LY::V, kL};
    const Tile tA{dsm + LY::A, kL}, tX{dsm + LY::X, kL};
    const Tile tQ2{dsm + LY::Q2, kL}, tK2{dsm + LY::K2, kL};  // Q and K of odd chunks (two buffers each)
    const Tile tS{dsm + LY::S, D};
    // normalised walk only
    const Tile tAl{dsm + LY::Alo, kL}, tXl{dsm + LY::Xlo, kL};
    auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == DA || i == DX || i == PX) cnt = kDrainWarps;
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
    if (NORM) {
        // the ones block of [V | 1] (bf16 1.0), 16 bytes per thread and step
        const uint32_t one2 = 0x3F803F80u;
        for (uint32_t i = (uint32_t)tid; i < kL * 8u; i += blockDim.x)
            st_shared_v4(tV.base + tV.block_bytes() + i * 16u, one2, one2, one2, one2);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // tensor-memory regions (column offsets); NORM: P and C are D + 16
    // columns wide, P += X^T [V | 1] and C += Q^T [V | 1] leaving p and m in
    // their column D
    constexpr uint32_t kWide = NORM ? 32u * ((D + 16 + 31) / 32) : D;
    const uint32_t tA_ = tmem + 0;  // A, then X
    const uint32_t tS_ = tmem + 128;
    const uint32_t tP_ = tS_ + D;
    const uint32_t tC_ = tP_ + kWide;
    const uint32_t tPn_ = tP_ + D;  // NORM: p
    const uint32_t tM_ = tC_ + D;   // NORM: m
    static_assert(128 + D + 2 * kWide <= kTmemCols, "tensor-memory columns");
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int c128 = half * 64;      // this drain warp's columns in a 128-wide region
    const int cD = half * (D / 2);   // ... and in a D-wide region

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
    LoadLedger<5> loads(bar(0));  // LQ, LK, LV, LQ2, LK2
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
    // split drains (normalised walks): hi to one tile, lo to another
    auto drain128s = [&](uint32_t treg, const Tile& hi, const Tile& lo, bool mask) {
        uint32_t r[64];
        tmem_ld_cols<64>(treg + lane_off + c128, r);
        put_row32_split2(hi, lo, row, c128, r, mask);
        put_row32_split2(hi, lo, row, c128 + 32, r + 32, mask);
    };
    auto drainDs = [&](uint32_t treg, const Tile& hi, const Tile& lo) {
        uint32_t r[64];
        tmem_ld_cols<D / 2>(treg + lane_off + cD, r);
        put_row32_split2(hi, lo, row, cD, r, false);
        if (D == 128) put_row32_split2(hi, lo, row, cD + 32, r + 32, false);
    };

    const int nchunks = c_end - c_begin;
    // The first chunk's tiles start moving now (the barriers were initialised
    // before the first __syncthreads, so the load warp may use them).
    if (producer && lane == 0 && nchunks > 0) {
        issue_load(LQ, &mQ, tQ, c_begin);
        issue_load(LK, &mK, tK0, c_begin);
        issue_load(LV, &mV, tV, c_begin);
        if (nchunks > 1) {
            issue_load(LQ2, &mQ, tQ2, c_begin + 1);
            issue_load(LK2, &mK, tK2, c_begin + 1);
        }
        for (int a = 1; a < kAhead && a < nchunks; ++a) prefetch(c_begin + a);
    }

    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    constexpr uint32_t iSq = idesc_bf16(128, 128, false, false);   // 128 x 128, both K-major
    constexpr uint32_t iKK = idesc_bf16(128, D, false, false);     // N = D, both K-major
    constexpr uint32_t iKM = idesc_bf16(128, D, false, true);      // A K-major, B MN-major
    constexpr uint32_t iMM = idesc_bf16(128, D, true, true);       // both MN-major
    constexpr uint32_t iMME = idesc_bf16(128, NORM ? D + 16 : D, true, true);  // NORM: N = D + 16, [V | 1]

    constexpr bool kDeferP = LY::kSepX;
    // P += X^T V of chunk j (NORM: [P | p] += X_hi^T [V | 1] + X_lo^T [V | 1])
    auto issue_p = [&](int j) {
        for (int ks = 0; ks < kL / 16; ++ks)
            mma_bf16(tP_, tX.mnmaj(ks), tV.mnmaj(ks), iMME, (j > 0 || ks > 0) ? 1u : 0u);
        if (NORM)
            for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tP_, tXl.mnmaj(ks), tV.mnmaj(ks), iMME, 1);
        mma_commit(bar(CP));
    };

    if (issuer) {
        // ============================ issuer ============================
        if (lane == 0 && nchunks > 0) {
            int it = 0;
            for (; it < nchunks; ++it) {
                const uint32_t ph = it & 1, pph = (it + 1) & 1;
                // two Q and two K buffers: chunk it uses buffer it & 1
                const bool qodd = it & 1;
                const Tile& tQc = qodd ? tQ2 : tQ;
                const Tile& tK = qodd ? tK2 : tK0;
                const uint32_t qph = (uint32_t)((it >> 1) & 1);
                if (!wait_bar(qodd ? LQ2 : LQ, qph) || !wait_bar(qodd ? LK2 : LK, qph)) break;
                if (it > 0) {
                    if (!wait_bar(DX, pph)) break;  // TMEM A (X of the previous chunk) read
                    tc_fence_after();
                }
                // A = Q K^T
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQc.kmaj(ks), tK.kmaj(ks), iSq, ks > 0);
                mma_commit(bar(CA));
                if (kDeferP && it > 0) issue_p(it - 1);  // X and V of the previous chunk are in place
                if (it > 0) {
                    if (!wait_bar(DS, pph)) break;  // sS = S_local of this chunk; TMEM S read
                    tc_fence_after();
                }
                // S += K^T K
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tS_, tK.mnmaj(ks), tK.mnmaj(ks), iMM, (it > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bar(CXS));
                if (!wait_bar(DA, ph)) break;  // sA = A; TMEM A read
                tc_fence_after();
                // X = Q S_local + A K   (no S_local term on the segment's first chunk)
                if (it > 0)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQc.kmaj(ks), tS.kmaj(ks), iKK, ks > 0);
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tA_, tA.kmaj(ks), tK.mnmaj(ks), iKM, (it > 0 || ks > 0) ? 1u : 0u);
                if (NORM)
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tA_, tAl.kmaj(ks), tK.mnmaj(ks), iKM, 1);
                mma_commit(bar(CX2));
                if (!wait_bar(LV, ph)) break;
                tc_fence_after();
                // C += Q^T V  (NORM: [C | m] += Q^T [V | 1])
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tC_, tQc.mnmaj(ks), tV.mnmaj(ks), iMME, (it > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bar(CQ));
                if (!kDeferP) {
                    if (!wait_bar(DX, ph)) break;  // sX = X
                    tc_fence_after();
                    issue_p(it);
                }
            }
            if (kDeferP && it == nchunks && wait_bar(DX, (uint32_t)((nchunks - 1) & 1))) {
                tc_fence_after();
                issue_p(nchunks - 1);
            }
            if (!mma_wait_all(bar(FIN))) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else if (producer) {
        // ============================ loads ============================
        // V of chunk c once the previous chunk's X^T V (V's last reader)
        // completed; K of chunk c + 2 into its buffer once A K (of chunk c,
        // the buffer's last reader) completed, Q of chunk c + 2 once Q^T V
        // completed (and, with XP, the column-sum warp has read it); tiles
        // kAhead chunks ahead move into L2 early
        if (lane == 0) {
            for (int it = 0; it < nchunks; ++it) {
                const int c = c_begin + it;
                const uint32_t ph = it & 1, pph = (it + 1) & 1;
                if (kAhead > 0 && it + kAhead < nchunks) prefetch(c + kAhead);
                if (it > 0) {
                    if (!wait_bar(CP, pph)) break;
                    issue_load(LV, &mV, tV, c);
                }
                if (it + 2 < nchunks) {
                    const bool qodd = it & 1;
                    if (!wait_bar(CX2, ph)) break;
                    issue_load(qodd ? LK2 : LK, &mK, qodd ? tK2 : tK0, c + 2);
                    if (!wait_bar(CQ, ph)) break;
                    if (XP && !wait_bar(qodd ? DQ2 : DQ, (uint32_t)((it >> 1) & 1))) break;
                    issue_load(qodd ? LQ2 : LQ, &mQ, qodd ? tQ2 : tQ, c + 2);
                }
            }
            if (!loads.settle()) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else if (msum) {
        // ================ Q column sums (XP summary walk) ================
        // lane l: bf16 pairs l + 32 g of every row (columns 2l + 64g, + 1);
        // a warp's loads cover 128 contiguous bytes of one row
        float macc[D / 32] = {};
        for (int it = 0; it < nchunks; ++it) {
            const bool qodd = it & 1;
            if (!wait_bar(qodd ? LQ2 : LQ, (uint32_t)((it >> 1) & 1))) break;
            const Tile& tQc = qodd ? tQ2 : tQ;
            const uint32_t boff = (uint32_t)(lane & 3) << 2;
#pragma unroll
            for (int g = 0; g < D / 64; ++g)
#pragma unroll 1
                for (int r0 = 0; r0 < kL; r0 += 16) {
                    uint32_t v[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = ld_shared_u32(tQc.chunk(r0 + j, g, lane >> 2) + boff);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        macc[2 * g] += __uint_as_float(v[j] << 16);
                        macc[2 * g + 1] += __uint_as_float(v[j] & 0xFFFF0000u);
                    }
                }
            __syncwarp();
            if (lane == 0)
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(qodd ? DQ2 : DQ)) : "memory");
        }
        if (nchunks > 0 && !abort_flag) {
            const size_t R = (size_t)D * D + 2 * (size_t)D * D + 2 * (size_t)D;
            float* out = p.summ + ((size_t)head * p.nseg + seg) * R + 2 * (size_t)D * D;
#pragma unroll
            for (int g = 0; g < D / 64; ++g) {
                out[64 * g + 2 * lane] = macc[2 * g];
                out[64 * g + 2 * lane + 1] = macc[2 * g + 1];
            }
        }
    } else {
        // ========================== drain warps ==========================
        // XP: running sums of this thread's X row (columns cD .. cD + D/2)
        float xacc[XP ? D / 2 : 1] = {};
        for (int it = 0; it < nchunks; ++it) {
            const uint32_t ph = it & 1;
            const bool has_next = it + 1 < nchunks;
            if (!wait_bar(CA, ph)) break;
            tc_fence_after();
            if (NORM) drain128s(tA_, tA, tAl, true);
            else drain128(tA_, tA, true);  // A -> sA (masked)
            drained(DA);
            if (!wait_bar(CX2, ph)) break;
            tc_fence_after();
            if constexpr (NORM) {
                drainDs(tA_, tX, tXl);
                drained(DX);
            } else if constexpr (XP) {
                uint32_t xr[64];
                tmem_ld_cols<D / 2>(tA_ + lane_off + cD, xr);  // X -> sX, then into this row's sums
                put_row32(tX, row, cD, xr, false);
                if (D == 128) put_row32(tX, row, cD + 32, xr + 32, false);
                drained(DX);
#pragma unroll
                for (int j = 0; j < D / 2; ++j) xacc[j] += __uint_as_float(xr[j]);
            } else {
                drainD(tA_, tX);  // X -> sX
                drained(DX);
            }
            if (state_rows && has_next) {
                drainD(tS_, tS);  // S_local of the next chunk -> sS
                drained(DS);
            }
        }
        // ---- segment summary out: S | C | m | P | p records, fp32 ----
        if (state_rows && nchunks > 0 && wait_bar(CP, (nchunks - 1) & 1)) {
            tc_fence_after();
            const size_t R = (size_t)D * D + 2 * (size_t)D * D + 2 * (size_t)D;
            float* out = p.summ + ((size_t)head * p.nseg + seg) * R;
            // S, C, P leave through 32 x 32 boxes and bulk tensor stores (mR maps
            // the records as (3D + 2) rows of D floats: S at row 0, C at row D,
            // P at row 2D + 1).  Every tile is dead now: the last MMAs completed
            // and no load is in flight, so each warp stages its boxes in its own
            // 3 * D / 16 KB of the tile area.
            const uint32_t src[3] = {tS_, tC_, tP_};
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
            if (NORM && half == 0) {
                // m (after C) and p (after P), one value per state row
                const uint32_t mv = tmem_ld1(tM_ + lane_off);
                const uint32_t pv = tmem_ld1(tPn_ + lane_off);
                tmem_ld_wait();
                out[2 * (size_t)D * D + row] = __uint_as_float(mv);
                out[3 * (size_t)D * D + D + row] = __uint_as_float(pv);
            }
        }
        if (XP && nchunks > 0 && wait_bar(CP, (nchunks - 1) & 1)) {
            // p of the segment: each warp leaves the column sums of its 32 rows
            // in the (dead) S tile, and the quarter-0 warps add the four quarters
            float pacc[2];
            {
                uint32_t xb[32];
#pragma unroll
                for (int g = 0; g < D / 64; ++g) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) xb[j] = __float_as_uint(xacc[32 * g + j]);
                    pacc[g] = warp_colsum32(xb, lane);
                }
            }
            float* px = reinterpret_cast<float*>(dsm_raw + (dsm + LY::S - smem_u32(dsm_raw)));
            px[quarter * D + cD + lane] = pacc[0];
            if (D == 128) px[quarter * D + cD + 32 + lane] = pacc[1];
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(PX)) : "memory");
            if (quarter == 0 && wait_bar(PX, 0)) {
                const size_t R = (size_t)D * D + 2 * (size_t)D * D + 2 * (size_t)D;
                float* out = p.summ + ((size_t)head * p.nseg + seg) * R;
#pragma unroll
                for (int j = 0; j < D / 2; j += 32) {
                    const int c = cD + j + lane;
                    out[3 * (size_t)D * D + D + c] = ((px[c] + px[D + c]) + px[2 * D + c]) + px[3 * D + c];
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


// ------------------------------------------------------- cross products ----
// out[b] = alpha base[b] + A[b] B[b] for a batch of fp32 D x D matrices (the
// scan's S_<r C_r terms).  Each fp32 operand x is split into bf16 parts
// hi = bf16(x), lo = bf16(x - hi), and the product is taken as
// A_hi B_hi + A_hi B_lo + A_lo B_hi on the tensor cores (fp32 accumulation),
// which keeps about 16 significant bits of every operand.  The optional
// column outx[b] = alpha basex[b] + A[b] bx[b] (the normaliser's matrix-vector
// term) is formed in fp32 on the CUDA cores from the A rows as they arrive.
template <int D>
struct CrossLayout {
    static constexpr uint32_t kA = 128u * D * 2u;  // A tiles keep 128 rows (MMA M = 128)
    static constexpr uint32_t kB = (uint32_t)D * D * 2u;
    static constexpr uint32_t Ahi = 0, Alo = kA, Bhi = 2 * kA, Blo = 2 * kA + kB;
    static constexpr uint32_t kBytes = 2 * kA + 2 * kB;
};

template <int D>
__global__ void __launch_bounds__(256, 1) tc_cross_kernel(CrossArgs a) {
    using CL = CrossLayout<D>;
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    __shared__ __align__(8) unsigned long long bar_mma;
    __shared__ uint32_t tmem_slot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const long long b = blockIdx.x;
    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tAh{dsm + CL::Ahi, 128}, tAl{dsm + CL::Alo, 128}, tBh{dsm + CL::Bhi, D}, tBl{dsm + CL::Blo, D};
    const float* A = a.A + b * a.sA;
    const float* B = a.B + b * a.sB;
    constexpr uint32_t kCols = D < 32 ? 32 : D;

    if (tid == 0) {
        mbar_init(smem_u32(&bar_mma), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // operands: A rows a (K-major, rows >= D zero), B rows b (read MN-major).
    // All of a thread's loads are issued before any conversion so that they
    // overlap (the shared-memory stores are compiler barriers).
    constexpr int kPer = D * D / 4 / 256;  // float4s of one D x D matrix per thread
    {
        float4 xa[kPer], xb[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = tid + j * 256;
            xa[j] = __ldg(reinterpret_cast<const float4*>(A) + i);
            xb[j] = __ldg(reinterpret_cast<const float4*>(B) + i);
        }
        if (a.bx && a.outx) {
            // D / 4 consecutive lanes hold one row of A (256 is a multiple of
            // D / 4, so a lane keeps its column quad for every j)
            const float4 m = __ldg(reinterpret_cast<const float4*>(a.bx + b * a.sbx) + (tid % (D / 4)));
            const float* basex = a.basex ? a.basex + b * a.sbasex : nullptr;
            float* outx = a.outx + b * a.soutx;
            const float sc = a.pscale ? a.pscale[(a.pscale_off + b) % a.pscale_mod] : 1.f;
            float part[kPer];
#pragma unroll
            for (int j = 0; j < kPer; ++j)
                part[j] = fmaf(xa[j].x, m.x, fmaf(xa[j].y, m.y, fmaf(xa[j].z, m.z, xa[j].w * m.w)));
#pragma unroll
            for (int o = D / 8; o > 0; o >>= 1)
#pragma unroll
                for (int j = 0; j < kPer; ++j) part[j] += __shfl_xor_sync(0xffffffffu, part[j], o);
            if (tid % (D / 4) == 0)
#pragma unroll
                for (int j = 0; j < kPer; ++j) {
                    const int r = (tid + j * 256) / (D / 4);
                    outx[r] = fmaf(a.alpha, basex ? basex[r] : 0.f, sc * part[j]);
                }
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = tid + j * 256;
            const int r = i / (D / 4), c = (i % (D / 4)) * 4;
            put4_split(tAh, tAl, r, c, xa[j]);
            put4_split(tBh, tBl, r, c, xb[j]);
        }
        if (D < 128)
            for (int i = D * D / 4 + tid; i < 128 * D / 4; i += 256)
                put4_split(tAh, tAl, i / (D / 4), (i % (D / 4)) * 4, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    constexpr uint32_t idesc = idesc_bf16(128, D, false, true);
    if (tid == 0) {
        for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tmem, tAh.kmaj(ks), tBh.mnmaj(ks), idesc, ks > 0);
        for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tmem, tAh.kmaj(ks), tBl.mnmaj(ks), idesc, 1);
        for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tmem, tAl.kmaj(ks), tBh.mnmaj(ks), idesc, 1);
        mma_commit(smem_u32(&bar_mma));
    }
    __syncwarp();
    // this thread's part of base (row `row`, columns cD .. cD + D/2), loaded
    // while the products run
    const bool out_rows = (D == 128) || quarter < D / 32;
    const int cD = half * (D / 2);
    float4 bv[D / 8];
    if (out_rows) {
        const float* base = a.base + b * a.sbase;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) bv[j] = __ldg(reinterpret_cast<const float4*>(base + (size_t)row * D + cD) + j);
    }
    // bounded wait for the products
    bool ok = mbar_try(smem_u32(&bar_mma), 0);
    if (!ok) {
        const unsigned long long t0 = globaltimer();
        while (!(ok = mbar_try(smem_u32(&bar_mma), 0)))
            if (globaltimer() - t0 > kWaitNs) break;
        if (!ok && lane == 0) atomicExch(a.status, (int)kDevWaitTimeout);
    }
    tc_fence_after();
    if (ok && out_rows) {
        uint32_t r[64];
        tmem_ld_cols<D / 2>(tmem + ((uint32_t)(quarter * 32) << 16) + cD, r);
        float* out = a.out + b * a.sout;
        const float sc = a.pscale ? a.pscale[(a.pscale_off + b) % a.pscale_mod] : 1.f;
#pragma unroll
        for (int j = 0; j < D / 2; j += 4) {
            const float4 x = bv[j / 4];
            *reinterpret_cast<float4*>(out + (size_t)row * D + cD + j) =
                make_float4(fmaf(a.alpha, x.x, sc * __uint_as_float(r[j])),
                            fmaf(a.alpha, x.y, sc * __uint_as_float(r[j + 1])),
                            fmaf(a.alpha, x.z, sc * __uint_as_float(r[j + 2])),
                            fmaf(a.alpha, x.w, sc * __uint_as_float(r[j + 3])));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
}

template <int D>
cudaError_t launch_cross_t(const CrossArgs& a, cudaStream_t s) {
    const size_t smem = CrossLayout<D>::kBytes + 1024;
    auto kern = tc_cross_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<a.nb, 256, smem, s>>>(a);
    note_launches(1);
    return cudaGetLastError();
}


template <int D, bool NORM, bool XP = false>
cudaError_t launch_t(const void* Q, const void* K, const void* V, float* summ, int BH, int T, SegPlan plan, int* status,
                     cudaStream_t s) {
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mk, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mv, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64))
        return cudaErrorInvalidValue;
    // mR: the segment summary records as (3D + 2) rows of D floats, 32 x 32 boxes
    CUtensorMap mr;
    if (!make_map(&mr, summ, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, 3 * D + 2, BH * plan.nseg, 32, 32))
        return cudaErrorInvalidValue;
    TCParams prm{T, plan.nseg, plan.nchunk, plan.seglen, summ, status};
    const size_t smem = Layout<D, NORM>::kBytes + 1024;
    auto kern = tc_walk_kernel<D, NORM, XP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.nseg, BH);
    kern<<<grid, walk_threads<XP>(), smem, s>>>(mq, mk, mv, mr, prm);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int d, int dv, int dtype, int normalized, int device) {
    if (d != dv || (d != 64 && d != 128) || dtype != 1) return false;
    if (normalized && d != 64) return false;  // the split operands fit in shared memory at d = 64
    static int cached[64] = {0};  // 0 unknown, 1 yes, 2 no
    if (device < 0 || device >= 64) return false;
    if (!cached[device]) {
        cudaDeviceProp prop;
        bool ok = cudaGetDeviceProperties(&prop, device) == cudaSuccess && prop.major == 10 && prop.minor == 3 &&
                  encode_fn() != nullptr;
        cached[device] = ok ? 1 : 2;
    }
    return cached[device] == 1;
}

cudaError_t launch_tc_walk(int mode, const void* Q, const void* K, const void* V, float* O, const float* prefix,
                           float* summ, int BH, int T, int d, int dv, int normalized, SegPlan plan, int* status,
                           cudaStream_t s, bool with_p) {
    if (BH == 0 || plan.nseg == 0) return cudaSuccess;
    if (plan.granule != kL || d != dv) return cudaErrorInvalidValue;
    // outputs: the walk pipelined across chunks (hla2_tc_out.cu)
    if (mode == 1) return launch_tc_out(Q, K, V, O, prefix, BH, T, d, dv, normalized != 0, plan, status, s);
    if (normalized) {
        if (d != 64) return cudaErrorInvalidValue;
        return launch_t<64, true>(Q, K, V, summ, BH, T, plan, status, s);
    }
    if (with_p) {
        if (d == 128) return launch_t<128, false, true>(Q, K, V, summ, BH, T, plan, status, s);
        if (d == 64) return launch_t<64, false, true>(Q, K, V, summ, BH, T, plan, status, s);
        return cudaErrorInvalidValue;
    }
    if (d == 128) return launch_t<128, false>(Q, K, V, summ, BH, T, plan, status, s);
    if (d == 64) return launch_t<64, false>(Q, K, V, summ, BH, T, plan, status, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_tc_cross(const CrossArgs& a, cudaStream_t s) {
    if (a.nb == 0) return cudaSuccess;
    if (a.d != a.dv) return cudaErrorInvalidValue;
    if (a.d == 128) return launch_cross_t<128>(a, s);
    if (a.d == 64) return launch_cross_t<64>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace hla2
