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
//   alpha: A, then W (each packed to bf16 in place, the A operand of A K and
//          of W V)          beta: X (= Q S0 + A K), then O
// so that X and O never wait for alpha, and nothing on the chain waits for
// shared memory: the drains of A and W stay in tensor memory, X goes to its
// own tile (the B operand of W and the A operand of X^T V), and O leaves
// through staging boxes that the next drains do not touch.  Q is
// double-buffered, and each chunk's V starts loading as soon as the previous
// O has completed (loads come from their own warp).  The bf16 operand copies of S0 and P0 share one tile: S0
// is read by Q S0 early in a chunk, P0 by Q P0 late in it.
//
// Precision: products take bf16 operands with fp32 accumulation; the running
// S and P stay fp32 in tensor memory.  On a head's first chunk, where an
// output can be a single product (t = 0 gives (q.k)^2 v) and roundings do not
// average out, X and W are split into bf16 hi + lo parts (W = Q X_hi^T +
// Q X_lo^T, O = W_hi V + W_lo V; W_lo packed next to W_hi in alpha).
//
// NORM (ratio-normalised variant, D = 64): o_t = q_t^T P_t / q_t^T p_t with
// p = S m - h.  The fp32 values that feed a product are split into bf16 hi +
// lo and both parts enter it (A, X, W, P0, p0), which keeps about 16
// significant bits of those operands; S0 is rounded to bf16 alone (its
// rounding stays two orders below the 1e-4 bound on the outputs, where any
// of the others would come within a factor of three of it or exceed it).
// p and the denominators ride along as one more value column: V is read as
// [V | 1] and P0 as [P0 | p0] (N = 80 products, the extra 64-column block of
// each operand holding the ones or p0), so P += X^T [V | 1] grows p in P's
// column D and O = Q [P0 | p0] + W [V | 1] leaves the denominators in O's
// column D.  X_lo sits in the X tile's second 64-column block.
//
// DECAY (exponentially decayed operator, gamma in the tensor-core range):
// the same pipeline on the decayed chunk form of hla2_decay_tc.cu.  A~ =
// tril(Q K^T) g^{-(i+1)} (column factors in the pack of A, split on a head's
// first chunk), X' = Q S0 + A~ K drained as sX = g^{2L-1-t} X', W~ =
// g^{-2L} tril(Q sX^T) split into hi + lo on every chunk (packed by every
// drain warp at D = 128), o_t = g^{2(t+1)} O'_t in the O drain; the beta
// warps scale K in place to K' = diag(sqrt(b)) K once A and A~ K have read it
// (S += K'^T K' then waits for them), and multiply tensor-memory P by
// g^{2L} when they hand P0 over and S by g^{L} after they hand S0 over.
#include "hla2_tc_common.cuh"

namespace hla2 {
namespace {

struct OutParams {
    int T, nseg, nchunk, seglen;
    const float* prefix;  // segment prefix records (S and P read)
    int* status;
    float lg;  // DECAY: log2(gamma)
};

template <int D, bool NORM>
struct OutLayout {
    static constexpr uint32_t kTok = kL * D * 2;  // Q, K, V tiles
    static constexpr uint32_t kSq = kL * kL * 2;  // X tile (and, at D = 128, the first O staging box of each warp)
    static constexpr uint32_t kSt = D * D * 2;    // S0 / P0 tile
    // O staging (the other box of each warp at D = 128, the only one at
    // D = 64; eight 4 KB boxes) and, on a head's first chunk, X_lo (kL x D)
    static constexpr uint32_t kO = kSq;
    // NORM: the V tile's second block holds the ones ([V | 1]), the S0 / P0
    // tile's second block p0 ([P0 | p0], column 0), then the same pair for
    // the lo parts of P0 and p0; X_lo in the X tile's second block
    static constexpr uint32_t Q0 = 0, Q1 = kTok, K = 2 * kTok, V = 3 * kTok, X = (NORM ? 5 : 4) * kTok;
    static constexpr uint32_t O = X + kSq, SP = O + kO, XL = X + kL * 128u;
    static constexpr uint32_t SPL = SP + 2 * kSt;
    static constexpr uint32_t kBytes = NORM ? SPL + 2 * kSt : SP + kSt;
    static_assert(!NORM || D == 64, "the normalised walk's extended tiles fit at D = 64");
};

// Warp roles: the drain warps move results out of tensor memory (warp w
// owns lane quarter w % 4 and, in every region, a share of the columns:
// 32 of a D-wide region, 128 / (D / 32) of alpha), one warp (lane 0) issues
// every MMA, another every tile load, so that MMA issue never waits behind a
// busy bulk-copy queue; the roles meet only on mbarriers.  There are D / 8
// drain warps (16 at D = 128), so that each drain is short.  At D = 128 they
// form two groups of eight (two warps per lane quarter): the alpha warps
// pack A and W, the beta warps drain X, O and the state, so that packing the
// next chunk's A never waits behind the previous chunk's O stores.  At D = 64
// every drain warp does both, except in the normalised walk (D = 64, bf16
// hi + lo packs twice as long), which has four warps per quarter: two of them
// also drain X, O and the state, and all four pack A and W, one 32-column
// group each (the split packs are the longest steps of its chunk).  Columns
// go in groups of 32: an alpha warp takes kAG groups of alpha, a beta warp
// kBG groups of each D-wide region.
template <int D, bool NORM>
struct OutRoles {
    static constexpr int kParts = NORM ? 4 : D / 32;   // drain warps per lane quarter
    static constexpr int kDrain = 4 * kParts;          // drain warps
    static constexpr bool kSplit = kParts == 4;        // alpha and beta warps apart
    static constexpr int kAPer = kSplit ? kParts / 2 : kParts;  // alpha warps per quarter
    static constexpr int kBPer = kSplit ? kParts / 2 : kParts;  // beta warps per quarter
    static constexpr int kBeta0 = kParts - kBPer;               // first beta part
    static constexpr int kAG = 4 / kAPer;              // alpha groups per alpha warp
    static constexpr int kBG = (D / 32) / kBPer;       // D-wide groups per beta warp
    static constexpr int kAlpha = 4 * kAPer, kBeta = 4 * kBPer;
    static constexpr int kState = (D / 32) * kBPer;    // beta warps holding state rows (< D)
    static constexpr int kThreads = (kDrain + 2) * 32;
};

// 16 fp32 TMEM columns of this thread's lane, stored / loaded with one call.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

template <int D, bool NORM, bool DECAY>
__global__ void __launch_bounds__(OutRoles<D, NORM>::kThreads, 1)
tc_out_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
              const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mO,
              const __grid_constant__ CUtensorMap mR, OutParams p) {
    using LY = OutLayout<D, NORM>;
    using RO = OutRoles<D, NORM>;
    constexpr int NDW = RO::kDrain, AG = RO::kAG, BG = RO::kBG;
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    // loads | MMA commits | drains | the S += K^T K commit | final wait |
    // drain warp w's prefix boxes
    // (DK: DECAY, K scaled in place by the beta warps)
    enum { LQ0, LQ1, LK, LV, CA_, CQS, CX, CW, CP, CO, DA, DP, DX, DW, DO, DS, CK, DK, FIN, PB, NBAR = PB + NDW };
    static_assert(!(NORM && DECAY), "one operator per walk");
    __shared__ __align__(8) unsigned long long bars[NBAR];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const bool drainer = warp < NDW;
    const bool issuer = warp == NDW;
    const bool producer = warp == NDW + 1;
    const int quarter = warp & 3;
    const int part = (warp >> 2) % RO::kParts;
    const int row = quarter * 32 + lane;  // TMEM lane / tile row owned by a drain thread
    int head, seg;
    const SegPlan plan{kL, p.nchunk, p.nseg, p.seglen};
    block_segment(plan, gridDim.y, (long long)blockIdx.y * gridDim.x + blockIdx.x, head, seg);
    const int c_begin = seg_chunk_begin(plan, seg);
    const int c_end = seg_chunk_begin(plan, seg + 1);
    const int nchunks = c_end - c_begin;
    const bool alpha_w = drainer && part < RO::kAPer;      // packs A and W
    const bool beta_w = drainer && part >= RO::kBeta0;     // drains X, O and the state
    const int aw = part, bw = part - RO::kBeta0;           // index among its kind in a quarter
    const bool state_rows = beta_w && quarter < D / 32;  // beta warp holding rows < D

    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tQ0{dsm + LY::Q0, kL}, tQ1{dsm + LY::Q1, kL}, tK{dsm + LY::K, kL}, tV{dsm + LY::V, kL};
    const Tile tX{dsm + LY::X, kL}, tO{dsm + LY::O, kL}, tSP{dsm + LY::SP, D};
    // NORM tiles (X_lo, the lo part of P0)
    const Tile tXL{dsm + LY::XL, kL}, tSPL{dsm + LY::SPL, D};
    auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == DA) cnt = NORM ? RO::kDrain : RO::kAlpha;  // NORM: every drain warp packs A
            // NORM, and DECAY at D = 128: every drain warp packs (split) W
            if (i == DW) cnt = (NORM || (DECAY && D == 128)) ? RO::kDrain : RO::kAlpha;
            if (i == DX || i == DO || i == DK) cnt = RO::kBeta;
            if (i == DS || i == DP) cnt = RO::kState;
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
        // the ones block of [V | 1] (bf16 1.0) and the zeroed p0 blocks of
        // [P0 | p0] (hi and lo), 16 bytes per thread and step
        const uint32_t one2 = 0x3F803F80u;
        for (uint32_t i = (uint32_t)tid; i < kL * 8u; i += blockDim.x)
            st_shared_v4(tV.base + tV.block_bytes() + i * 16u, one2, one2, one2, one2);
        for (uint32_t i = (uint32_t)tid; i < D * 8u; i += blockDim.x) {
            st_shared_v4(tSP.base + tSP.block_bytes() + i * 16u, 0u, 0u, 0u, 0u);
            st_shared_v4(tSPL.base + tSPL.block_bytes() + i * 16u, 0u, 0u, 0u, 0u);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // NORM: beta and P are D + 16 columns wide (O and P with the extra column)
    constexpr uint32_t kWide = NORM ? 32u * ((D + 16 + 31) / 32) : D;
    const uint32_t tAl_ = tmem + 0;                 // alpha: A, then W (packed bf16 in place; W_lo too on a first chunk)
    const uint32_t tBe_ = tmem + 128;               // beta: Q S0 + A K = X, then O
    const uint32_t tS_ = tmem + 128 + kWide;        // running S
    const uint32_t tP_ = tmem + 128 + kWide + D;    // running P
    const uint32_t tPn_ = tP_ + D;                  // NORM: running p (P's extra column)
    const uint32_t tDen_ = tBe_ + D;                // NORM: the chunk's denominators (O's extra column)
    static_assert(128 + 2 * kWide + D <= kTmemCols, "tensor-memory columns");
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int cD = part * 32;  // this drain warp's columns of the segment prefix (prologue)
    auto acol = [&](int g) { return (aw * AG + g) * 32; };  // alpha group g of this alpha warp
    auto bcol = [&](int g) { return (bw * BG + g) * 32; };  // D-wide group g of this beta warp
    // DECAY: g^n, and the real length of chunk c (the last one may be short)
    auto gp = [&](float n) { return exp2f(n * p.lg); };
    auto clen = [&](int c) { return (float)min(kL, p.T - c * kL); };

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
    // every tile load is issued by the producer's lane 0, which settles them
    // (waits for the last of each barrier) before the CTA exits
    LoadLedger<4> loads(bar(0));  // LQ0, LQ1, LK, LV
    static_assert(LQ0 == 0 && LQ1 == 1 && LK == 2 && LV == 3, "load barriers first");
    auto issue_load = [&](int b, const CUtensorMap* map, const Tile& t, int chunk) {
        loads.note(b);
        mbar_expect_tx(bar(b), kTileBytes);
#pragma unroll
        for (int k = 0; k < D / 64; ++k) tma_load_3d(t.base + k * t.block_bytes(), map, k * 64, chunk * kL, head, bar(b));
    };
    // a drain warp announces that its share of a region is done (after
    // shared-memory writes the async proxy will read: with a proxy fence)
    auto drained = [&](int b) {
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(b)) : "memory");
    };
    // ... after tensor-memory writes only (the packs of alpha)
    auto packed = [&](int b) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(b)) : "memory");
    };
    // this beta warp's groups of a D-wide fp32 region -> bf16 tile rows
    // (DECAY, wb: the tensor-memory copy is then multiplied by `decay` for
    // the next update)
    auto drainD = [&](uint32_t treg, const Tile& t, bool split, float decay = 1.f, bool wb = false) {
#pragma unroll
        for (int g = 0; g < BG; ++g) {
            uint32_t r[32];
            tmem_ld32(treg + lane_off + bcol(g), r);
            tmem_ld_wait();
            if (NORM && split) put_row32_split2(t, tSPL, row, bcol(g), r, false);  // t is the S0 / P0 tile
            else put_row32(t, row, bcol(g), r, false);
            if (DECAY && wb) {
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * decay);
                tmem_st32(treg + lane_off + bcol(g), r);
            }
        }
        if (DECAY && wb) tmem_st_wait();
    };
    // DECAY: this beta warp's groups of a D-wide region multiplied by `decay` in place
    auto rescale = [&](uint32_t treg, float decay) {
#pragma unroll
        for (int g = 0; g < BG; ++g) {
            uint32_t r[32];
            tmem_ld32(treg + lane_off + bcol(g), r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * decay);
            tmem_st32(treg + lane_off + bcol(g), r);
        }
        tmem_st_wait();
    };
    // NORM: p0 (one fp32 per state row d) into column D of [P0 | p0], hi and
    // lo (row d, first element of the second block)
    auto put_p0 = [&](float x) {
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(tSP.chunk(row, 1, 0)),
                     "h"(*reinterpret_cast<const unsigned short*>(&h)) : "memory");
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(tSPL.chunk(row, 1, 0)),
                     "h"(*reinterpret_cast<const unsigned short*>(&l)) : "memory");
    };
    // Packed bf16 operands in alpha: each 32-column group [c0, c0 + 32) of
    // alpha (A, or W and on a first chunk also W_lo) is packed in place, its
    // pairs into [c0, c0 + 16) and the lo parts into [c0 + 16, c0 + 32), by the
    // alpha warp that has itself just read the group, so no other warp's
    // pending read is overwritten.  K-step ks (16 tokens) of the product
    // reads 8 packed columns.
    auto pk_col = [](int ks) -> uint32_t { return (uint32_t)(32 * ((16 * ks) / 32) + ((16 * ks) % 32) / 2); };
    // this alpha warp's groups -> bf16 pairs (masked to columns <= row),
    // optionally with the lo parts, written back packed; `one` packs the
    // single group `part` instead (NORM's W, which every drain warp packs)
    // (DECAY: each value times s and, when colfac is set, its column factor
    // g^{-(col+1)}, stepped from the group's first column by 1 / g, before
    // the mask and the rounding)
    const float ginv = DECAY ? exp2f(-p.lg) : 1.f;
    auto pack_alpha = [&](bool split, bool one = false, bool colfac = false, float s = 1.f) {
        if (!split && AG == 2) {
            // both groups' loads in flight before the one wait (the common case)
            uint32_t r0[32], r1[32];
            tmem_ld32(tAl_ + lane_off + acol(0), r0);
            tmem_ld32(tAl_ + lane_off + acol(1), r1);
            tmem_ld_wait();
            auto pack16 = [&](const uint32_t (&r)[32], int c0) {
                uint32_t hi[16];
                float cf = (DECAY && colfac) ? exp2f(-(float)(c0 + 1) * p.lg) * s : s;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float x0 = __uint_as_float(r[2 * j]), x1 = __uint_as_float(r[2 * j + 1]);
                    if constexpr (DECAY) {
                        x0 *= cf;
                        if (colfac) cf *= ginv;
                        x1 *= cf;
                        if (colfac) cf *= ginv;
                    }
                    if (c0 + 2 * j > row) x0 = 0.f;
                    if (c0 + 2 * j + 1 > row) x1 = 0.f;
                    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                    hi[j] = *reinterpret_cast<const uint32_t*>(&h);
                }
                tmem_st16(tAl_ + lane_off + (uint32_t)c0, hi);
            };
            pack16(r0, acol(0));
            pack16(r1, acol(1));
            tmem_st_wait();
            return;
        }
#pragma unroll
        for (int g = 0; g < AG; ++g) {
            if (one && g > 0) break;
            const int c0 = one ? part * 32 : acol(g);
            uint32_t r[32];
            tmem_ld32(tAl_ + lane_off + c0, r);
            tmem_ld_wait();
            uint32_t hl[32];  // the pairs, then (split) the lo parts
            float cf = (DECAY && colfac) ? exp2f(-(float)(c0 + 1) * p.lg) * s : s;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float x0 = __uint_as_float(r[2 * j]), x1 = __uint_as_float(r[2 * j + 1]);
                if constexpr (DECAY) {
                    x0 *= cf;
                    if (colfac) cf *= ginv;
                    x1 *= cf;
                    if (colfac) cf *= ginv;
                }
                if (c0 + 2 * j > row) x0 = 0.f;
                if (c0 + 2 * j + 1 > row) x1 = 0.f;
                const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                hl[j] = *reinterpret_cast<const uint32_t*>(&h);
                hl[16 + j] = pack_bf16(x0 - __low2float(h), x1 - __high2float(h));
            }
            if (split) tmem_st32(tAl_ + lane_off + (uint32_t)c0, hl);
            else tmem_st16(tAl_ + lane_off + (uint32_t)c0, hl);
        }
        tmem_st_wait();
    };

    // ---- prologue: the first tiles start moving while the drain warps load
    // the segment prefix (S0, P0) into tensor memory and S0 into its tile ----
    if (producer && lane == 0 && nchunks > 0) {
        issue_load(LQ0, &mQ, tQ0, c_begin);
        issue_load(LK, &mK, tK, c_begin);
        issue_load(LV, &mV, tV, c_begin);
        if (nchunks > 1) issue_load(LQ1, &mQ, tQ1, c_begin + 1);
    }
    if (drainer && quarter < D / 32 && part < D / 32 && nchunks > 0) {  // rows < D, one box of columns each
        // S0 (record row 0) and P0 (record row 2D + 1) arrive as this warp's
        // 32 x 32 fp32 box by bulk tensor loads (mR maps the records as
        // (3D + 2) rows of D floats) into a private staging area in the X / O
        // tiles, which nothing else touches before the first chunk
        const int rec = head * p.nseg + seg;
        const uint32_t stage = dsm + LY::X + (uint32_t)warp * 4096u;
        LoadLedger<1> boxes(bar(PB + warp));
#pragma unroll 1
        for (int m = 0; m < 2; ++m) {
            if (lane == 0) {
                boxes.note(0);
                fence_proxy_async();
                mbar_expect_tx(bar(PB + warp), 4096u);
                tma_load_3d(stage, &mR, cD, (m == 0 ? 0 : 2 * D + 1) + quarter * 32, rec, bar(PB + warp));
            }
            __syncwarp();
            if (!wait_bar(PB + warp, (uint32_t)m)) break;
            uint32_t r[32];
            box32_read(stage, lane, r);
            if (m == 0) {  // bf16 S0; P0 follows once Q S0 has read it
                put_row32(tSP, row, cD, r, false);
                if constexpr (DECAY) {  // TMEM S decayed over the first chunk (the P0 drain decays P)
                    const float f = gp(clen(c_begin));
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
                }
            }
            tmem_st32((m == 0 ? tS_ : tP_) + lane_off + cD, r);
            __syncwarp();  // every lane has read the box before the next load reuses it
        }
        if (lane == 0 && !boxes.settle()) atomicExch(p.status, (int)kDevWaitTimeout);
        if (NORM && part == 0 && quarter < D / 32) {
            // p0 of the prefix (record slot after P), one value per state row
            const size_t R = 3 * (size_t)D * D + 2 * (size_t)D;
            const float p0 = p.prefix[((size_t)head * p.nseg + seg) * R + 3 * (size_t)D * D + D + row];
            tmem_st1(tPn_ + lane_off, __float_as_uint(p0));
        }
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
    constexpr int NE = NORM ? D + 16 : D;                           // NORM: [V | 1], [P0 | p0]
    constexpr uint32_t iKME = idesc_bf16(128, NE, false, true);     // N = NE, A K-major, B MN-major
    constexpr uint32_t iMME = idesc_bf16(128, NE, true, true);      // N = NE, both MN-major

    if (issuer) {
        // ============================ issuer ============================
        if (lane == 0 && nchunks > 0) {
            for (int it = 0; it < nchunks; ++it) {
                const int c = c_begin + it;
                const uint32_t ph = it & 1, pph = (it + 1) & 1;
                const bool first = c == 0;  // S0 = P0 = 0; X, W split
                const Tile& tQ = (it & 1) ? tQ1 : tQ0;
                if (!wait_bar((it & 1) ? LQ1 : LQ0, (uint32_t)((it >> 1) & 1)) || !wait_bar(LK, ph)) break;
                // alpha is free once the previous O has read W from it
                if (it > 0 && !wait_bar(CO, pph)) break;
                tc_fence_after();
                // A = Q K^T
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tAl_, tQ.kmaj(ks), tK.kmaj(ks), iSq, ks > 0);
                mma_commit(bar(CA_));
                if (it > 0) {
                    // beta free (O read out) and S0 of this chunk in its tile
                    if (!wait_bar(DO, pph) || !wait_bar(DS, pph)) break;
                    tc_fence_after();
                }
                // X = Q S0 (S0 symmetric: its tile read K-major)
                if (!first) {
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tBe_, tQ.kmaj(ks), tSP.kmaj(ks), iKK, ks > 0);
                }
                mma_commit(bar(CQS));
                if (!wait_bar(DA, ph)) break;  // A packed in alpha
                tc_fence_after();
                // X += A K  (A from tensor memory)
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16_tmem_a(tBe_, tAl_ + pk_col(ks), tK.mnmaj(ks), iKM, (!first || ks > 0) ? 1u : 0u);
                if (NORM || (DECAY && first))  // + A_lo K
                    for (int ks = 0; ks < kL / 16; ++ks)
                        mma_bf16_tmem_a(tBe_, tAl_ + pk_col(ks) + 16u, tK.mnmaj(ks), iKM, 1);
                mma_commit(bar(CX));
                // S += K^T K after A K: it then runs beside the X drain, not
                // beside the pack of A, whose tensor-memory traffic it slowed
                // (K's last reader now, so the next K waits for CK).  DECAY:
                // S += K'^T K' once the beta warps have scaled K, after W
                if (!DECAY) {
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tS_, tK.mnmaj(ks), tK.mnmaj(ks), iMM, 1);
                    mma_commit(bar(CK));
                }
                if (!wait_bar(DX, ph)) break;  // sX = X (and sO = X_lo on a head's first chunk); beta free
                tc_fence_after();
                // W = Q X^T (+ Q X_lo^T) into alpha (A there was read by A K)
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tAl_, tQ.kmaj(ks), tX.kmaj(ks), iSq, ks > 0);
                if (first || NORM)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tAl_, tQ.kmaj(ks), (NORM ? tXL : tO).kmaj(ks), iSq, 1);
                mma_commit(bar(CW));
                if (DECAY) {
                    // S += K'^T K', K' = diag(sqrt(b)) K scaled in place by the beta warps
                    if (!wait_bar(DK, ph)) break;
                    tc_fence_after();
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tS_, tK.mnmaj(ks), tK.mnmaj(ks), iMM, 1);
                    mma_commit(bar(CK));
                }
                // P += X^T V once P0 of this chunk has left TMEM P
                if (!wait_bar(LV, ph) || !wait_bar(DP, ph)) break;
                tc_fence_after();
                for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tP_, tX.mnmaj(ks), tV.mnmaj(ks), iMME, 1);
                if (NORM)  // [P | p] += X_lo^T [V | 1]
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tP_, tXL.mnmaj(ks), tV.mnmaj(ks), iMME, 1);
                mma_commit(bar(CP));
                if (!wait_bar(DW, ph)) break;  // W packed in alpha (and W_lo on a head's first chunk)
                tc_fence_after();
                // O = Q P0 + W V (+ W_lo V)  (W from tensor memory)
                // (NORM: [O | den] = Q [P0 | p0] (hi, lo) + W [V | 1] (hi, lo))
                if (!first) {
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tBe_, tQ.kmaj(ks), tSP.mnmaj(ks), iKME, ks > 0);
                    if (NORM)
                        for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tBe_, tQ.kmaj(ks), tSPL.mnmaj(ks), iKME, 1);
                }
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16_tmem_a(tBe_, tAl_ + pk_col(ks), tV.mnmaj(ks), iKME, (!first || ks > 0) ? 1u : 0u);
                if (first || NORM || DECAY)
                    for (int ks = 0; ks < kL / 16; ++ks)
                        mma_bf16_tmem_a(tBe_, tAl_ + pk_col(ks) + 16u, tV.mnmaj(ks), iKME, 1);
                mma_commit(bar(CO));
            }
            if (!mma_wait_all(bar(FIN))) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else if (producer) {
        // =========================== producer ===========================
        // each tile loads as soon as its buffer is free: the next K once
        // S += K^T K (its last reader) completed, the next V and the Q after
        // next once O (the last reader of this chunk's V and Q) completed
        if (lane == 0) {
            for (int it = 0; it + 1 < nchunks; ++it) {
                const int c = c_begin + it;
                const uint32_t ph = it & 1;
                if (!wait_bar(CK, ph)) break;
                issue_load(LK, &mK, tK, c + 1);
                if (!wait_bar(CO, ph)) break;
                issue_load(LV, &mV, tV, c + 1);
                if (it + 2 < nchunks) issue_load((it & 1) ? LQ1 : LQ0, &mQ, (it & 1) ? tQ1 : tQ0, c + 2);
            }
            if (!loads.settle()) atomicExch(p.status, (int)kDevWaitTimeout);
        }
    } else if (drainer) {
        // ========================== drain warps ==========================
        // A beta warp's O staging box (32 rows x 32 fp32 columns, 4 KB) is its
        // own region of sO (rows 32 quarter.., block bw); its O groups pass
        // through it one after the other, each once the previous one has
        // been read out by its bulk store.  (On a head's first chunk the X
        // drain puts this warp's X_lo rows in the same region, before any O.)
        const uint32_t box = tO.base + (uint32_t)(bw & 1) * (kL * 128u) + (uint32_t)(quarter * 32) * 128u;
        int o_row0 = 0;  // first token of this warp's O rows in the current chunk
        // DECAY: o_t = g^{2(t+1)} O'_t
        auto scale_o = [&](uint32_t (&r)[32]) {
            const float os = gp(2.f * (float)(row + 1));
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * os);
        };
        auto stage_o = [&](const uint32_t (&r)[32], int g) {
            if (lane == 0) tma_store_wait_read();  // the box's previous content has left
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 8; ++q)
                st_shared_v4(box + (uint32_t)lane * 128u + (uint32_t)((q ^ (lane & 7)) << 4), r[4 * q], r[4 * q + 1],
                             r[4 * q + 2], r[4 * q + 3]);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&mO, box, bcol(g), o_row0, head);
                tma_store_commit();
            }
        };
        for (int it = 0; it < nchunks; ++it) {
            const uint32_t ph = it & 1;
            const int c = c_begin + it;
            const bool has_next = it + 1 < nchunks;
            const bool first = c == 0;
            static_assert(BG <= 2, "a beta warp holds at most one O group while it drains S");
            if (alpha_w || NORM) {
                // A packed in place (masked; hi and lo in the normalised walk,
                // where every drain warp packs one group)
                if (!wait_bar(CA_, ph)) break;
                tc_fence_after();
                // (DECAY: A~ = A g^{-(i+1)} by columns, split on a head's first chunk)
                pack_alpha(NORM || (DECAY && first), NORM, DECAY, 1.f);
                packed(DA);
            }
            if (beta_w) {
                // P0 of this chunk -> the S0 / P0 tile, once Q S0 has read S0 (a
                // head's first chunk has P0 = 0 and skips Q P0)
                if (!wait_bar(CQS, ph)) break;
                tc_fence_after();
                if (state_rows) {
                    if (!first) {
                        drainD(tP_, tSP, true, DECAY ? gp(2.f * clen(c)) : 1.f, DECAY);  // DECAY: TMEM P decayed
                        if (NORM && bw == 0) {  // p0 of this chunk -> its operand tiles
                            const uint32_t pv = tmem_ld1(tPn_ + lane_off);
                            tmem_ld_wait();
                            put_p0(__uint_as_float(pv));
                        }
                    }
                    drained(DP);
                }
                // X -> sX (bf16); on a head's first chunk split into hi (sX) and
                // lo (sO)
                if (!wait_bar(CX, ph)) break;
                tc_fence_after();
#pragma unroll
                for (int g = 0; g < BG; ++g) {
                    uint32_t x[32];
                    tmem_ld32(tBe_ + lane_off + bcol(g), x);
                    tmem_ld_wait();
                    if constexpr (DECAY) {  // sX = g^{2L-1-t} X'
                        const float xs = gp(2.f * clen(c) - 1.f - (float)row);
#pragma unroll
                        for (int j = 0; j < 32; ++j) x[j] = __float_as_uint(__uint_as_float(x[j]) * xs);
                    }
                    if (NORM) put_row32_split2(tX, tXL, row, bcol(g), x, false);
                    else if (first) put_row32_split2(tX, tO, row, bcol(g), x, false);
                    else put_row32(tX, row, bcol(g), x, false);
                }
                drained(DX);
                if constexpr (DECAY) {
                    // K' = diag(sqrt(b)) K in place (row = token, b = g^{L-1-t}):
                    // A and A~ K, its other readers, have completed
                    const float kf = gp(0.5f * (clen(c) - 1.f - (float)row));
#pragma unroll
                    for (int g = 0; g < BG; ++g)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int col = bcol(g) + 8 * q;
                            const uint32_t a = tK.chunk(row, col >> 6, (col & 63) >> 3);
                            uint32_t w[4];
                            ld_shared_v4(a, w[0], w[1], w[2], w[3]);
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&w[h]);
                                w[h] = pack_bf16(__low2float(v2) * kf, __high2float(v2) * kf);
                            }
                            st_shared_v4(a, w[0], w[1], w[2], w[3]);
                        }
                    drained(DK);
                }
            }
            if (alpha_w || NORM || DECAY) {
                // W packed in place (masked; hi and lo on a head's first chunk
                // and in the normalised walk, where every drain warp packs one
                // group; DECAY: W~ = g^{-2L} tril(W'), split on every chunk, by
                // every drain warp at D = 128)
                if (!wait_bar(CW, ph)) break;
                tc_fence_after();
                pack_alpha(first || NORM || DECAY, NORM || (DECAY && D == 128), false,
                           DECAY ? gp(-2.f * clen(c)) : 1.f);
                packed(DW);
            }
            if (beta_w) {
                // O: the first group through the staging box, the last one into
                // registers, then beta is free; the next chunk's S0 into its
                // tile (Q P0 has read P0); then the last group through the box
                // (X_lo, in the box region on a head's first chunk, was last
                // read by W, complete once O is)
                if (!wait_bar(CO, ph)) break;
                tc_fence_after();
                o_row0 = c * kL + quarter * 32;
                uint32_t r[32];
                tmem_ld32(tBe_ + lane_off + bcol(0), r);
                if constexpr (BG == 1) {
                    // one group: beta is free once it sits in registers, and the
                    // next S0 goes out before the group is staged
                    float den = 1.f;
                    if (NORM) den = __uint_as_float(tmem_ld1(tDen_ + lane_off));
                    tmem_ld_wait();
                    drained(DO);
                    if (state_rows && has_next) {
                        drainD(tS_, tSP, false);
                        drained(DS);
                    }
                    if (NORM) {
                        // ratio normalisation: o = num * (1 / den), the reciprocal
                        // correctly rounded (within one more rounding of num / den)
                        const float inv = __frcp_rn(den);
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * inv);
                    }
                    if (DECAY) scale_o(r);
                    stage_o(r, 0);
                    // DECAY: TMEM S decayed for the next update (S += K'^T K'
                    // waits for K', which this warp scales after it)
                    if (DECAY && state_rows && has_next) rescale(tS_, gp(clen(c + 1)));
                } else {
                    static_assert(NORM == false, "the normalised walk has one O group per beta warp");
                    tmem_ld_wait();
                    if (DECAY) scale_o(r);
                    stage_o(r, 0);
                    tmem_ld32(tBe_ + lane_off + bcol(1), r);  // BG == 2: the last group
                    tmem_ld_wait();
                    if (DECAY) scale_o(r);
                    drained(DO);
                    if (state_rows && has_next) {
                        drainD(tS_, tSP, false);
                        drained(DS);
                    }
                    stage_o(r, 1);
                    if (DECAY && state_rows && has_next) rescale(tS_, gp(clen(c + 1)));  // as above
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

template <int D, bool NORM, bool DECAY = false>
cudaError_t launch_out_t(const void* Q, const void* K, const void* V, float* O, const float* prefix, int BH, int T,
                         SegPlan plan, int* status, cudaStream_t s, float lg = 0.f) {
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
    OutParams prm{T, plan.nseg, plan.nchunk, plan.seglen, prefix, status, lg};
    const size_t smem = OutLayout<D, NORM>::kBytes + 1024;
    auto kern = tc_out_kernel<D, NORM, DECAY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.nseg, BH);
    kern<<<grid, OutRoles<D, NORM>::kThreads, smem, s>>>(mq, mk, mv, mo, mr, prm);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_out(const void* Q, const void* K, const void* V, float* O, const float* prefix, int BH, int T,
                          int d, int dv, bool normalized, SegPlan plan, int* status, cudaStream_t s) {
    if (BH == 0 || plan.nseg == 0) return cudaSuccess;
    if (plan.granule != kL || d != dv) return cudaErrorInvalidValue;
    if (normalized) return d == 64 ? launch_out_t<64, true>(Q, K, V, O, prefix, BH, T, plan, status, s)
                                   : cudaErrorInvalidValue;
    if (d == 128) return launch_out_t<128, false>(Q, K, V, O, prefix, BH, T, plan, status, s);
    if (d == 64) return launch_out_t<64, false>(Q, K, V, O, prefix, BH, T, plan, status, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_tc_out_decay(const void* Q, const void* K, const void* V, float* O, const float* prefix, int BH,
                                int T, int d, int dv, float lg, SegPlan plan, int* status, cudaStream_t s) {
    if (BH == 0 || plan.nseg == 0) return cudaSuccess;
    if (plan.granule != kL || d != dv) return cudaErrorInvalidValue;
    if (d == 128) return launch_out_t<128, false, true>(Q, K, V, O, prefix, BH, T, plan, status, s, lg);
    if (d == 64) return launch_out_t<64, false, true>(Q, K, V, O, prefix, BH, T, plan, status, s, lg);
    return cudaErrorInvalidValue;
}

}  // namespace hla2
