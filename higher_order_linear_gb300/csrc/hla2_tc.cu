// hla2_tc.cu -- tensor-core segment walks of masked second-order HLA on
// GB300 (sm_103a): tcgen05.mma with TMEM accumulators, TMA-staged tiles.
//
// HLA summary (arXiv 2510.27258): section 1 "Second-order HLA" (o_t =
// q_t^T (S_t C_t - G_t), the causal A A^T V structure of section 2) and
// section 4 "Parallel training via associative scans" (chunk-parallel form:
// segment summaries, exclusive scan, restart from the prefix).
//
// One CTA walks one segment of one head in chunks of L = 128 tokens.  With
// P = S C - G ("P-form"), the state entering a chunk is (S0, P0) and, for the
// chunk's Q, K, V (128 x d, 128 x d, 128 x dv):
//   A = tril(Q K^T)                     (i <= t, diagonal kept)
//   X = Q S0 + A K                      (so that P grows by X^T V)
//   W = tril(A A^T + (Q S0) Q^T)        (j <= t)
//   O = Q P0 + W V                      (the chunk's outputs)
//   P0 += X^T V,   S0 += K^T K
// Summary mode (from a zero state) also accumulates C = Q^T V and emits the
// segment's S, C, P.  Every product is a dense 128-row contraction issued as
// tcgen05.mma kind::f16 (bf16 operands from shared memory, fp32 accumulators
// in tensor memory).  fp32 results that feed a later product (A, X, W, S0,
// P0) are rounded to bf16 when written back to shared memory; the running S
// and P stay fp32 in tensor memory for the whole segment.
//
// Operand layout: every tile lives in shared memory as rows of 128 bytes
// (64 bf16) in the 128-byte-swizzled pattern TMA writes, split into 64-column
// blocks.  A tile whose rows are the product's M (or N) index is read as a
// K-major operand; a tile whose rows are the contraction index is read as an
// MN-major operand.  This lets every tensor-memory drain write whole rows.
#include <cuda.h>

#include "hla2_internal.h"

namespace hla2 {
namespace {

constexpr int kL = 128;          // tokens per chunk (MMA M)
constexpr int kThreadsTC = 256;  // eight warps: two per 32-lane quarter of TMEM
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kWaitNs = 2000000000ull;  // bounded waits: 2 s

// ------------------------------------------------------------------ PTX ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    return ok != 0;
}
// 3-D tiled TMA load into shared memory, completion counted on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar)
        : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;  // SWIZZLE_128B
    return d;
}
// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                     // D format: f32
           | (1u << 7)                   // A format: bf16
           | (1u << 10)                  // B format: bf16
           | ((a_mn ? 1u : 0u) << 15)    // A major-ness: 0 K-major, 1 MN-major
           | ((b_mn ? 1u : 0u) << 16)    // B major-ness
           | ((uint32_t)(N >> 3) << 17)  // N / 8
           | ((uint32_t)(M >> 4) << 24); // M / 16
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// -------------------------------------------------------------- tiles ----
// A tile of R rows x C bf16 columns, stored as C/64 blocks of R x 128 bytes,
// 128-byte swizzled (16-byte chunk c of row r at position c ^ (r & 7)).
struct Tile {
    uint32_t base;  // shared address, 1024-byte aligned
    int rows;
    __device__ uint32_t block_bytes() const { return (uint32_t)rows * 128u; }
    // K-major operand (rows are the M/N index): descriptor for K-step ks (16 columns)
    __device__ uint64_t kmaj(int ks) const {
        return sdesc(base + (uint32_t)(ks >> 2) * block_bytes() + (uint32_t)(ks & 3) * 32u, 16u, 1024u);
    }
    // MN-major operand (rows are the contraction index): K-step ks (16 rows)
    __device__ uint64_t mnmaj(int ks) const { return sdesc(base + (uint32_t)ks * 2048u, block_bytes(), 1024u); }
    // byte address of 16-byte chunk `c` (0..7) of row r in column block b
    __device__ uint32_t chunk(int r, int b, int c) const {
        return base + (uint32_t)b * block_bytes() + (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) << 4);
    }
};

// Write 32 fp32 values (columns col0..col0+31 of row r) to a bf16 tile,
// optionally zeroing columns > r (causal mask).
__device__ __forceinline__ void put_row32(const Tile& t, int r, int col0, const uint32_t* v, bool mask) {
    const int b = col0 >> 6;
    const int c0 = (col0 & 63) >> 3;  // 0 or 4
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int j = q * 8 + h * 2;
            float x0 = __uint_as_float(v[j]), x1 = __uint_as_float(v[j + 1]);
            if (mask) {
                if (col0 + j > r) x0 = 0.f;
                if (col0 + j + 1 > r) x1 = 0.f;
            }
            w[h] = pack_bf16(x0, x1);
        }
        st_shared_v4(t.chunk(r, b, c0 + q), w[0], w[1], w[2], w[3]);
    }
}

// Same, splitting each masked value x into hi = bf16(x) (written to the tile)
// and lo = bf16(x - hi), returned as 16 packed bf16 pairs.
__device__ __forceinline__ void put_row32_split(const Tile& t, int r, int col0, const uint32_t* v, bool mask,
                                                uint32_t* lo) {
    const int b = col0 >> 6;
    const int c0 = (col0 & 63) >> 3;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int j = q * 8 + h * 2;
            float x0 = __uint_as_float(v[j]), x1 = __uint_as_float(v[j + 1]);
            if (mask) {
                if (col0 + j > r) x0 = 0.f;
                if (col0 + j + 1 > r) x1 = 0.f;
            }
            const __nv_bfloat162 hv = __floats2bfloat162_rn(x0, x1);
            w[h] = *reinterpret_cast<const uint32_t*>(&hv);
            lo[q * 4 + h] = pack_bf16(x0 - __low2float(hv), x1 - __high2float(hv));
        }
        st_shared_v4(t.chunk(r, b, c0 + q), w[0], w[1], w[2], w[3]);
    }
}

// Load NC (32 or 64) consecutive TMEM columns of this thread's lane, one wait.
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[64]) {
    tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    if (NC == 64) tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
    tmem_ld_wait();
}

__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// ------------------------------------------------------------- kernel ----
struct TCParams {
    int T, nseg, nchunk;
    float* summ;          // mode 0 output records
    const float* prefix;  // mode 1 input records
    int* status;
};

template <int D, int MODE>
struct Layout {
    // byte offsets of the tiles inside the 1024-aligned dynamic shared memory
    static constexpr uint32_t kTok = kL * D * 2;      // Q, K, V, X tiles
    static constexpr uint32_t kSq = kL * kL * 2;      // A / W tile
    static constexpr uint32_t kSt = D * D * 2;        // S0 / P0 tiles
    static constexpr uint32_t Q = 0, K = Q + kTok, V = K + kTok, A = V + kTok, X = A + kSq;
    static constexpr uint32_t P = X + kTok;                       // mode 1 only
    static constexpr uint32_t S = (MODE == 1) ? P + kSt : X + kTok;
    // MN-major operands read with M = 128 > D see a second 64-column block
    // one block past the tile: keep valid memory there when D = 64.
    static constexpr uint32_t kPad = (D < 128) ? 16384u : 0u;
    static constexpr uint32_t kBytes = S + kSt + kPad;
};

// Eight warps: warp w drains TMEM lanes 32*(w%4).. (its lane quarter) and the
// w/4-th half of each region's columns.  Thread 0 issues TMA and MMAs.
template <int D, int MODE>
__global__ void __launch_bounds__(kThreadsTC, 1)
tc_walk_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mO, TCParams p) {
    using LY = Layout<D, MODE>;
    extern __shared__ __align__(1024) unsigned char dsm_raw[];
    __shared__ __align__(8) unsigned long long bars[5];  // Q, K, V loads; MMA completion; Q released
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int row = quarter * 32 + (tid & 31);  // TMEM lane / tile row owned by this thread
    const int seg = blockIdx.x;
    const int head = blockIdx.y;
    const int c_begin = (int)((long long)seg * p.nchunk / p.nseg);
    const int c_end = (int)((long long)(seg + 1) * p.nchunk / p.nseg);
    const bool state_rows = (D == 128) || quarter < D / 32;  // warp holds rows < D

    const uint32_t dsm = (smem_u32(dsm_raw) + 1023u) & ~1023u;
    const Tile tQ{dsm + LY::Q, kL}, tK{dsm + LY::K, kL}, tV{dsm + LY::V, kL};
    const Tile tA{dsm + LY::A, kL}, tX{dsm + LY::X, kL};
    const Tile tS{dsm + LY::S, D}, tP{dsm + LY::P, D};
    const uint32_t bQ = smem_u32(&bars[0]), bK = smem_u32(&bars[1]), bV = smem_u32(&bars[2]), bM = smem_u32(&bars[3]);
    const uint32_t bR = smem_u32(&bars[4]);

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bQ, 1);
        mbar_init(bK, 1);
        mbar_init(bV, 1);
        mbar_init(bM, 1);
        mbar_init(bR, 1);
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
    const uint32_t tA_ = tmem + 0;           // A, then W, then O (mode 1); A then X (mode 0)
    const uint32_t tX_ = tmem + 128;         // X, then packed bf16 W_lo (mode 1)
    const uint32_t tS_ = tmem + (MODE == 1 ? 256 : 128);
    const uint32_t tP_ = tmem + (MODE == 1 ? 256 + D : 128 + D);
    const uint32_t tC_ = tmem + 128 + 2 * D;  // mode 0 only
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // this warp's column window in a 128-wide and in a D-wide region
    const int c128 = half * 64;
    const int cD = half * (D / 2);

    uint32_t ph_load = 0, ph_mma = 0, ph_rel = 0;
    constexpr uint32_t kTileBytes = kL * D * 2;
    auto wait_bar = [&](uint32_t bar, uint32_t parity) -> bool {
        if (abort_flag) return false;
        if (mbar_try(bar, parity)) return true;
        const unsigned long long t0 = globaltimer();
        while (!mbar_try(bar, parity)) {
            if (abort_flag) return false;
            if (globaltimer() - t0 > kWaitNs) {
                abort_flag = 1;
                atomicExch(p.status, (int)kDevWaitTimeout);
                return false;
            }
        }
        return true;
    };
    auto issue_load = [&](uint32_t bar, const CUtensorMap* map, const Tile& t, int chunk) {
        mbar_expect_tx(bar, kTileBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b) tma_load_3d(t.base + b * t.block_bytes(), map, b * 64, chunk * kL, head, bar);
    };
    // drain this warp's share of a 128-wide fp32 region into a bf16 tile
    auto drain128 = [&](uint32_t treg, const Tile& t, bool mask) {
        uint32_t r[64];
        tmem_ld_cols<64>(treg + lane_off + c128, r);
        put_row32(t, row, c128, r, mask);
        put_row32(t, row, c128 + 32, r + 32, mask);
    };
    // drain this warp's share of a D-wide fp32 region into a bf16 tile
    auto drainD = [&](uint32_t treg, const Tile& t) {
        uint32_t r[64];
        tmem_ld_cols<D / 2>(treg + lane_off + cD, r);
        put_row32(t, row, cD, r, false);
        if (D == 128) put_row32(t, row, cD + 32, r + 32, false);
    };

    // ---- initial state ----
    if (MODE == 1 && state_rows) {
        // S0, P0 from the segment's exclusive prefix: fp32 into TMEM, bf16 into smem
        const size_t R = (size_t)D * D + 2 * (size_t)D * D + 2 * (size_t)D;
        const float* pre = p.prefix + ((size_t)head * p.nseg + seg) * R;
        const float* S0 = pre;                          // S at offset 0
        const float* P0 = pre + 2 * (size_t)D * D + D;  // P after S, C, m
#pragma unroll 1
        for (int cb = cD; cb < cD + D / 2; cb += 32) {
            uint32_t r[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 x = *reinterpret_cast<const float4*>(S0 + (size_t)row * D + cb + j);
                r[j] = __float_as_uint(x.x); r[j + 1] = __float_as_uint(x.y);
                r[j + 2] = __float_as_uint(x.z); r[j + 3] = __float_as_uint(x.w);
            }
            tmem_st32(tS_ + lane_off + cb, r);
            put_row32(tS, row, cb, r, false);
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 x = *reinterpret_cast<const float4*>(P0 + (size_t)row * D + cb + j);
                r[j] = __float_as_uint(x.x); r[j + 1] = __float_as_uint(x.y);
                r[j + 2] = __float_as_uint(x.z); r[j + 3] = __float_as_uint(x.w);
            }
            tmem_st32(tP_ + lane_off + cb, r);
            put_row32(tP, row, cb, r, false);
        }
        tmem_st_wait();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0 && c_begin < c_end) {
        issue_load(bQ, &mQ, tQ, c_begin);
        issue_load(bK, &mK, tK, c_begin);
        issue_load(bV, &mV, tV, c_begin);
    }

    constexpr uint32_t iSq = idesc_bf16(128, 128, false, false);   // 128 x 128, both K-major
    constexpr uint32_t iKK = idesc_bf16(128, D, false, false);     // N = D, both K-major
    constexpr uint32_t iKM = idesc_bf16(128, D, false, true);      // A K-major, B MN-major
    constexpr uint32_t iMM = idesc_bf16(128, D, true, true);       // both MN-major
    bool first = true;

    for (int c = c_begin; c < c_end; ++c) {
        const bool has_next = c + 1 < c_end;
        // ================= phase 1 =================
        if (tid == 0) {
            if (MODE == 1) tma_store_wait_read();  // previous O tile has left sA|sX
            wait_bar(bQ, ph_load);
            wait_bar(bK, ph_load);
            tc_fence_after();
            if (!abort_flag) {
                // A = Q K^T
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQ.kmaj(ks), tK.kmaj(ks), iSq, ks > 0);
                if (MODE == 1) {
                    // X = Q S0
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tX_, tQ.kmaj(ks), tS.kmaj(ks), iKK, ks > 0);
                }
                // S += K^T K
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tS_, tK.mnmaj(ks), tK.mnmaj(ks), iMM, (MODE == 1 || !first || ks > 0) ? 1u : 0u);
                mma_commit(bM);
            }
        }
        __syncwarp();
        wait_bar(bM, ph_mma);
        ph_mma ^= 1;
        tc_fence_after();
        // drain 1: A -> sA (masked); mode 1 also X -> sX and S -> sS
        if (!abort_flag) {
            drain128(tA_, tA, true);
            if (MODE == 1) {
                drainD(tX_, tX);
                if (state_rows) drainD(tS_, tS);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ================= phase 2 =================
        if (tid == 0 && !abort_flag) {
            tc_fence_after();
            if (MODE == 1) {
                // W = A A^T + X Q^T   (X holds Q S0 here)
                for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tA_, tA.kmaj(ks), tA.kmaj(ks), iSq, ks > 0);
                for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tX.kmaj(ks), tQ.kmaj(ks), iSq, 1);
                // X = Q S0 + A K  (accumulate onto the fp32 Q S0 still in TMEM)
                for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tX_, tA.kmaj(ks), tK.mnmaj(ks), iKM, 1);
            } else {
                // X = Q S_local + A K   (no S_local term on the segment's first chunk)
                if (!first)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQ.kmaj(ks), tS.kmaj(ks), iKK, ks > 0);
                for (int ks = 0; ks < kL / 16; ++ks)
                    mma_bf16(tA_, tA.kmaj(ks), tK.mnmaj(ks), iKM, (!first || ks > 0) ? 1u : 0u);
            }
            mma_commit(bM);
        }
        __syncwarp();
        wait_bar(bM, ph_mma);
        ph_mma ^= 1;
        tc_fence_after();
        // drain 2
        if (!abort_flag) {
            if (MODE == 1) {
                // X -> sX; W -> hi in sA (masked), lo packed into the X region of TMEM
                drainD(tX_, tX);
                uint32_t lo[32];
                {
                    uint32_t r[64];
                    tmem_ld_cols<64>(tA_ + lane_off + c128, r);
                    put_row32_split(tA, row, c128, r, true, lo);
                    put_row32_split(tA, row, c128 + 32, r + 32, true, lo + 16);
                }
                // both warps of this lane quarter have read X before it is overwritten
                asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
                tmem_st32(tX_ + lane_off + half * 32, lo);
                tmem_st_wait();
            } else {
                // X -> sX ; S -> sS (S_local for the next chunk)
                drainD(tA_, tX);
                if (has_next && state_rows) drainD(tS_, tS);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // ================= phase 3 =================
        if (tid == 0 && !abort_flag) {
            if (has_next) issue_load(bK, &mK, tK, c + 1);  // sK was last read in phase 2
            wait_bar(bV, ph_load);
            tc_fence_after();
            if (!abort_flag) {
                // the products that read Q go first, with their own commit, so
                // that the next chunk's Q can load while the rest runs
                if (MODE == 1) {
                    // O = Q P0 (+ W_hi V + W_lo V below)
                    for (int ks = 0; ks < D / 16; ++ks) mma_bf16(tA_, tQ.kmaj(ks), tP.mnmaj(ks), iKM, ks > 0);
                } else {
                    // C += Q^T V
                    for (int ks = 0; ks < kL / 16; ++ks)
                        mma_bf16(tC_, tQ.mnmaj(ks), tV.mnmaj(ks), iMM, (!first || ks > 0) ? 1u : 0u);
                }
                mma_commit(bR);
                if (MODE == 1) {
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tA_, tA.kmaj(ks), tV.mnmaj(ks), iKM, 1);
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16_tmem_a(tA_, tX_ + ks * 8, tV.mnmaj(ks), iKM, 1);
                    // P += X^T V
                    for (int ks = 0; ks < kL / 16; ++ks) mma_bf16(tP_, tX.mnmaj(ks), tV.mnmaj(ks), iMM, 1);
                } else {
                    // P += X^T V
                    for (int ks = 0; ks < kL / 16; ++ks)
                        mma_bf16(tP_, tX.mnmaj(ks), tV.mnmaj(ks), iMM, (!first || ks > 0) ? 1u : 0u);
                }
                mma_commit(bM);
                const bool q_free = wait_bar(bR, ph_rel);
                ph_rel ^= 1;
                if (has_next && q_free) issue_load(bQ, &mQ, tQ, c + 1);
            }
        }
        ph_load ^= 1;
        __syncwarp();
        wait_bar(bM, ph_mma);
        ph_mma ^= 1;
        tc_fence_after();
        if (tid == 0 && has_next && !abort_flag) issue_load(bV, &mV, tV, c + 1);  // sV is free
        if (MODE == 1 && !abort_flag) {
            // drain 3: O -> fp32 staging in sA|sX (TMA store boxes of 32 columns);
            // P -> sP (P0 of the next chunk)
            {
                uint32_t r[64];
                tmem_ld_cols<D / 2>(tA_ + lane_off + cD, r);
#pragma unroll
                for (int g = 0; g < D / 64; ++g) {
                    const int cb = (cD >> 5) + g;
                    const uint32_t box = tA.base + (uint32_t)cb * 16384u + (uint32_t)row * 128u;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st_shared_v4(box + (uint32_t)((q ^ (row & 7)) << 4), r[32 * g + 4 * q], r[32 * g + 4 * q + 1],
                                     r[32 * g + 4 * q + 2], r[32 * g + 4 * q + 3]);
                }
            }
            if (has_next && state_rows) drainD(tP_, tP);
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && !abort_flag) {
            if (MODE == 1) {
#pragma unroll
                for (int cb = 0; cb < D / 32; ++cb) tma_store_3d(&mO, tA.base + (uint32_t)cb * 16384u, cb * 32, c * kL, head);
                tma_store_commit();
            }
        }
        first = false;
    }

    // ---- segment summary out (mode 0): S | C | m | P | p records, fp32 ----
    if (MODE == 0 && !abort_flag && state_rows) {
        const size_t R = (size_t)D * D + 2 * (size_t)D * D + 2 * (size_t)D;
        float* out = p.summ + ((size_t)head * p.nseg + seg) * R;
        float* dst[3] = {out, out + (size_t)D * D, out + 2 * (size_t)D * D + D};  // S, C, P
        const uint32_t src[3] = {tS_, tC_, tP_};
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            uint32_t r[64];
            tmem_ld_cols<D / 2>(src[m] + lane_off + cD, r);
#pragma unroll
            for (int j = 0; j < D / 2; j += 4)
                *reinterpret_cast<float4*>(dst[m] + (size_t)row * D + cD + j) =
                    make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                                __uint_as_float(r[j + 3]));
        }
    }
    if (MODE == 1 && tid == 0) tma_store_wait_all();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// ------------------------------------------------------------ host side ----
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 3-D map over [BH][T][cols] (innermost first), box {box_x, 128, 1}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int cols, int T, int BH, int box_x) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols * esize, (cuuint64_t)T * cols * esize};
    cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)kL, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int MODE>
cudaError_t launch_t(const void* Q, const void* K, const void* V, float* O, const float* prefix, float* summ, int BH,
                     int T, SegPlan plan, int* status, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mk, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64) ||
        !make_map(&mv, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, T, BH, 64))
        return cudaErrorInvalidValue;
    if (MODE == 1) {
        if (!make_map(&mo, O, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, T, BH, 32)) return cudaErrorInvalidValue;
    } else {
        mo = mq;  // unused
    }
    TCParams prm{T, plan.nseg, plan.nchunk, summ, prefix, status};
    const size_t smem = Layout<D, MODE>::kBytes + 1024;
    auto kern = tc_walk_kernel<D, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.nseg, BH);
    kern<<<grid, kThreadsTC, smem, s>>>(mq, mk, mv, mo, prm);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int d, int dv, int dtype, int normalized, int device) {
    if (d != dv || (d != 64 && d != 128) || dtype != 1 || normalized) return false;
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
