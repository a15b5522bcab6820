// hla2_tc_common.cuh -- building blocks shared by the tcgen05 segment walks
// (hla2_tc.cu for HLA, hla2_ahla_tc.cu for AHLA): inline-PTX wrappers for
// mbarriers, TMA, tcgen05 MMA / tensor-memory access, the swizzled bf16
// tile addressing, tensor-memory drains and the host-side tensor-map encoder.
// Everything sits in an anonymous namespace: each translation unit that
// includes this file gets its own copy.
#pragma once

#include <cuda.h>

#include "hla2_internal.h"

namespace hla2 {
namespace {

constexpr int kL = 128;          // tokens per chunk (MMA M)
constexpr int kDrainWarps = 8;   // two per 32-lane quarter of TMEM
constexpr int kThreadsTC = (kDrainWarps + 1) * 32;  // plus one issuing warp
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
// Pull a tile into L2 ahead of its TMA load (no shared memory involved).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global [%0, {%1, %2, %3}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until at most the most recent bulk store group of this thread still
// reads shared memory (the older ones have left it).
__device__ __forceinline__ void tma_store_wait_read_all_but_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
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

__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
    return r;
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r) : "memory");
}
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

// Same split, hi to tile `hi` and lo to tile `lo` (both bf16 operands).
__device__ __forceinline__ void put_row32_split2(const Tile& hi, const Tile& lo, int r, int col0, const uint32_t* v,
                                                 bool mask) {
    uint32_t l[16];
    put_row32_split(hi, r, col0, v, mask, l);
    const int b = col0 >> 6;
    const int c0 = (col0 & 63) >> 3;
#pragma unroll
    for (int q = 0; q < 4; ++q) st_shared_v4(lo.chunk(r, b, c0 + q), l[4 * q], l[4 * q + 1], l[4 * q + 2], l[4 * q + 3]);
}

// Column sums over a warp: lane i holds row i's 32 fp32 values (as bits) in
// r[0..31]; lane j gets the sum over all lanes of column j.  A transposing
// butterfly: at step w the lanes with bit w set keep the upper w of their
// remaining columns and trade the lower w with lane ^ w, so each step halves
// the columns a lane holds (31 shuffles for the 32 columns).
__device__ __forceinline__ float warp_colsum32(const uint32_t* r, int lane) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int k = 0; k < w; ++k) {
            const float send = up ? v[k] : v[k + w];
            const float keep = up ? v[k + w] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return v[0];
}

// Write the bf16 hi and lo parts of 4 fp32 values (columns c..c+3 of row r).
__device__ __forceinline__ void put4_split(const Tile& hi, const Tile& lo, int r, int c, float4 x) {
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(x.x, x.y), h1 = __floats2bfloat162_rn(x.z, x.w);
    const uint32_t l0 = pack_bf16(x.x - __low2float(h0), x.y - __high2float(h0));
    const uint32_t l1 = pack_bf16(x.z - __low2float(h1), x.w - __high2float(h1));
    const uint32_t off = (uint32_t)((c & 7) >> 2) * 8u;  // which half of the 16-byte chunk
    const uint32_t ah = hi.chunk(r, c >> 6, (c & 63) >> 3) + off;
    const uint32_t al = lo.chunk(r, c >> 6, (c & 63) >> 3) + off;
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(ah), "r"(*reinterpret_cast<const uint32_t*>(&h0)),
                 "r"(*reinterpret_cast<const uint32_t*>(&h1))
                 : "memory");
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(al), "r"(l0), "r"(l1) : "memory");
}

// Commits every tcgen05 operation this thread issued to `mbar` (one arrival,
// used for nothing else, phase 0) and waits for them, at most kWaitNs, so that
// no MMA is still writing tensor memory or reading shared memory when the CTA
// releases them.  False when the wait ran out.
__device__ __forceinline__ bool mma_wait_all(uint32_t mbar) {
    mma_commit(mbar);
    const unsigned long long t0 = globaltimer();
    while (!mbar_try(mbar, 0))
        if (globaltimer() - t0 > kWaitNs) return false;
    return true;
}

// Bulk tensor loads that one thread issued on its load barriers (one phase
// per load, nobody else arrives there).  Before the CTA exits, that thread
// calls settle(): it waits, at most kWaitNs in all and whatever the abort
// state, until the last phase it armed on each barrier has completed, so that
// no copy is still writing this CTA's shared memory when a wait elsewhere ran
// out and the CTA unwinds early.  In a normal run every load has long landed.
template <int N>
struct LoadLedger {
    static_assert(N <= 16, "two bits per barrier in one word");
    uint32_t bar0;   // shared address of barrier index 0
    uint32_t state;  // per barrier i: bit 2i = armed at least once, bit 2i + 1 = parity of its last phase
    __device__ explicit LoadLedger(uint32_t b0) : bar0(b0), state(0u) {}
    __device__ void note(int b) {
        const uint32_t armed = 1u << (2 * b);
        if (state & armed) state ^= armed << 1;
        else state |= armed;
    }
    __device__ bool settle() const {
        const unsigned long long t0 = globaltimer();
#pragma unroll
        for (int i = 0; i < N; ++i) {
            if (!((state >> (2 * i)) & 1u)) continue;
            const uint32_t a = bar0 + 8u * (uint32_t)i, parity = (state >> (2 * i + 1)) & 1u;
            while (!mbar_try(a, parity))
                if (globaltimer() - t0 > kWaitNs) return false;
        }
        return true;
    }
};

// Load NC (32 or 64) consecutive TMEM columns of this thread's lane, one wait.
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[64]) {
    tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    if (NC == 64) tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
    tmem_ld_wait();
}

// One lane-row of 32 fp32 values per lane (the warp's 32 lanes are the box's
// 32 rows) written as a 4 KB box in the 128-byte-swizzled layout a tensor map
// with SWIZZLE_128B expects, then sent to global memory by a bulk tensor store
// at (x, y, z) that lane 0 issues and commits.  The caller waits for the bulk
// group before reusing `scratch` and before the CTA exits.
__device__ __forceinline__ void box32_store(const CUtensorMap* map, uint32_t scratch, const uint32_t* v, int lane,
                                            int x, int y, int z) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
        st_shared_v4(scratch + (uint32_t)lane * 128u + (uint32_t)((q ^ (lane & 7)) << 4), v[4 * q], v[4 * q + 1],
                     v[4 * q + 2], v[4 * q + 3]);
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(map, scratch, x, y, z);
        tma_store_commit();
    }
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr) : "memory");
}

// Reads back this lane's row (32 fp32 values) of a 32 x 32 box that a tensor
// load with SWIZZLE_128B wrote at `scratch` (the layout box32_store writes).
__device__ __forceinline__ void box32_read(uint32_t scratch, int lane, uint32_t* v) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
        ld_shared_v4(scratch + (uint32_t)lane * 128u + (uint32_t)((q ^ (lane & 7)) << 4), v[4 * q], v[4 * q + 1],
                     v[4 * q + 2], v[4 * q + 3]);
}

__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
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

// 3-D map over [BH][T][cols] (innermost first), box {box_x, box_y, 1}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int cols, int T, int BH, int box_x,
              int box_y = kL) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols * esize, (cuuint64_t)T * cols * esize};
    cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)box_y, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace hla2
