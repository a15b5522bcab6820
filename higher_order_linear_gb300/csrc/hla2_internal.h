// hla2_internal.h -- launch wrappers shared between the CUDA translation
// units of libhla2.  Host-only declarations; no torch types anywhere.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

namespace hla2 {

// Device-side error codes written into the library's status word.
enum DeviceError : int {
    kDevOk = 0,
    kDevWaitTimeout = 1,   // a bounded mbarrier wait ran out
    kDevBounds = 2,        // an index check failed; the access was skipped
    kDevTmemAlloc = 3,     // tensor-memory allocation returned an unexpected address
};

// Address of this device's status word (looked up once per device).
int* device_status_word();

// Counts kernel launches issued by the library (for instrumentation).
void note_launches(int n);

// Records a formatted reason for hla2_last_error_detail and returns `code`.
int set_error(int code, const char* fmt, ...);

// Length (in floats) of one summary / decode-state record:
// d*d + 2*d*dv + 2*d.
__host__ __device__ inline size_t record_len(int d, int dv) {
    return (size_t)d * d + 2 * (size_t)d * dv + 2 * (size_t)d;
}
// Offsets inside a summary record S | C | m | X | x (X = G or P, x = h or p).
struct RecOff {
    size_t S, C, m, X, x, R;
};
__host__ __device__ inline RecOff summary_offsets(int d, int dv) {
    RecOff o;
    o.S = 0;
    o.C = (size_t)d * d;
    o.m = o.C + (size_t)d * dv;
    o.X = o.m + d;
    o.x = o.X + (size_t)d * dv;
    o.R = o.x + d;
    return o;
}
// Offsets inside a decode-state record S | C | G | m | h.
__host__ __device__ inline RecOff decode_offsets(int d, int dv) {
    RecOff o;
    o.S = 0;
    o.C = (size_t)d * d;
    o.X = o.C + (size_t)d * dv;  // G
    o.m = o.X + (size_t)d * dv;
    o.x = o.m + d;               // h
    o.R = o.x + d;
    return o;
}

// Segment partition: a head's nchunk = ceil(T/granule) chunks are split into
// nseg contiguous runs of seglen chunks; the last run may be shorter.
// Segment s owns chunks [seg_chunk_begin(s), seg_chunk_begin(s + 1)).
struct SegPlan {
    int granule;  // tokens per chunk
    int nchunk;   // chunks per head
    int nseg;     // segments per head
    int seglen;   // chunks per segment (all but the last)
};
__host__ __device__ inline int seg_chunk_begin(const SegPlan& p, int s) {
    const long long c = (long long)s * p.seglen;
    return c < p.nchunk ? (int)c : p.nchunk;
}
// The (head, segment) a CTA of a (nseg, BH) grid works on, from its linear
// block index b.  When each head's last segment is shorter than the others,
// the CTAs of all full-length segments come first (head-major) and the short
// ones last, so that the short segments go to the SMs that free up first.
__host__ __device__ inline void block_segment(const SegPlan& p, int BH, long long b, int& head, int& seg) {
    const bool short_tail = p.nseg > 1 && (long long)p.nseg * p.seglen > p.nchunk;
    if (!short_tail) {
        head = (int)(b / p.nseg);
        seg = (int)(b % p.nseg);
        return;
    }
    const long long nfull = (long long)BH * (p.nseg - 1);
    if (b < nfull) {
        head = (int)(b / (p.nseg - 1));
        seg = (int)(b % (p.nseg - 1));
    } else {
        head = (int)(b - nfull);
        seg = p.nseg - 1;
    }
}

// ---- decode step (hla2_decode.cu) ----
cudaError_t launch_step(float* state, const float* q, const float* k, const float* v, float* o,
                        int n, int d, int dv, int normalized, cudaStream_t s);
// Same step on the compact P-form state S | P | p.
cudaError_t launch_step_pform(float* state, const float* q, const float* k, const float* v, float* o,
                              int n, int d, int dv, int normalized, cudaStream_t s);
// The same with per-token decay gamma of every prefix moment.
cudaError_t launch_step_pform_decay(float* state, const float* q, const float* k, const float* v, float* o,
                                    int n, int d, int dv, int normalized, float gamma, cudaStream_t s);

// Unmasked operator o = q^T S C on the state S | C | m.
cudaError_t launch_step_unmasked(float* state, const float* q, const float* k, const float* v, float* o,
                                 int n, int d, int dv, int normalized, cudaStream_t s);

// ---- segment walks on CUDA cores (hla2_walk.cu) ----
// mode 0: P-form segment summary  S|C|m|P|p from zero state.
// mode 1: outputs, starting from the prefix record S|.|.|P|p of the segment.
// mode 2: G-form summary S|C|m|G|h from zero state (chunk summaries).
// unmasked (modes 0, 1): o_t = q_t^T S_t C_t; mode 0 keeps S|C|m only, mode 1
// starts from the prefix S|C|m.  gamma (modes 0, 1, P-form): per-token decay
// of every prefix moment (1 = none).
cudaError_t launch_walk(int mode, const void* Q, const void* K, const void* V, int dtype,
                        float* O, const float* prefix, float* summ,
                        int BH, int T, int d, int dv, int normalized, int unmasked, float gamma, SegPlan plan,
                        cudaStream_t s);

// Decay factors of the segment plan: fac[r] = gamma^{n_r} and
// fac[nseg + r] = gamma^{2 n_r}, n_r the tokens of segment r.
cudaError_t launch_decay_factors(float* fac, int T, float gamma, SegPlan plan, cudaStream_t s);

// Decayed exclusive running sum along the record axis over the element range
// [off, off+len): out[b][0][i] = 0, out[b][n+1][i] = fac[n] out[b][n][i] + in[b][n][i].
// in may equal out; total (if not null) receives the inclusive sums.
cudaError_t launch_decay_exscan(const float* in, float* out, int BH, int N, size_t R, size_t off, size_t len,
                                float* total, size_t total_stride, const float* fac, cudaStream_t s);

// ---- scans (hla2_scan.cu) ----
// Exclusive running sum along the record axis for the element range
// [off, off+len) of every record: out[b][n][i] = sum_{r<n} in[b][r][i].
// in may equal out.  If total != nullptr, total[b*total_stride + i] receives
// the inclusive sum (element i relative to off); with out == nullptr only
// the totals are written.
cudaError_t launch_exscan(const float* in, float* out, int BH, int N, size_t R, size_t off, size_t len,
                          float* total, size_t total_stride, cudaStream_t s);

// Batched out = alpha*base + A * [B | bx] for nb matrices:
//   A d x d (row stride d), B d x dv (row stride dv), bx a d-vector taken as
//   column dv; base/out split the same way (main d x dv + extra vector).
//   Element strides between consecutive batch items are given per operand.
struct CrossArgs {
    const float* A;  long long sA;
    const float* B;  long long sB;
    const float* bx; long long sbx;
    const float* base;  long long sbase;
    const float* basex; long long sbasex;
    float* out;  long long sout;
    float* outx; long long soutx;
    float alpha;
    int d, dv, nb;
    int* status;  // device status word (tensor-core variant's bounded wait)
    // optional per-item scale of the product: item i of the batch uses
    // pscale[(pscale_off + i) % pscale_mod]
    const float* pscale;
    long long pscale_off;
    int pscale_mod;
};
cudaError_t launch_cross(const CrossArgs& a, cudaStream_t s);

// Copy `len` floats from each of nb records (strided) to another layout.
// The final decode state S|C|G|m|h of each of BH heads from its P-form
// totals S|C|m|P|p (records of summary_offsets(d, dv)): G = S C - P,
// h = S m - p in fp32.
cudaError_t launch_state_tail(const float* tot, float* state, int BH, int d, int dv, cudaStream_t s);
cudaError_t launch_copy_strided(const float* src, long long s_src, float* dst, long long s_dst,
                                size_t len, int nb, cudaStream_t s);

// ---- AHLA on CUDA cores (hla2_ahla.cu) ----
// mode 0: segment summary M|P|m|E|n (at the S|C|m|X|x offsets) from zero.
// mode 1: outputs from the segment's prefix P, E (and m, n when normalised).
cudaError_t launch_ahla_walk(int mode, const void* Q, const void* K, const void* V, int dtype,
                             float* O, const float* prefix, float* summ,
                             int BH, int T, int d, int dv, int normalized, SegPlan plan,
                             cudaStream_t s);
// One decode step on n heads, state P|E|m|n per head.
cudaError_t launch_ahla_step(float* state, const float* q, const float* k, const float* v, float* o,
                             int n, int d, int dv, int normalized, cudaStream_t s);

// ---- tensor-core segment walks (hla2_tc.cu) ----
// mode 0 writes the segment summaries S|C|.|P|. (and m, p when normalised or
// with_p), mode 1 the outputs from the prefixes S|.|.|P|(p).
bool tc_supported(int d, int dv, int dtype, int normalized, int device);
cudaError_t launch_tc_walk(int mode, const void* Q, const void* K, const void* V,
                           float* O, const float* prefix, float* summ,
                           int BH, int T, int d, int dv, int normalized, SegPlan plan, int* status,
                           cudaStream_t s, bool with_p = false);
// Chunk summaries S|C|m|G|h on tensor cores (hla2_tc_chunk.cu): bf16 inputs,
// d = dv in {64, 128}, chunk length L in {64, 128}.
bool tc_chunk_supported(int d, int dv, int L, int dtype, int device);
cudaError_t launch_tc_chunk(const void* Q, const void* K, const void* V, float* summ, int BH, int T, int d, int L,
                            int* status, cudaStream_t s);
// The HLA output walk pipelined across chunks (hla2_tc_out.cu), d = dv in
// {64, 128} (normalised: d = 64), bf16: outputs of every segment from its
// prefix S|.|.|P|.|p.
cudaError_t launch_tc_out(const void* Q, const void* K, const void* V, float* O, const float* prefix, int BH, int T,
                          int d, int dv, bool normalized, SegPlan plan, int* status, cudaStream_t s);
// The same walk for the decayed operator (lg = log2(gamma), gamma in the
// tensor-core range): outputs from the decayed prefix S|.|.|P|.
cudaError_t launch_tc_out_decay(const void* Q, const void* K, const void* V, float* O, const float* prefix, int BH,
                                int T, int d, int dv, float lg, SegPlan plan, int* status, cudaStream_t s);
// AHLA on tensor cores (hla2_ahla_tc.cu), d = dv in {64, 128}, bf16, unnormalised:
// mode 0 writes the M|P|.|E|. parts of the segment summaries, mode 1 outputs.
cudaError_t launch_ahla_tc_walk(int mode, const void* Q, const void* K, const void* V,
                                float* O, const float* prefix, float* summ,
                                int BH, int T, int d, int dv, SegPlan plan, int* status, cudaStream_t s);
// Unmasked operator on tensor cores (hla2_unm_tc.cu), d = dv in {64, 128}, bf16,
// unnormalised: mode 0 writes the S|C parts of the segment sums, mode 1 outputs
// from the prefix S|C.
cudaError_t launch_unm_tc_walk(int mode, const void* Q, const void* K, const void* V,
                               float* O, const float* prefix, float* summ,
                               int BH, int T, int d, int dv, SegPlan plan, int* status, cudaStream_t s);
// Decayed operator on tensor cores (hla2_decay_tc.cu), d = dv in {64, 128},
// bf16, unnormalised, gamma in [kDecayTcMinGamma, 1]: mode 0 writes the S|C|.|P|.
// parts of the segment summaries, mode 1 outputs from the prefix S|.|.|P|.
constexpr float kDecayTcMinGamma = 0.8f;
bool decay_tc_gamma_ok(float gamma);
cudaError_t launch_decay_tc_walk(int mode, const void* Q, const void* K, const void* V,
                                 float* O, const float* prefix, float* summ,
                                 int BH, int T, int d, int dv, float gamma, SegPlan plan, int* status,
                                 cudaStream_t s);
// Batched out = alpha*base + A*B on tensor cores with split-bf16 operands
// (d = dv in {64, 128}); the optional column outx = alpha*basex + A*bx is
// taken in fp32 on the CUDA cores.
cudaError_t launch_tc_cross(const CrossArgs& a, cudaStream_t s);

// The forward's exclusive scan over segment summaries (hla2_tc_scan.cu),
// d = dv in {64, 128}: CTA (head, r) folds the product factor of records
// 0..r-1 (S_<r, or P_<r for AHLA, the prefix's final value) and takes the
// cross products on tensor cores (split-bf16 operands).  Up to
// tc_scan_full_max_segments() segments it writes complete prefixes; above,
// it leaves record r's term X_r in prefix record r, and an exclusive running
// sum of the X field (launch_exscan / launch_decay_exscan with fac + nseg)
// completes them.  Fields written (terms, or their exclusive sums):
//   kScanHLA:   S_<r (S), X_r = P_r + S_<r C_r (X); with extra, x_r = p_r + S_<r m_r (x)
//   kScanDecay: S_<r (S, decayed fold), X_r = P_r + f_r S_<r C_r (X)
//   kScanAHLA:  P_<r (C), X_r = E_r + M_r P_<r (X), from M (S), P (C), E (X)
enum ScanOpKind { kScanHLA = 0, kScanDecay = 1, kScanAHLA = 2 };
struct ScanArgs {
    const float* summ;
    float* prefix;
    int nseg;
    size_t R;
    RecOff ro;
    const float* fac;  // decayed: fac[r] = gamma^{n_r}, fac[nseg + r] = gamma^{2 n_r}
    int* status;
    bool extra;
    bool terms_only = false;  // always leave terms (no complete prefixes), whatever nseg
    // optional: tot[head * R + i] = sum over the records of summ[..][i] for
    // i < tot_len (the plain sums S | C | m of a final state), formed by
    // extra CTAs of the same launch
    float* tot = nullptr;
    size_t tot_len = 0;
};
cudaError_t launch_tc_scan(int op, const ScanArgs& a, int BH, int d, int dv, cudaStream_t s);
// Scans of at most this many segments complete every prefix inside
// launch_tc_scan (no running-sum pass is needed afterwards).
int tc_scan_full_max_segments();

// A bounded device wait that runs out on purpose (hla2_selftest.cu): one CTA
// waits wait_ns on an mbarrier nothing arrives on, sets *status, writes 0 to
// *out (1 had the wait completed) and releases its tensor memory.
cudaError_t launch_selftest_runout(int* status, unsigned long long wait_ns, int* out, cudaStream_t s);

}  // namespace hla2
