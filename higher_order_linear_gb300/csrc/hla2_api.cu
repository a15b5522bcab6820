// hla2_api.cu -- the C ABI of libhla2 (declared in include/hla2.h).
//
// Host code only: argument checks, the segment plan, workspace carving and
// the launch sequence.  Every step of the computation runs in the CUDA
// kernels of this library; there is no host or CPU fallback.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <queue>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/hla2.h"
#include "hla2_internal.h"

namespace hla2 {

// Device-side error word (one per device that loads the library).
__device__ int g_status_word;

namespace {

thread_local std::string t_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* where) {
    return fail(HLA2_ERR_LAUNCH, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;
int* g_status_addr[kMaxDevices] = {};
std::mutex g_status_mu;

// Segments per head for the forward.  Every segment is one CTA, and a
// tensor-core walk holds a whole SM (its shared memory).  A head's chunks are
// cut into runs of seglen chunks (the last run may be shorter); the CTAs of
// full runs are dispatched first and the short ones last (block_segment).
// The plan takes the run length that minimises
//   makespan + nseg / 2          (in units of one chunk)
// where the makespan comes from dispatching every CTA, in that order, to the
// first free of the device's SMs, a CTA costing its chunks plus two for its
// ramp (prefix and first tiles), and nseg / 2 stands for the scan work a
// segment adds.  Plans are cached per (BH, T, SM count).
constexpr int kGranule = 128;
// SM count assumed when no device can be queried (a machine without a
// visible GPU asking for a workspace size): GB300's 152.  A forward always
// plans with the count of the device it runs on, queried once per device.
constexpr int kFallbackSMs = 152;

int current_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();  // clear the (non-sticky) error of a machine without a device
        return kFallbackSMs;
    }
    static std::atomic<int> cache[kMaxDevices];
    const int known = cache[dev].load(std::memory_order_relaxed);
    if (known > 0) return known;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return kFallbackSMs;
    }
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {
long long plan_makespan2(long long BH, int nchunk, int seglen, int nseg, int sms) {
    // twice the makespan, in chunk units (a CTA costs its chunks + 2)
    const int tail = nchunk - (nseg - 1) * seglen;
    const bool short_tail = nseg > 1 && tail < seglen;
    const long long full = short_tail ? BH * (nseg - 1) : BH * nseg;
    const long long a = seglen + 2, b = tail + 2;
    // full-length CTAs first: equal jobs fill the SMs round by round
    const long long q = full / sms, r = full % sms;
    long long span = (r > 0 ? q + 1 : q) * a;
    if (!short_tail) return 2 * span;
    if (BH > 20000) {  // too many to place one by one: treat them as one more round
        return 2 * (span + ((BH + sms - 1) / sms) * b);
    }
    std::priority_queue<long long, std::vector<long long>, std::greater<long long>> load;
    for (long long i = 0; i < sms; ++i) load.push(i < r ? (q + 1) * a : q * a);
    for (long long i = 0; i < BH; ++i) {
        const long long t = load.top() + b;
        load.pop();
        load.push(t);
        if (t > span) span = t;
    }
    return 2 * span;
}
}  // namespace

SegPlan forward_plan(int BH, int T, int sms) {
    if (sms <= 0) sms = current_sm_count();
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, SegPlan> cache;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find({BH, T, sms});
        if (it != cache.end()) return it->second;
    }
    SegPlan p;
    p.granule = kGranule;
    p.nchunk = (T + kGranule - 1) / kGranule;
    long long best_cost = -1;
    p.nseg = 1;
    p.seglen = p.nchunk;
    const int len0 = (p.nchunk + 4095) / 4096;  // at most 4096 segments per head
    for (int len = len0 > 0 ? len0 : 1; len <= p.nchunk; ++len) {
        const int nseg = (p.nchunk + len - 1) / len;
        const long long cost2 = plan_makespan2(BH, p.nchunk, len, nseg, sms) + nseg;
        if (best_cost < 0 || cost2 < best_cost) {
            best_cost = cost2;
            p.nseg = nseg;
            p.seglen = len;
        }
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[{BH, T, sms}] = p;
    return p;
}

struct FwdWorkspace {
    float* summ;    // [BH][nseg][R]
    float* prefix;  // [BH][nseg][R]
    float* tot;     // [BH][R]
    float* fac;     // [2][nseg] decay factors of the segments (decayed operator)
    size_t bytes;
};

FwdWorkspace carve(void* base, int BH, SegPlan p, int d, int dv) {
    const size_t R = record_len(d, dv);
    const size_t seg_floats = (size_t)BH * p.nseg * R;
    auto up = [](size_t n) { return (n + 63) & ~size_t(63); };  // 256-byte granules
    FwdWorkspace w;
    char* c = static_cast<char*>(base);
    w.summ = reinterpret_cast<float*>(c);
    w.prefix = reinterpret_cast<float*>(c + up(seg_floats) * 4);
    w.tot = reinterpret_cast<float*>(c + 2 * up(seg_floats) * 4);
    w.fac = reinterpret_cast<float*>(c + (2 * up(seg_floats) + up((size_t)BH * R)) * 4);
    w.bytes = (2 * up(seg_floats) + up((size_t)BH * R) + up(2 * (size_t)p.nseg)) * 4;
    return w;
}

int check_common(const void* Q, const void* K, const void* V, int B, int H, int T, int d, int dv, int dtype) {
    if (!Q || !K || !V) return fail(HLA2_ERR_INVALID, "null input pointer");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V)) return fail(HLA2_ERR_INVALID, "input pointer not 16-byte aligned");
    if (B <= 0 || H <= 0 || T <= 0 || d <= 0 || dv <= 0)
        return fail(HLA2_ERR_INVALID, "sizes must be positive (B=%d H=%d T=%d d=%d dv=%d)", B, H, T, d, dv);
    if (dtype != HLA2_DTYPE_F32 && dtype != HLA2_DTYPE_BF16) return fail(HLA2_ERR_UNSUPPORTED, "unknown dtype %d", dtype);
    if (d > 128 || dv > 128) return fail(HLA2_ERR_UNSUPPORTED, "d=%d dv=%d: this build supports d, dv <= 128", d, dv);
    const long long BH = (long long)B * H;
    if (BH > 65535) return fail(HLA2_ERR_UNSUPPORTED, "B*H=%lld exceeds 65535", BH);
    if (BH * T * (long long)(d > dv ? d : dv) > (1LL << 40)) return fail(HLA2_ERR_UNSUPPORTED, "problem too large");
    return HLA2_OK;
}

}  // namespace

// ---- instrumentation: launch counter and per-phase events ----
namespace {
std::atomic<long long> g_launches{0};
std::atomic<int> g_profile_on{0};
std::mutex g_prof_mu;
struct PhaseEvents {
    cudaEvent_t ev[4];
};
std::vector<PhaseEvents> g_prof_pending;  // recorded, not yet read
std::vector<PhaseEvents> g_prof_pool;     // reusable

bool prof_begin(PhaseEvents& pe) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_pool.empty()) {
        pe = g_prof_pool.back();
        g_prof_pool.pop_back();
        return true;
    }
    for (int i = 0; i < 4; ++i)
        if (cudaEventCreate(&pe.ev[i]) != cudaSuccess) return false;
    return true;
}
void prof_commit(const PhaseEvents& pe) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_pending.push_back(pe);
}
}  // namespace

void note_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int set_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int* device_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_addr[dev] = static_cast<int*>(p);
    }
    return g_status_addr[dev];
}

// Runs the P-form scan over the segment summaries in ws (see hla2_scan.cu),
// leaving every segment's exclusive prefix in ws.prefix and, when wanted,
// the inclusive totals in ws.tot.
static int forward_scan(const FwdWorkspace& ws, int BH, SegPlan plan, int d, int dv, bool want_extra,
                        bool want_tot, bool use_tc, int* status, cudaStream_t s) {
    const RecOff ro = summary_offsets(d, dv);
    const size_t R = ro.R;
    cudaError_t e;
    // 1. exclusive sums of S (the walks read only S and P from a prefix;
    //    C and m are summed too when the final state is wanted)
    e = launch_exscan(ws.summ, ws.prefix, BH, plan.nseg, R, 0, want_tot ? ro.X : (size_t)d * d,
                      want_tot ? ws.tot : nullptr, R, s);
    if (e != cudaSuccess) return cuda_fail(e, "scan: prefix sums of S, C, m");
    // 2. X_r = P_r + S_<r C_r  (and p_r + S_<r m_r)
    CrossArgs a{};
    a.A = ws.prefix + ro.S; a.sA = (long long)R;
    a.B = ws.summ + ro.C;   a.sB = (long long)R;
    a.bx = want_extra ? ws.summ + ro.m : nullptr; a.sbx = (long long)R;
    a.base = ws.summ + ro.X; a.sbase = (long long)R;
    a.basex = ws.summ + ro.x; a.sbasex = (long long)R;
    a.out = ws.prefix + ro.X; a.sout = (long long)R;
    a.outx = want_extra ? ws.prefix + ro.x : nullptr; a.soutx = (long long)R;
    a.alpha = 1.f; a.d = d; a.dv = dv; a.status = status;
    for (long long b0 = 0; b0 < (long long)BH * plan.nseg; b0 += 65535) {
        CrossArgs c = a;
        const long long nb = (long long)BH * plan.nseg - b0;
        c.nb = (int)(nb < 65535 ? nb : 65535);
        c.A += b0 * R; c.B += b0 * R; if (c.bx) c.bx += b0 * R;
        c.base += b0 * R; c.basex += b0 * R; c.out += b0 * R; if (c.outx) c.outx += b0 * R;
        // tensor cores (split-bf16 operands) on the tensor-core path; exact fp32 otherwise
        e = (use_tc && !want_extra) ? launch_tc_cross(c, s) : launch_cross(c, s);
        if (e != cudaSuccess) return cuda_fail(e, "scan: cross terms");
    }
    // 3. exclusive sums of the corrected part P | p (in place)
    const size_t xlen = want_extra ? R - ro.X : (size_t)d * dv;
    e = launch_exscan(ws.prefix, ws.prefix, BH, plan.nseg, R, ro.X, xlen, want_tot ? ws.tot + ro.X : nullptr, R, s);
    if (e != cudaSuccess) return cuda_fail(e, "scan: prefix sums of P");
    return HLA2_OK;
}

// AHLA scan over the segment summaries M|P|m|E|n (HLA summary, section 2 for
// the summaries, section 4 for the combine).  E_AB = E_A + E_B + M_B P_A makes
// the exclusive prefix unroll to E_<n = sum_{r<n} (E_r + M_r P_<r):
//   1. exclusive sums of P (and m),
//   2. Y_r = E_r + M_r P_<r (and n_r + M_r m_<r), one product per record,
//   3. exclusive sums of Y in place.
// M itself is never summed: no prefix or final state needs it.
static int forward_scan_ahla(const FwdWorkspace& ws, int BH, SegPlan plan, int d, int dv, bool want_extra,
                             bool want_tot, bool use_tc, int* status, cudaStream_t s) {
    const RecOff ro = summary_offsets(d, dv);
    const size_t R = ro.R;
    cudaError_t e;
    const size_t plen = want_extra ? (size_t)d * dv + d : (size_t)d * dv;  // P (| m)
    e = launch_exscan(ws.summ, ws.prefix, BH, plan.nseg, R, ro.C, plen, want_tot ? ws.tot + ro.C : nullptr, R, s);
    if (e != cudaSuccess) return cuda_fail(e, "ahla scan: prefix sums of P, m");
    CrossArgs a{};
    a.A = ws.summ + ro.S;   a.sA = (long long)R;      // M_r
    a.B = ws.prefix + ro.C; a.sB = (long long)R;      // P_<r
    a.bx = want_extra ? ws.prefix + ro.m : nullptr; a.sbx = (long long)R;  // m_<r
    a.base = ws.summ + ro.X; a.sbase = (long long)R;  // E_r
    a.basex = ws.summ + ro.x; a.sbasex = (long long)R;  // n_r
    a.out = ws.prefix + ro.X; a.sout = (long long)R;
    a.outx = want_extra ? ws.prefix + ro.x : nullptr; a.soutx = (long long)R;
    a.alpha = 1.f; a.d = d; a.dv = dv; a.status = status;
    for (long long b0 = 0; b0 < (long long)BH * plan.nseg; b0 += 65535) {
        CrossArgs c = a;
        const long long nb = (long long)BH * plan.nseg - b0;
        c.nb = (int)(nb < 65535 ? nb : 65535);
        c.A += b0 * R; c.B += b0 * R; if (c.bx) c.bx += b0 * R;
        c.base += b0 * R; c.basex += b0 * R; c.out += b0 * R; if (c.outx) c.outx += b0 * R;
        e = (use_tc && !want_extra) ? launch_tc_cross(c, s) : launch_cross(c, s);
        if (e != cudaSuccess) return cuda_fail(e, "ahla scan: cross terms");
    }
    const size_t elen = want_extra ? (size_t)d * dv + d : (size_t)d * dv;  // E (| n)
    e = launch_exscan(ws.prefix, ws.prefix, BH, plan.nseg, R, ro.X, elen, want_tot ? ws.tot + ro.X : nullptr, R, s);
    if (e != cudaSuccess) return cuda_fail(e, "ahla scan: prefix sums of E, n");
    return HLA2_OK;
}

}  // namespace hla2

using namespace hla2;

extern "C" {

size_t hla2_forward_workspace(int B, int H, int T, int d, int dv, int dtype) {
    if (B <= 0 || H <= 0 || T <= 0 || d <= 0 || dv <= 0 || d > 128 || dv > 128) return 0;
    if (dtype != HLA2_DTYPE_F32 && dtype != HLA2_DTYPE_BF16) return 0;
    if ((long long)B * H > 65535) return 0;
    const int BH = B * H;
    SegPlan p = forward_plan(BH, T, 0);
    return carve(nullptr, BH, p, d, dv).bytes;
}

int hla2_forward_plan(int B, int H, int T, int sm_count, int* nseg, int* chunks_per_segment, int* sm_count_used) {
    if (B <= 0 || H <= 0 || T <= 0) return fail(HLA2_ERR_INVALID, "sizes must be positive (B=%d H=%d T=%d)", B, H, T);
    if (!nseg || !chunks_per_segment) return fail(HLA2_ERR_INVALID, "null output pointer");
    if ((long long)B * H > 65535) return fail(HLA2_ERR_UNSUPPORTED, "B*H=%lld exceeds 65535", (long long)B * H);
    const int sms = sm_count > 0 ? sm_count : current_sm_count();
    const SegPlan p = forward_plan(B * H, T, sms);
    *nseg = p.nseg;
    *chunks_per_segment = p.seglen;
    if (sm_count_used) *sm_count_used = sms;
    return HLA2_OK;
}

int hla2_forward(const void* Q, const void* K, const void* V, float* O, int B, int H, int T, int d, int dv,
                 int normalized, int dtype, void* workspace, size_t ws_bytes, float* state_out,
                 hla2_stream_t stream) {
    int rc = check_common(Q, K, V, B, H, T, d, dv, dtype);
    if (rc) return rc;
    if (!O) return fail(HLA2_ERR_INVALID, "null output pointer");
    if (!aligned16(O) || (state_out && !aligned16(state_out))) return fail(HLA2_ERR_INVALID, "output pointer not 16-byte aligned");
    const size_t need = hla2_forward_workspace(B, H, T, d, dv, dtype);
    if (!workspace || ws_bytes < need)
        return fail(HLA2_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace ? ws_bytes : (size_t)0, need);
    if (!aligned16(workspace)) return fail(HLA2_ERR_INVALID, "workspace not 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int BH = B * H;
    const SegPlan plan = forward_plan(BH, T, 0);
    const FwdWorkspace ws = carve(workspace, BH, plan, d, dv);
    const bool want_extra = normalized || state_out;  // p (and m) needed
    int dev = 0;
    cudaGetDevice(&dev);
    const bool use_tc = tc_supported(d, dv, dtype, normalized, dev);
    int* status = device_status_word();
    if (!status) return fail(HLA2_ERR_LAUNCH, "cannot resolve the device status word");
    cudaError_t e;
    PhaseEvents pe;
    const bool prof = g_profile_on.load() && prof_begin(pe);
    if (prof) cudaEventRecord(pe.ev[0], s);

    // segment summaries (with the final state wanted the tensor-core walk
    // also forms m and p, which the normalised walk always does)
    const RecOff ro = summary_offsets(d, dv);
    if (use_tc) {
        e = launch_tc_walk(0, Q, K, V, nullptr, nullptr, ws.summ, BH, T, d, dv, normalized, plan, status, s,
                           state_out && !normalized);
    } else {
        e = launch_walk(0, Q, K, V, dtype, nullptr, nullptr, ws.summ, BH, T, d, dv, normalized, 0, 1.0f, plan, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "segment summaries");
    if (prof) cudaEventRecord(pe.ev[1], s);
    // exclusive scan of the summaries: one launch on the tensor-core path
    // (plus the running sums of the terms for long scans or a final state)
    if (use_tc) {
        const bool extra = normalized || state_out;
        ScanArgs sa{ws.summ, ws.prefix, plan.nseg, ro.R, ro, nullptr, status, extra};
        if (state_out) {
            sa.terms_only = true;
            sa.tot = ws.tot;  // plain totals of S | C | m
            sa.tot_len = ro.X;
        }
        e = launch_tc_scan(kScanHLA, sa, BH, d, dv, s);
        if (e == cudaSuccess && (state_out || plan.nseg > tc_scan_full_max_segments()))
            // exclusive sums of the terms X_r (and x_r), with their totals
            e = launch_exscan(ws.prefix, ws.prefix, BH, plan.nseg, ro.R, ro.X, (size_t)d * dv + (extra ? (size_t)d : 0),
                              state_out ? ws.tot + ro.X : nullptr, ro.R, s);
        if (e != cudaSuccess) return cuda_fail(e, "scan");
    } else {
        rc = forward_scan(ws, BH, plan, d, dv, want_extra, state_out != nullptr, use_tc, status, s);
        if (rc) return rc;
    }
    if (prof) cudaEventRecord(pe.ev[2], s);
    // outputs
    if (use_tc) e = launch_tc_walk(1, Q, K, V, O, ws.prefix, nullptr, BH, T, d, dv, normalized, plan, status, s);
    else e = launch_walk(1, Q, K, V, dtype, O, ws.prefix, nullptr, BH, T, d, dv, normalized, 0, 1.0f, plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "segment outputs");
    if (prof) {
        cudaEventRecord(pe.ev[3], s);
        prof_commit(pe);
    }

    if (state_out) {
        // final state in decode order S|C|G|m|h: G = S C - P, h = S m - p
        e = launch_state_tail(ws.tot, state_out, BH, d, dv, s);
        if (e != cudaSuccess) return cuda_fail(e, "state_out");
    }
    return HLA2_OK;
}

int hla2_step(float* state, const float* q, const float* k, const float* v, float* o, int n, int d, int dv,
              int normalized, hla2_stream_t stream) {
    if (!state || !q || !k || !v || !o) return fail(HLA2_ERR_INVALID, "null pointer");
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return fail(HLA2_ERR_INVALID, "pointer not 16-byte aligned");
    if (n <= 0 || d <= 0 || dv <= 0) return fail(HLA2_ERR_INVALID, "sizes must be positive (n=%d d=%d dv=%d)", n, d, dv);
    auto pow2_4_128 = [](int x) { return x >= 4 && x <= 128 && (x & (x - 1)) == 0; };
    if (!pow2_4_128(d) || !pow2_4_128(dv))
        return fail(HLA2_ERR_UNSUPPORTED, "hla2_step needs d, dv powers of two in [4, 128] (d=%d dv=%d)", d, dv);
    if (n > 2147483647 / 2) return fail(HLA2_ERR_UNSUPPORTED, "n too large");
    cudaError_t e = launch_step(state, q, k, v, o, n, d, dv, normalized, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "hla2_step");
    return HLA2_OK;
}

int hla2_step_pform(float* state, const float* q, const float* k, const float* v, float* o, int n, int d, int dv,
                    int normalized, hla2_stream_t stream) {
    if (!state || !q || !k || !v || !o) return fail(HLA2_ERR_INVALID, "null pointer");
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return fail(HLA2_ERR_INVALID, "pointer not 16-byte aligned");
    if (n <= 0 || d <= 0 || dv <= 0) return fail(HLA2_ERR_INVALID, "sizes must be positive (n=%d d=%d dv=%d)", n, d, dv);
    auto pow2_4_128 = [](int x) { return x >= 4 && x <= 128 && (x & (x - 1)) == 0; };
    if (!pow2_4_128(d) || !pow2_4_128(dv))
        return fail(HLA2_ERR_UNSUPPORTED, "hla2_step_pform needs d, dv powers of two in [4, 128] (d=%d dv=%d)", d, dv);
    cudaError_t e = launch_step_pform(state, q, k, v, o, n, d, dv, normalized, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "hla2_step_pform");
    return HLA2_OK;
}

int hla2_state_to_pform(const float* gstate, float* pstate, int n, int d, int dv, hla2_stream_t stream) {
    if (!gstate || !pstate) return fail(HLA2_ERR_INVALID, "null pointer");
    if (!aligned16(gstate) || !aligned16(pstate)) return fail(HLA2_ERR_INVALID, "pointer not 16-byte aligned");
    if (n <= 0 || d <= 0 || dv <= 0) return fail(HLA2_ERR_INVALID, "sizes must be positive (n=%d d=%d dv=%d)", n, d, dv);
    if (d > 128 || dv > 128) return fail(HLA2_ERR_UNSUPPORTED, "d, dv must be <= 128");
    const RecOff g = decode_offsets(d, dv);
    const long long Rg = (long long)g.R;
    const long long Rp = (long long)d * d + (long long)d * dv + d;
    if (gstate < pstate + n * Rp && pstate < gstate + n * Rg) return fail(HLA2_ERR_INVALID, "gstate and pstate overlap");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (long long b0 = 0; b0 < n; b0 += 65535) {
        const int nb = (int)((n - b0) < 65535 ? (n - b0) : 65535);
        const float* gs = gstate + b0 * Rg;
        float* ps = pstate + b0 * Rp;
        cudaError_t e = launch_copy_strided(gs + g.S, Rg, ps, Rp, (size_t)d * d, nb, s);
        if (e != cudaSuccess) return cuda_fail(e, "hla2_state_to_pform: copy S");
        CrossArgs a{};
        a.A = gs + g.S; a.sA = Rg;                 // S
        a.B = gs + g.C; a.sB = Rg;                 // C
        a.bx = gs + g.m; a.sbx = Rg;               // m (extra column)
        a.base = gs + g.X; a.sbase = Rg;           // G
        a.basex = gs + g.x; a.sbasex = Rg;         // h
        a.out = ps + (size_t)d * d; a.sout = Rp;   // P = S C - G
        a.outx = ps + (size_t)d * d + (size_t)d * dv; a.soutx = Rp;  // p = S m - h
        a.alpha = -1.f; a.d = d; a.dv = dv; a.nb = nb;
        e = launch_cross(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "hla2_state_to_pform: products");
    }
    return HLA2_OK;
}

int hla2_chunk_summaries(const void* Q, const void* K, const void* V, float* summ, int B, int H, int T, int d,
                         int dv, int L, int dtype, hla2_stream_t stream) {
    int rc = check_common(Q, K, V, B, H, T, d, dv, dtype);
    if (rc) return rc;
    if (!summ) return fail(HLA2_ERR_INVALID, "null summary pointer");
    if (!aligned16(summ)) return fail(HLA2_ERR_INVALID, "summary pointer not 16-byte aligned");
    if (L <= 0) return fail(HLA2_ERR_INVALID, "chunk length must be positive (L=%d)", L);
    SegPlan p;
    p.granule = L;
    p.nchunk = (T + L - 1) / L;
    p.nseg = p.nchunk;  // one chunk per segment
    p.seglen = 1;
    if (p.nseg > 65535) return fail(HLA2_ERR_UNSUPPORTED, "%d chunks per head exceeds 65535", p.nseg);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e;
    if (tc_chunk_supported(d, dv, L, dtype, dev)) {
        int* status = device_status_word();
        if (!status) return fail(HLA2_ERR_LAUNCH, "cannot resolve the device status word");
        e = launch_tc_chunk(Q, K, V, summ, B * H, T, d, L, status, s);
    } else {
        e = launch_walk(2, Q, K, V, dtype, nullptr, nullptr, summ, B * H, T, d, dv, 0, 0, 1.0f, p, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "hla2_chunk_summaries");
    return HLA2_OK;
}

int hla2_scan(const float* summ, float* prefix, int B, int H, int N, int d, int dv, hla2_stream_t stream) {
    if (!summ || !prefix) return fail(HLA2_ERR_INVALID, "null pointer");
    if (!aligned16(summ) || !aligned16(prefix)) return fail(HLA2_ERR_INVALID, "pointer not 16-byte aligned");
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0 || dv <= 0)
        return fail(HLA2_ERR_INVALID, "sizes must be positive (B=%d H=%d N=%d d=%d dv=%d)", B, H, N, d, dv);
    if (d > 128 || dv > 128) return fail(HLA2_ERR_UNSUPPORTED, "d, dv must be <= 128");
    if ((long long)B * H > 65535) return fail(HLA2_ERR_UNSUPPORTED, "B*H exceeds 65535");
    const RecOff ro = summary_offsets(d, dv);
    const size_t R = ro.R;
    const long long BH = (long long)B * H;
    const long long total = BH * N * (long long)R;
    if (summ < prefix + total && prefix < summ + total) return fail(HLA2_ERR_INVALID, "summ and prefix overlap");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // 1. exclusive sums of S | C | m
    cudaError_t e = launch_exscan(summ, prefix, (int)BH, N, R, 0, ro.X, nullptr, 0, s);
    if (e != cudaSuccess) return cuda_fail(e, "hla2_scan: prefix sums");
    // 2. Y_r = G_r + S_r C_<r, y_r = h_r + S_r m_<r (tensor cores with
    //    split-bf16 operands where they apply, exact fp32 otherwise)
    int dev = 0;
    cudaGetDevice(&dev);
    const bool use_tc = tc_supported(d, dv, HLA2_DTYPE_BF16, 0, dev);
    int* status = use_tc ? device_status_word() : nullptr;
    if (use_tc && !status) return fail(HLA2_ERR_LAUNCH, "cannot resolve the device status word");
    CrossArgs a{};
    a.A = summ + ro.S; a.sA = (long long)R;
    a.B = prefix + ro.C; a.sB = (long long)R;
    a.bx = prefix + ro.m; a.sbx = (long long)R;
    a.base = summ + ro.X; a.sbase = (long long)R;
    a.basex = summ + ro.x; a.sbasex = (long long)R;
    a.out = prefix + ro.X; a.sout = (long long)R;
    a.outx = prefix + ro.x; a.soutx = (long long)R;
    a.alpha = 1.f; a.d = d; a.dv = dv; a.status = status;
    for (long long b0 = 0; b0 < BH * N; b0 += 65535) {
        CrossArgs c = a;
        const long long nb = BH * N - b0;
        c.nb = (int)(nb < 65535 ? nb : 65535);
        c.A += b0 * R; c.B += b0 * R; c.bx += b0 * R;
        c.base += b0 * R; c.basex += b0 * R; c.out += b0 * R; c.outx += b0 * R;
        e = use_tc ? launch_tc_cross(c, s) : launch_cross(c, s);
        if (e != cudaSuccess) return cuda_fail(e, "hla2_scan: cross terms");
    }
    // 3. exclusive sums of G | h (in place)
    e = launch_exscan(prefix, prefix, (int)BH, N, R, ro.X, R - ro.X, nullptr, 0, s);
    if (e != cudaSuccess) return cuda_fail(e, "hla2_scan: prefix sums of G");
    return HLA2_OK;
}

int hla2_selftest_wait_runout(int* flag, int wait_us, hla2_stream_t stream) {
    if (!flag) return fail(HLA2_ERR_INVALID, "null flag pointer");
    if (reinterpret_cast<uintptr_t>(flag) % 4 != 0) return fail(HLA2_ERR_INVALID, "flag pointer not 4-byte aligned");
    if (wait_us < 1 || wait_us > 2000000) return fail(HLA2_ERR_INVALID, "wait_us must be in [1, 2000000] (got %d)", wait_us);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(HLA2_ERR_LAUNCH, "no current device");
    if (!tc_supported(64, 64, HLA2_DTYPE_BF16, 0, dev))
        return fail(HLA2_ERR_UNSUPPORTED, "the self-test needs tensor memory (sm_103)");
    int* status = device_status_word();
    if (!status) return fail(HLA2_ERR_LAUNCH, "cannot resolve the device status word");
    cudaError_t e = launch_selftest_runout(status, 1000ull * (unsigned long long)wait_us, flag,
                                           reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "self-test");
    return HLA2_OK;
}

int hla2_forward_path(int d, int dv, int dtype, int normalized, int with_state_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    (void)with_state_out;  // the tensor-core forward also hands over the final state
    return tc_supported(d, dv, dtype, normalized, dev) ? 1 : 0;
}

int hla2_chunk_summaries_path(int d, int dv, int L, int dtype) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return tc_chunk_supported(d, dv, L, dtype, dev) ? 1 : 0;
}

int hla2_profile_enable(int on) {
    g_profile_on.store(on ? 1 : 0);
    return HLA2_OK;
}

int hla2_profile_read(float* ms_out, int n, int* forwards, long long* launches) {
    std::vector<PhaseEvents> pend;
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        pend.swap(g_prof_pending);
    }
    float acc[3] = {0.f, 0.f, 0.f};
    int rc = HLA2_OK;
    for (auto& pe : pend) {
        if (cudaEventSynchronize(pe.ev[3]) != cudaSuccess) rc = fail(HLA2_ERR_LAUNCH, "profile event sync failed");
        for (int i = 0; i < 3; ++i) {
            float ms = 0.f;
            if (cudaEventElapsedTime(&ms, pe.ev[i], pe.ev[i + 1]) == cudaSuccess) acc[i] += ms;
        }
    }
    for (int i = 0; i < n && i < 3; ++i) ms_out[i] = acc[i];
    if (forwards) *forwards = (int)pend.size();
    if (launches) *launches = g_launches.exchange(0);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto& pe : pend) g_prof_pool.push_back(pe);
    return rc;
}

int hla2_last_error_detail(char* buf, size_t n) {
    const std::string& m = t_last_error;
    if (buf && n) {
        size_t c = m.size() < n - 1 ? m.size() : n - 1;
        memcpy(buf, m.data(), c);
        buf[c] = '\0';
    }
    return (int)m.size();
}

int hla2_device_status(hla2_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "hla2_device_status: stream synchronize");
    int* w = device_status_word();
    if (!w) return fail(HLA2_ERR_LAUNCH, "cannot resolve the device status word");
    int v = 0;
    e = cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "hla2_device_status: read");
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "hla2_device_status: clear");
        return fail(HLA2_ERR_DEVICE, "device reported error %d (%s)", v,
                    v == kDevWaitTimeout ? "bounded wait ran out" : v == kDevBounds ? "bounds check failed"
                                                                           : v == kDevTmemAlloc ? "tensor memory allocation"
                                                                                                : "unknown");
    }
    return HLA2_OK;
}


int hla2_ahla_forward(const void* Q, const void* K, const void* V, float* O, int B, int H, int T, int d, int dv,
                      int normalized, int dtype, void* workspace, size_t ws_bytes, float* state_out,
                      hla2_stream_t stream) {
    int rc = check_common(Q, K, V, B, H, T, d, dv, dtype);
    if (rc) return rc;
    if (!O) return fail(HLA2_ERR_INVALID, "null output pointer");
    if (!aligned16(O) || (state_out && !aligned16(state_out))) return fail(HLA2_ERR_INVALID, "output pointer not 16-byte aligned");
    const size_t need = hla2_forward_workspace(B, H, T, d, dv, dtype);
    if (!workspace || ws_bytes < need)
        return fail(HLA2_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace ? ws_bytes : (size_t)0, need);
    if (!aligned16(workspace)) return fail(HLA2_ERR_INVALID, "workspace not 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int BH = B * H;
    const SegPlan plan = forward_plan(BH, T, 0);
    const FwdWorkspace ws = carve(workspace, BH, plan, d, dv);
    const bool want_extra = normalized || state_out;  // m and n needed
    int* status = device_status_word();
    if (!status) return fail(HLA2_ERR_LAUNCH, "cannot resolve the device status word");
    const bool use_tc = hla2_ahla_forward_path(d, dv, dtype, normalized, state_out != nullptr) == 1;
    cudaError_t e = use_tc ? launch_ahla_tc_walk(0, Q, K, V, nullptr, nullptr, ws.summ, BH, T, d, dv, plan, status, s)
                           : launch_ahla_walk(0, Q, K, V, dtype, nullptr, nullptr, ws.summ, BH, T, d, dv, normalized,
                                              plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "ahla segment summaries");
    if (use_tc) {
        const RecOff ro = summary_offsets(d, dv);
        const ScanArgs sa{ws.summ, ws.prefix, plan.nseg, ro.R, ro, nullptr, status, false};
        e = launch_tc_scan(kScanAHLA, sa, BH, d, dv, s);
        if (e == cudaSuccess && plan.nseg > tc_scan_full_max_segments())  // exclusive sums of the terms Y_r
            e = launch_exscan(ws.prefix, ws.prefix, BH, plan.nseg, ro.R, ro.X, (size_t)d * dv, nullptr, 0, s);
        if (e != cudaSuccess) return cuda_fail(e, "ahla scan");
    } else {
        rc = forward_scan_ahla(ws, BH, plan, d, dv, want_extra, state_out != nullptr, use_tc, status, s);
        if (rc) return rc;
    }
    e = use_tc ? launch_ahla_tc_walk(1, Q, K, V, O, ws.prefix, nullptr, BH, T, d, dv, plan, status, s)
               : launch_ahla_walk(1, Q, K, V, dtype, O, ws.prefix, nullptr, BH, T, d, dv, normalized, plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "ahla segment outputs");
    if (state_out) {
        // final state in decode order P|E|m|n from the scan totals
        const RecOff so = summary_offsets(d, dv);
        const long long R = (long long)so.R;
        const long long Rs = 2LL * d * dv + 2LL * d;
        const size_t nC = (size_t)d * dv;
        e = launch_copy_strided(ws.tot + so.C, R, state_out, Rs, nC, BH, s);
        if (e == cudaSuccess) e = launch_copy_strided(ws.tot + so.X, R, state_out + nC, Rs, nC, BH, s);
        if (e == cudaSuccess) e = launch_copy_strided(ws.tot + so.m, R, state_out + 2 * nC, Rs, (size_t)d, BH, s);
        if (e == cudaSuccess) e = launch_copy_strided(ws.tot + so.x, R, state_out + 2 * nC + d, Rs, (size_t)d, BH, s);
        if (e != cudaSuccess) return cuda_fail(e, "ahla state_out copy");
    }
    return HLA2_OK;
}

int hla2_ahla_forward_path(int d, int dv, int dtype, int normalized, int with_state_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return (!normalized && !with_state_out && tc_supported(d, dv, dtype, 0, dev)) ? 1 : 0;
}

int hla2_ahla_step(float* state, const float* q, const float* k, const float* v, float* o, int n, int d, int dv,
                   int normalized, hla2_stream_t stream) {
    if (!state || !q || !k || !v || !o) return fail(HLA2_ERR_INVALID, "null pointer");
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return fail(HLA2_ERR_INVALID, "pointer not 16-byte aligned");
    if (n <= 0 || d <= 0 || dv <= 0) return fail(HLA2_ERR_INVALID, "sizes must be positive (n=%d d=%d dv=%d)", n, d, dv);
    auto pow2_4_128 = [](int x) { return x >= 4 && x <= 128 && (x & (x - 1)) == 0; };
    if (!pow2_4_128(d) || !pow2_4_128(dv))
        return fail(HLA2_ERR_UNSUPPORTED, "hla2_ahla_step needs d, dv powers of two in [4, 128] (d=%d dv=%d)", d, dv);
    cudaError_t e = launch_ahla_step(state, q, k, v, o, n, d, dv, normalized, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "hla2_ahla_step");
    return HLA2_OK;
}


int hla2_unmasked_forward(const void* Q, const void* K, const void* V, float* O, int B, int H, int T, int d, int dv,
                          int normalized, int dtype, void* workspace, size_t ws_bytes, float* state_out,
                          hla2_stream_t stream) {
    int rc = check_common(Q, K, V, B, H, T, d, dv, dtype);
    if (rc) return rc;
    if (!O) return fail(HLA2_ERR_INVALID, "null output pointer");
    if (!aligned16(O) || (state_out && !aligned16(state_out))) return fail(HLA2_ERR_INVALID, "output pointer not 16-byte aligned");
    const size_t need = hla2_forward_workspace(B, H, T, d, dv, dtype);
    if (!workspace || ws_bytes < need)
        return fail(HLA2_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace ? ws_bytes : (size_t)0, need);
    if (!aligned16(workspace)) return fail(HLA2_ERR_INVALID, "workspace not 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int BH = B * H;
    const SegPlan plan = forward_plan(BH, T, 0);
    const FwdWorkspace ws = carve(workspace, BH, plan, d, dv);
    const RecOff ro = summary_offsets(d, dv);
    const bool use_tc = hla2_unmasked_forward_path(d, dv, dtype, normalized, state_out != nullptr) == 1;
    int* status = nullptr;
    if (use_tc && !(status = device_status_word())) return fail(HLA2_ERR_LAUNCH, "cannot resolve the device status word");
    // segment sums S|C|m (S|C on tensor cores), their exclusive prefix sums
    // (the combine has no cross term here), then the walks from the prefixes
    cudaError_t e = use_tc ? launch_unm_tc_walk(0, Q, K, V, nullptr, nullptr, ws.summ, BH, T, d, dv, plan, status, s)
                           : launch_walk(0, Q, K, V, dtype, nullptr, nullptr, ws.summ, BH, T, d, dv, normalized, 1, 1.0f,
                                         plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "unmasked segment sums");
    e = launch_exscan(ws.summ, ws.prefix, BH, plan.nseg, ro.R, 0, use_tc ? ro.m : ro.X, state_out ? ws.tot : nullptr,
                      ro.R, s);
    if (e != cudaSuccess) return cuda_fail(e, "unmasked prefix sums");
    e = use_tc ? launch_unm_tc_walk(1, Q, K, V, O, ws.prefix, nullptr, BH, T, d, dv, plan, status, s)
               : launch_walk(1, Q, K, V, dtype, O, ws.prefix, nullptr, BH, T, d, dv, normalized, 1, 1.0f, plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "unmasked segment outputs");
    if (state_out) {
        // final state S|C|m: the first d*d + d*dv + d floats of the totals
        e = launch_copy_strided(ws.tot, (long long)ro.R, state_out, (long long)ro.X, ro.X, BH, s);
        if (e != cudaSuccess) return cuda_fail(e, "unmasked state_out copy");
    }
    return HLA2_OK;
}

int hla2_decay_forward_path(int d, int dv, int dtype, int normalized, int with_state_out, float gamma) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return (!normalized && !with_state_out && decay_tc_gamma_ok(gamma) && tc_supported(d, dv, dtype, 0, dev)) ? 1 : 0;
}

int hla2_unmasked_forward_path(int d, int dv, int dtype, int normalized, int with_state_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return (!normalized && !with_state_out && tc_supported(d, dv, dtype, 0, dev)) ? 1 : 0;
}

int hla2_unmasked_step(float* state, const float* q, const float* k, const float* v, float* o, int n, int d, int dv,
                       int normalized, hla2_stream_t stream) {
    if (!state || !q || !k || !v || !o) return fail(HLA2_ERR_INVALID, "null pointer");
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return fail(HLA2_ERR_INVALID, "pointer not 16-byte aligned");
    if (n <= 0 || d <= 0 || dv <= 0) return fail(HLA2_ERR_INVALID, "sizes must be positive (n=%d d=%d dv=%d)", n, d, dv);
    auto pow2_4_128 = [](int x) { return x >= 4 && x <= 128 && (x & (x - 1)) == 0; };
    if (!pow2_4_128(d) || !pow2_4_128(dv))
        return fail(HLA2_ERR_UNSUPPORTED, "hla2_unmasked_step needs d, dv powers of two in [4, 128] (d=%d dv=%d)", d, dv);
    cudaError_t e = launch_step_unmasked(state, q, k, v, o, n, d, dv, normalized, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "hla2_unmasked_step");
    return HLA2_OK;
}


int hla2_decay_forward(const void* Q, const void* K, const void* V, float* O, int B, int H, int T, int d, int dv,
                       int normalized, float gamma, int dtype, void* workspace, size_t ws_bytes, float* state_out,
                       hla2_stream_t stream) {
    int rc = check_common(Q, K, V, B, H, T, d, dv, dtype);
    if (rc) return rc;
    if (!O) return fail(HLA2_ERR_INVALID, "null output pointer");
    if (!(gamma >= 0.f && gamma <= 1.f)) return fail(HLA2_ERR_INVALID, "gamma must lie in [0, 1] (got %g)", (double)gamma);
    if (!aligned16(O) || (state_out && !aligned16(state_out))) return fail(HLA2_ERR_INVALID, "output pointer not 16-byte aligned");
    const size_t need = hla2_forward_workspace(B, H, T, d, dv, dtype);
    if (!workspace || ws_bytes < need)
        return fail(HLA2_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace ? ws_bytes : (size_t)0, need);
    if (!aligned16(workspace)) return fail(HLA2_ERR_INVALID, "workspace not 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int BH = B * H;
    const SegPlan plan = forward_plan(BH, T, 0);
    const FwdWorkspace ws = carve(workspace, BH, plan, d, dv);
    const bool use_tc = hla2_decay_forward_path(d, dv, dtype, normalized, state_out != nullptr, gamma) == 1;
    int* status = nullptr;
    if (use_tc && !(status = device_status_word())) return fail(HLA2_ERR_LAUNCH, "cannot resolve the device status word");
    if (use_tc) {
        // tensor cores: segment summaries S|C|.|P|. from the walks, the segment
        // factors, the decayed scan (one launch: S_<r and P_<r with the cross
        // terms f_r S_<r C_r on tensor cores), then the output walks
        const RecOff ro = summary_offsets(d, dv);
        cudaError_t e = launch_decay_tc_walk(0, Q, K, V, nullptr, nullptr, ws.summ, BH, T, d, dv, gamma, plan, status, s);
        if (e != cudaSuccess) return cuda_fail(e, "decay segment summaries");
        e = launch_decay_factors(ws.fac, T, gamma, plan, s);
        if (e != cudaSuccess) return cuda_fail(e, "decay scan: segment factors");
        const ScanArgs sa{ws.summ, ws.prefix, plan.nseg, ro.R, ro, ws.fac, status, false};
        e = launch_tc_scan(kScanDecay, sa, BH, d, dv, s);
        if (e == cudaSuccess && plan.nseg > tc_scan_full_max_segments())  // decayed sums of the terms X_r with f_r^2
            e = launch_decay_exscan(ws.prefix, ws.prefix, BH, plan.nseg, ro.R, ro.X, (size_t)d * dv, nullptr, ro.R,
                                    ws.fac + plan.nseg, s);
        if (e != cudaSuccess) return cuda_fail(e, "decay scan");
        e = launch_decay_tc_walk(1, Q, K, V, O, ws.prefix, nullptr, BH, T, d, dv, gamma, plan, status, s);
        if (e != cudaSuccess) return cuda_fail(e, "decay segment outputs");
        return HLA2_OK;
    }
    // P-form segment summaries with decay, the decayed scan, walks
    cudaError_t e = launch_walk(0, Q, K, V, dtype, nullptr, nullptr, ws.summ, BH, T, d, dv, normalized, 0, gamma,
                                plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "decay segment summaries");
    // decayed scan (f_r = gamma^{n_r}, segment r spanning n_r tokens):
    //   S_<r+1 = f_r S_<r + S_r (C, m likewise),
    //   P_<r+1 = f_r^2 P_<r + P_r + f_r S_<r C_r (p likewise with m_r),
    // as decayed running sums of (S, C, m), one product per record, and
    // decayed running sums of the corrected part with f_r^2
    {
        const RecOff ro = summary_offsets(d, dv);
        float* tot = state_out ? ws.tot : nullptr;
        e = launch_decay_factors(ws.fac, T, gamma, plan, s);
        if (e == cudaSuccess)
            e = launch_decay_exscan(ws.summ, ws.prefix, BH, plan.nseg, ro.R, 0, ro.X, tot, ro.R, ws.fac, s);
        if (e != cudaSuccess) return cuda_fail(e, "decay scan: prefix sums of S, C, m");
        CrossArgs a{};
        a.A = ws.prefix + ro.S; a.sA = (long long)ro.R;
        a.B = ws.summ + ro.C;   a.sB = (long long)ro.R;
        a.bx = ws.summ + ro.m;  a.sbx = (long long)ro.R;
        a.base = ws.summ + ro.X; a.sbase = (long long)ro.R;
        a.basex = ws.summ + ro.x; a.sbasex = (long long)ro.R;
        a.out = ws.prefix + ro.X; a.sout = (long long)ro.R;
        a.outx = ws.prefix + ro.x; a.soutx = (long long)ro.R;
        a.alpha = 1.f; a.d = d; a.dv = dv;
        a.pscale = ws.fac; a.pscale_mod = plan.nseg;
        for (long long b0 = 0; b0 < (long long)BH * plan.nseg; b0 += 65535) {
            CrossArgs c = a;
            const long long nb = (long long)BH * plan.nseg - b0;
            c.nb = (int)(nb < 65535 ? nb : 65535);
            c.pscale_off = b0;
            c.A += b0 * ro.R; c.B += b0 * ro.R; c.bx += b0 * ro.R;
            c.base += b0 * ro.R; c.basex += b0 * ro.R; c.out += b0 * ro.R; c.outx += b0 * ro.R;
            e = launch_cross(c, s);
            if (e != cudaSuccess) return cuda_fail(e, "decay scan: cross terms");
        }
        e = launch_decay_exscan(ws.prefix, ws.prefix, BH, plan.nseg, ro.R, ro.X, ro.R - ro.X,
                                tot ? tot + ro.X : nullptr, ro.R, ws.fac + plan.nseg, s);
        if (e != cudaSuccess) return cuda_fail(e, "decay scan: prefix sums of P, p");
    }
    e = launch_walk(1, Q, K, V, dtype, O, ws.prefix, nullptr, BH, T, d, dv, normalized, 0, gamma, plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "decay segment outputs");
    if (state_out) {
        // final compact state S|P|p from the totals S|C|m|P|p
        const RecOff so = summary_offsets(d, dv);
        const long long R = (long long)so.R;
        const long long Rp = (long long)d * d + (long long)d * dv + d;
        e = launch_copy_strided(ws.tot + so.S, R, state_out, Rp, (size_t)d * d, BH, s);
        if (e == cudaSuccess)
            e = launch_copy_strided(ws.tot + so.X, R, state_out + (size_t)d * d, Rp, (size_t)d * dv + d, BH, s);
        if (e != cudaSuccess) return cuda_fail(e, "decay state_out copy");
    }
    return HLA2_OK;
}

int hla2_decay_step(float* state, const float* q, const float* k, const float* v, float* o, int n, int d, int dv,
                    int normalized, float gamma, hla2_stream_t stream) {
    if (!state || !q || !k || !v || !o) return fail(HLA2_ERR_INVALID, "null pointer");
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return fail(HLA2_ERR_INVALID, "pointer not 16-byte aligned");
    if (n <= 0 || d <= 0 || dv <= 0) return fail(HLA2_ERR_INVALID, "sizes must be positive (n=%d d=%d dv=%d)", n, d, dv);
    if (!(gamma >= 0.f && gamma <= 1.f)) return fail(HLA2_ERR_INVALID, "gamma must lie in [0, 1] (got %g)", (double)gamma);
    auto pow2_4_128 = [](int x) { return x >= 4 && x <= 128 && (x & (x - 1)) == 0; };
    if (!pow2_4_128(d) || !pow2_4_128(dv))
        return fail(HLA2_ERR_UNSUPPORTED, "hla2_decay_step needs d, dv powers of two in [4, 128] (d=%d dv=%d)", d, dv);
    cudaError_t e = launch_step_pform_decay(state, q, k, v, o, n, d, dv, normalized, gamma,
                                            reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "hla2_decay_step");
    return HLA2_OK;
}

}  // extern "C"
