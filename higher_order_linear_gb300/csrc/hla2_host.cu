// hla2_host.cu -- the masked forward on host buffers: heads are independent,
// so the batch is cut into groups of heads and each group's host-to-device
// copy, forward and device-to-host copy run as a three-stage pipeline on a
// copy-in stream, the caller's stream and a copy-out stream.  Two device
// slots hold the Q, K, V and O of the groups in flight; the forward of each
// group is hla2_forward itself (one workspace, shared, since the forwards run
// in order on the caller's stream).
#include <mutex>

#include "hla2_internal.h"
#include "../../include/hla2.h"

namespace hla2 {
namespace {

constexpr int kMaxDev = 64;
constexpr size_t kAlign = 256;

size_t up(size_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, in_ready[2] = {}, computed[2] = {}, out_done[2] = {};
};
HostPipe g_pipe[kMaxDev];
std::mutex g_pipe_mu;

// Streams and events of the device, created on first use and kept for the
// life of the process (no device memory is allocated).
bool pipe_init(HostPipe& p) {
    if (p.ready) return true;
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess) return false;
    cudaEvent_t* evs[7] = {&p.start, &p.in_ready[0], &p.in_ready[1], &p.computed[0], &p.computed[1],
                           &p.out_done[0], &p.out_done[1]};
    for (cudaEvent_t* e : evs)
        if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
    p.ready = true;
    return true;
}

int group_heads(int BH, int heads_per_group) {
    if (heads_per_group > 0) return heads_per_group < BH ? heads_per_group : BH;
    const int g = (BH + 7) / 8;  // eight groups when there are enough heads
    return g > 0 ? g : 1;
}

struct HostLayout {
    int G, ngroups;
    size_t q, k, v, o;  // bytes of one slot's buffers
    size_t slot, ws, bytes;
};

HostLayout host_layout(int B, int H, int T, int d, int dv, int dtype, int heads_per_group) {
    HostLayout L{};
    const int BH = B * H;
    const size_t es = dtype == HLA2_DTYPE_BF16 ? 2 : 4;
    L.G = group_heads(BH, heads_per_group);
    L.ngroups = (BH + L.G - 1) / L.G;
    L.q = up((size_t)L.G * T * d * es);
    L.k = L.q;
    L.v = up((size_t)L.G * T * dv * es);
    L.o = up((size_t)L.G * T * dv * 4);
    L.slot = L.q + L.k + L.v + L.o;
    // the forward's workspace for a full group and for the last (possibly smaller) one
    const int last = BH - (L.ngroups - 1) * L.G;
    const size_t w1 = hla2_forward_workspace(1, L.G, T, d, dv, dtype);
    const size_t w2 = hla2_forward_workspace(1, last, T, d, dv, dtype);
    L.ws = up(w1 > w2 ? w1 : w2);
    L.bytes = 2 * L.slot + L.ws;
    return L;
}

}  // namespace
}  // namespace hla2

using namespace hla2;

extern "C" {

size_t hla2_forward_host_workspace(int B, int H, int T, int d, int dv, int dtype, int heads_per_group) {
    if (B <= 0 || H <= 0 || T <= 0 || d <= 0 || dv <= 0 || heads_per_group < 0) return 0;
    if (hla2_forward_workspace(B, H, T, d, dv, dtype) == 0) return 0;
    return host_layout(B, H, T, d, dv, dtype, heads_per_group).bytes;
}

int hla2_forward_host(const void* Qh, const void* Kh, const void* Vh, float* Oh, int B, int H, int T, int d, int dv,
                      int normalized, int dtype, int heads_per_group, void* dev, size_t dev_bytes,
                      hla2_stream_t stream) {
    if (!Qh || !Kh || !Vh || !Oh) return set_error(HLA2_ERR_INVALID, "null host pointer");
    if (heads_per_group < 0) return set_error(HLA2_ERR_INVALID, "heads_per_group must be >= 0 (got %d)", heads_per_group);
    if (B <= 0 || H <= 0 || T <= 0 || d <= 0 || dv <= 0)
        return set_error(HLA2_ERR_INVALID, "sizes must be positive (B=%d H=%d T=%d d=%d dv=%d)", B, H, T, d, dv);
    const size_t need = hla2_forward_host_workspace(B, H, T, d, dv, dtype, heads_per_group);
    if (need == 0) return set_error(HLA2_ERR_UNSUPPORTED, "unsupported problem (B=%d H=%d T=%d d=%d dv=%d dtype=%d)",
                                    B, H, T, d, dv, dtype);
    if (!dev || dev_bytes < need)
        return set_error(HLA2_ERR_WORKSPACE, "device buffer %zu bytes, need %zu", dev ? dev_bytes : (size_t)0, need);
    if (reinterpret_cast<uintptr_t>(dev) % kAlign) return set_error(HLA2_ERR_INVALID, "device buffer not 256-byte aligned");
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDev)
        return set_error(HLA2_ERR_LAUNCH, "cannot resolve the current device");
    const HostLayout Lh = host_layout(B, H, T, d, dv, dtype, heads_per_group);
    const int BH = B * H;
    const size_t es = dtype == HLA2_DTYPE_BF16 ? 2 : 4;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(dev);
    char* ws = base + 2 * Lh.slot;

    // One enqueue at a time per device: the pipeline's streams and events are shared.
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe& P = g_pipe[device];
    if (!pipe_init(P)) return set_error(HLA2_ERR_LAUNCH, "cannot create the copy streams and events");
    auto ck = [](cudaError_t e, const char* what) -> int {
        return e == cudaSuccess ? HLA2_OK : set_error(HLA2_ERR_LAUNCH, "%s: %s", what, cudaGetErrorString(e));
    };
    int rc;
    // both copy streams start after the work already on the caller's stream
    if ((rc = ck(cudaEventRecord(P.start, s), "event record"))) return rc;
    if ((rc = ck(cudaStreamWaitEvent(P.in, P.start, 0), "stream wait"))) return rc;
    if ((rc = ck(cudaStreamWaitEvent(P.out, P.start, 0), "stream wait"))) return rc;
    for (int g = 0; g < Lh.ngroups; ++g) {
        const int slot = g & 1;
        const int h0 = g * Lh.G;
        const int hn = BH - h0 < Lh.G ? BH - h0 : Lh.G;
        char* sq = base + slot * Lh.slot;
        char* sk = sq + Lh.q;
        char* sv = sk + Lh.k;
        float* so = reinterpret_cast<float*>(sv + Lh.v);
        const size_t nq = (size_t)hn * T * d * es, nv = (size_t)hn * T * dv * es, no = (size_t)hn * T * dv * 4;
        // copy in: the slot is free once its previous group's O has been copied out
        if (g >= 2 && (rc = ck(cudaStreamWaitEvent(P.in, P.out_done[slot], 0), "stream wait"))) return rc;
        if ((rc = ck(cudaMemcpyAsync(sq, static_cast<const char*>(Qh) + (size_t)h0 * T * d * es, nq,
                                     cudaMemcpyHostToDevice, P.in), "copy of Q")))
            return rc;
        if ((rc = ck(cudaMemcpyAsync(sk, static_cast<const char*>(Kh) + (size_t)h0 * T * d * es, nq,
                                     cudaMemcpyHostToDevice, P.in), "copy of K")))
            return rc;
        if ((rc = ck(cudaMemcpyAsync(sv, static_cast<const char*>(Vh) + (size_t)h0 * T * dv * es, nv,
                                     cudaMemcpyHostToDevice, P.in), "copy of V")))
            return rc;
        if ((rc = ck(cudaEventRecord(P.in_ready[slot], P.in), "event record"))) return rc;
        // forward on the caller's stream
        if ((rc = ck(cudaStreamWaitEvent(s, P.in_ready[slot], 0), "stream wait"))) return rc;
        rc = hla2_forward(sq, sk, sv, so, 1, hn, T, d, dv, normalized, dtype, ws, Lh.ws, nullptr, stream);
        if (rc) return rc;
        if ((rc = ck(cudaEventRecord(P.computed[slot], s), "event record"))) return rc;
        // copy out
        if ((rc = ck(cudaStreamWaitEvent(P.out, P.computed[slot], 0), "stream wait"))) return rc;
        if ((rc = ck(cudaMemcpyAsync(reinterpret_cast<char*>(Oh) + (size_t)h0 * T * dv * 4, so, no,
                                     cudaMemcpyDeviceToHost, P.out), "copy of O")))
            return rc;
        if ((rc = ck(cudaEventRecord(P.out_done[slot], P.out), "event record"))) return rc;
    }
    // the caller's stream ends after the last copies out
    if ((rc = ck(cudaStreamWaitEvent(s, P.out_done[(Lh.ngroups - 1) & 1], 0), "stream wait"))) return rc;
    if (Lh.ngroups > 1 && (rc = ck(cudaStreamWaitEvent(s, P.out_done[Lh.ngroups & 1], 0), "stream wait"))) return rc;
    return HLA2_OK;
}

}  // extern "C"
