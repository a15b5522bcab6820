// hla2_noalloc.cu -- a forward entry point that needs no caller workspace.
//
// Some callers cannot allocate device memory at the point where they call
// the forward: a host framework that owns a fixed device arena and forbids
// cudaMalloc from its execution callbacks, an embedding runtime that only
// hands its plugins input and output buffers, or a latency-critical loop
// where allocation is banned after start-up.  hla2_forward_noalloc serves
// them: it runs exactly hla2_forward, but takes its scratch from a
// file-scope device array of fixed size instead of a caller workspace.
//
// The array is a static __device__ object, so every GPU that loads this
// library holds it (kNoallocScratchBytes) until the process exits.  Its
// device address is looked up once per device, on the first call made with
// that device current; make that first call before any stream capture.
// All calls share the array: two calls whose work overlaps on the GPU (for
// example on two streams) race on it and must be serialised by the caller.
// The forward writes every scratch element before it reads it, so nothing
// has to start at zero and the contents left by earlier calls are harmless.
#include <mutex>

#include "../../include/hla2.h"
#include "hla2_internal.h"

namespace hla2 {
namespace {

constexpr size_t kNoallocScratchBytes = (size_t)64 << 20;  // 64 MiB per device

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev] = {};
std::mutex g_scratch_mu;

}  // namespace
}  // namespace hla2

extern "C" {

int hla2_forward_noalloc(const void* Q, const void* K, const void* V, float* O, int B, int H, int T, int d, int dv,
                         int normalized, int dtype, hla2_stream_t stream) {
    using namespace hla2;
    const size_t need = hla2_forward_workspace(B, H, T, d, dv, dtype);
    if (need == 0) {
        // let hla2_forward report the precise argument error
        return hla2_forward(Q, K, V, O, B, H, T, d, dv, normalized, dtype, nullptr, 0, nullptr, stream);
    }
    if (need > kNoallocScratchBytes)
        return set_error(HLA2_ERR_UNSUPPORTED,
                         "hla2_forward_noalloc: this problem needs %zu bytes of scratch, more than the library's "
                         "fixed %zu-byte array; call hla2_forward with a workspace instead",
                         need, kNoallocScratchBytes);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return set_error(HLA2_ERR_LAUNCH, "hla2_forward_noalloc: no usable current device");
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        if (!g_scratch_addr[dev]) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p)
                return set_error(HLA2_ERR_LAUNCH, "hla2_forward_noalloc: cudaGetSymbolAddress of the scratch array "
                                 "failed: %s", cudaGetErrorString(e));
            g_scratch_addr[dev] = p;
        }
        scratch = g_scratch_addr[dev];
    }
    return hla2_forward(Q, K, V, O, B, H, T, d, dv, normalized, dtype, scratch, kNoallocScratchBytes, nullptr, stream);
}

}  // extern "C"
