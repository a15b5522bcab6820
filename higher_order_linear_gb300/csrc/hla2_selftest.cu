// hla2_selftest.cu -- a run-out of the bounded device wait, on purpose and
// without any fault: one CTA takes tensor memory, waits on an mbarrier that
// nothing arrives on, gives up after the given time exactly as the walks'
// waits do (abort flag, device status word), releases its tensor memory and
// returns.  The host then reads the status word through hla2_device_status,
// and the context stays usable.  No counterpart on the pages: it tests the
// library's error path.
#include "hla2_tc_common.cuh"

namespace hla2 {
namespace {

__global__ void __launch_bounds__(64, 1) selftest_runout_kernel(int* status, unsigned long long wait_ns, int* out) {
    __shared__ __align__(8) unsigned long long bar_never;
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar_never), 1);  // nothing ever arrives
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(32u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // the walks' wait: try, then poll until the phase completes, the CTA's
    // abort flag is set, or the time runs out (then set both)
    bool done = false;
    if (warp == 1) {
        const uint32_t a = smem_u32(&bar_never);
        const unsigned long long t0 = globaltimer();
        while (!(done = mbar_try(a, 0))) {
            if (abort_flag) break;
            if (globaltimer() - t0 > wait_ns) {
                abort_flag = 1;
                if (lane == 0) atomicExch(status, (int)kDevWaitTimeout);
                break;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) out[0] = done ? 1 : 0;  // 0: the wait gave up
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(32u) : "memory");
}

}  // namespace

cudaError_t launch_selftest_runout(int* status, unsigned long long wait_ns, int* out, cudaStream_t s) {
    selftest_runout_kernel<<<1, 64, 0, s>>>(status, wait_ns, out);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace hla2
