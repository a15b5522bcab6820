// hla2_tc.cu -- tensor-core (tcgen05) segment walks; placeholder until the
// kernels land: reports "not supported" so the CUDA-core walks run.
#include "hla2_internal.h"

namespace hla2 {

bool tc_supported(int, int, int, int, int) { return false; }

cudaError_t launch_tc_walk(int, const void*, const void*, const void*, float*, const float*, float*, int, int, int,
                           int, SegPlan, int*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace hla2
