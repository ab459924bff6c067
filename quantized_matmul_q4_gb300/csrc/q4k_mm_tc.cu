// Q4_K prefill on tcgen05 tensor cores: not built yet.
#include "kernels.h"

namespace q4mm {

cudaError_t launch_q4k_mm_tc(const LaunchCtx &, const float *, const uint8_t *, float *, int, int,
                             int) {
    return cudaErrorNotSupported;
}

}  // namespace q4mm
