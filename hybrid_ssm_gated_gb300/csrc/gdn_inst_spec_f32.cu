// Instantiations of the speculative-step kernel for f32 states (dk x window size).
#include "gdn_dispatch.h"
#include "gdn_launch_spec.cuh"

namespace gdn {

cudaError_t dispatch_spec_f32(int dk, int tmax, SpecArgs& a, cudaStream_t s, bool& too_big) {
    return dispatch_spec_t<float>(dk, tmax, a, s, too_big);
}

}  // namespace gdn
