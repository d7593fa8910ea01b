// Instantiations of the decode kernel for the Mamba2 recurrence (state dtype x d_state).
#include "gdn_dispatch.h"
#include "gdn_launch.cuh"

namespace gdn {

cudaError_t dispatch_mamba2_decode(int state_dtype, int dk, const DecodeArgs& a, cudaStream_t s) {
#define GDN_DEC(CODE, ST)                                                  \
    if (state_dtype == CODE) {                                             \
        if (dk == 32) return launch_decode<ST, 32, RULE_MAMBA2>(a, s);     \
        if (dk == 64) return launch_decode<ST, 64, RULE_MAMBA2>(a, s);     \
        if (dk == 128) return launch_decode<ST, 128, RULE_MAMBA2>(a, s);   \
    }
    GDN_DEC(GDN_F32, float)
    GDN_DEC(GDN_BF16, __nv_bfloat16)
    GDN_DEC(GDN_F16, __half)
#undef GDN_DEC
    return cudaErrorNotSupported;
}

}  // namespace gdn
