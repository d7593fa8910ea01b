// Instantiations of the replay kernel for f32 checkpoints (dk x window size).
#include "gdn_dispatch.h"
#include "gdn_launch_replay.cuh"

namespace gdn {

cudaError_t dispatch_replay_f32(int dk, int tmax, ReplayArgs& a, cudaStream_t s, bool& too_big) {
#define GDN_REP(DK)                                                            \
    if (dk == DK) {                                                            \
        if (tmax == 1) return launch_replay_io<float, DK, 1>(a, s, too_big);      \
        if (tmax == 4) return launch_replay_io<float, DK, 4>(a, s, too_big);      \
        if (tmax == 8) return launch_replay_io<float, DK, 8>(a, s, too_big);      \
    }
    GDN_REP(32)
    GDN_REP(64)
    GDN_REP(128)
#undef GDN_REP
    return cudaErrorNotSupported;
}

}  // namespace gdn
