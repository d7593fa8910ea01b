// Instantiations of the decode kernel (state dtype x dk) and the rollback launch.
#include "gdn_dispatch.h"
#include "gdn_launch.cuh"

namespace gdn {

// gdn_rollback: keep 1 + accepted[b] of the T window tokens of sequence b. The window's first ring
// record carries its length T in field 3 (written when the window was appended); a rollback whose T
// differs, or one that finds no such window (already rolled back), is refused with
// GDN_DEVERR_ACCEPT. A rollback clears the field, so a second one is refused.
__global__ void rollback_kernel(int32_t* pos, const int32_t* ckpt_pos, float* ring_rec, const int32_t* slots,
                                const int32_t* accepted, int B, int Hv, int T, int L, int rec_floats,
                                int64_t num_slots, int32_t* dev_err) {
    for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < B * Hv; u += gridDim.x * blockDim.x) {
        const int b = u / Hv, h = u - b * Hv;
        const int s = slots[b];
        if (s < 0) continue;
        if (s >= num_slots) {
            if (h == 0) set_error(dev_err, GDN_DEVERR_SLOT);
            continue;
        }
        const int acc = accepted[b];
        if (acc < 0 || acc > T - 1) {
            if (h == 0) set_error(dev_err, GDN_DEVERR_ACCEPT);
            continue;
        }
        const int64_t idx = (int64_t)s * Hv + h;
        const int p0 = pos[idx] - T;  // the window's first position
        const int ck = ckpt_pos[idx];
        if (p0 < ck || pos[idx] - ck > L) {
            set_error(dev_err, GDN_DEVERR_RING);
            continue;
        }
        float* mark = ring_rec + (idx * L + p0 % L) * (int64_t)rec_floats + 3;
        if (!in_bounds(mark, 4, ring_rec, (uint64_t)num_slots * Hv * L * rec_floats * 4, dev_err)) continue;
        if (*mark != (float)T) {
            set_error(dev_err, GDN_DEVERR_ACCEPT);
            continue;
        }
        *mark = 0.f;
        pos[idx] = p0 + 1 + acc;
    }
}

cudaError_t dispatch_decode(int state_dtype, int dk, const DecodeArgs& a, cudaStream_t s) {
#define GDN_DEC(CODE, ST)                                  \
    if (state_dtype == CODE) {                             \
        if (dk == 32) return launch_decode<ST, 32>(a, s);  \
        if (dk == 64) return launch_decode<ST, 64>(a, s);  \
        if (dk == 128) return launch_decode<ST, 128>(a, s); \
    }
    GDN_DEC(GDN_F32, float)
    GDN_DEC(GDN_BF16, __nv_bfloat16)
    GDN_DEC(GDN_F16, __half)
#undef GDN_DEC
    return cudaErrorNotSupported;
}

cudaError_t launch_rollback(int32_t* pos, const int32_t* ckpt_pos, float* ring_rec, const int32_t* slots,
                            const int32_t* accepted, int B, int Hv, int T, int L, int dv, int64_t num_slots,
                            int32_t* dev_err, cudaStream_t s) {
    const int n = B * Hv;
    const int threads = 256;
    int blocks = (n + threads - 1) / threads;
    if (blocks > 1024) blocks = 1024;
    rollback_kernel<<<blocks, threads, 0, s>>>(pos, ckpt_pos, ring_rec, slots, accepted, B, Hv, T, L, 4 + dv,
                                               num_slots, dev_err);
    return cudaGetLastError();
}

}  // namespace gdn
