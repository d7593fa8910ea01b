// gdn_launch_spec.cuh -- host-side launch of the speculative-step kernel:
// consumer warp counts, the shared-memory layout (head and chunk rings) and
// the persistent grid.
#pragma once

#include "gdn_launch.cuh"
#include "gdn_spec.cuh"

namespace gdn {

// Registers are granted per group of four warps: 12 warps leave 168 registers a
// thread, 8 leave 255 (the window's normalised keys and queries stay in registers).
template <int TMAX>
constexpr int spec_warps() {
    return TMAX <= 4 ? 11 : 7;
}

// Fill the layout fields of `a` (needs T, dv, in_dtype); total dynamic shared
// memory in bytes, or -1 if it cannot fit.
template <int DK>
int spec_layout(SpecArgs& a, int smem_limit) {
    const int in_sz = dtype_size(a.in_dtype);
    // head stage: meta | window q rows | k rows | v rows
    a.off_q = SPEC_META;
    a.off_k = a.off_q + a.T * DK * in_sz;
    a.off_v = a.off_k + a.T * DK * in_sz;
    a.head_bytes = align_up(a.off_v + a.T * a.dv * in_sz, 128);
    auto total = [&](int ns, int nh) { return ns * CHUNK_BYTES + nh * a.head_bytes + (2 * ns + 2 * nh) * 8; };
    int nh = 4;
    while (nh > 2 && total(2, nh) > smem_limit) --nh;
    if (total(2, nh) > smem_limit) return -1;
    int ns = 2;
    while (ns < 12 && total(ns + 1, nh) <= smem_limit) ++ns;
    a.nstage = ns, a.nhead = nh;
    a.heads_off = ns * CHUNK_BYTES;
    a.bars_off = a.heads_off + nh * a.head_bytes;
    return total(ns, nh);
}

template <typename ST, int DK, int TMAX, int IO>
cudaError_t launch_spec(SpecArgs& a, cudaStream_t stream, bool& too_big) {
    constexpr int NCW = spec_warps<TMAX>();
    using C = SpecCfg<ST, DK, TMAX, NCW>;
    auto kern = spec_kernel<ST, DK, TMAX, NCW, IO>;
    DeviceInfo di;
    cudaError_t e = device_info(di);
    if (e != cudaSuccess) return e;
    const int smem = spec_layout<DK>(a, di.smem_optin);
    too_big = smem < 0;
    if (too_big) return cudaSuccess;
    int bps = 0;
    if ((e = prepare_kernel(kern, C::THREADS, smem, bps)) != cudaSuccess) return e;
    const int units = a.B * a.Hv;
    const int grid = units < di.sms * bps ? units : di.sms * bps;
    kern<<<grid, C::THREADS, smem, stream>>>(a);
    return cudaGetLastError();
}

// The bf16-in / fp32-out instantiation when the arguments match it, the generic one otherwise.
template <typename ST, int DK, int TMAX>
cudaError_t launch_spec_io(SpecArgs& a, cudaStream_t stream, bool& too_big) {
    if (io_mode(a.in_dtype, a.out_dtype) == IO_BF16_F32)
        return launch_spec<ST, DK, TMAX, IO_BF16_F32>(a, stream, too_big);
    return launch_spec<ST, DK, TMAX, IO_ANY>(a, stream, too_big);
}

// The window size's kernel (tmax 4 or 8) for one state type, by dk.
template <typename ST>
cudaError_t dispatch_spec_t(int dk, int tmax, SpecArgs& a, cudaStream_t s, bool& too_big) {
#define GDN_SPEC(DK)                                                     \
    if (dk == DK) {                                                      \
        if (tmax == 4) return launch_spec_io<ST, DK, 4>(a, s, too_big);  \
        if (tmax == 8) return launch_spec_io<ST, DK, 8>(a, s, too_big);  \
    }
    GDN_SPEC(32)
    GDN_SPEC(64)
    GDN_SPEC(128)
#undef GDN_SPEC
    return cudaErrorNotSupported;
}

}  // namespace gdn
