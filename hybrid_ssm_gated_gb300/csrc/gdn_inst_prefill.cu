// Instantiations of the prefill kernel (state dtype x dk) and its launch.
#include "gdn_dispatch.h"
#include "gdn_launch.cuh"
#include "gdn_prefill.cuh"
#include "gdn_prefill_tc.cuh"

namespace gdn {

template <typename ST, int DK, int IO>
cudaError_t launch_prefill(PrefillArgs& a, cudaStream_t stream) {
    auto kern = prefill_kernel<ST, DK, IO>;
    const int isz = dtype_size(a.in_dtype);
    a.raw_bytes = PF_TC * (2 * DK + PF_ROWS) * isz;
    a.off_kqn = 2 * a.raw_bytes;
    a.off_qk = a.off_kqn + PF_TC * 2 * DK * 4;
    a.off_vf = a.off_qk + align_up(PF_TC * 4, 16);
    a.off_of = a.off_vf + PF_TC * PF_ROWS * 4;
    a.off_gates = a.off_of + PF_TC * PF_ROWS * 4;
    const int smem = a.off_gates + 2 * PF_TC * 16;
    int bps = 0;
    cudaError_t e = prepare_kernel(kern, PF_WARPS * 32, smem, bps);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)a.B * a.Hv * a.row_blocks;
    if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, PF_WARPS * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

// The chunked tensor-core prefill: one CTA per (sequence, value head, 128 state rows).
template <typename ST, int IO>
cudaError_t launch_prefill_tc(PrefillArgs& a, cudaStream_t stream) {
    auto kern = prefill_tc_kernel<ST, IO>;
    int bps = 0;
    cudaError_t e = prepare_kernel(kern, tc::THREADS, tc::SMEM, bps);
    if (e != cudaSuccess) return e;
    a.row_blocks = a.dv / tc::ROWS;
    const int64_t grid = (int64_t)a.B * a.Hv * a.row_blocks;
    if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, tc::THREADS, tc::SMEM, stream>>>(a);
    return cudaGetLastError();
}

// The bf16-in / fp32-out instantiation when the arguments match it, the generic one otherwise. 16-bit
// states with dk = 128 and dv a multiple of 128 take the chunked tensor-core kernel; FP32 states (whose
// tolerance one TF32 pass does not meet) and other shapes the sequential one.
template <typename ST, int DK>
cudaError_t launch_prefill_io(PrefillArgs& a, cudaStream_t stream) {
    const bool bf16_f32 = io_mode(a.in_dtype, a.out_dtype) == IO_BF16_F32;
    if constexpr (sizeof(ST) == 2 && DK == tc::DKT) {
        if (a.dv % tc::ROWS == 0)
            return bf16_f32 ? launch_prefill_tc<ST, IO_BF16_F32>(a, stream) : launch_prefill_tc<ST, IO_ANY>(a, stream);
    }
    if (bf16_f32) return launch_prefill<ST, DK, IO_BF16_F32>(a, stream);
    return launch_prefill<ST, DK, IO_ANY>(a, stream);
}

cudaError_t dispatch_prefill(int state_dtype, int dk, PrefillArgs& a, cudaStream_t s) {
#define GDN_PF(CODE, ST)                                       \
    if (state_dtype == CODE) {                                 \
        if (dk == 32) return launch_prefill_io<ST, 32>(a, s);   \
        if (dk == 64) return launch_prefill_io<ST, 64>(a, s);   \
        if (dk == 128) return launch_prefill_io<ST, 128>(a, s); \
    }
    GDN_PF(GDN_F32, float)
    GDN_PF(GDN_BF16, __nv_bfloat16)
    GDN_PF(GDN_F16, __half)
#undef GDN_PF
    return cudaErrorNotSupported;
}

}  // namespace gdn
