// gdn_launch_replay.cuh -- host-side launch of the replay kernel: warps per CTA
// by window size, the per-warp shared memory, and the persistent grid.
#pragma once

#include "gdn_launch.cuh"
#include "gdn_replay_rows.cuh"
#include "gdn_replay_warp.cuh"

namespace gdn {

// Warps per CTA by window size. The kernel is launched with one CTA per SM at this size, so a thread
// may use 65536 / (32 * warps) registers: 12 warps leave 168 (one token, with E = 16 elements a lane
// and four rows in flight, spills at 128; windows of up to 4 tokens, whose keys and queries take 64
// registers), 8 leave 255 (windows of up to 8 tokens).
#ifndef GDN_REPLAY_WARPS_STEP
#define GDN_REPLAY_WARPS_STEP 12
#endif
#ifndef GDN_REPLAY_WARPS_W4
#define GDN_REPLAY_WARPS_W4 12
#endif
#ifndef GDN_REPLAY_WARPS_W8
#define GDN_REPLAY_WARPS_W8 8
#endif
template <int TMAX>
constexpr int replay_warps() {
    return TMAX == 1 ? GDN_REPLAY_WARPS_STEP : (TMAX <= 4 ? GDN_REPLAY_WARPS_W4 : GDN_REPLAY_WARPS_W8);
}
// The row-per-lane kernel: its shared memory (17, 21 and 26 KB a warp at L = 16, d = 128, for
// windows of 1, 4 and 8 tokens) allows 13, 10 and 8 warps. Registers are granted per SM
// sub-partition, a warp of each four on each, so 13 to 16 warps leave 128 registers a thread, 9 to 12
// leave 168 and 5 to 8 leave 255: compiled for 16, 8 and 8.
template <int TMAX>
constexpr int replay_rows_warps() {
    return TMAX == 1 ? 16 : 8;
}

// ST: the checkpoint steps read; MT: the one folds update (a wider master, or ST);
// RULE: the recurrence (gated delta rule or Mamba2). too_big is set when not even one warp's shared
// memory (copy stages, staged ring columns, row-sum tile, coefficient table) fits.
template <typename ST, int DK, int TMAX, typename MT = ST, int RULE = RULE_GDN, int IO = IO_ANY>
cudaError_t launch_replay(ReplayArgs& a, cudaStream_t stream, bool& too_big) {
    constexpr bool MIXED = !std::is_same<ST, MT>::value;
    // one checkpoint: a row per lane (gdn_replay_rows.cuh); two: rows split over lanes, whose whole
    // rows a sequential fold needs (gdn_replay_warp.cuh)
    constexpr int NW = MIXED ? replay_warps<TMAX>() : replay_rows_warps<TMAX>();
    auto kern = [] {
        if constexpr (MIXED)
            return replay_warp_kernel<ST, DK, TMAX, NW, MT, RULE, IO>;
        else
            return replay_rows_kernel<ST, DK, TMAX, NW, RULE, IO>;
    }();
    DeviceInfo di;
    cudaError_t e = device_info(di);
    if (e != cudaSuccess) return e;
    // as many of the NW warps as the per-warp shared memory allows (fewer only for long rings)
    const int wb = MIXED ? replay_warp_layout<ST, MT, DK, TMAX, RULE>(a.L, dtype_size(a.in_dtype)).bytes
                         : replay_rows_layout<ST, DK, TMAX, RULE>(a.L, dtype_size(a.in_dtype)).bytes;
    int nw = (di.smem_optin - REPLAY_SMEM_HEAD) / wb;
    if (nw > NW) nw = NW;
    too_big = nw < 1;
    if (too_big) return cudaSuccess;
    const int smem = REPLAY_SMEM_HEAD + nw * wb;
    int bps = 0;
    if ((e = prepare_kernel(kern, nw * 32, smem, bps)) != cudaSuccess) return e;
    const int units = a.B * a.Hv;
    const int grid = units < di.sms * bps ? units : di.sms * bps;
    kern<<<grid, nw * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

// The bf16-in / fp32-out instantiation when the arguments match it, the generic one otherwise.
template <typename ST, int DK, int TMAX, typename MT = ST, int RULE = RULE_GDN>
cudaError_t launch_replay_io(ReplayArgs& a, cudaStream_t stream, bool& too_big) {
    if (io_mode(a.in_dtype, a.out_dtype) == IO_BF16_F32)
        return launch_replay<ST, DK, TMAX, MT, RULE, IO_BF16_F32>(a, stream, too_big);
    return launch_replay<ST, DK, TMAX, MT, RULE, IO_ANY>(a, stream, too_big);
}

}  // namespace gdn
