// gdn_launch_replay.cuh -- host-side launch of the replay kernels: which one a
// call takes, warps per CTA, shared-memory layouts and the persistent grid.
#pragma once

#include "gdn_launch.cuh"
#include "gdn_replay_producer.cuh"
#include "gdn_replay_rows.cuh"
#include "gdn_replay_warp.cuh"

namespace gdn {

// The row-per-lane kernel: its shared memory (18, 21 and 26 KB a warp at L = 16, d = 128 with bf16
// activations, for windows of 1, 4 and 8 tokens) allows 12, 10 and 8 warps. Registers are granted
// per SM sub-partition, a warp of each four on each, so 13 to 16 warps leave 128 registers a thread,
// 9 to 12 leave 168 and 5 to 8 leave 255: compiled for 16, 12 and 8.
template <int TMAX>
constexpr int replay_rows_warps() {
    return TMAX == 1 ? 16 : (TMAX <= 4 ? 12 : 8);
}

// The two-checkpoint warp kernel (the producer kernel's fallback): warps by window size. The kernel
// is launched with one CTA per SM at this size, so a thread may use 65536 / (32 * warps) registers:
// 12 warps leave 168, 8 leave 255 (windows of up to 8 tokens).
template <int TMAX>
constexpr int replay_warp_warps() {
    return TMAX <= 4 ? 12 : 8;
}

// The producer kernel: consumer warps per window size. Registers are granted per group of
// four warps, so producer + consumers is kept a multiple of four: 16 warps
// leave 128 registers a thread, 12 leave 168, 8 leave 255.
#ifndef GDN_REPLAY_WARPS_STEP
#define GDN_REPLAY_WARPS_STEP 11
#endif
#ifndef GDN_REPLAY_WARPS_W4
#define GDN_REPLAY_WARPS_W4 11
#endif
#ifndef GDN_REPLAY_WARPS_W8
#define GDN_REPLAY_WARPS_W8 7
#endif
template <int TMAX>
constexpr int producer_warps() {
    return TMAX == 1 ? GDN_REPLAY_WARPS_STEP : (TMAX <= 4 ? GDN_REPLAY_WARPS_W4 : GDN_REPLAY_WARPS_W8);
}

#ifndef GDN_REPLAY_MAX_HEADS
#define GDN_REPLAY_MAX_HEADS 6
#endif
#ifndef GDN_REPLAY_MIN_CHUNKS
#define GDN_REPLAY_MIN_CHUNKS 8
#endif

// Fill the shared-memory layout fields of `a` (needs T, L, dv, in_dtype, nchunk, mnchunk, ckpt_copy).
// Returns the total dynamic shared memory in bytes, or -1 if it cannot fit. The chunk ring holds at
// least one whole unit: a unit's head barrier completes only once every chunk of the unit is armed,
// so a unit with more chunks than stages could never complete.
template <int DK, int TMAX>
int producer_layout(ReplayArgs& a, int smem_limit, int sums_bytes) {
    const int need = a.nchunk > a.mnchunk ? a.nchunk : a.mnchunk;
    const int in_sz = dtype_size(a.in_dtype);
    const int T = a.T, L = a.L;
    // head stage: meta | window q, k, v rows | ring keys | ring records | ring values (two-checkpoint
    // folds only) | coefficient table
    a.off_wq = REPLAY_META;
    a.off_wk = a.off_wq + T * DK * in_sz;
    a.off_wv = a.off_wk + T * DK * in_sz;
    a.off_rk = align_up(a.off_wv + T * a.dv * in_sz, 16);
    a.off_rec = a.off_rk + L * DK * in_sz;
    a.off_rv = a.off_rec + L * (4 + a.dv) * 4;
    a.off_coef = a.off_rv + (a.ckpt_copy ? L * a.dv * in_sz : 0);
    a.head_bytes = align_up(a.off_coef + (L + TMAX) * 2 * TMAX * 4, 128);
    auto total = [&](int ns, int nh) {
        // mbarriers: 2 per chunk stage, 3 per head stage; a 4-byte counter per head stage
        return ns * CHUNK_BYTES + nh * a.head_bytes + sums_bytes + (2 * ns + 3 * nh) * 8 + align_up(nh * 4, 16);
    };
    // deepest head ring (units in flight) that leaves GDN_REPLAY_MIN_CHUNKS chunk stages (and at
    // least a unit's), then more chunk stages
    const int floor_ns = need > 2 ? need : 2;
    int ns = 0, nh = 0;
    for (int min_ns = GDN_REPLAY_MIN_CHUNKS > floor_ns ? GDN_REPLAY_MIN_CHUNKS : floor_ns; min_ns >= floor_ns && !ns;
         min_ns -= 2)
        for (int h = GDN_REPLAY_MAX_HEADS; h >= 1 && !ns; --h)
            if (total(min_ns, h) <= smem_limit) ns = min_ns, nh = h;
    if (!ns && total(floor_ns, 1) <= smem_limit) ns = floor_ns, nh = 1;
    if (!ns) return -1;
    while (ns < 12 && total(ns + 1, nh) <= smem_limit) ++ns;
    a.nstage = ns, a.nhead = nh;
    a.heads_off = ns * CHUNK_BYTES;
    a.sums_off = a.heads_off + nh * a.head_bytes;  // one row-sum tile per consumer warp (wide windows)
    a.bars_off = a.sums_off + sums_bytes;
    return total(ns, nh);
}

template <typename ST, int DK, int TMAX, int RULE, int IO>
cudaError_t launch_replay_rows(ReplayArgs& a, cudaStream_t stream, bool& too_big) {
    constexpr int NW = replay_rows_warps<TMAX>();
    auto kern = replay_rows_kernel<ST, DK, TMAX, NW, RULE, IO>;
    DeviceInfo di;
    cudaError_t e = device_info(di);
    if (e != cudaSuccess) return e;
    // as many of the NW warps as the per-warp shared memory allows (fewer only for long rings)
    const int wb = replay_rows_layout<ST, DK, TMAX, RULE>(a.L, dtype_size(a.in_dtype)).bytes;
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

template <typename ST, int DK, int TMAX, typename MT, int RULE, int IO>
cudaError_t launch_replay_producer(ReplayArgs& a, cudaStream_t stream, bool& too_big) {
    constexpr int NCW = producer_warps<TMAX>();
    using C = ReplayCfg<ST, DK, TMAX, NCW>;
    auto kern = replay_producer_kernel<ST, DK, TMAX, NCW, MT, RULE, IO>;
    DeviceInfo di;
    cudaError_t e = device_info(di);
    if (e != cudaSuccess) return e;
    const int smem = producer_layout<DK, TMAX>(a, di.smem_optin, NCW * C::SUMS * 4);
    too_big = smem < 0;
    if (too_big) return cudaSuccess;
    int bps = 0;
    if ((e = prepare_kernel(kern, C::THREADS, smem, bps)) != cudaSuccess) return e;
    const int units = a.B * a.Hv;
    const int grid = units < di.sms * bps ? units : di.sms * bps;
    kern<<<grid, C::THREADS, smem, stream>>>(a);
    return cudaGetLastError();
}

template <typename ST, int DK, int TMAX, typename MT, int RULE, int IO>
cudaError_t launch_replay_warp(ReplayArgs& a, cudaStream_t stream, bool& too_big) {
    constexpr int NW = replay_warp_warps<TMAX>();
    auto kern = replay_warp_kernel<ST, DK, TMAX, NW, MT, RULE, IO>;
    DeviceInfo di;
    cudaError_t e = device_info(di);
    if (e != cudaSuccess) return e;
    const int wb = replay_warp_layout<ST, MT, DK, TMAX, RULE>(a.L, dtype_size(a.in_dtype)).bytes;
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

// ST: the checkpoint steps read; MT: the one folds update (a wider master, or ST); RULE: the
// recurrence (gated delta rule or Mamba2). The producer kernel takes the two-checkpoint mode and one
// fp32 checkpoint's single tokens (gated delta rule), where its deep chunk ring measured faster
// (B = 256, d = 128, L = 16: 117 against 129 us a step; two checkpoints 135 against 154 us); the
// row kernel takes the rest, where it measured faster (a bf16 step 94 against 112 us, windows of
// four 253 / 203 against 286 / 285 us, Mamba2 steps). A two-checkpoint call whose unit does not fit
// the producer kernel's shared memory (long rings with dv = 256: a fold streams 8 master chunks beside
// a head stage of the ring's keys, records and values) runs on the warp kernel, which streams rows a
// warp at a time. too_big is set when not even that fits.
template <typename ST, int DK, int TMAX, typename MT = ST, int RULE = RULE_GDN, int IO = IO_ANY>
cudaError_t launch_replay(ReplayArgs& a, cudaStream_t stream, bool& too_big) {
    constexpr bool MIXED = !std::is_same<ST, MT>::value;
    too_big = false;
    if constexpr (MIXED) {
        const cudaError_t e = launch_replay_producer<ST, DK, TMAX, MT, RULE, IO>(a, stream, too_big);
        if (e != cudaSuccess || !too_big) return e;
        return launch_replay_warp<ST, DK, TMAX, MT, RULE, IO>(a, stream, too_big);
    } else {
        if constexpr (std::is_same<ST, float>::value && TMAX == 1 && RULE == RULE_GDN)
            if (a.T == 1) return launch_replay_producer<ST, DK, TMAX, MT, RULE, IO>(a, stream, too_big);
        return launch_replay_rows<ST, DK, TMAX, RULE, IO>(a, stream, too_big);
    }
}

// The bf16-in / fp32-out instantiation when the arguments match it, the generic one otherwise.
template <typename ST, int DK, int TMAX, typename MT = ST, int RULE = RULE_GDN>
cudaError_t launch_replay_io(ReplayArgs& a, cudaStream_t stream, bool& too_big) {
    if (io_mode(a.in_dtype, a.out_dtype) == IO_BF16_F32)
        return launch_replay<ST, DK, TMAX, MT, RULE, IO_BF16_F32>(a, stream, too_big);
    return launch_replay<ST, DK, TMAX, MT, RULE, IO_ANY>(a, stream, too_big);
}

}  // namespace gdn
