// gdn_launch.cuh -- host-side launch helpers for the decode and replay
// kernels: per-device caching of SM count / occupancy / shared-memory opt-in,
// persistent grid sizing, and the replay shared-memory layout.
#pragma once

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "gdn_decode.cuh"
#include "gdn_replay.cuh"

namespace gdn {

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
};

inline cudaError_t device_info(DeviceInfo& out) {
    static std::mutex mu;
    static std::map<int, DeviceInfo> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(dev);
    if (it == cache.end()) {
        DeviceInfo d;
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess)
            return e;
        it = cache.emplace(dev, d).first;
    }
    out = it->second;
    return cudaSuccess;
}

// Opt a kernel into the device's full dynamic shared memory (once per device
// and kernel) and return how many CTAs using `smem` bytes fit on one SM.
template <typename Kernel>
cudaError_t prepare_kernel(Kernel kern, int threads, int smem, int& blocks_per_sm) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void*, int>, int> cache;
    DeviceInfo di;
    cudaError_t e = device_info(di);
    if (e != cudaSuccess) return e;
    if (smem > di.smem_optin) return cudaErrorInvalidValue;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    std::lock_guard<std::mutex> g(mu);
    const void* kp = reinterpret_cast<const void*>(kern);
    const auto opted = std::make_tuple(dev, kp, -1);
    if (cache.find(opted) == cache.end()) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin)) !=
            cudaSuccess)
            return e;
        cache.emplace(opted, 0);
    }
    const auto key = std::make_tuple(dev, kp, smem);
    auto it = cache.find(key);
    if (it == cache.end()) {
        int bps = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, threads, smem)) != cudaSuccess) return e;
        if (bps < 1) return cudaErrorInvalidConfiguration;
        it = cache.emplace(key, bps).first;
    }
    blocks_per_sm = it->second;
    return cudaSuccess;
}

// Decode: consumer warps, 16 KB chunk stages and head stages per CTA.
#ifndef GDN_DECODE_CONSUMER_WARPS
#define GDN_DECODE_CONSUMER_WARPS 16
#endif
#ifndef GDN_DECODE_CHUNK_STAGES
#define GDN_DECODE_CHUNK_STAGES 6
#endif
#ifndef GDN_DECODE_HEAD_STAGES
#define GDN_DECODE_HEAD_STAGES 4
#endif
constexpr int DEC_NCW = GDN_DECODE_CONSUMER_WARPS, DEC_NS = GDN_DECODE_CHUNK_STAGES, DEC_NH = GDN_DECODE_HEAD_STAGES;

template <typename ST, int DK>
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    using C = DecodeCfg<ST, DK, DEC_NCW, DEC_NS, DEC_NH>;
    auto kern = decode_kernel<ST, DK, DEC_NCW, DEC_NS, DEC_NH>;
    DeviceInfo di;
    cudaError_t e = device_info(di);
    if (e != cudaSuccess) return e;
    int bps = 0;
    if ((e = prepare_kernel(kern, C::THREADS, C::SMEM, bps)) != cudaSuccess) return e;
    const int units = a.B * a.Hv;
    const int grid = units < di.sms * bps ? units : di.sms * bps;
    kern<<<grid, C::THREADS, C::SMEM, stream>>>(a);
    return cudaGetLastError();
}

// Replay: consumer warps per window size. Registers are granted per group of
// four warps, so producer + consumers is kept a multiple of four: 16 warps
// leave 128 registers a thread, 12 leave 168, 8 leave 255.
#ifndef GDN_REPLAY_WARPS_STEP
#define GDN_REPLAY_WARPS_STEP 15
#endif
#ifndef GDN_REPLAY_WARPS_W4
#define GDN_REPLAY_WARPS_W4 11
#endif
#ifndef GDN_REPLAY_WARPS_W8
#define GDN_REPLAY_WARPS_W8 7
#endif
template <int TMAX>
constexpr int replay_warps() {
    return TMAX == 1 ? GDN_REPLAY_WARPS_STEP : (TMAX <= 4 ? GDN_REPLAY_WARPS_W4 : GDN_REPLAY_WARPS_W8);
}

#ifndef GDN_REPLAY_MAX_HEADS
#define GDN_REPLAY_MAX_HEADS 6
#endif
#ifndef GDN_REPLAY_MIN_CHUNKS
#define GDN_REPLAY_MIN_CHUNKS 6
#endif

// Fill the shared-memory layout fields of `a` (needs T, L, dv, in_dtype).
// Returns the total dynamic shared memory in bytes, or -1 if it cannot fit.
template <int DK, int TMAX>
int replay_layout(ReplayArgs& a, int smem_limit) {
    const int in_sz = dtype_size(a.in_dtype);
    const int T = a.T, L = a.L;
    // head stage: meta | window q, k, v rows | ring keys | ring records | coefficient table
    a.off_wq = REPLAY_META;
    a.off_wk = a.off_wq + T * DK * in_sz;
    a.off_wv = a.off_wk + T * DK * in_sz;
    a.off_rk = align_up(a.off_wv + T * a.dv * in_sz, 16);
    a.off_rec = a.off_rk + L * DK * in_sz;
    a.off_coef = a.off_rec + L * (4 + a.dv) * 4;
    a.head_bytes = align_up(a.off_coef + (L + TMAX) * 2 * TMAX * 4, 128);
    auto total = [&](int ns, int nh) {
        // mbarriers: 2 per chunk stage, 3 per head stage; a 4-byte counter per head stage
        return ns * CHUNK_BYTES + nh * a.head_bytes + (2 * ns + 3 * nh) * 8 + align_up(nh * 4, 16);
    };
    // deepest head ring (units in flight) that leaves GDN_REPLAY_MIN_CHUNKS chunk stages, then more
    // chunk stages
    int ns = 0, nh = 0;
    for (int min_ns = GDN_REPLAY_MIN_CHUNKS; min_ns >= 2 && !ns; min_ns -= 2)
        for (int h = GDN_REPLAY_MAX_HEADS; h >= 2 && !ns; --h)
            if (total(min_ns, h) <= smem_limit) ns = min_ns, nh = h;
    if (!ns) return -1;
    while (ns < 12 && total(ns + 1, nh) <= smem_limit) ++ns;
    a.nstage = ns, a.nhead = nh;
    a.heads_off = ns * CHUNK_BYTES;
    a.bars_off = a.heads_off + nh * a.head_bytes;
    return total(ns, nh);
}

template <typename ST, int DK, int TMAX>
cudaError_t launch_replay(ReplayArgs& a, cudaStream_t stream, bool& too_big) {
    constexpr int NCW = replay_warps<TMAX>();
    using C = ReplayCfg<ST, DK, TMAX, NCW>;
    auto kern = replay_kernel<ST, DK, TMAX, NCW>;
    DeviceInfo di;
    cudaError_t e = device_info(di);
    if (e != cudaSuccess) return e;
    const int smem = replay_layout<DK, TMAX>(a, di.smem_optin);
    too_big = smem < 0;
    if (too_big) return cudaSuccess;
    int bps = 0;
    if ((e = prepare_kernel(kern, C::THREADS, smem, bps)) != cudaSuccess) return e;
    const int units = a.B * a.Hv;
    const int grid = units < di.sms * bps ? units : di.sms * bps;
    kern<<<grid, C::THREADS, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
