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

// Replay: prep warps and row warps beside the two producer warps.
#ifndef GDN_REPLAY_PREP_WARPS
#define GDN_REPLAY_PREP_WARPS 2
#endif
#ifndef GDN_REPLAY_ROW_WARPS
#define GDN_REPLAY_ROW_WARPS 8
#endif
constexpr int REP_NPW = GDN_REPLAY_PREP_WARPS, REP_NRW = GDN_REPLAY_ROW_WARPS;

// Fill the shared-memory layout fields of `a` (needs T, L, dv, in_dtype).
// Returns the total dynamic shared memory in bytes, or -1 if it cannot fit.
template <int DK, int TMAX, int NPW>
int replay_layout(ReplayArgs& a, int smem_limit) {
    const int in_sz = dtype_size(a.in_dtype);
    const int T = a.T, L = a.L;
    a.off_wq = REPLAY_META;
    a.off_wk = a.off_wq + T * DK * in_sz;
    a.off_wv = a.off_wk + T * DK * in_sz;
    a.off_rk = align_up(a.off_wv + T * a.dv * in_sz, 16);
    a.off_rec = a.off_rk + L * DK * in_sz;
    a.head_bytes = align_up(a.off_rec + L * (4 + a.dv) * 4, 128);
    a.off_kw = 0;
    a.off_qw = TMAX * DK * 4;
    a.off_coef = 2 * TMAX * DK * 4;
    const int coef_floats = 2 * TMAX * (L + TMAX) + 2 * TMAX + 1 + L;
    a.scratch_bytes = align_up(a.off_coef + coef_floats * 4, 128);
    // scratch slot s serves units n = s mod nscr, all prepared by warp s mod NPW
    a.nscr = 2 * NPW;
    auto total = [&](int ns, int nh) {
        // mbarriers: 2 per chunk and head stage, 1 per scratch slot; tags: 16 B per chunk stage, 4 B per slot
        return ns * CHUNK_BYTES + nh * a.head_bytes + a.nscr * a.scratch_bytes + (2 * ns + 2 * nh + a.nscr) * 8 +
               ns * 16 + align_up((a.nscr + nh) * 4, 16);
    };
    // deepest head ring first (prep lookahead, at least NPW), then chunk stages
    int ns = 0, nh = 0;
    for (int min_ns = 4; min_ns >= 2 && !ns; --min_ns)
        for (int h = NPW + 3; h >= NPW && h >= 2 && !ns; --h)
            if (total(min_ns, h) <= smem_limit) ns = min_ns, nh = h;
    if (!ns) return -1;
    while (ns < 12 && total(ns + 1, nh) <= smem_limit) ++ns;
    a.nstage = ns, a.nhead = nh;
    a.heads_off = ns * CHUNK_BYTES;
    a.scratch_off = a.heads_off + nh * a.head_bytes;
    a.bars_off = a.scratch_off + a.nscr * a.scratch_bytes;
    return total(ns, nh);
}

template <typename ST, int DK, int TMAX>
cudaError_t launch_replay(ReplayArgs& a, cudaStream_t stream, bool& too_big) {
    using C = ReplayCfg<ST, DK, TMAX, REP_NPW, REP_NRW>;
    auto kern = replay_kernel<ST, DK, TMAX, REP_NPW, REP_NRW>;
    DeviceInfo di;
    cudaError_t e = device_info(di);
    if (e != cudaSuccess) return e;
    const int smem = replay_layout<DK, TMAX, REP_NPW>(a, di.smem_optin);
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
