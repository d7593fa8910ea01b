// gdn_launch.cuh -- host-side launch helpers: per-device caching of SM count /
// occupancy / shared-memory opt-in, persistent grid sizing, and the decode
// launch. The replay launch and its shared-memory layout are in
// gdn_launch_replay.cuh.
#pragma once

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "gdn_decode.cuh"

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
// chunk stages for fp32 states and for 16-bit states (measured best: 6 and 8)
#ifndef GDN_DECODE_CHUNK_STAGES
#define GDN_DECODE_CHUNK_STAGES 6
#endif
#ifndef GDN_DECODE_CHUNK_STAGES_NARROW
#define GDN_DECODE_CHUNK_STAGES_NARROW 8
#endif
// head stages: units in flight per CTA (6 measured best for 16-bit states: 4 left them short of data)
#ifndef GDN_DECODE_HEAD_STAGES
#define GDN_DECODE_HEAD_STAGES 6
#endif
constexpr int DEC_NCW = GDN_DECODE_CONSUMER_WARPS, DEC_NH = GDN_DECODE_HEAD_STAGES;
template <typename ST>
constexpr int decode_stages() {
    return sizeof(ST) == 4 ? GDN_DECODE_CHUNK_STAGES : GDN_DECODE_CHUNK_STAGES_NARROW;
}

template <typename ST, int DK, int RULE = RULE_GDN>
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    constexpr int NS = decode_stages<ST>();
    using C = DecodeCfg<ST, DK, DEC_NCW, NS, DEC_NH, RULE>;
    auto kern = decode_kernel<ST, DK, DEC_NCW, NS, DEC_NH, RULE>;
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

}  // namespace gdn
