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

// Decode: 8 consumer warps, 8 chunk stages of 16 KB, 4 head stages.
constexpr int DEC_NCW = 8, DEC_NS = 8, DEC_NH = 4;

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

// Replay: 8 consumer warps; chunk stages as many as fit (2..6).
constexpr int REP_NCW = 8, REP_NS_MAX = 6;

// Fill the shared-memory layout fields of `a` (needs dk, T, L, dv, in_dtype).
// Returns the total dynamic shared memory in bytes, or -1 if it cannot fit.
template <int DK, int TMAX>
int replay_layout(ReplayArgs& a, int smem_limit) {
    const int in_sz = dtype_size(a.in_dtype);
    const int T = a.T, L = a.L;
    a.off_wq = REPLAY_META;
    a.off_wk = a.off_wq + T * DK * in_sz;
    a.off_wv = a.off_wk + T * DK * in_sz;
    a.off_rk = align_up(a.off_wv + T * a.dv * in_sz, 16);
    a.off_rec = a.off_rk + L * DK * in_sz;
    a.head_bytes = align_up(a.off_rec + L * (4 + a.dv) * 4, 128);
    a.off_khat = 0;
    a.off_qhat = (L + TMAX) * DK * 4;
    a.off_coef = a.off_qhat + TMAX * DK * 4;
    const int coef_floats = 2 * TMAX * (L + TMAX) + 2 * TMAX + 1 + L;
    a.scratch_bytes = align_up(a.off_coef + coef_floats * 4, 128);
    const int fixed = REPLAY_NH * a.head_bytes + 2 * a.scratch_bytes;
    int ns = REP_NS_MAX;
    auto total = [&](int n) { return n * CHUNK_BYTES + fixed + (2 * n + 2 * REPLAY_NH + 2) * 8; };
    while (ns >= 2 && total(ns) > smem_limit) --ns;
    if (ns < 2) return -1;
    a.nstage = ns;
    a.heads_off = ns * CHUNK_BYTES;
    a.scratch_off = a.heads_off + REPLAY_NH * a.head_bytes;
    a.bars_off = a.scratch_off + 2 * a.scratch_bytes;
    return total(ns);
}

template <typename ST, int DK, int TMAX>
cudaError_t launch_replay(ReplayArgs& a, cudaStream_t stream, bool& too_big) {
    using C = ReplayCfg<ST, DK, TMAX, REP_NCW>;
    auto kern = replay_kernel<ST, DK, TMAX, REP_NCW>;
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
