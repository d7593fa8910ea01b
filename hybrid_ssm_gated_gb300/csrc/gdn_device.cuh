// gdn_device.cuh -- device-side building blocks shared by the decode and
// replay kernels: mbarrier / bulk-copy (TMA engine) wrappers in inline PTX,
// bounded waits, element conversions and lane-group reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr unsigned FULL_MASK = 0xffffffffu;
// A pipeline wait that has not completed after this long gives up, records
// GDN_DEVERR_TIMEOUT and lets the kernel return (no trap, no hang).
constexpr uint64_t WAIT_LIMIT_NS = 1000ull * 1000ull * 1000ull;  // 1 s

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrival that counts as `n` arrivals.
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(n) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Test for completion of the phase with the given parity. A thread whose
// phase is not complete is suspended until it completes or `hint_ns` pass,
// so a waiting warp does not take issue slots from working warps.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns = 100000) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete; false after
// WAIT_LIMIT_NS without completion.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
    return true;
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned), tracked
// by commit groups; cp_async_wait<N> returns once at most N groups of this
// thread are still in flight (the copies always complete: no flag is polled).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// L2 policy for data read once (state tiles): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 policy for data that later steps read again (replay ring entries).
__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Bulk global->shared copy through the TMA engine, completing `bytes`
// transaction bytes on `bar`. dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
        "[%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// ------------------------------------------------------------------ reductions

// Sum over aligned groups of G consecutive lanes (G a power of two <= 32).
template <int G>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) x += __shfl_xor_sync(FULL_MASK, x, off);
    return x;
}

// Reduce-scatter of x[0..N) over aligned groups of N lanes: afterwards lane
// (group position g) holds the group total of x[g].
template <int N>
__device__ __forceinline__ float reduce_scatter(float (&x)[N], int g) {
#pragma unroll
    for (int half = N / 2; half >= 1; half >>= 1) {
        const bool upper = (g & half) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? x[i] : x[i + half];
            const float keep = upper ? x[i + half] : x[i];
            x[i] = keep + __shfl_xor_sync(FULL_MASK, send, half);
        }
    }
    return x[0];
}

// ------------------------------------------------------------------ elements

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ float2 f16x2_to_f2(uint32_t x) {
    __half2 h = *reinterpret_cast<__half2*>(&x);
    return __half22float2(h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Storage traits: one 16-byte vector holds VEC elements.
template <typename T>
struct Store;

template <>
struct Store<float> {
    static constexpr int VEC = 4;
    static constexpr int code = GDN_F32;
    __device__ static __forceinline__ void unpack(const uint4& r, float* x) {
        x[0] = __uint_as_float(r.x);
        x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z);
        x[3] = __uint_as_float(r.w);
    }
    __device__ static __forceinline__ uint4 pack(const float* x) {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                          __float_as_uint(x[3]));
    }
};

template <>
struct Store<__nv_bfloat16> {
    static constexpr int VEC = 8;
    static constexpr int code = GDN_BF16;
    __device__ static __forceinline__ void unpack(const uint4& r, float* x) {
        x[0] = bf16_lo(r.x), x[1] = bf16_hi(r.x);
        x[2] = bf16_lo(r.y), x[3] = bf16_hi(r.y);
        x[4] = bf16_lo(r.z), x[5] = bf16_hi(r.z);
        x[6] = bf16_lo(r.w), x[7] = bf16_hi(r.w);
    }
    __device__ static __forceinline__ uint4 pack(const float* x) {
        return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                          pack_bf16x2(x[6], x[7]));
    }
};

template <>
struct Store<__half> {
    static constexpr int VEC = 8;
    static constexpr int code = GDN_F16;
    __device__ static __forceinline__ void unpack(const uint4& r, float* x) {
        float2 f;
        f = f16x2_to_f2(r.x), x[0] = f.x, x[1] = f.y;
        f = f16x2_to_f2(r.y), x[2] = f.x, x[3] = f.y;
        f = f16x2_to_f2(r.z), x[4] = f.x, x[5] = f.y;
        f = f16x2_to_f2(r.w), x[6] = f.x, x[7] = f.y;
    }
    __device__ static __forceinline__ uint4 pack(const float* x) {
        return make_uint4(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]), pack_f16x2(x[4], x[5]),
                          pack_f16x2(x[6], x[7]));
    }
};

__host__ __device__ constexpr int dtype_size(int dt) { return dt == GDN_F32 ? 4 : 2; }

// One element of a runtime-typed activation array.
__device__ __forceinline__ float load_elem(const void* base, int64_t idx, int dt) {
    if (dt == GDN_F32) return static_cast<const float*>(base)[idx];
    const uint16_t h = static_cast<const uint16_t*>(base)[idx];
    if (dt == GDN_BF16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ void store_elem(void* base, int64_t idx, int dt, float x) {
    if (dt == GDN_F32) {
        static_cast<float*>(base)[idx] = x;
    } else if (dt == GDN_BF16) {
        static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(x);
    } else {
        static_cast<__half*>(base)[idx] = __float2half_rn(x);
    }
}

// N consecutive elements of type T at element `first` of a 16-byte aligned
// row (first * sizeof(T) a multiple of 16, N a multiple of Store<T>::VEC).
template <typename T, int N>
__device__ __forceinline__ void load_row_run(const unsigned char* row, int first, float* x) {
#pragma unroll
    for (int e = 0; e < N; e += Store<T>::VEC)
        Store<T>::unpack(*reinterpret_cast<const uint4*>(row + (first + e) * (int)sizeof(T)), x + e);
}

// Store x rounded to T at element `first` of a row (as load_row_run), and
// replace x by the stored values.
template <typename T, int N>
__device__ __forceinline__ void store_row_run(unsigned char* row, int first, float* x) {
#pragma unroll
    for (int e = 0; e < N; e += Store<T>::VEC) {
        const uint4 packed = Store<T>::pack(x + e);
        *reinterpret_cast<uint4*>(row + (first + e) * (int)sizeof(T)) = packed;
        Store<T>::unpack(packed, x + e);
    }
}

// N consecutive runtime-typed elements from shared memory, starting at
// element `first` (first * size aligned to N * size, N in {4, 8}).
template <int N>
__device__ __forceinline__ void load_run(const unsigned char* base, int first, int dt, float* x) {
    if (dt == GDN_F32) {
#pragma unroll
        for (int e = 0; e < N; e += 4) {
            const float4 f = *reinterpret_cast<const float4*>(base + (first + e) * 4);
            x[e] = f.x, x[e + 1] = f.y, x[e + 2] = f.z, x[e + 3] = f.w;
        }
    } else if (N == 8) {
        const uint4 r = *reinterpret_cast<const uint4*>(base + first * 2);
        if (dt == GDN_BF16)
            Store<__nv_bfloat16>::unpack(r, x);
        else
            Store<__half>::unpack(r, x);
    } else {
        const uint2 r = *reinterpret_cast<const uint2*>(base + first * 2);
        if (dt == GDN_BF16) {
            x[0] = bf16_lo(r.x), x[1] = bf16_hi(r.x), x[2] = bf16_lo(r.y), x[3] = bf16_hi(r.y);
        } else {
            float2 f = f16x2_to_f2(r.x);
            x[0] = f.x, x[1] = f.y;
            f = f16x2_to_f2(r.y);
            x[2] = f.x, x[3] = f.y;
        }
    }
}

// Gates of the rule, in FP32:
//   alpha = exp(-exp(A_log) * softplus(a + dt_bias)),  beta = sigmoid(b)
// softplus(x) = x above 20, log(1 + e^x) otherwise.
__device__ __forceinline__ void gates(float A_log, float dt_bias, float a, float b, float& alpha, float& beta) {
    const float x = a + dt_bias;
    const float sp = x > 20.f ? x : log1pf(expf(x));
    alpha = expf(-expf(A_log) * sp);
    beta = 1.f / (1.f + expf(-b));
}

// The recurrence a kernel runs. GDN: the gated delta rule above. MAMBA2: the
// Mamba2 decode recurrence with the same state layout (key = B, value = x,
// query = C; no normalisation, no prediction term, plus the skip term D x):
//   delta = softplus(dt + dt_bias),  alpha = exp(-exp(A_log) delta)
//   S_t = alpha S_{t-1} + delta B x^T,   y_t = S_t^T C + D x
enum Rule : int { RULE_GDN = 0, RULE_MAMBA2 = 1 };

// Gates of one (sequence, head): GDN takes (a, b); Mamba2 takes dt in `a` and
// returns delta in `beta`.
template <int RULE>
__device__ __forceinline__ void rule_gates(float A_log, float dt_bias, const void* a, const void* b, int64_t i,
                                           int dt, float& alpha, float& beta) {
    if constexpr (RULE == RULE_GDN) {
        gates(A_log, dt_bias, load_elem(a, i, dt), load_elem(b, i, dt), alpha, beta);
    } else {
        const float x = load_elem(a, i, dt) + dt_bias;
        beta = x > 20.f ? x : log1pf(expf(x));
        alpha = expf(-expf(A_log) * beta);
    }
}

__device__ __forceinline__ void set_error(int32_t* dev_err, int bits) { atomicOr(dev_err, bits); }

// Complete `bytes` of a barrier's expected transaction with no copy. A bounds-checking build's
// skipped bulk copy does this, so that the copy's waiters see the phase complete (and read stale
// data, flagged by the error bit) instead of waiting out the timeout.
__device__ __forceinline__ void mbar_complete_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// Bounds-checking builds (compiled with GDN_DEBUG_BOUNDS): an access of `bytes` at `p` must lie in
// [base, base + extent); otherwise GDN_DEVERR_BOUNDS is set and the caller skips the access, so a
// wrong index shows as an error bit, never as a fault. In other builds the check is compiled out.
__device__ __forceinline__ bool in_bounds(const void* p, uint64_t bytes, const void* base, uint64_t extent,
                                          int32_t* dev_err) {
#ifdef GDN_DEBUG_BOUNDS
    const uint64_t a = reinterpret_cast<uint64_t>(p), b0 = reinterpret_cast<uint64_t>(base);
    if (a < b0 || a + bytes > b0 + extent) {
        set_error(dev_err, GDN_DEVERR_BOUNDS);
        return false;
    }
#else
    (void)p, (void)bytes, (void)base, (void)extent, (void)dev_err;
#endif
    return true;
}

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

}  // namespace gdn

namespace gdn {

// Bulk copies with the bounds check of bounds-checking builds: the source range must lie in
// [base, base + extent); a skipped copy completes its bytes on the barrier.
__device__ __forceinline__ void bulk_load_checked(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                  const void* base, uint64_t extent, int32_t* dev_err) {
    if (in_bounds(src, bytes, base, extent, dev_err))
        bulk_load(dst, src, bytes, bar);
    else
        mbar_complete_tx(bar, bytes);
}

__device__ __forceinline__ void bulk_load_hint_checked(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                       uint64_t policy, const void* base, uint64_t extent,
                                                       int32_t* dev_err) {
    if (in_bounds(src, bytes, base, extent, dev_err))
        bulk_load_hint(dst, src, bytes, bar, policy);
    else
        mbar_complete_tx(bar, bytes);
}

}  // namespace gdn
