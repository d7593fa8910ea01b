// gdn_replay_common.cuh -- what the two ReplaySSM kernels share: the
// launch arguments, the unit scheduling and a few copy and reduction helpers.
//
// Mode (AREX article on ReplaySSM, section "缓存输入而非状态：checkpoint 每
// L 步才更新一次"): keep a checkpoint S0 and the state-building inputs of the
// tokens since it in an L-entry ring; compute each output from S0 and the
// ring without writing the state; fold the ring into S0 when it is full;
// roll back rejected drafts by moving the ring pointer; verify a whole draft
// window in one pass.
//
// Arithmetic. Each buffered entry e (gates alpha_e, beta_e, unit key k_e)
// applies S_e = alpha_e S_{e-1} + k_e w_e^T with the correction vector
// w_e = beta_e (v_e - alpha_e S_{e-1}^T k_e). Unrolled from the checkpoint,
//   S_e = G(e) S0 + sum_{f<=e} A(f,e) k_f w_f^T,
//   G(e) = prod_{g<=e} alpha_g,   A(f,e) = prod_{f<g<=e} alpha_g.
// So for a window token e (query q):
//   S_{e-1}^T k_e = G(e-1) S0^T k_e + sum_{f<e}  A(f,e-1) (k_f.k_e) w_f
//   w_e           = beta_e (v_e - alpha_e S_{e-1}^T k_e)
//   o_e = S_e^T q = G(e)   S0^T q   + sum_{f<=e} A(f,e)   (k_f.q)   w_f
// The ring keeps w_f (fp32) and the key's inverse norm beside each entry's raw
// inputs, so one pass over S0 -- 2T dot products per state row -- and O(count)
// vector work give every output; S_t itself is only materialised (in FP32
// registers) when the ring is folded: S0 <- round(G S0 + sum A k w^T).
//
// The kernels: gdn_replay_rows.cuh (one checkpoint, a warp per unit and a
// state row per lane) and gdn_replay_producer.cuh (a producer warp feeding
// consumer warps through shared-memory rings; the two-checkpoint mode, and one
// fp32 checkpoint's single tokens). gdn_launch_replay.cuh picks one per call.
#pragma once

#include <type_traits>

#include "gdn_device.cuh"
#include "gdn_io.cuh"

namespace gdn {

constexpr int L_MAX = 64;
constexpr int WINDOW_MAX = 8;

struct ReplayArgs {
    void* ckpt;
    void* ring_k;
    void* ring_v;
    float* ring_rec;
    int32_t* pos;
    int32_t* ckpt_pos;
    const int32_t* slots;
    const void* q;
    const void* k;
    const void* v;
    const void* a;
    const void* b;
    const float* A_log;
    const float* dt_bias;
    const float* D;  // Mamba2 skip weights [Hv]; unused by the gated delta rule
    void* out;
    int32_t* dev_err;
    int64_t num_slots;
    int B, Hk, Hv, dv, L, T, force;
    int in_dtype, out_dtype;
    // Two-checkpoint mode (master type MT wider than the read type ST): ckpt is the master, which
    // only folds read and write; ckpt_copy is the read copy, which every other unit reads and
    // every fold rewrites from the stored master rows.
    void* ckpt_copy;
    float q_scale;
    // the producer kernel's chunking and shared-memory layout (set by its launch)
    int rows, nchunk;    // S0 rows per 16 KB chunk and chunks per unit, read type
    int mrows, mnchunk;  // the same for the master (equal to rows, nchunk with one checkpoint)
    int nstage, nhead;   // chunk and head ring depths
    int head_bytes, off_wq, off_wk, off_wv, off_rk, off_rec, off_rv, off_coef;  // inside a head stage, bytes
    int heads_off, sums_off, bars_off;                                          // inside the CTA's buffer
};

// Reduce-scatter of V values over aligned groups of G lanes (powers of two):
// halving steps while a lane holds more than one value, then butterfly
// steps. Afterwards lane g holds group totals in x[0..max(1, V/G)): values
// g*(V/G) + i when V >= G, value g/(G/V) when V < G (G/V lanes share it).
template <int NV, int D>
struct ScatterStep {
    template <int V>
    __device__ static __forceinline__ void run(float (&x)[V], int g) {
        if constexpr (D >= 1) {
            if constexpr (NV > 1) {
                const bool upper = (g & D) != 0;
#pragma unroll
                for (int i = 0; i < NV / 2; ++i) {
                    const float send = upper ? x[i] : x[i + NV / 2];
                    const float keep = upper ? x[i + NV / 2] : x[i];
                    x[i] = keep + __shfl_xor_sync(FULL_MASK, send, D);
                }
                ScatterStep<NV / 2, D / 2>::run(x, g);
            } else {
                x[0] += __shfl_xor_sync(FULL_MASK, x[0], D);
                ScatterStep<1, D / 2>::run(x, g);
            }
        }
    }
};

template <int V, int G>
__device__ __forceinline__ void reduce_scatter_values(float (&x)[V], int g) {
    ScatterStep<V, G / 2>::run(x, g);
}

// Store x rounded to T (round-to-nearest-even) at element `first` of a row, and replace x by
// the stored values.
template <typename T, int N>
__device__ __forceinline__ void st_state(unsigned char* row, int first, float* x) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int e = 0; e < N; e += 4)
            *reinterpret_cast<float4*>(row + (first + e) * 4) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
    } else if constexpr (N == 4) {
        const bool bf = std::is_same<T, __nv_bfloat16>::value;
        const uint2 r = bf ? make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]))
                           : make_uint2(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]));
        *reinterpret_cast<uint2*>(row + first * 2) = r;
        if (bf) {
            x[0] = bf16_lo(r.x), x[1] = bf16_hi(r.x), x[2] = bf16_lo(r.y), x[3] = bf16_hi(r.y);
        } else {
            float2 f = f16x2_to_f2(r.x);
            x[0] = f.x, x[1] = f.y;
            f = f16x2_to_f2(r.y);
            x[2] = f.x, x[3] = f.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < N; e += 8) {
            const uint4 packed = Store<T>::pack(x + e);
            *reinterpret_cast<uint4*>(row + (first + e) * 2) = packed;
            Store<T>::unpack(packed, x + e);
        }
    }
}


// Asynchronous copy of BYTES (16, 8 or 4) from global to shared memory, tracked
// by this thread's commit groups (cp_async_commit / cp_async_wait<N>): the
// copies always complete, no flag or barrier is polled.
template <int BYTES>
__device__ __forceinline__ void cp_async_piece(void* smem_dst, const void* gsrc) {
    if constexpr (BYTES == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_addr(smem_dst)), "l"(gsrc), "n"(BYTES)
                     : "memory");
}

// Unit scheduling of the row kernel: a CTA takes its units blockIdx.x + n * gridDim.x in rounds
// of REPLAY_ROUND. A round starts with every thread loading one unit's slot and pointers and listing
// the unit, fold units first; then the warps take the list's units one at a time from a counter, so
// the heavier fold units never trail a round and no warp waits on a unit's pointer loads. The head of
// the dynamic shared memory holds the counters and the two lists.
constexpr int REPLAY_ROUND = 256;
constexpr int REPLAY_SMEM_HEAD = 16 + 2 * REPLAY_ROUND * 16;

// One round's unit lists (REPLAY_ROUND, above): units blockIdx.x + (r0 + i) * gridDim.x, i < nr, as
// {unit, slot, pos, ckpt_pos}, fold units in lfold (ctr[1] of them), the others in lrest (ctr[2]);
// ctr[0], the warps' next list index, starts at 0. Called by every thread of the CTA.
__device__ __forceinline__ void replay_list_round(const ReplayArgs& p, int T, int L, int r0, int nr, int* ctr,
                                                  int4* lfold, int4* lrest) {
    if (threadIdx.x == 0) ctr[0] = ctr[1] = ctr[2] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < nr; i += blockDim.x) {
        const int u = blockIdx.x + (r0 + i) * gridDim.x;
        const int sl = p.slots[u / p.Hv];
        int ps = 0, ck = 0;
        bool heavy = false;  // folds (whether its pointers are valid is checked when it is run)
        if (sl >= 0 && sl < p.num_slots) {
            const int64_t idx = (int64_t)sl * p.Hv + (u - u / p.Hv * p.Hv);
            ps = p.pos[idx], ck = p.ckpt_pos[idx];
            heavy = T > 0 ? ps - ck + T > L : (p.force ? ps - ck > 0 : ps - ck + 1 > L);
        }
        if (heavy)
            lfold[atomicAdd(&ctr[1], 1)] = make_int4(u, sl, ps, ck);
        else
            lrest[atomicAdd(&ctr[2], 1)] = make_int4(u, sl, ps, ck);
    }
    __syncthreads();
}

}  // namespace gdn
