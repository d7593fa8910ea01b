// gdn_prefill_tc.cuh -- prefill of the gated delta rule in its chunked form on
// the tcgen05 tensor cores (16-bit states, dk = 128, dv a multiple of 128).
//
// Same semantics as prefill_kernel (vLLM PR #52191 summary, section 实现拆解
// items 3-4): the state is rounded to its dtype after every `interval` tokens
// and after the last one; outputs come from the unrounded FP32 state. Chunks
// end at those rounding points (and after at most 64 tokens), so a chunk
// starts from exactly the state the sequential rule would continue from.
//
// The chunked form (Gated DeltaNet paper, section 3, the WY/UT form of the
// delta rule with decays). With g_t the cumulative log-decay of the chunk's
// tokens up to t (inclusive) and S0 the state [dv rows j][dk columns i] at the
// chunk's start, the rule's corrections delta_t = beta_t (v_t - alpha_t S_{t-1}
// k_t) solve the unit lower-triangular system
//   delta_t + sum_{s<t} A[t][s] delta_s = beta_t (v_t - e^{g_t} S0 k_t),
//   A[t][s] = beta_t e^{g_t - g_s} (k_t . k_s),
// and then
//   o_t = e^{g_t} S0 q_t + sum_{s<=t} e^{g_t - g_s} (q_t . k_s) delta_s,
//   S_C = e^{g_C} S0 + sum_s delta_s (e^{g_C - g_s} k_s)^T.
//
// Kernel shape: one CTA per (sequence, value head, 128 state rows), 8 warps.
// The FP32 state stays in shared memory for the whole sequence, in the
// K-major layout of a tensor-core operand. Per chunk:
//  1. gates as cumulative base-2 log-decays (warp 0); keys and queries,
//     normalised, into [K; Q] (128 x dk); the decayed keys transposed into
//     K~ (dk x 64). The chunk's rows were loaded into registers, and its values
//     copied into shared memory, while the previous chunk computed;
//  2. tcgen05 MMAs into TMEM: S0 [K; Q]^T (128 x 128) and [K; Q] K^T (128 x 64);
//  3. Y = V - 2^g (S0 K^T) by one thread per state row (its TMEM lane), A and
//     P[t][s] = 2^{g_t - g_s} (q_t . k_s) (s <= t) beside it; the triangular
//     system's inverse T = (I + A)^{-1} diag(beta), shared by all rows, blockwise
//     (16 x 16 diagonal blocks by forward substitution, then the off-diagonal
//     blocks block row by block row) by all threads; delta^T = Y T^T on the
//     tensor cores;
//  4. tcgen05 MMAs: delta^T P^T (the outputs' intra-chunk part) and delta^T K~
//     (the state update);
//  5. outputs and the new state (rounded at a rounding point) by the threads.
// Operands are FP32 values in shared memory of which the MMA (kind::tf32)
// takes the TF32 part; accumulation is FP32 (rounding the operands to TF32
// first measured 4% slower, with the same parity). One TF32 pass keeps 16-bit states within their own rounding (in an
// emulation of this form over 2048-token sequences: state max-abs 2.2e-3 with a
// bf16 state, outputs 4.7e-5); FP32 states stay on prefill_kernel.
//
// tcgen05 use (PTX ISA, tcgen05 sections): TMEM allocated by warp 0 (512
// columns; one CTA per SM by its shared memory) and freed on every path; MMAs
// issued by one thread, completion through tcgen05.commit on an mbarrier whose
// waits are bounded; operands in shared memory without swizzle, K-major, as
// 8-row x 16-byte core matrices with the K-direction core matrices outermost
// (leading-dimension byte offset = rows x 16, stride-dimension byte offset =
// 128); accumulators read back with tcgen05.ld (32x32b: a warp reads the 32
// lanes of its sub-partition).
#pragma once

#include "gdn_device.cuh"
#include "gdn_io.cuh"
#include "gdn_prefill.cuh"

namespace gdn {

namespace tc {

constexpr int CH = 64;    // tokens per chunk at most
constexpr int DKT = 128;  // key dimension
constexpr int ROWS = 128;  // state rows per CTA (the MMAs' M)
constexpr int THREADS = 256;
// shared memory, bytes
constexpr int OFF_S = 0;                     // S0: FP32 [128 j][128 i], operand layout
constexpr int OFF_KQ = OFF_S + 128 * 128 * 4;  // [K; Q]: [128 n][128 i]
constexpr int OFF_D = OFF_KQ + 128 * 128 * 4;  // delta^T: [128 j][64 s]
constexpr int OFF_A = OFF_D + 128 * 64 * 4;    // A: [64 t][68] row-major (padded)
constexpr int A_LD = 68;
constexpr int OFF_P = OFF_A + 64 * A_LD * 4;   // P: [64 t][64 s], operand layout
constexpr int OFF_KT = OFF_P + 64 * 64 * 4;    // K~: [128 i][64 s], operand layout
constexpr int OFF_G = OFF_KT + 128 * 64 * 4;   // per token: g, beta, 2^g, alpha, 2^(g_C - g) [5][64]
constexpr int OFF_BAR = OFF_G + 5 * 64 * 4;    // mbarrier, TMEM address
constexpr int SMEM = OFF_BAR + 16;
static_assert(SMEM <= 232448, "shared memory");
// TMEM columns
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t C_SKQ = 0;    // S0 [K; Q]^T: [j][s] keys at 0..63, queries at 64..127
constexpr uint32_t C_G = 128;    // [K; Q] K^T: lane t < 64 keys, 64 + t queries; column s
constexpr uint32_t C_O = 192;    // delta^T P^T: [j][t]
constexpr uint32_t C_U = 256;    // delta^T K~: [j][i]
constexpr uint32_t C_D = 384;    // Y T^T = delta^T: [j][t]

// Byte offset of element (r, k) in a K-major operand of `rows` rows: core matrix (r / 8, k / 4) of 8
// rows x 16 bytes, the K-direction core matrices outermost.
__device__ __forceinline__ int op_off(int r, int k, int rows) {
    return ((k >> 2) * (rows >> 3) + (r >> 3)) * 128 + (r & 7) * 16 + (k & 3) * 4;
}

// Shared-memory matrix descriptor: start address, leading-dimension byte offset (between K-direction
// core matrices), stride-dimension byte offset (between 8-row groups), descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | (uint64_t)((lbo >> 4) & 0x3FFF) << 16 |
           (uint64_t)((sbo >> 4) & 0x3FFF) << 32 | (uint64_t)1 << 46;
}

// Instruction descriptor, kind::tf32: FP32 accumulator, TF32 A and B, both K-major, N and M.
__device__ __forceinline__ uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (TMEM) = / += A B^T over `ksteps` steps of 8: A `arows` x K, B `brows` x K (brows = N), both operands
// laid out by op_off with the given row counts.
__device__ __forceinline__ void mma_chain(uint32_t d, uint32_t a, int arows, uint32_t b, int brows, int N, int ksteps,
                                          bool accumulate) {
    const uint32_t idesc = idesc_tf32(128, N);
    for (int s = 0; s < ksteps; ++s) {
        const uint64_t ad = smem_desc(a + s * 2 * arows * 16, arows * 16, 128);
        const uint64_t bd = smem_desc(b + s * 2 * brows * 16, brows * 16, 128);
        const uint32_t acc = (accumulate || s > 0) ? 1u : 0u;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
            : "memory");
    }
}

__device__ __forceinline__ void commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// N consecutive TMEM columns of this thread's lane (the warp's sub-partition), as floats; the load and
// its wait in one statement, so that the destination registers are only read once they hold the data.
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v);
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void tmem_ld<64>(uint32_t taddr, float* v) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// x rounded to the 16-bit state dtype (nearest even), as FP32.
template <typename ST>
__device__ __forceinline__ float round_to(float x) {
    if constexpr (std::is_same<ST, __nv_bfloat16>::value)
        return __bfloat162float(__float2bfloat16_rn(x));
    else
        return __half2float(__float2half_rn(x));
}

// 2^x (PTX ex2.approx.ftz: relative error near 2^-22; the decays are kept as base-2 logarithms)
__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}


}  // namespace tc

template <typename ST, int IO = IO_ANY>
__global__ void __launch_bounds__(tc::THREADS, 1) prefill_tc_kernel(const PrefillArgs p) {
    using namespace tc;
    constexpr int DK = DKT;
    constexpr int SZ = (int)sizeof(ST);
    const int in_dt = io_in<IO>(p.in_dtype), out_dt = io_out<IO>(p.out_dtype);
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rb = blockIdx.x % p.row_blocks;
    const int unit = blockIdx.x / p.row_blocks;
    const int bseq = unit / p.Hv, h = unit - bseq * p.Hv, kh = h / (p.Hv / p.Hk);
    const int slot = p.slots[bseq];
    const int t0 = p.cu_seqlens[bseq], t1 = p.cu_seqlens[bseq + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.total) {
        if (tid == 0 && rb == 0 && h == 0) set_error(p.dev_err, GDN_DEVERR_SEQLEN);
        return;
    }
    const int T = t1 - t0;
    const int osz = dtype_size(out_dt), isz = dtype_size(in_dt);
    const uint64_t ext_out = (uint64_t)p.total * p.Hv * p.dv * osz;
    const uint64_t ext_state = (uint64_t)p.num_slots * p.Hv * p.dv * DK * SZ;
    const uint64_t ext_qk = (uint64_t)p.total * p.Hk * DK * isz;
    const uint64_t ext_v = (uint64_t)p.total * p.Hv * p.dv * isz;
    const int row0 = rb * ROWS;
    if (slot < 0 || slot >= p.num_slots) {
        if (slot >= p.num_slots && tid == 0 && rb == 0) set_error(p.dev_err, GDN_DEVERR_SLOT);
        for (int i = tid; i < T * ROWS; i += blockDim.x) {
            const int t = i / ROWS, r = i - t * ROWS;
            const int64_t oi = ((int64_t)(t0 + t) * p.Hv + h) * p.dv + row0 + r;
            if (in_bounds(static_cast<char*>(p.out) + oi * osz, osz, p.out, ext_out, p.dev_err))
                store_elem(p.out, oi, out_dt, 0.f);
        }
        return;
    }
    if (T == 0) return;

    unsigned char* sS = smem + OFF_S;
    unsigned char* sKQ = smem + OFF_KQ;
    unsigned char* sD = smem + OFF_D;
    float* sA = reinterpret_cast<float*>(smem + OFF_A);
    unsigned char* sP = smem + OFF_P;
    unsigned char* sKT = smem + OFF_KT;
    float* sg = reinterpret_cast<float*>(smem + OFF_G);  // cumulative base-2 log-decay g_t (inclusive)
    float* sbeta = sg + 64;                              // beta_t
    float* seg = sg + 128;                               // 2^{g_t}
    float* salpha = sg + 192;                            // alpha_t = 2^{g_t - g_{t-1}}
    float* skt = sg + 256;                               // 2^{g_C - g_t}
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tm_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8);
    unsigned char* gstate =
        static_cast<unsigned char*>(p.pool) + (((int64_t)slot * p.Hv + h) * p.dv + row0) * (int64_t)(DK * SZ);

    // ---- setup: barrier, TMEM, the initial state into the operand layout
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tm_slot)),
                     "r"(TM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    {
        // warp w: rows 16 w .. 16 w + 15 in two groups of 8; lane (rr, qq): row rr of the group, elements
        // 32 qq .. 32 qq + 31 (four 16-byte pieces of a 16-bit row)
        const int rr = lane & 7, qq = lane >> 3;
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            const int j = 16 * warp + 8 * grp + rr;
            float x[32];
            const unsigned char* src = gstate + (int64_t)j * DK * SZ + 32 * qq * SZ;
#pragma unroll
            for (int c = 0; c < 32 * SZ / 16; ++c) {
                uint4 raw = make_uint4(0, 0, 0, 0);
                if (in_bounds(src + 16 * c, 16, p.pool, ext_state, p.dev_err))
                    raw = *reinterpret_cast<const uint4*>(src + 16 * c);
                Store<ST>::unpack(raw, x + c * (16 / SZ));
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<float4*>(sS + op_off(j, 32 * qq + 4 * c, 128)) =
                    make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tm_slot;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float eA = -expf(p.A_log[h]) * 1.4426950408889634f, dtb = p.dt_bias[h];  // log2 of a decay per softplus
    uint32_t phase = 0;
    bool failed = false;
    auto wait_mma = [&]() {
        bool ok = mbar_wait(bar, phase);
        if (!ok) {
            if (tid == 0) set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
            mbar_wait(bar, phase);  // let MMAs still in flight finish before TMEM is freed
        }
        phase ^= 1;
        fence_after();
        return __syncthreads_or(!ok) == 0;
    };

    // Chunks end after 64 tokens, at a rounding point, or at the sequence's end. A chunk's key and query
    // rows and gate inputs are loaded into registers while the previous chunk computes, and its value rows
    // are copied into shared memory (cp.async) once the previous chunk's last MMAs have read that space.
    auto chunk_len = [&](int c) { return min(min(CH, T - c), p.interval - c % p.interval); };
    const int rr = lane & 7, qq = lane >> 3;  // [K; Q] row rr of a group of 8, elements 32 qq .. 32 qq + 31
    // raw bytes as loaded (converted where used, so that a load issued a chunk early does not wait):
    uint4 xr[2][8];      // warp w: rows 16 w + 8 grp + rr of [K; Q], 32 elements (4 pieces when 16-bit)
    uint32_t gr[2][2];   // warp 0: gate inputs a, b of tokens lane, 32 + lane
    auto load_kq = [&](int c, int Cn) {
        const int np = 2 * isz;  // 16-byte pieces of 32 elements
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            const int n = 16 * warp + 8 * grp + rr;
            const int t = n < 64 ? n : n - 64;
#pragma unroll
            for (int i = 0; i < 8; ++i) xr[grp][i] = make_uint4(0, 0, 0, 0);
            if (t < Cn) {
                const void* arr = n < 64 ? p.k : p.q;
                const int64_t row = (((int64_t)t0 + c + t) * p.Hk + kh) * DK + 32 * qq;
                const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(arr) + row * isz);
                if (in_bounds(src, 32 * isz, arr, ext_qk, p.dev_err)) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (i < np) xr[grp][i] = src[i];
                }
            }
        }
        if (warp == 0) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int t = lane + 32 * hf;
                gr[hf][0] = gr[hf][1] = 0;
                if (t < Cn) {
                    const int64_t gi = ((int64_t)t0 + c + t) * p.Hv + h;
                    if (isz == 4) {
                        gr[hf][0] = static_cast<const uint32_t*>(p.a)[gi], gr[hf][1] = static_cast<const uint32_t*>(p.b)[gi];
                    } else {
                        gr[hf][0] = static_cast<const uint16_t*>(p.a)[gi], gr[hf][1] = static_cast<const uint16_t*>(p.b)[gi];
                    }
                }
            }
        }
    };
    // a raw gate input as a float
    auto gate_in = [&](uint32_t r) {
        if (isz == 4) return __uint_as_float(r);
        if (in_dt == GDN_BF16) return __uint_as_float(r << 16);
        return __half2float(__ushort_as_half(static_cast<unsigned short>(r)));
    };
    auto stage_v = [&](int c, int Cn) {
        const int vpieces = ROWS * isz / 16;  // 16-byte pieces of a token's value row
        for (int i = tid; i < Cn * vpieces; i += THREADS) {
            const int t = i / vpieces, pc = i - t * vpieces;
            const char* src =
                static_cast<const char*>(p.v) + ((((int64_t)t0 + c + t) * p.Hv + h) * p.dv + row0) * isz + pc * 16;
            if (in_bounds(src, 16, p.v, ext_v, p.dev_err)) cp_async16(sD + t * ROWS * isz + pc * 16, src);
        }
        cp_async_commit();
    };

    int c0 = 0, C = chunk_len(0);
    load_kq(0, C);
    stage_v(0, C);
    while (c0 < T && !failed) {
        const bool round_end = (c0 + C) % p.interval == 0 || c0 + C == T;
        const int64_t tok0 = (int64_t)t0 + c0;
        const int c1 = c0 + C, C1 = c1 < T ? chunk_len(c1) : 0;

        // ---- 1a. gates: warp 0, lane l tokens l and 32 + l; inclusive scan of the base-2 log-decays (sg)
        if (warp == 0) {
            float la[2], be[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const bool live = lane + 32 * hf < C;
                const float xa = gate_in(gr[hf][0]) + dtb;
                const float sp = xa > 20.f ? xa : log1pf(expf(xa));
                la[hf] = live ? eA * sp : 0.f;
                be[hf] = live ? 1.f / (1.f + expf(-gate_in(gr[hf][1]))) : 0.f;
            }
            const float step[2] = {la[0], la[1]};  // each token's own log-decay
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(FULL_MASK, la[hf], off);
                    if (lane >= off) la[hf] += o;
                }
            la[1] += __shfl_sync(FULL_MASK, la[0], 31);
            const float gc = __shfl_sync(FULL_MASK, (C - 1) >> 5 ? la[1] : la[0], (C - 1) & 31);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int t = lane + 32 * hf;
                sg[t] = la[hf], sbeta[t] = be[hf];
                seg[t] = ex2(la[hf]), salpha[t] = ex2(step[hf]), skt[t] = ex2(gc - la[hf]);
            }
        }
        __syncthreads();

        // ---- 1b. [K; Q] normalised (rows n < 64 keys, 64 + t queries), K~ = 2^{g_C - g_s} k_s transposed
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            const int n = 16 * warp + 8 * grp + rr;
            const bool key = n < 64;
            const int t = key ? n : n - 64;
            float x[32];
            if (isz == 4) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    x[4 * i] = __uint_as_float(xr[grp][i].x), x[4 * i + 1] = __uint_as_float(xr[grp][i].y),
                    x[4 * i + 2] = __uint_as_float(xr[grp][i].z), x[4 * i + 3] = __uint_as_float(xr[grp][i].w);
            } else if (in_dt == GDN_BF16) {
#pragma unroll
                for (int i = 0; i < 4; ++i) Store<__nv_bfloat16>::unpack(xr[grp][i], x + 8 * i);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) Store<__half>::unpack(xr[grp][i], x + 8 * i);
            }
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) ss = fmaf(x[e], x[e], ss);
            ss += __shfl_xor_sync(FULL_MASK, ss, 8);
            ss += __shfl_xor_sync(FULL_MASK, ss, 16);
            const float sc = rsqrtf(ss + 1e-6f) * (key ? 1.f : p.q_scale);
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] *= sc;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<float4*>(sKQ + op_off(n, 32 * qq + 4 * c, 128)) =
                    make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
            if (key) {
                // K~ element (i, t): store k of the lane writes element e = 8 (k / 8) + ((k ^ key3) & 7), key3
                // = 2 qq + rr / 4, so that the 32 lanes of a store hit 32 banks (bank: (e & 7) 4 + t & 3). The
                // lane's registers are first permuted by XOR with key3 within groups of 8 (three conditional
                // swap stages), so that store k reads register k.
                const float dk = t < C ? skt[t] : 0.f;
                const int key3 = (2 * qq + (rr >> 2)) & 7;
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] *= dk;
#pragma unroll
                for (int bit = 1; bit < 8; bit <<= 1) {
                    const bool sw = key3 & bit;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (!(e & bit)) {
                            const float a0 = x[e], a1 = x[e | bit];
                            x[e] = sw ? a1 : a0, x[e | bit] = sw ? a0 : a1;
                        }
                }
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int e = (k & ~7) | ((k ^ key3) & 7);
                    *reinterpret_cast<float*>(sKT + op_off(32 * qq + e, t, 128)) = x[k];
                }
            }
        }
        cp_async_wait<0>();  // this thread's value pieces (visible to all after the barrier below)
        fence_async_smem();
        fence_before();
        __syncthreads();

        // ---- 2. S0 [K; Q]^T and [K; Q] K^T; meanwhile the next chunk's rows and gate inputs
        if (tid == 0) {
            fence_after();
            mma_chain(tmem + C_SKQ, smem_addr(sS), 128, smem_addr(sKQ), 128, 128, DK / 8, false);
            mma_chain(tmem + C_G, smem_addr(sKQ), 128, smem_addr(sKQ), 128, 64, DK / 8, false);
            commit(bar);
        }
        if (C1 > 0) load_kq(c1, C1);
        if (!wait_mma()) {
            failed = true;
            break;
        }

        // ---- 3. The triangular system through its inverse, shared by the block's rows: Y[j][s] = v_s[j] -
        // 2^{g_s} (S0 k_s)[j] (warps 0-3, row j = TMEM lane), A (warps 4, 5) and P (warps 6, 7) from
        // [K; Q] K^T; T = (I + A)^{-1} diag(beta) blockwise (16 x 16 blocks) by all threads; then
        // delta^T = Y T^T on the tensor cores. [K; Q] is free once its MMAs are done: it holds Y (an
        // operand), T (an operand; first the products of the off-diagonal stages) and the inverse.
        unsigned char* sY = sKQ;                                        // [128 j][64 s], operand layout
        unsigned char* sT = sKQ + 128 * 64 * 4;                         // [64 t][64 s], operand layout
        float* sM = reinterpret_cast<float*>(sT);                       // [6][16][16] products B_IK
        float* sTi = reinterpret_cast<float*>(sKQ + 128 * 64 * 4 + 64 * 64 * 4);  // (I + A)^{-1}, [64][64]
        {
            float v[CH];
            if (warp >= 4) {
                // TMEM lane t of [K; Q] K^T: warps 4, 5 keys (rows of A), warps 6, 7 queries (rows of P)
                const int n = 32 * (warp & 3) + lane;
                const bool key = n < 64;
                const int t = key ? n : n - 64;
                const float bt = key ? sbeta[t] : 1.f;
                tmem_ld<64>(tmem + lane_base + C_G, v);
                // 2^{g_t - g_s} = alpha_{s+1} ... alpha_t, built downwards from s = t
                float f = 1.f;
#pragma unroll
                for (int s_ = CH - 1; s_ >= 0; --s_) {
                    f = s_ >= t ? 1.f : f * salpha[s_ + 1];
                    const float e = bt * f * v[s_];
                    v[s_] = key ? (s_ < t ? e : 0.f) : (s_ <= t ? e : 0.f);
                }
                if (key) {
#pragma unroll
                    for (int i = 0; i < CH; i += 4)
                        *reinterpret_cast<float4*>(sA + t * A_LD + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                } else {
#pragma unroll
                    for (int i = 0; i < CH; i += 4)
                        *reinterpret_cast<float4*>(sP + op_off(t, i, 64)) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                }
            } else {
                const int j = 32 * warp + lane;
                tmem_ld<64>(tmem + lane_base + C_SKQ, v);
                // the staged values by explicit shared-memory loads (16-bit inputs) and the decays four at a time
                const uint32_t vrow = smem_addr(sD) + j * isz;
#pragma unroll
                for (int s4 = 0; s4 < CH; s4 += 4) {
                    const float4 e4 = *reinterpret_cast<const float4*>(seg + s4);
                    const float ev[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int s_ = s4 + u;
                        float vs;
                        if (isz == 2) {
                            uint16_t hraw;
                            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(hraw) : "r"(vrow + s_ * ROWS * 2));
                            vs = in_dt == GDN_BF16 ? __uint_as_float(static_cast<uint32_t>(hraw) << 16)
                                                   : __half2float(__ushort_as_half(hraw));
                        } else {
                            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(vs) : "r"(vrow + s_ * ROWS * 4));
                        }
                        v[s_] = s_ < C ? vs - ev[u] * v[s_] : 0.f;
                    }
                }
#pragma unroll
                for (int i = 0; i < CH; i += 4)
                    *reinterpret_cast<float4*>(sY + op_off(j, i, 128)) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            }
        }
        __syncthreads();
        // diagonal blocks: thread (k, c) < 64 inverts column c of block k by forward substitution
        if (tid < 64) {
            const int k = tid >> 4, c = tid & 15;
            float xv[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s4 = 0; s4 < r; s4 += 4) {
                    const float4 av = *reinterpret_cast<const float4*>(sA + (16 * k + r) * A_LD + 16 * k + s4);
                    acc[0] = fmaf(av.x, xv[s4], acc[0]);
                    if (s4 + 1 < r) acc[1] = fmaf(av.y, xv[s4 + 1], acc[1]);
                    if (s4 + 2 < r) acc[2] = fmaf(av.z, xv[s4 + 2], acc[2]);
                    if (s4 + 3 < r) acc[3] = fmaf(av.w, xv[s4 + 3], acc[3]);
                }
                xv[r] = r == c ? 1.f : -((acc[0] + acc[1]) + (acc[2] + acc[3]));  // zero above the diagonal
                sTi[(16 * k + r) * 64 + 16 * k + c] = xv[r];
            }
        }
        __syncthreads();
        // off-diagonal blocks: B_IK = Tinv[I][I] A[I][K] for every K < I at once, then block row by block row
        // Tinv[I][J] = -sum_{K=J}^{I-1} B_IK Tinv[K][J] (J < I); B_IK at sM[(I (I - 1) / 2 + K) 256]
        for (int o = tid; o < 6 * 256; o += THREADS) {
            const int pr = o >> 8, r = (o >> 4) & 15, c = o & 15;
            const int I = pr == 0 ? 1 : (pr < 3 ? 2 : 3), K = pr - I * (I - 1) / 2;
            const float* drow = sTi + (16 * I + r) * 64 + 16 * I;
            const float* acol = sA + (16 * I) * A_LD + 16 * K + c;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int u4 = 0; u4 < 16; u4 += 4) {
                const float4 d = *reinterpret_cast<const float4*>(drow + u4);
                acc[0] = fmaf(d.x, acol[(u4 + 0) * A_LD], acc[0]);
                acc[1] = fmaf(d.y, acol[(u4 + 1) * A_LD], acc[1]);
                acc[2] = fmaf(d.z, acol[(u4 + 2) * A_LD], acc[2]);
                acc[3] = fmaf(d.w, acol[(u4 + 3) * A_LD], acc[3]);
            }
            sM[o] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        }
        __syncthreads();
        for (int I = 1; I < 4; ++I) {
            for (int o = tid; o < I * 256; o += THREADS) {
                const int J = o >> 8, r = (o >> 4) & 15, c = o & 15;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                for (int K = J; K < I; ++K) {
                    const float* brow = sM + (I * (I - 1) / 2 + K) * 256 + r * 16;
                    const float* tcol = sTi + (16 * K) * 64 + 16 * J + c;
#pragma unroll
                    for (int s4 = 0; s4 < 16; s4 += 4) {
                        const float4 bv = *reinterpret_cast<const float4*>(brow + s4);
                        acc[0] = fmaf(bv.x, tcol[(s4 + 0) * 64], acc[0]);
                        acc[1] = fmaf(bv.y, tcol[(s4 + 1) * 64], acc[1]);
                        acc[2] = fmaf(bv.z, tcol[(s4 + 2) * 64], acc[2]);
                        acc[3] = fmaf(bv.w, tcol[(s4 + 3) * 64], acc[3]);
                    }
                }
                sTi[(16 * I + r) * 64 + 16 * J + c] = -((acc[0] + acc[1]) + (acc[2] + acc[3]));
            }
            __syncthreads();
        }
        // T[t][s] = Tinv[t][s] beta_s (zero above the diagonal), the operand of delta^T = Y T^T
        for (int o = tid; o < 64 * 16; o += THREADS) {
            const int t = o >> 4, s4 = (o & 15) * 4;
            float4 v = *reinterpret_cast<const float4*>(sTi + t * 64 + s4);
            v.x = s4 + 0 <= t ? v.x * sbeta[s4 + 0] : 0.f;
            v.y = s4 + 1 <= t ? v.y * sbeta[s4 + 1] : 0.f;
            v.z = s4 + 2 <= t ? v.z * sbeta[s4 + 2] : 0.f;
            v.w = s4 + 3 <= t ? v.w * sbeta[s4 + 3] : 0.f;
            *reinterpret_cast<float4*>(sT + op_off(t, s4, 64)) = v;
        }
        fence_async_smem();
        fence_before();
        __syncthreads();
        if (tid == 0) {
            fence_after();
            mma_chain(tmem + C_D, smem_addr(sY), 128, smem_addr(sT), 64, 64, CH / 8, false);
            commit(bar);
        }
        if (!wait_mma()) {
            failed = true;
            break;
        }
        // delta^T into the operand of the next MMAs (warps 0-3 tokens 0..31, warps 4-7 tokens 32..63)
        {
            const int j = 32 * (warp & 3) + lane, tb = 32 * (warp >> 2);
            float v[32];
            tmem_ld<32>(tmem + lane_base + C_D + tb, v);
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(sD + op_off(j, tb + i, 128)) =
                    make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
        fence_async_smem();
        fence_before();
        __syncthreads();

        // ---- 4. delta^T P^T (outputs) and delta^T K~ (state update)
        if (tid == 0) {
            fence_after();
            mma_chain(tmem + C_O, smem_addr(sD), 128, smem_addr(sP), 64, 64, CH / 8, false);
            mma_chain(tmem + C_U, smem_addr(sD), 128, smem_addr(sKT), 128, 128, CH / 8, false);
            commit(bar);
        }
        if (!wait_mma()) {
            failed = true;
            break;
        }
        if (C1 > 0) stage_v(c1, C1);  // the MMAs are done with delta^T

        // ---- 5. outputs (warps 0-3 tokens 0..31, warps 4-7 tokens 32..63) and the state (columns split alike)
        {
            const int j = 32 * (warp & 3) + lane;
            const int hw = warp >> 2;
            const int tb = 32 * hw;
            if (tb < C) {
                float sq[32], oi[32];
                tmem_ld<32>(tmem + lane_base + C_SKQ + 64 + tb, sq);
                tmem_ld<32>(tmem + lane_base + C_O + tb, oi);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int t = tb + i;
                    if (t < C) {
                        const float o = fmaf(seg[t], sq[i], oi[i]);
                        const int64_t idx = ((tok0 + t) * p.Hv + h) * p.dv + row0 + j;
                        if (in_bounds(static_cast<char*>(p.out) + idx * osz, osz, p.out, ext_out, p.dev_err))
                            store_elem(p.out, idx, out_dt, o);
                    }
                }
            }
            const float eg = seg[C - 1];
            const bool last = c0 + C == T;
            const int i0 = 64 * hw;
            float u[64];
            tmem_ld<64>(tmem + lane_base + C_U + i0, u);
#pragma unroll
            for (int q4 = 0; q4 < 64; q4 += 4) {
                float4* sp = reinterpret_cast<float4*>(sS + op_off(j, i0 + q4, 128));
                float4 sv = *sp;
                sv.x = fmaf(eg, sv.x, u[q4]), sv.y = fmaf(eg, sv.y, u[q4 + 1]);
                sv.z = fmaf(eg, sv.z, u[q4 + 2]), sv.w = fmaf(eg, sv.w, u[q4 + 3]);
                if (round_end) {
                    sv.x = round_to<ST>(sv.x), sv.y = round_to<ST>(sv.y);
                    sv.z = round_to<ST>(sv.z), sv.w = round_to<ST>(sv.w);
                }
                *sp = sv;
                u[q4] = sv.x, u[q4 + 1] = sv.y, u[q4 + 2] = sv.z, u[q4 + 3] = sv.w;
            }
            if (last) {
                unsigned char* dst = gstate + (int64_t)j * DK * SZ + i0 * SZ;
#pragma unroll
                for (int e = 0; e < 64; e += 16 / SZ)
                    if (in_bounds(dst + e * SZ, 16, p.pool, ext_state, p.dev_err))
                        *reinterpret_cast<uint4*>(dst + e * SZ) = Store<ST>::pack(u + e);
            }
        }
        fence_before();
        __syncthreads();
        c0 = c1, C = C1;
    }

    // ---- TMEM back (every path after the allocation comes here)
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TM_COLS) : "memory");
    }
}

}  // namespace gdn
