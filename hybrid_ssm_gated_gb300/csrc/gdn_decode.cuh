// gdn_decode.cuh -- the gated delta-rule decode step (gdn_decode_step).
//
// Rule (standard gated delta rule; the vLLM PR #52191 summary, section
// 实现拆解 items 3-4, fixes its numeric contract: FP32 arithmetic, state
// stored as fp32/bf16/fp16 and rounded once per write-back):
//   S_t = alpha S_{t-1} + beta k (v - alpha S_{t-1}^T k)^T,   o_t = S_t^T q.
// A dk x dv state is stored as dv rows ("columns of S") of dk contiguous
// elements, so for row j:
//   u_j = S[:,j].k   p_j = S[:,j].q   delta_j = beta (v_j - alpha u_j)
//   S'[:,j] = alpha S[:,j] + k delta_j     o_j = alpha p_j + (q.k) delta_j
// One read and one write of the state; ~4 FP32 ops per state element, so the
// step is bound by HBM bandwidth, not by arithmetic.
//
// Kernel shape: persistent CTAs over (sequence, value head) units, one
// producer warp + NCW consumer warps.
//  - The producer warp (two, taking alternate units, for 16-bit states)
//    fetches slot indices and gates for 32 units at a time (one lane per
//    unit), then streams each unit's state in 16 KB chunks
//    into an NS-deep shared-memory ring with bulk copies on the TMA engine
//    (cp.async.bulk + mbarrier transaction counts), together with the unit's
//    q/k/v rows into an NH-deep "head" ring; a unit's copies are spread over
//    the producer's lanes.
//  - Consumer warps read the chunk from shared memory (128-bit, conflict
//    free), do the fused update in FP32 registers, and store the new state
//    (packed to the storage type) and the output straight to global memory.
//    A row is covered by LPR = dk/16 lanes holding 16 elements each; the two
//    row dot products are reduced with log2(LPR) xor-shuffles.
//  - The consumer warps form groups of UW that take units in turn: a unit's
//    passes go to one group, so each warp normalises q and k for only its
//    group's units. Every warp still waits for and releases every chunk in
//    order, so no parity wait can alias.
//  - Every wait is bounded (GDN_DEVERR_TIMEOUT, then return).
// The same kernel runs the Mamba2 decode step (RULE_MAMBA2, gdn_device.cuh):
// k, q and v rows carry B, C and x, nothing is normalised, delta_j = beta x_j
// (beta being Mamba2's softplus step size), and o_j gains D x_j.
#pragma once

#include "gdn_device.cuh"

namespace gdn {

struct DecodeArgs {
    void* pool;
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
    int B, Hk, Hv, dv;
    int in_dtype, out_dtype;
    int rows;    // state rows per chunk
    int nchunk;  // dv / rows
    float q_scale;
};

#ifndef GDN_DECODE_UNIT_WARPS
#define GDN_DECODE_UNIT_WARPS 4
#endif
#ifndef GDN_DECODE_UNIT_WARPS_MAMBA2
#define GDN_DECODE_UNIT_WARPS_MAMBA2 2  // Mamba2 has no per-unit normalisation: smaller groups measured best
#endif

constexpr int CHUNK_BYTES = 16384;
constexpr int DV_MAX = 256;

template <typename ST, int DK, int NCW, int NS, int NH, int RULE = RULE_GDN>
struct DecodeCfg {
    static constexpr int VEC = Store<ST>::VEC;  // elements per 16-byte vector
    static constexpr int E = 16;                // state elements per lane per row
    static constexpr int NC = E / VEC;          // 16-byte vectors per lane per row
    static constexpr int LPR = DK / E;          // lanes per row
    static constexpr int RPP = 32 / LPR;        // rows per warp pass
    static constexpr int ROW_BYTES = DK * (int)sizeof(ST);
    // head stage: meta (16 B) | q row | k row (DK fp32 max each) | v row (DV_MAX fp32 max)
    static constexpr int OFF_Q = 16;
    static constexpr int OFF_K = OFF_Q + DK * 4;
    static constexpr int OFF_V = OFF_K + DK * 4;
    static constexpr int HEAD = align_up(OFF_V + DV_MAX * 4, 128);
    static constexpr int SMEM = NS * CHUNK_BYTES + NH * HEAD + (2 * NS + 2 * NH) * 8;
    // producer warps: units of a 16-bit state are small enough that one warp's per-unit issue latency
    // (about 0.75 us) bounds the step, so two warps take alternate units
    static constexpr int NP = sizeof(ST) == 2 ? 2 : 1;
    static_assert(NH % NP == 0, "each head stage is filled by one producer warp");
    static constexpr int THREADS = (NCW + NP) * 32;
    // warps per unit: a unit's passes are dealt over UW warps, the NG = NCW / UW groups taking
    // units in turn
    static constexpr int UW_ = RULE == RULE_GDN ? GDN_DECODE_UNIT_WARPS : GDN_DECODE_UNIT_WARPS_MAMBA2;
    static constexpr int UW = UW_ < NCW ? UW_ : NCW;
    static constexpr int NG = NCW / UW;
    static_assert(NCW % UW == 0, "unit warps must divide the consumer warps");
    static_assert(DK % E == 0 && LPR <= 32, "dk must be a multiple of 16 and at most 512");
};

template <typename ST, int DK, int NCW, int NS, int NH, int RULE = RULE_GDN>
__global__ void __launch_bounds__((NCW + (sizeof(ST) == 2 ? 2 : 1)) * 32, 1) decode_kernel(const DecodeArgs p) {
    using C = DecodeCfg<ST, DK, NCW, NS, NH, RULE>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* chunks = smem;
    unsigned char* heads = smem + NS * CHUNK_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(heads + NH * C::HEAD);
    uint64_t* cfull = bars;
    uint64_t* cempty = bars + NS;
    uint64_t* hfull = bars + 2 * NS;
    uint64_t* hempty = bars + 2 * NS + NH;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&cfull[s], 1), mbar_init(&cempty[s], NCW);
        for (int s = 0; s < NH; ++s) mbar_init(&hfull[s], 1), mbar_init(&hempty[s], NCW);
        fence_barrier_init();
    }
    __syncthreads();

    const int total = p.B * p.Hv;
    // store extents, for the bounds-checking build
    const uint64_t ext_state = (uint64_t)p.num_slots * p.Hv * p.dv * C::ROW_BYTES;
    const uint64_t ext_out = (uint64_t)total * p.dv * dtype_size(p.out_dtype);
    auto out_ok = [&](int64_t i) {
        return in_bounds(static_cast<char*>(p.out) + i * dtype_size(p.out_dtype), dtype_size(p.out_dtype), p.out,
                         ext_out, p.dev_err);
    };
    const int in_sz = dtype_size(p.in_dtype);
    const int group = p.Hv / p.Hk;

    if (warp < C::NP) {
        // ---------------------------------------------------------------- producer(s)
        // With NP warps, warp w provisions units n = w (mod NP). Unit n's chunks take the fills after
        // those of every earlier valid unit, whichever warp issued them; both warps count the valid
        // units of every batch. A warp waits for a chunk stage only after the head stage of its unit
        // was released, i.e. after the consumers finished unit n - NH: every fill older than one round
        // of the ring has then been consumed, so the parity wait cannot alias.
        const uint64_t pol = policy_evict_first();
        const uint32_t qbytes = DK * in_sz, vbytes = p.dv * in_sz;
        const uint32_t cbytes = p.rows * C::ROW_BYTES;
        // source extents, for the bounds-checking build
        const uint64_t ext_pool = (uint64_t)p.num_slots * p.Hv * p.dv * C::ROW_BYTES;
        const uint64_t ext_qk = (uint64_t)p.B * p.Hk * qbytes, ext_v = (uint64_t)p.B * p.Hv * vbytes;
        uint32_t m = 0;   // chunk fills issued (one producer: all; several: up to the last one this warp issued)
        uint32_t nh = 0;  // head fills issued (likewise)
        uint32_t vb = 0;  // valid units in earlier batches
        int n = 0;        // units visited
        bool ok = true;
        for (int n0 = 0; ok && blockIdx.x + n0 * gridDim.x < total; n0 += 32) {
            // lane l fetches the slot and gates of unit n0 + l
            const int my_unit = blockIdx.x + (n0 + lane) * gridDim.x;
            int slot = -1;
            float alpha = 0.f, beta = 0.f, dskip = 0.f;
            if (my_unit < total) {
                const int b = my_unit / p.Hv, h = my_unit - b * p.Hv;
                const int s = p.slots[b];
                if (s >= p.num_slots) {
                    set_error(p.dev_err, GDN_DEVERR_SLOT);
                } else if (s >= 0) {
                    slot = s;
                    rule_gates<RULE>(p.A_log[h], p.dt_bias[h], p.a, p.b, my_unit, p.in_dtype, alpha, beta);
                    if constexpr (RULE == RULE_MAMBA2) dskip = p.D[h];
                }
            }
            if constexpr (C::NP > 1) {
                const unsigned valid = __ballot_sync(FULL_MASK, slot >= 0);
                for (int i = warp; i < 32; i += C::NP) {
                    n = n0 + i;
                    const int unit = blockIdx.x + n * gridDim.x;
                    if (unit >= total) break;
                    const int s_i = __shfl_sync(FULL_MASK, slot, i);
                    const float al = __shfl_sync(FULL_MASK, alpha, i);
                    const float be = __shfl_sync(FULL_MASK, beta, i);
                    const float dsk = RULE == RULE_MAMBA2 ? __shfl_sync(FULL_MASK, dskip, i) : 0.f;
                    const int hs = n % NH;
                    unsigned char* head = heads + hs * C::HEAD;
                    if (lane == 0) {
                        if (n >= NH) ok = mbar_wait(&hempty[hs], ((n / NH) + 1) & 1);
                        if (ok) {
                            reinterpret_cast<int*>(head)[0] = s_i;
                            reinterpret_cast<float*>(head)[1] = al;
                            reinterpret_cast<float*>(head)[2] = be;
                            if constexpr (RULE == RULE_MAMBA2) reinterpret_cast<float*>(head)[3] = dsk;
                            if (s_i >= 0)
                                mbar_arrive_expect_tx(&hfull[hs], 2 * qbytes + vbytes);
                            else
                                mbar_arrive(&hfull[hs]);
                        }
                    }
                    ok = __shfl_sync(FULL_MASK, ok, 0);
                    if (!ok) break;
                    nh = n + 1;
                    if (s_i < 0) continue;
                    const int b = unit / p.Hv, h = unit - b * p.Hv, kh = h / group;
                    const int64_t qrow = (int64_t)b * p.Hk + kh;
                    {
                        const char* src = lane == 0   ? static_cast<const char*>(p.q) + qrow * qbytes
                                          : lane == 1 ? static_cast<const char*>(p.k) + qrow * qbytes
                                                      : static_cast<const char*>(p.v) + (int64_t)unit * vbytes;
                        unsigned char* dst = head + (lane == 0 ? C::OFF_Q : lane == 1 ? C::OFF_K : C::OFF_V);
                        if (lane < 3)
                            bulk_load_checked(dst, src, lane == 2 ? vbytes : qbytes, &hfull[hs],
                                              lane == 0 ? p.q : lane == 1 ? p.k : p.v, lane == 2 ? ext_v : ext_qk,
                                              p.dev_err);
                    }
                    // this unit's first fill: after those of the valid units before it
                    const uint32_t m0 = (vb + __popc(valid & ((1u << i) - 1u))) * (uint32_t)p.nchunk;
                    for (int c0 = 0; c0 < p.nchunk && ok; c0 += NS) {
                        const int c = c0 + lane;
                        if (lane < NS && c < p.nchunk) {
                            const uint32_t mc = m0 + c;
                            const int cs = mc % NS;
                            ok = mc < NS || mbar_wait(&cempty[cs], ((mc / NS) + 1) & 1);
                            if (ok) {
                                const char* src = static_cast<const char*>(p.pool) +
                                                  ((int64_t)s_i * p.Hv + h) * p.dv * C::ROW_BYTES + (int64_t)c * cbytes;
                                mbar_arrive_expect_tx(&cfull[cs], cbytes);
                                bulk_load_hint_checked(chunks + cs * CHUNK_BYTES, src, cbytes, &cfull[cs], pol, p.pool,
                                                       ext_pool, p.dev_err);
                            }
                        }
                        ok = __all_sync(FULL_MASK, ok);
                    }
                    m = m0 + p.nchunk;
                    if (!ok) break;
                }
                vb += __popc(valid);
                continue;
            }
            for (int i = 0; i < 32; ++i, ++n) {
                const int unit = blockIdx.x + n * gridDim.x;
                if (unit >= total) break;
                const int s_i = __shfl_sync(FULL_MASK, slot, i);
                const float al = __shfl_sync(FULL_MASK, alpha, i);
                const float be = __shfl_sync(FULL_MASK, beta, i);
                const float dsk = RULE == RULE_MAMBA2 ? __shfl_sync(FULL_MASK, dskip, i) : 0.f;
                // A single thread issues a bulk copy only every ~0.25 us, so the unit's
                // copies are spread over lanes: lanes 0-2 the q/k/v rows, lane c chunk c.
                const int hs = n % NH;
                unsigned char* head = heads + hs * C::HEAD;
                if (lane == 0) {
                    if (n >= NH) ok = mbar_wait(&hempty[hs], ((n / NH) + 1) & 1);
                    if (ok) {
                        reinterpret_cast<int*>(head)[0] = s_i;
                        reinterpret_cast<float*>(head)[1] = al;
                        reinterpret_cast<float*>(head)[2] = be;
                        if constexpr (RULE == RULE_MAMBA2) reinterpret_cast<float*>(head)[3] = dsk;
                        if (s_i >= 0)
                            mbar_arrive_expect_tx(&hfull[hs], 2 * qbytes + vbytes);
                        else
                            mbar_arrive(&hfull[hs]);
                        ++nh;
                    }
                }
                ok = __shfl_sync(FULL_MASK, ok, 0);
                if (!ok) break;
                if (s_i >= 0) {
                    const int b = unit / p.Hv, h = unit - b * p.Hv, kh = h / group;
                    const int64_t qrow = (int64_t)b * p.Hk + kh;
                    // the q/k/v rows first, in one convergent copy instruction (lanes 0-2)
                    {
                        const char* src = lane == 0   ? static_cast<const char*>(p.q) + qrow * qbytes
                                          : lane == 1 ? static_cast<const char*>(p.k) + qrow * qbytes
                                                      : static_cast<const char*>(p.v) + (int64_t)unit * vbytes;
                        unsigned char* dst = head + (lane == 0 ? C::OFF_Q : lane == 1 ? C::OFF_K : C::OFF_V);
                        if (lane < 3)
                            bulk_load_checked(dst, src, lane == 2 ? vbytes : qbytes, &hfull[hs],
                                              lane == 0 ? p.q : lane == 1 ? p.k : p.v, lane == 2 ? ext_v : ext_qk,
                                              p.dev_err);
                    }
                    // then the chunks, each lane's as soon as its stage is free (a wait for every stage
                    // first delays the early chunks); at most NS lanes at a time, so no lane waits for a
                    // stage another lane is about to fill
                    for (int c0 = 0; c0 < p.nchunk && ok; c0 += NS) {
                        const int c = c0 + lane;
                        if (lane < NS && c < p.nchunk) {
                            const uint32_t mc = m + c;
                            const int cs = mc % NS;
                            ok = mc < NS || mbar_wait(&cempty[cs], ((mc / NS) + 1) & 1);
                            if (ok) {
                                const char* src = static_cast<const char*>(p.pool) +
                                                  ((int64_t)s_i * p.Hv + h) * p.dv * C::ROW_BYTES + (int64_t)c * cbytes;
                                mbar_arrive_expect_tx(&cfull[cs], cbytes);
                                bulk_load_hint_checked(chunks + cs * CHUNK_BYTES, src, cbytes, &cfull[cs], pol, p.pool,
                                                       ext_pool, p.dev_err);
                            }
                        }
                        ok = __all_sync(FULL_MASK, ok);
                    }
                    m += p.nchunk;
                    if (!ok) break;
                }
            }
        }
        if (!ok && lane == 0) {
            set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
            // let every copy already issued land before the CTA can exit
            for (uint32_t s = 0; s < NS && s < m; ++s) mbar_wait(&cfull[s], ((m - 1 - s) / NS) & 1);
            for (uint32_t s = 0; s < NH && s < nh; ++s) mbar_wait(&hfull[s], ((nh - 1 - s) / NH) & 1);
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int cw = warp - C::NP;
    const int pg = lane % C::LPR;        // lane's position within its row group
    const int rsub = lane / C::LPR;      // row within the warp pass
    const int passes = p.rows / C::RPP;  // warp passes per chunk
    uint32_t m = 0;
    for (int n = 0;; ++n) {
        const int unit = blockIdx.x + n * gridDim.x;
        if (unit >= total) break;
        const int hs = n % NH;
        if (!mbar_wait(&hfull[hs], (n / NH) & 1)) {
            if (lane == 0) set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
            return;
        }
        const unsigned char* head = heads + hs * C::HEAD;
        const int slot = reinterpret_cast<const int*>(head)[0];
        const float alpha = reinterpret_cast<const float*>(head)[1];
        const float beta = reinterpret_cast<const float*>(head)[2];
        const float dskip = reinterpret_cast<const float*>(head)[3];  // Mamba2's D[h]
        if (slot < 0) {
            for (int j = cw * 32 + lane; j < p.dv; j += NCW * 32)
                if (out_ok((int64_t)unit * p.dv + j)) store_elem(p.out, (int64_t)unit * p.dv + j, p.out_dtype, 0.f);
        } else {
            // A unit's passes go to one group of UW warps (groups alternate by unit), so each warp
            // normalises the window for only its group's units; every warp still waits for and
            // releases every chunk, in order.
            const bool mine = (n % C::NG) == cw / C::UW;
            const int gw = cw % C::UW;
            // normalised k and q at this lane's 16 key positions, in packed FP32x2 pairs
            float2 kn2[C::E / 2], qn2[C::E / 2];
            float qk = 0.f;
            if (mine) {
                float kn[C::E], qn[C::E];
#pragma unroll
                for (int c = 0; c < C::NC; ++c) {
                    const int first = (c * C::LPR + pg) * C::VEC;
                    load_run<C::VEC>(head + C::OFF_K, first, p.in_dtype, kn + c * C::VEC);
                    load_run<C::VEC>(head + C::OFF_Q, first, p.in_dtype, qn + c * C::VEC);
                }
                float2 sk = make_float2(0.f, 0.f), sq = sk;
#pragma unroll
                for (int e = 0; e < C::E / 2; ++e) {
                    kn2[e] = make_float2(kn[2 * e], kn[2 * e + 1]), qn2[e] = make_float2(qn[2 * e], qn[2 * e + 1]);
                    sk = __ffma2_rn(kn2[e], kn2[e], sk), sq = __ffma2_rn(qn2[e], qn2[e], sq);
                }
                // Mamba2 takes B and C as they are
                const float ik = RULE == RULE_GDN ? rsqrtf(group_sum<C::LPR>(sk.x + sk.y) + 1e-6f) : 1.f;
                const float iq = RULE == RULE_GDN ? rsqrtf(group_sum<C::LPR>(sq.x + sq.y) + 1e-6f) * p.q_scale : 1.f;
                const float2 ik2 = make_float2(ik, ik), iq2 = make_float2(iq, iq);
                float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < C::E / 2; ++e) {
                    if constexpr (RULE == RULE_GDN) kn2[e] = __fmul2_rn(kn2[e], ik2), qn2[e] = __fmul2_rn(qn2[e], iq2);
                    d2 = __ffma2_rn(kn2[e], qn2[e], d2);
                }
                qk = group_sum<C::LPR>(d2.x + d2.y);
            }

            const int b = unit / p.Hv, h = unit - b * p.Hv;
            char* gstate = static_cast<char*>(p.pool) + ((int64_t)slot * p.Hv + h) * p.dv * C::ROW_BYTES;
            for (int c = 0; c < p.nchunk; ++c, ++m) {
                const int cs = m % NS;
                if (!mbar_wait(&cfull[cs], (m / NS) & 1)) {
                    if (lane == 0) set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
                    return;
                }
                const unsigned char* tile = chunks + cs * CHUNK_BYTES;
                // the unit's warp passes are spread over its group's warps across chunks
                for (int ps = mine ? ((gw - c * passes) % C::UW + C::UW) % C::UW : passes; ps < passes;
                     ps += C::UW) {
                    const int r = ps * C::RPP + rsub;
                    const int j = c * p.rows + r;
                    float s[C::E];
#pragma unroll
                    for (int cc = 0; cc < C::NC; ++cc) {
                        const uint4 raw = *reinterpret_cast<const uint4*>(tile + r * C::ROW_BYTES +
                                                                          (cc * C::LPR + pg) * 16);
                        Store<ST>::unpack(raw, s + cc * C::VEC);
                    }
                    float2 u2 = make_float2(0.f, 0.f), p2 = u2;
#pragma unroll
                    for (int e = 0; e < C::E / 2; ++e) {
                        const float2 s2 = make_float2(s[2 * e], s[2 * e + 1]);
                        if constexpr (RULE == RULE_GDN) u2 = __ffma2_rn(s2, kn2[e], u2);
                        p2 = __ffma2_rn(s2, qn2[e], p2);
                    }
                    const float u = RULE == RULE_GDN ? group_sum<C::LPR>(u2.x + u2.y) : 0.f;
                    const float pq = group_sum<C::LPR>(p2.x + p2.y);
                    const float vj = load_elem(head + C::OFF_V, j, p.in_dtype);
                    const float delta = RULE == RULE_GDN ? beta * (vj - alpha * u) : beta * vj;
                    const float2 al2 = make_float2(alpha, alpha), d2 = make_float2(delta, delta);
#pragma unroll
                    for (int e = 0; e < C::E / 2; ++e) {
                        const float2 r2 = __ffma2_rn(kn2[e], d2, __fmul2_rn(make_float2(s[2 * e], s[2 * e + 1]), al2));
                        s[2 * e] = r2.x, s[2 * e + 1] = r2.y;
                    }
                    char* dst = gstate + (int64_t)j * C::ROW_BYTES;
#pragma unroll
                    for (int cc = 0; cc < C::NC; ++cc)
                        if (in_bounds(dst + (cc * C::LPR + pg) * 16, 16, p.pool, ext_state, p.dev_err))
                            *reinterpret_cast<uint4*>(dst + (cc * C::LPR + pg) * 16) = Store<ST>::pack(s + cc * C::VEC);
                    if (pg == 0) {
                        float o = fmaf(alpha, pq, qk * delta);
                        if constexpr (RULE == RULE_MAMBA2) o = fmaf(dskip, vj, o);
                        if (out_ok((int64_t)unit * p.dv + j)) store_elem(p.out, (int64_t)unit * p.dv + j, p.out_dtype, o);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&cempty[cs]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hempty[hs]);
    }
}

}  // namespace gdn
