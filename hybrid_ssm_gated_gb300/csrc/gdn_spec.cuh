// gdn_spec.cuh -- speculative step with one state copy per window token
// (gdn_spec_step): the baseline that a ReplaySSM verify window replaces.
//
// Each sequence takes a window of T tokens (the last verified token and T-1
// drafts) from the state in its source slot. After token t the state is
// written, rounded once, to the token's own destination slot, so that after
// verification the state of the last accepted token is already stored; the
// recursion itself continues in FP32 registers. It costs one state read and
// T state writes per sequence and head, where the ReplaySSM verify window
// (gdn_replay_rows.cuh) reads the checkpoint once and writes no state: this kernel
// is the comparison point for that claim. The AREX article on ReplaySSM
// describes the baseline in its section "每步写回完整循环状态：SSM 解码的两个
// 瓶颈" (a recurrent state kept per draft token, about (1 + num_spec) times
// the state memory) and its removal in section "缓存输入而非状态".
//
// Per state row j (a column of S, dk contiguous) and token t:
//   u = S[:,j].k_t   p = S[:,j].q_t   delta = beta_t (v_t[j] - alpha_t u)
//   S[:,j] <- alpha_t S[:,j] + k_t delta    o_t[j] = alpha_t p + (q_t.k_t) delta
//
// Kernel shape: the decode kernel's. A persistent CTA runs one producer warp
// and NCW consumer warps over (sequence, value head) units. The producer
// writes a unit's metadata (slots, gates) to an NH-deep head ring and issues
// the window's q/k/v rows and the source state's 16 KB chunks in one
// convergent bulk-copy instruction (one copy per lane). Every consumer warp
// visits every unit and every chunk in order. A warp pass is RPP state rows,
// each taken through all T tokens, with LPR lanes per row and E elements per
// lane, and the unit's passes are dealt over the warps. Every wait is bounded
// (GDN_DEVERR_TIMEOUT, then return).
#pragma once

#include "gdn_decode.cuh"
#include "gdn_device.cuh"
#include "gdn_io.cuh"

namespace gdn {

constexpr int SPEC_WINDOW_MAX = 8;
constexpr int SPEC_META = 128;  // bytes of per-unit metadata at the start of a head stage

struct SpecArgs {
    void* pool;
    const int32_t* src_slots;
    const int32_t* dst_slots;
    const void* q;
    const void* k;
    const void* v;
    const void* a;
    const void* b;
    const float* A_log;
    const float* dt_bias;
    void* out;
    int32_t* dev_err;
    int64_t num_slots;
    int B, Hk, Hv, dv, T;
    int in_dtype, out_dtype;
    int rows, nchunk;  // state rows per chunk, chunks per state
    int nstage, nhead;
    float q_scale;
    int head_bytes, off_q, off_k, off_v;  // head stage layout, bytes
    int heads_off, bars_off;              // inside the CTA's buffer
};

struct SpecMeta {
    int src;  // >= 0 work; < 0 padding or refused (zero outputs)
    int pad[3];
    int dst[SPEC_WINDOW_MAX];
    float alpha[SPEC_WINDOW_MAX];
    float beta[SPEC_WINDOW_MAX];
};
static_assert(sizeof(SpecMeta) <= SPEC_META, "meta too large");

template <typename ST, int DK, int TMAX, int NCW>
struct SpecCfg {
    static constexpr int VEC = Store<ST>::VEC;
    static constexpr int E = 8;  // state elements per lane per row (the window's vectors stay in registers)
    static constexpr int NC = E / VEC > 0 ? E / VEC : 1;
    static constexpr int LPR = DK / E;
    static constexpr int RPP = 32 / LPR;
    static constexpr int ROW_BYTES = DK * (int)sizeof(ST);
    static constexpr int THREADS = (NCW + 1) * 32;
    static_assert(E % VEC == 0 && DK % E == 0 && LPR >= 2 && LPR <= 32, "unsupported dk");
};

template <typename ST, int DK, int TMAX, int NCW, int IO = IO_ANY>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) spec_kernel(const SpecArgs p) {
    using C = SpecCfg<ST, DK, TMAX, NCW>;
    const int in_dt = io_in<IO>(p.in_dtype), out_dt = io_out<IO>(p.out_dtype);
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* chunks = smem;
    unsigned char* heads = smem + p.heads_off;
    const int NS = p.nstage, NH = p.nhead;
    uint64_t* cfull = reinterpret_cast<uint64_t*>(smem + p.bars_off);
    uint64_t* cempty = cfull + NS;
    uint64_t* hfull = cempty + NS;
    uint64_t* hempty = hfull + NH;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&cfull[s], 1), mbar_init(&cempty[s], NCW);
        for (int s = 0; s < NH; ++s) mbar_init(&hfull[s], 1), mbar_init(&hempty[s], NCW);
        fence_barrier_init();
    }
    __syncthreads();

    const int total = p.B * p.Hv;
    const int in_sz = dtype_size(in_dt);
    const int group = p.Hv / p.Hk;
    const int T = p.T;
    // array extents in bytes, for the bounds-checking build
    const uint64_t ext_pool = (uint64_t)p.num_slots * p.Hv * p.dv * C::ROW_BYTES;
    const uint64_t ext_qk = (uint64_t)p.B * T * p.Hk * DK * in_sz, ext_v = (uint64_t)p.B * T * p.Hv * p.dv * in_sz;
    const uint64_t ext_out = (uint64_t)p.B * T * p.Hv * p.dv * dtype_size(out_dt);
    auto out_ok = [&](int64_t i) {
        return in_bounds(static_cast<char*>(p.out) + i * dtype_size(out_dt), dtype_size(out_dt), p.out, ext_out,
                         p.dev_err);
    };

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        const uint64_t pol = policy_evict_first();
        const uint32_t qbytes = DK * in_sz, vbytes = p.dv * in_sz;
        const uint32_t cbytes = p.rows * C::ROW_BYTES;
        uint32_t m = 0;   // chunk fills issued
        uint32_t nh = 0;  // head fills issued
        int n = 0;
        bool ok = true;
        for (int n0 = 0; ok && blockIdx.x + n0 * gridDim.x < total; n0 += 32) {
            // lane l fetches the slots and gates of unit n0 + l
            const int my_unit = blockIdx.x + (n0 + lane) * gridDim.x;
            int src = -1;
            int dst[TMAX];
            float al[TMAX], be[TMAX];
#pragma unroll
            for (int t = 0; t < TMAX; ++t) dst[t] = -1, al[t] = 0.f, be[t] = 0.f;
            if (my_unit < total) {
                const int b = my_unit / p.Hv, h = my_unit - b * p.Hv;
                const int s = p.src_slots[b];
                bool in_range = s < p.num_slots;
#pragma unroll
                for (int t = 0; t < TMAX; ++t)
                    if (t < T) {
                        dst[t] = p.dst_slots[(int64_t)b * T + t];
                        in_range = in_range && dst[t] < p.num_slots;
                    }
                if (s >= 0 && !in_range) {
                    set_error(p.dev_err, GDN_DEVERR_SLOT);
                } else if (s >= 0) {
                    src = s;
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        if (t < T) {
                            const int64_t gi = ((int64_t)b * T + t) * p.Hv + h;
                            gates(p.A_log[h], p.dt_bias[h], load_elem(p.a, gi, in_dt),
                                  load_elem(p.b, gi, in_dt), al[t], be[t]);
                        }
                    }
                }
            }
            for (int i = 0; i < 32; ++i, ++n) {
                const int unit = blockIdx.x + n * gridDim.x;
                if (unit >= total) break;
                const int s_i = __shfl_sync(FULL_MASK, src, i);
                const int hs = n % NH;
                unsigned char* head = heads + hs * p.head_bytes;
                if (lane == 0) {
                    if (n >= NH) ok = mbar_wait(&hempty[hs], ((n / NH) + 1) & 1);
                    if (ok) {
                        SpecMeta* meta = reinterpret_cast<SpecMeta*>(head);
                        meta->src = s_i;
                    }
                }
                ok = __shfl_sync(FULL_MASK, ok, 0);
                if (!ok) break;
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                    const int d = __shfl_sync(FULL_MASK, dst[t], i);
                    const float a_t = __shfl_sync(FULL_MASK, al[t], i), b_t = __shfl_sync(FULL_MASK, be[t], i);
                    if (lane == 0) {
                        SpecMeta* meta = reinterpret_cast<SpecMeta*>(head);
                        meta->dst[t] = d, meta->alpha[t] = a_t, meta->beta[t] = b_t;
                    }
                }
                if (lane == 0) {
                    if (s_i >= 0)
                        mbar_arrive_expect_tx(&hfull[hs], T * (2 * qbytes + vbytes));
                    else
                        mbar_arrive(&hfull[hs]);
                    ++nh;
                }
                if (s_i < 0) continue;
                const int b = unit / p.Hv, h = unit - b * p.Hv, kh = h / group;
                // one convergent bulk copy per round: lanes 0..3T-1 the window's q/k/v rows, then the
                // source state's chunks, at most NS per round so that no lane waits for a stage
                // another lane is about to fill
                const int hj = 3 * T;
                for (int c0 = 0, round = 0; ok && (round == 0 || c0 < p.nchunk); ++round) {
                    const int cl0 = round == 0 ? hj : 0;
                    const int per = min(NS, 32 - cl0);
                    const char* srcp = nullptr;
                    unsigned char* dstp = nullptr;
                    uint32_t bytes = 0;
                    uint64_t* bar = &hfull[hs];
                    const void* sbase = p.pool;  // the source's array and its extent (bounds-checking builds)
                    uint64_t sext = ext_pool;
                    if (round == 0 && lane < hj) {
                        const int t = lane / 3, kind = lane - 3 * t;
                        const int64_t qrow = ((int64_t)b * T + t) * p.Hk + kh;
                        const int64_t vrow = ((int64_t)b * T + t) * p.Hv + h;
                        srcp = kind == 0   ? static_cast<const char*>(p.q) + qrow * qbytes
                               : kind == 1 ? static_cast<const char*>(p.k) + qrow * qbytes
                                           : static_cast<const char*>(p.v) + vrow * vbytes;
                        dstp = head + (kind == 0 ? p.off_q + t * qbytes : kind == 1 ? p.off_k + t * qbytes
                                                                                    : p.off_v + t * vbytes);
                        bytes = kind == 2 ? vbytes : qbytes;
                        sbase = kind == 0 ? p.q : kind == 1 ? p.k : p.v;
                        sext = kind == 2 ? ext_v : ext_qk;
                    }
                    const int c = c0 + lane - cl0;
                    if (lane >= cl0 && lane - cl0 < per && c < p.nchunk) {
                        const uint32_t mc = m + c;
                        const int cs = mc % NS;
                        ok = mc < (uint32_t)NS || mbar_wait(&cempty[cs], ((mc / NS) + 1) & 1);
                        if (ok) {
                            mbar_arrive_expect_tx(&cfull[cs], cbytes);
                            srcp = static_cast<const char*>(p.pool) + ((int64_t)s_i * p.Hv + h) * p.dv * C::ROW_BYTES +
                                   (int64_t)c * cbytes;
                            dstp = chunks + cs * CHUNK_BYTES;
                            bytes = cbytes;
                            bar = &cfull[cs];
                        }
                    }
                    ok = __all_sync(FULL_MASK, ok);
                    if (ok && bytes) bulk_load_hint_checked(dstp, srcp, bytes, bar, pol, sbase, sext, p.dev_err);
                    c0 += per;
                }
                m += p.nchunk;
                if (!ok) break;
            }
        }
        if (!ok && lane == 0) {
            set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
            // let every copy already issued land before the CTA can exit
            for (uint32_t s = 0; s < (uint32_t)NS && s < m; ++s) mbar_wait(&cfull[s], ((m - 1 - s) / NS) & 1);
            for (uint32_t s = 0; s < (uint32_t)NH && s < nh; ++s) mbar_wait(&hfull[s], ((nh - 1 - s) / NH) & 1);
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int pg = lane % C::LPR;        // lane's position within its row group
    const int rsub = lane / C::LPR;      // row within the warp pass
    const int passes = p.rows / C::RPP;  // warp passes per chunk
    auto pos_of = [&](int cc) { return (cc * C::LPR + pg) * C::VEC; };
    uint32_t m = 0;
    for (int n = 0;; ++n) {
        const int unit = blockIdx.x + n * gridDim.x;
        if (unit >= total) break;
        const int hs = n % NH;
        if (!mbar_wait(&hfull[hs], (n / NH) & 1)) {
            if (lane == 0) set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
            return;
        }
        const unsigned char* head = heads + hs * p.head_bytes;
        const SpecMeta* meta = reinterpret_cast<const SpecMeta*>(head);
        const int src = meta->src;
        const int b = unit / p.Hv, h = unit - b * p.Hv;
        if (src < 0) {
            for (int x = cw * 32 + lane; x < T * p.dv; x += NCW * 32) {
                const int t = x / p.dv, j = x - t * p.dv;
                const int64_t oi = (((int64_t)b * T + t) * p.Hv + h) * p.dv + j;
                if (out_ok(oi)) store_elem(p.out, oi, out_dt, 0.f);
            }
        } else {
            // the window's keys and queries, normalised, at this lane's key positions; q_t.k_t
            float2 kw2[TMAX][C::E / 2], qw2[TMAX][C::E / 2];
            float qk[TMAX];
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
                float xk[C::E], xq[C::E];
#pragma unroll
                for (int e = 0; e < C::E; ++e) xk[e] = 0.f, xq[e] = 0.f;
                qk[t] = 0.f;
                if (t < T) {
#pragma unroll
                    for (int cc = 0; cc < C::NC; ++cc) {
                        load_run<C::VEC>(head + p.off_k + t * DK * in_sz, pos_of(cc), in_dt, xk + cc * C::VEC);
                        load_run<C::VEC>(head + p.off_q + t * DK * in_sz, pos_of(cc), in_dt, xq + cc * C::VEC);
                    }
                    float ssk = 0.f, ssq = 0.f;
#pragma unroll
                    for (int e = 0; e < C::E; ++e) ssk = fmaf(xk[e], xk[e], ssk), ssq = fmaf(xq[e], xq[e], ssq);
                    const float ik = rsqrtf(group_sum<C::LPR>(ssk) + 1e-6f);
                    const float iq = rsqrtf(group_sum<C::LPR>(ssq) + 1e-6f) * p.q_scale;
                    float d = 0.f;
#pragma unroll
                    for (int e = 0; e < C::E; ++e) xk[e] *= ik, xq[e] *= iq, d = fmaf(xk[e], xq[e], d);
                    qk[t] = group_sum<C::LPR>(d);
                }
#pragma unroll
                for (int e = 0; e < C::E / 2; ++e)
                    kw2[t][e] = make_float2(xk[2 * e], xk[2 * e + 1]), qw2[t][e] = make_float2(xq[2 * e], xq[2 * e + 1]);
            }
            for (int c = 0; c < p.nchunk; ++c, ++m) {
                const int cs = m % NS;
                if (!mbar_wait(&cfull[cs], (m / NS) & 1)) {
                    if (lane == 0) set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
                    return;
                }
                const unsigned char* tile = chunks + cs * CHUNK_BYTES;
                // the unit's warp passes are spread over the consumer warps across chunks
                for (int ps = ((cw - c * passes) % NCW + NCW) % NCW; ps < passes; ps += NCW) {
                    const int r = ps * C::RPP + rsub;
                    const int j = c * p.rows + r;
                    float s[C::E];
#pragma unroll
                    for (int cc = 0; cc < C::NC; ++cc)
                        Store<ST>::unpack(
                            *reinterpret_cast<const uint4*>(tile + r * C::ROW_BYTES + pos_of(cc) * (int)sizeof(ST)),
                            s + cc * C::VEC);
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        if (t < T) {
                            float2 u2 = make_float2(0.f, 0.f), p2 = u2;
#pragma unroll
                            for (int e = 0; e < C::E / 2; ++e) {
                                const float2 s2 = make_float2(s[2 * e], s[2 * e + 1]);
                                u2 = __ffma2_rn(s2, kw2[t][e], u2);
                                p2 = __ffma2_rn(s2, qw2[t][e], p2);
                            }
                            const float u = group_sum<C::LPR>(u2.x + u2.y);
                            const float pq = group_sum<C::LPR>(p2.x + p2.y);
                            const float alpha = meta->alpha[t], beta = meta->beta[t];
                            const float vj = load_elem(head + p.off_v + t * p.dv * in_sz, j, in_dt);
                            const float delta = beta * (vj - alpha * u);
                            const float2 al2 = make_float2(alpha, alpha), d2 = make_float2(delta, delta);
#pragma unroll
                            for (int e = 0; e < C::E / 2; ++e) {
                                const float2 r2 =
                                    __ffma2_rn(kw2[t][e], d2, __fmul2_rn(make_float2(s[2 * e], s[2 * e + 1]), al2));
                                s[2 * e] = r2.x, s[2 * e + 1] = r2.y;
                            }
                            const int64_t oi = (((int64_t)b * T + t) * p.Hv + h) * p.dv + j;
                            if (pg == 0 && out_ok(oi)) store_elem(p.out, oi, out_dt, fmaf(alpha, pq, qk[t] * delta));
                            const int d = meta->dst[t];
                            if (d >= 0) {  // this token's state copy, rounded once
                                char* dst = static_cast<char*>(p.pool) + (((int64_t)d * p.Hv + h) * p.dv + j) * C::ROW_BYTES;
#pragma unroll
                                for (int cc = 0; cc < C::NC; ++cc)
                                    if (in_bounds(dst + pos_of(cc) * (int)sizeof(ST), 16, p.pool, ext_pool, p.dev_err))
                                        *reinterpret_cast<uint4*>(dst + pos_of(cc) * (int)sizeof(ST)) =
                                            Store<ST>::pack(s + cc * C::VEC);
                            }
                        }
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
