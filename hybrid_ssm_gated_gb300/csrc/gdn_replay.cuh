// gdn_replay.cuh -- ReplaySSM for the gated delta rule: standard decode step,
// speculative verify window and fold (flush).
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
// So for a new token e (query q):
//   S_{e-1}^T k_e = G(e-1) S0^T k_e + sum_{f<e}  A(f,e-1) (k_f.k_e) w_f
//   w_e           = beta_e (v_e - alpha_e S_{e-1}^T k_e)
//   o_e = S_e^T q = G(e)   S0^T q   + sum_{f<=e} A(f,e)   (k_f.q)   w_f
// The ring keeps w_f (fp32) and the key's inverse norm beside each entry's raw
// inputs, so one pass over S0 -- two dot products per state element per
// window token -- and O(count) vector work give every output; S_t itself is
// only materialised (in FP32 registers) when the ring is folded:
// S0 <- round(G S0 + sum A k w^T).
//
// Kernel shape: persistent CTAs over (sequence, value head) units, four warp
// roles, so the per-unit scalar work never stalls the state stream:
//   warp 0       head producer: per-unit metadata (slot, pointers, gates) for
//                32 units at a time, then the unit's window rows and buffered
//                ring entries into a head ring (bulk copies, one per lane);
//   warp 1       chunk producer: streams S0 in 16 KB chunks into a chunk ring
//                (lane c issues chunk c of a unit) and tags each stage with
//                its unit; after the last chunk it posts one stop tag per row
//                warp;
//   NPW warps    prep: one warp prepares one whole unit into a scratch slot --
//                normalised window keys/queries, one lane per buffered entry
//                for its dot products with the window, decay products by a
//                suffix-product scan across lanes -- then appends the window
//                to the ring and moves the pointers;
//   NRW warps    rows: each takes whole chunks, round robin. Window size 1:
//                eight row passes of partial dot products, then one
//                reduce-scatter across the row's lanes leaves every lane
//                owning one row, so the w recursion, output and w store run
//                once per row, coalesced. Larger windows reduce per pass.
// Hand-offs: an mbarrier parity wait cannot tell a phase from the one two
// rounds earlier, so it is used alone only where the waiter sees every phase
// of that barrier in order (the producers; prep warps on their own scratch
// slots, the scratch ring depth being a multiple of the prep-warp count).
// Elsewhere the filler first publishes a unit / chunk number tag and the
// waiter checks the tag before the barrier (prep warps and head stages; row
// warps, which take every NRW-th chunk, and chunk stages / scratch slots).
// Every wait is bounded (GDN_DEVERR_TIMEOUT, then return).
#pragma once

#include "gdn_decode.cuh"
#include "gdn_device.cuh"

namespace gdn {

constexpr int L_MAX = 32;
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
    void* out;
    int32_t* dev_err;
    int64_t num_slots;
    int B, Hk, Hv, dv, L, T, force;
    int in_dtype, out_dtype;
    int rows, nchunk;
    int nstage, nhead, nscr;  // chunk, head and scratch ring depths
    float q_scale;
    // shared-memory layout, bytes
    int head_bytes, off_wq, off_wk, off_wv, off_rk, off_rec;  // inside a head stage
    int heads_off, scratch_off, scratch_bytes, bars_off;      // inside the CTA's buffer
    int off_kw, off_qw, off_coef;                             // inside a scratch slot
};

constexpr int REPLAY_META = 128;  // bytes of per-unit metadata at the start of a head stage

template <typename ST, int DK, int TMAX, int NPW, int NRW>
struct ReplayCfg {
    static constexpr int VEC = Store<ST>::VEC;
    static constexpr int E = TMAX <= 2 ? 16 : 8;  // state elements per lane per row
    static constexpr int NC = E / VEC;
    static constexpr int LPR = DK / E;    // lanes per row
    static constexpr int RPP = 32 / LPR;  // rows per warp pass
    static constexpr int ROW_BYTES = DK * (int)sizeof(ST);
    static constexpr int THREADS = (2 + NPW + NRW) * 32;
    static constexpr bool KW_REG = TMAX <= 4;  // window vectors held in registers by the row warps
    static constexpr bool FAST = TMAX == 1;    // one row per lane after a reduce-scatter
    static_assert(E % VEC == 0 && DK % E == 0 && LPR <= 32 && DK % 32 == 0, "unsupported dk");
};

// Per-unit metadata written by the head producer at the start of a head stage.
struct ReplayMeta {
    int slot;  // >= 0 work; -1 invalid (zero outputs); -2 nothing to do (flush)
    int count;
    int fold;
    int pos0;
    int ckpt0;
    int pad[3];
    float alpha[WINDOW_MAX];
    float beta[WINDOW_MAX];
};
static_assert(sizeof(ReplayMeta) <= REPLAY_META, "meta too large");

__device__ __forceinline__ float warp_sum(float x) { return group_sum<32>(x); }

__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(n) : "memory");
}

// Reduce-scatter of x[0..G) over aligned groups of G lanes: afterwards lane
// (group position g) holds the group total of x[g]. G lanes, G values.
template <int G>
__device__ __forceinline__ float reduce_scatter(float (&x)[G], int g) {
#pragma unroll
    for (int half = G / 2; half >= 1; half >>= 1) {
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

template <typename ST, int DK, int TMAX, int NPW, int NRW>
__global__ void __launch_bounds__((2 + NPW + NRW) * 32, 1) replay_kernel(const ReplayArgs p) {
    using C = ReplayCfg<ST, DK, TMAX, NPW, NRW>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* chunks = smem;
    unsigned char* heads = smem + p.heads_off;
    const int NS = p.nstage, NH = p.nhead, NSC = p.nscr;
    uint64_t* cfull = reinterpret_cast<uint64_t*>(smem + p.bars_off);
    uint64_t* cempty = cfull + NS;
    uint64_t* hfull = cempty + NS;
    uint64_t* hempty = hfull + NH;
    uint64_t* sempty = hempty + NH;
    // per chunk stage: {global chunk number, unit number (-1: stop), chunk of the unit, 0}
    int4* ctag = reinterpret_cast<int4*>(sempty + NSC);
    int* stag = reinterpret_cast<int*>(ctag + NS);  // per scratch slot: unit number prepared in it
    int* htag = stag + NSC;                          // per head stage: unit number it is being filled with

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&cfull[s], 1), mbar_init(&cempty[s], 1);
        for (int s = 0; s < NH; ++s) mbar_init(&hfull[s], 1), mbar_init(&hempty[s], p.nchunk + 2);
        for (int s = 0; s < NSC; ++s) mbar_init(&sempty[s], p.nchunk), stag[s] = -1;
        for (int s = 0; s < NS; ++s) ctag[s] = make_int4(-1, -1, 0, 0);
        for (int s = 0; s < NH; ++s) htag[s] = -1;
        fence_barrier_init();
    }
    __syncthreads();

    const int total = p.B * p.Hv;
    const int in_sz = dtype_size(p.in_dtype);
    const int group = p.Hv / p.Hk;
    const int T = p.T, L = p.L;
    const int rec_floats = 4 + p.dv;
    const int LT = L + TMAX;  // row stride of the coefficient tables

    if (warp == 0) {
        // ---------------------------------------------------------------- head producer
        const uint32_t qbytes = DK * in_sz, vbytes = p.dv * in_sz, recbytes = rec_floats * 4;
        uint32_t nh = 0;
        int n = 0;
        bool ok = true;
        for (int n0 = 0; ok && blockIdx.x + n0 * gridDim.x < total; n0 += 32) {
            const int my_unit = blockIdx.x + (n0 + lane) * gridDim.x;
            int slot = -1, count = 0, fold = 0, pos0 = 0, ck0 = 0;
            float al[TMAX], be[TMAX];
#pragma unroll
            for (int t = 0; t < TMAX; ++t) al[t] = 0.f, be[t] = 0.f;
            if (my_unit < total) {
                const int b = my_unit / p.Hv, h = my_unit - b * p.Hv;
                const int s = p.slots[b];
                if (s >= p.num_slots) {
                    set_error(p.dev_err, GDN_DEVERR_SLOT);
                } else if (s >= 0) {
                    const int64_t idx = (int64_t)s * p.Hv + h;
                    pos0 = p.pos[idx];
                    ck0 = p.ckpt_pos[idx];
                    count = pos0 - ck0;
                    if (ck0 < 0 || count < 0 || count > L) {
                        set_error(p.dev_err, GDN_DEVERR_RING);
                    } else if (T > 0) {
                        slot = s;
                        fold = count + T > L;
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) {
                            if (t < T) {
                                const int64_t gi = ((int64_t)b * T + t) * p.Hv + h;
                                gates(p.A_log[h], p.dt_bias[h], load_elem(p.a, gi, p.in_dtype),
                                      load_elem(p.b, gi, p.in_dtype), al[t], be[t]);
                            }
                        }
                    } else {
                        fold = p.force ? count > 0 : count == L;
                        slot = fold ? s : -2;
                    }
                }
            }
            for (int i = 0; i < 32; ++i, ++n) {
                const int unit = blockIdx.x + n * gridDim.x;
                if (unit >= total) break;
                const int s_i = __shfl_sync(FULL_MASK, slot, i);
                const int c_i = __shfl_sync(FULL_MASK, count, i);
                const int f_i = __shfl_sync(FULL_MASK, fold, i);
                const int p_i = __shfl_sync(FULL_MASK, pos0, i);
                const int k_i = __shfl_sync(FULL_MASK, ck0, i);
                float al_i[TMAX], be_i[TMAX];
#pragma unroll
                for (int t = 0; t < TMAX; ++t)
                    al_i[t] = __shfl_sync(FULL_MASK, al[t], i), be_i[t] = __shfl_sync(FULL_MASK, be[t], i);
                // One thread issues a bulk copy only every ~0.25 us: lane 0 posts the
                // transaction count, then each lane issues one of the unit's copies
                // (3 rows per window token, up to 4 ring ranges).
                const int hs = n % NH;
                unsigned char* head = heads + hs * p.head_bytes;
                const int rbase = k_i % L;
                const int n1 = min(c_i, L - rbase);
                if (lane == 0) {
                    if (n >= NH) ok = mbar_wait(&hempty[hs], ((n / NH) + 1) & 1);
                    if (ok) {
                        ReplayMeta* meta = reinterpret_cast<ReplayMeta*>(head);
                        meta->slot = s_i, meta->count = c_i, meta->fold = f_i, meta->pos0 = p_i, meta->ckpt0 = k_i;
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) meta->alpha[t] = al_i[t], meta->beta[t] = be_i[t];
                        *reinterpret_cast<volatile int*>(htag + hs) = n;  // before the stage is armed
                        if (s_i >= 0)
                            mbar_arrive_expect_tx(&hfull[hs], T * (2 * qbytes + vbytes) + c_i * (qbytes + recbytes));
                        else
                            mbar_arrive(&hfull[hs]);
                        ++nh;
                    }
                }
                ok = __shfl_sync(FULL_MASK, ok, 0);
                if (!ok) break;
                if (s_i >= 0) {
                    const int b = unit / p.Hv, h = unit - b * p.Hv, kh = h / group;
                    const int64_t unit_ring = ((int64_t)s_i * p.Hv + h) * L;
                    if (lane < 3 * T) {
                        const int t = lane / 3, kind = lane - 3 * t;
                        const int64_t qrow = ((int64_t)b * T + t) * p.Hk + kh;
                        const int64_t vrow = ((int64_t)b * T + t) * p.Hv + h;
                        if (kind == 0)
                            bulk_load(head + p.off_wq + t * qbytes, static_cast<const char*>(p.q) + qrow * qbytes, qbytes,
                                      &hfull[hs]);
                        else if (kind == 1)
                            bulk_load(head + p.off_wk + t * qbytes, static_cast<const char*>(p.k) + qrow * qbytes, qbytes,
                                      &hfull[hs]);
                        else
                            bulk_load(head + p.off_wv + t * vbytes, static_cast<const char*>(p.v) + vrow * vbytes, vbytes,
                                      &hfull[hs]);
                    } else if (lane < 3 * T + 4) {
                        const int job = lane - 3 * T;  // 0/1: first ring range (k, rec); 2/3: wrapped range
                        const int first = job < 2 ? 0 : n1, cnt = job < 2 ? n1 : c_i - n1, ridx = job < 2 ? rbase : 0;
                        if (cnt > 0) {
                            if ((job & 1) == 0)
                                bulk_load(head + p.off_rk + first * qbytes,
                                          static_cast<const char*>(p.ring_k) + (unit_ring + ridx) * qbytes, cnt * qbytes,
                                          &hfull[hs]);
                            else
                                bulk_load(head + p.off_rec + first * recbytes, p.ring_rec + (unit_ring + ridx) * rec_floats,
                                          cnt * recbytes, &hfull[hs]);
                        }
                    }
                }
            }
        }
        if (!ok && lane == 0) {
            set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
            for (uint32_t s = 0; s < (uint32_t)NH && s < nh; ++s) mbar_wait(&hfull[s], ((nh - 1 - s) / NH) & 1);
        }
        return;
    }

    if (warp == 1) {
        // ---------------------------------------------------------------- chunk producer
        // lane c waits for its stage and issues chunk c of the unit
        const uint64_t pol = policy_evict_first();
        const uint32_t cbytes = p.rows * C::ROW_BYTES;
        uint32_t m = 0;
        bool ok = true;
        for (int n = 0; ok; ++n) {
            const int unit = blockIdx.x + n * gridDim.x;
            if (unit >= total) break;
            const int hs = n % NH;
            if (!(ok = __all_sync(FULL_MASK, wait_tag(htag + hs, n) && mbar_wait(&hfull[hs], (n / NH) & 1)))) break;
            const int slot = reinterpret_cast<const ReplayMeta*>(heads + hs * p.head_bytes)->slot;
            __syncwarp();
            if (lane == 0) mbar_arrive(&hempty[hs]);  // done reading the unit's metadata
            if (slot < 0) continue;
            const int h = unit % p.Hv;
            // at most NS lanes at a time, so no lane waits for a stage another lane is about to fill
            for (int c0 = 0; c0 < p.nchunk && ok; c0 += NS) {
                const int c = c0 + lane;
                if (lane < NS && c < p.nchunk) {
                    const uint32_t mc = m + c;
                    const int cs = mc % NS;
                    ok = mc < (uint32_t)NS || mbar_wait(&cempty[cs], ((mc / NS) + 1) & 1);
                    if (ok) {
                        const char* src = static_cast<const char*>(p.ckpt) +
                                          ((int64_t)slot * p.Hv + h) * p.dv * C::ROW_BYTES + (int64_t)c * cbytes;
                        ctag[cs] = make_int4(mc, n, c, 0);
                        mbar_arrive_expect_tx(&cfull[cs], cbytes);
                        bulk_load_hint(chunks + cs * CHUNK_BYTES, src, cbytes, &cfull[cs], pol);
                    }
                }
                ok = __all_sync(FULL_MASK, ok);
            }
            m += p.nchunk;
        }
        if (ok && lane == 0) {  // one stop tag per row warp, posted in order by one lane
            for (int i = 0; i < NRW && ok; ++i) {
                const uint32_t mc = m + i;
                const int cs = mc % NS;
                ok = mc < (uint32_t)NS || mbar_wait(&cempty[cs], ((mc / NS) + 1) & 1);
                if (ok) {
                    ctag[cs] = make_int4(mc, -1, 0, 0);
                    mbar_arrive(&cfull[cs]);
                }
            }
        }
        if (!__all_sync(FULL_MASK, ok) && lane == 0) {
            set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
            for (uint32_t s = 0; s < (uint32_t)NS && s < m; ++s) mbar_wait(&cfull[s], ((m - 1 - s) / NS) & 1);
        }
        return;
    }

    if (warp < 2 + NPW) {
        // ---------------------------------------------------------------- prep warps
        const int pw = warp - 2;
        bool ok = true;
        for (int n = pw; ok; n += NPW) {
            const int unit = blockIdx.x + n * gridDim.x;
            if (unit >= total) break;
            const int hs = n % NH, ss = n % NSC;
            // the head stage may still hold an older unit's fill: wait for this unit's tag first
            if (!(ok = wait_tag(htag + hs, n) && mbar_wait(&hfull[hs], (n / NH) & 1))) break;
            if (n >= NSC && !(ok = mbar_wait(&sempty[ss], ((n / NSC) + 1) & 1))) break;
            const unsigned char* head = heads + hs * p.head_bytes;
            const ReplayMeta* meta = reinterpret_cast<const ReplayMeta*>(head);
            const int slot = meta->slot;
            const int b = unit / p.Hv, h = unit - b * p.Hv;
            if (slot < 0) {
                // no chunks will come for this unit: zero its outputs and release on the rows' behalf
                if (slot == -1 && T > 0) {
                    for (int x = lane; x < T * p.dv; x += 32) {
                        const int t = x / p.dv, j = x - t * p.dv;
                        store_elem(p.out, (((int64_t)b * T + t) * p.Hv + h) * p.dv + j, p.out_dtype, 0.f);
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_n(&sempty[ss], p.nchunk);
                    mbar_arrive_n(&hempty[hs], p.nchunk + 1);
                }
                continue;
            }
            unsigned char* scr = smem + p.scratch_off + ss * p.scratch_bytes;
            float* kw = reinterpret_cast<float*>(scr + p.off_kw);      // [TMAX][DK] window keys
            float* qw = reinterpret_cast<float*>(scr + p.off_qw);      // [TMAX][DK] window queries
            float* ckk = reinterpret_cast<float*>(scr + p.off_coef);   // [TMAX][LT]
            float* ckq = ckk + TMAX * LT;                              // [TMAX][LT]
            float* G1 = ckq + TMAX * LT;                               // [TMAX]
            float* G2 = G1 + TMAX;                                     // [TMAX]
            float* Gf = G2 + TMAX;                                     // [1]
            float* cf = Gf + 1;                                        // [L]
            const int count = meta->count, fold = meta->fold, pos0 = meta->pos0;
            const int cpr = fold ? 0 : count;  // ring entries in front of the window
            const float* rec = reinterpret_cast<const float*>(head + p.off_rec);
            const int64_t unit_ring = ((int64_t)slot * p.Hv + h) * L;
            // Lane groups as in the row warps: LPR lanes per vector, E elements per lane at
            // positions (cc * LPR + pg) * VEC + e; RPP vectors per warp pass.
            const int pg = lane % C::LPR, rsub = lane / C::LPR;
            auto pos_of = [&](int cc) { return (cc * C::LPR + pg) * C::VEC; };

            // window keys and queries, normalised; every group holds the whole vectors
            float kwn[C::KW_REG ? TMAX : 1][C::E], qwn[C::KW_REG ? TMAX : 1][C::E], ikw[TMAX];
            constexpr int KWN = C::KW_REG ? TMAX : 1;
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
                ikw[t] = 0.f;
                if (t < T) {
                    float xk[C::E], xq[C::E], ssk = 0.f, ssq = 0.f;
#pragma unroll
                    for (int cc = 0; cc < C::NC; ++cc) {
                        load_run<C::VEC>(head + p.off_wk + t * DK * in_sz, pos_of(cc), p.in_dtype, xk + cc * C::VEC);
                        load_run<C::VEC>(head + p.off_wq + t * DK * in_sz, pos_of(cc), p.in_dtype, xq + cc * C::VEC);
                    }
#pragma unroll
                    for (int e = 0; e < C::E; ++e) ssk = fmaf(xk[e], xk[e], ssk), ssq = fmaf(xq[e], xq[e], ssq);
                    const float ik = rsqrtf(group_sum<C::LPR>(ssk) + 1e-6f);
                    const float iq = rsqrtf(group_sum<C::LPR>(ssq) + 1e-6f) * p.q_scale;
                    ikw[t] = ik;
#pragma unroll
                    for (int e = 0; e < C::E; ++e) xk[e] *= ik, xq[e] *= iq;
                    if (rsub == 0) {
#pragma unroll
                        for (int cc = 0; cc < C::NC; ++cc) {
#pragma unroll
                            for (int u = 0; u < C::VEC; u += 4) {
                                const int e0 = cc * C::VEC + u;
                                *reinterpret_cast<float4*>(kw + t * DK + pos_of(cc) + u) =
                                    make_float4(xk[e0], xk[e0 + 1], xk[e0 + 2], xk[e0 + 3]);
                                *reinterpret_cast<float4*>(qw + t * DK + pos_of(cc) + u) =
                                    make_float4(xq[e0], xq[e0 + 1], xq[e0 + 2], xq[e0 + 3]);
                            }
                        }
                    }
                    if (C::KW_REG) {
#pragma unroll
                        for (int e = 0; e < C::E; ++e) kwn[t < KWN ? t : 0][e] = xk[e], qwn[t < KWN ? t : 0][e] = xq[e];
                    }
                }
            }
            __syncwarp();
            // window vector t at this lane's positions (registers, or the scratch table for wide windows)
            auto wk = [&](int t, int e) -> float {
                return C::KW_REG ? kwn[t < KWN ? t : 0][e] : kw[t * DK + pos_of(e / C::VEC) + e % C::VEC];
            };
            auto wq = [&](int t, int e) -> float {
                return C::KW_REG ? qwn[t < KWN ? t : 0][e] : qw[t * DK + pos_of(e / C::VEC) + e % C::VEC];
            };
            // window-window dot products (entries cpr + s): k_s.k_t for s < t, k_s.q_t for s <= t,
            // times the window decays between them
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
#pragma unroll
                for (int s = 0; s <= t; ++s) {
                    if (t < T) {
                        float dkk = 0.f, dkq = 0.f;
#pragma unroll
                        for (int e = 0; e < C::E; ++e) dkk = fmaf(wk(s, e), wk(t, e), dkk), dkq = fmaf(wk(s, e), wq(t, e), dkq);
                        dkk = group_sum<C::LPR>(dkk);
                        dkq = group_sum<C::LPR>(dkq);
                        if (lane == 0) {
                            float dec = 1.f;  // prod_{s < x < t} alpha_x
                            for (int x = s + 1; x < t; ++x) dec *= meta->alpha[x];
                            if (s < t) ckk[t * LT + cpr + s] = dkk * dec;
                            ckq[t * LT + cpr + s] = dkq * dec * (s < t ? meta->alpha[t] : 1.f);
                        }
                    }
                }
            }
            // buffered ring entries, RPP per warp pass: dot products with the window (scaled by the
            // entry's cached inverse norm), or the normalised key for a fold
            for (int f0 = 0; f0 < count; f0 += C::RPP) {
                const int f = min(f0 + rsub, count - 1);
                const float ik_f = rec[f * rec_floats + 2];
                float x[C::E];
#pragma unroll
                for (int cc = 0; cc < C::NC; ++cc)
                    load_run<C::VEC>(head + p.off_rk + f * DK * in_sz, pos_of(cc), p.in_dtype, x + cc * C::VEC);
                if (fold) {
                    // a fold reads the raw ring keys from the head stage with the cached inverse norms
                } else {
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        if (t < T) {
                            float2 a2 = make_float2(0.f, 0.f), b2 = a2;
#pragma unroll
                            for (int e = 0; e < C::E / 2; ++e) {
                                const float2 x2 = make_float2(x[2 * e], x[2 * e + 1]);
                                a2 = __ffma2_rn(x2, make_float2(wk(t, 2 * e), wk(t, 2 * e + 1)), a2);
                                b2 = __ffma2_rn(x2, make_float2(wq(t, 2 * e), wq(t, 2 * e + 1)), b2);
                            }
                            const float dkk = group_sum<C::LPR>(a2.x + a2.y);
                            const float dkq = group_sum<C::LPR>(b2.x + b2.y);
                            if (pg == 0 && f0 + rsub < count) ckk[t * LT + f] = dkk * ik_f, ckq[t * LT + f] = dkq * ik_f;
                        }
                    }
                }
            }
            __syncwarp();
            // decay products, one lane per ring entry: R(f) = prod_{f<g<count} alpha_g by a suffix scan
            const bool mine = lane < count;
            float suf = mine ? rec[lane * rec_floats] : 1.f;  // inclusive suffix product
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_down_sync(FULL_MASK, suf, off);
                if (lane + off < 32) suf *= o;
            }
            const float gring = __shfl_sync(FULL_MASK, suf, 0);  // prod of all ring alphas
            float R = __shfl_down_sync(FULL_MASK, suf, 1);
            if (lane == 31) R = 1.f;
            if (lane == 0) {
                float wp = 1.f;  // prod of window alphas before token t
                for (int t = 0; t < T; ++t) {
                    G1[t] = (fold ? 1.f : gring) * wp;
                    wp *= meta->alpha[t];
                    G2[t] = (fold ? 1.f : gring) * wp;
                }
                if (fold) Gf[0] = gring;
            }
            if (mine) {
                if (fold) {
                    cf[lane] = R;
                } else {
                    float wp = 1.f;  // A(f, cpr + t - 1) = R(f) * prod_{s<t} alpha_s
                    for (int t = 0; t < T; ++t) {
                        ckk[t * LT + lane] *= R * wp;
                        wp *= meta->alpha[t];
                        ckq[t * LT + lane] *= R * wp;
                    }
                }
            }
            // append the window's raw inputs, gates and key norms to the ring; move the pointers
            const int kvec = DK * in_sz / 16, vvec = p.dv * in_sz / 16;
            for (int t = 0; t < T; ++t) {
                const int64_t ent = unit_ring + (pos0 + t) % L;
                for (int x = lane; x < kvec; x += 32)
                    reinterpret_cast<uint4*>(static_cast<char*>(p.ring_k) + ent * DK * in_sz)[x] =
                        reinterpret_cast<const uint4*>(head + p.off_wk + t * DK * in_sz)[x];
                for (int x = lane; x < vvec; x += 32)
                    reinterpret_cast<uint4*>(static_cast<char*>(p.ring_v) + ent * p.dv * in_sz)[x] =
                        reinterpret_cast<const uint4*>(head + p.off_wv + t * p.dv * in_sz)[x];
            }
            if (lane < T) {
                float ikt = ikw[0];
#pragma unroll
                for (int t = 1; t < TMAX; ++t)
                    if (lane == t) ikt = ikw[t];
                const int64_t ent = unit_ring + (pos0 + lane) % L;
                *reinterpret_cast<float4*>(p.ring_rec + ent * rec_floats) =
                    make_float4(meta->alpha[lane], meta->beta[lane], ikt, 0.f);
            }
            if (lane == 0) {
                const int64_t idx = (int64_t)slot * p.Hv + h;
                p.pos[idx] = pos0 + T;
                if (fold) p.ckpt_pos[idx] = pos0;
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();  // scratch contents before the tag
                *reinterpret_cast<volatile int*>(stag + ss) = n;
                mbar_arrive(&hempty[hs]);
            }
        }
        if (!ok && lane == 0) set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
        return;
    }

    // -------------------------------------------------------------------- row warps
    const int rw = warp - 2 - NPW;
    const int pg = lane % C::LPR;
    const int rsub = lane / C::LPR;
    bool ok = true;
    for (uint32_t m = rw;; m += NRW) {
        const int cs = m % NS;
        // the stage's tag names the chunk first, so an older round of the stage is never taken for it
        if (!(ok = wait_tag(&ctag[cs].x, (int)m) && mbar_wait(&cfull[cs], (m / NS) & 1))) break;
        const int4 tag = ctag[cs];
        if (tag.y < 0) {  // stop: release the stage (a later stop tag may need it) and leave
            __syncwarp();
            if (lane == 0) mbar_arrive(&cempty[cs]);
            break;
        }
        const int n = tag.y, c = tag.z;
        const int hs = n % NH, ss = n % NSC;
        if (!(ok = wait_tag(stag + ss, n) && mbar_wait(&hfull[hs], (n / NH) & 1))) break;
        __threadfence_block();  // scratch contents after the tag
        const int unit = blockIdx.x + n * gridDim.x;
        const unsigned char* head = heads + hs * p.head_bytes;
        const ReplayMeta* meta = reinterpret_cast<const ReplayMeta*>(head);
        const int slot = meta->slot;
        const int b = unit / p.Hv, h = unit - b * p.Hv;
        const int count = meta->count, fold = meta->fold, pos0 = meta->pos0;
        const int cpr = fold ? 0 : count;
        const int64_t unit_ring = ((int64_t)slot * p.Hv + h) * L;
        const float* rec = reinterpret_cast<const float*>(head + p.off_rec);
        const unsigned char* scr = smem + p.scratch_off + ss * p.scratch_bytes;
        const float* kwp = reinterpret_cast<const float*>(scr + p.off_kw);
        const float* qwp = reinterpret_cast<const float*>(scr + p.off_qw);
        const float* ckk = reinterpret_cast<const float*>(scr + p.off_coef);
        const float* ckq = ckk + TMAX * LT;
        const float* G1 = ckq + TMAX * LT;
        const float* G2 = G1 + TMAX;
        const float gfold = fold ? G2[TMAX] : 1.f;  // Gf follows G2
        const float* cf = G2 + TMAX + 1;
        const unsigned char* tile = chunks + cs * CHUNK_BYTES;
        char* gck = static_cast<char*>(p.ckpt) + ((int64_t)slot * p.Hv + h) * p.dv * C::ROW_BYTES;

        // window vectors at this lane's key positions
        auto win = [&](const float* base, int t, int cc, int u) -> float4 {
            return *reinterpret_cast<const float4*>(base + t * DK + (cc * C::LPR + pg) * C::VEC + u);
        };
        constexpr int KWN = C::KW_REG ? TMAX : 1;
        float kw[KWN][C::E], qw[KWN][C::E];
        if (C::KW_REG) {
#pragma unroll
            for (int t = 0; t < KWN; ++t) {
#pragma unroll
                for (int cc = 0; cc < C::NC; ++cc) {
#pragma unroll
                    for (int u = 0; u < C::VEC; u += 4) {
                        float4 vk = make_float4(0.f, 0.f, 0.f, 0.f), vq = vk;
                        if (t < T) vk = win(kwp, t, cc, u), vq = win(qwp, t, cc, u);
                        const int e0 = cc * C::VEC + u;
                        kw[t][e0] = vk.x, kw[t][e0 + 1] = vk.y, kw[t][e0 + 2] = vk.z, kw[t][e0 + 3] = vk.w;
                        qw[t][e0] = vq.x, qw[t][e0 + 1] = vq.y, qw[t][e0 + 2] = vq.z, qw[t][e0 + 3] = vq.w;
                    }
                }
            }
        }

        // Load one state row of the chunk (this lane's E elements) and fold it if required.
        auto load_row = [&](int r, float (&s)[C::E]) {
#pragma unroll
            for (int cc = 0; cc < C::NC; ++cc) {
                const uint4 raw = *reinterpret_cast<const uint4*>(tile + r * C::ROW_BYTES + (cc * C::LPR + pg) * 16);
                Store<ST>::unpack(raw, s + cc * C::VEC);
            }
            if (fold) {
                // S0 <- round(G S0 + sum_f A(f, count-1) k_f w_f^T), row j
                const int j = c * p.rows + r;
#pragma unroll
                for (int e = 0; e < C::E; ++e) s[e] *= gfold;
                for (int f = 0; f < count; ++f) {
                    // k_f = raw key * 1/|k_f| (cached in the record)
                    const float cwf = cf[f] * rec[f * rec_floats + 4 + j] * rec[f * rec_floats + 2];
                    float kr[C::E];
#pragma unroll
                    for (int cc = 0; cc < C::NC; ++cc)
                        load_run<C::VEC>(head + p.off_rk + f * DK * in_sz, (cc * C::LPR + pg) * C::VEC, p.in_dtype,
                                         kr + cc * C::VEC);
#pragma unroll
                    for (int e = 0; e < C::E; ++e) s[e] = fmaf(kr[e], cwf, s[e]);
                }
                char* dst = gck + (int64_t)j * C::ROW_BYTES;
#pragma unroll
                for (int cc = 0; cc < C::NC; ++cc) {
                    const uint4 packed = Store<ST>::pack(s + cc * C::VEC);
                    *reinterpret_cast<uint4*>(dst + (cc * C::LPR + pg) * 16) = packed;
                    Store<ST>::unpack(packed, s + cc * C::VEC);  // continue from the stored values
                }
            }
        };

        if (T > 0 && C::FAST) {
            // window of one token: per 32-row block, LPR passes of partial dots, then a reduce-scatter
            // leaves lane (rsub, pg) with the sums of row pg * RPP + rsub of the block
            constexpr int MAXBLK = CHUNK_BYTES / C::ROW_BYTES / 32 > 0 ? CHUNK_BYTES / C::ROW_BYTES / 32 : 1;
            float2 kw2[C::E / 2], qw2[C::E / 2];
#pragma unroll
            for (int e = 0; e < C::E / 2; ++e)
                kw2[e] = make_float2(kw[0][2 * e], kw[0][2 * e + 1]), qw2[e] = make_float2(qw[0][2 * e], qw[0][2 * e + 1]);
            const float g1 = G1[0], g2 = G2[0], al = meta->alpha[0], be = meta->beta[0];
            const float cdiag = ckq[cpr];  // k_t.q_t
            const int nblk = p.rows / 32;
            float Yb[MAXBLK], Zb[MAXBLK];
#pragma unroll
            for (int blk = 0; blk < MAXBLK; ++blk) {
                if (blk < nblk) {
                    const int r0 = blk * 32;
                    float y[C::LPR], z[C::LPR];
                    if (fold) {
#pragma unroll
                        for (int ps = 0; ps < C::LPR; ++ps) {
                            float s[C::E];
                            load_row(r0 + ps * C::RPP + rsub, s);
                            float2 u2 = make_float2(0.f, 0.f), v2 = u2;
#pragma unroll
                            for (int e = 0; e < C::E / 2; ++e) {
                                const float2 s2 = make_float2(s[2 * e], s[2 * e + 1]);
                                u2 = __ffma2_rn(s2, kw2[e], u2);
                                v2 = __ffma2_rn(s2, qw2[e], v2);
                            }
                            y[ps] = u2.x + u2.y;
                            z[ps] = v2.x + v2.y;
                        }
                    } else {
                        // 16-byte vector cc of all LPR passes first, then their math: 2*LPR independent chains
                        float2 u2[C::LPR], v2[C::LPR];
#pragma unroll
                        for (int ps = 0; ps < C::LPR; ++ps) u2[ps] = make_float2(0.f, 0.f), v2[ps] = u2[ps];
#pragma unroll
                        for (int cc = 0; cc < C::NC; ++cc) {
                            uint4 raw[C::LPR];
#pragma unroll
                            for (int ps = 0; ps < C::LPR; ++ps)
                                raw[ps] = *reinterpret_cast<const uint4*>(tile + (r0 + ps * C::RPP + rsub) * C::ROW_BYTES +
                                                                          (cc * C::LPR + pg) * 16);
#pragma unroll
                            for (int ps = 0; ps < C::LPR; ++ps) {
                                float sv[C::VEC];
                                Store<ST>::unpack(raw[ps], sv);
#pragma unroll
                                for (int e = 0; e < C::VEC / 2; ++e) {
                                    const float2 s2 = make_float2(sv[2 * e], sv[2 * e + 1]);
                                    u2[ps] = __ffma2_rn(s2, kw2[cc * C::VEC / 2 + e], u2[ps]);
                                    v2[ps] = __ffma2_rn(s2, qw2[cc * C::VEC / 2 + e], v2[ps]);
                                }
                            }
                        }
#pragma unroll
                        for (int ps = 0; ps < C::LPR; ++ps) y[ps] = u2[ps].x + u2[ps].y, z[ps] = v2[ps].x + v2[ps].y;
                    }
                    Yb[blk] = reduce_scatter<C::LPR>(y, pg) * g1;
                    Zb[blk] = reduce_scatter<C::LPR>(z, pg) * g2;
                }
            }
            // the chunk's state rows are consumed: hand the stage back before the per-row tail
            __syncwarp();
            if (lane == 0) mbar_arrive(&cempty[cs]);
#pragma unroll
            for (int blk = 0; blk < MAXBLK; ++blk) {
                if (blk < nblk) {
                    const int r = blk * 32 + pg * C::RPP + rsub;
                    const int j = c * p.rows + r;
                    float Y = Yb[blk], Z = Zb[blk];
                    float Y1 = 0.f, Z1 = 0.f, Y2 = 0.f, Z2 = 0.f, Y3 = 0.f, Z3 = 0.f;
                    int f = 0;
                    for (; f + 4 <= cpr; f += 4) {
                        const float w0 = rec[f * rec_floats + 4 + j], w1 = rec[(f + 1) * rec_floats + 4 + j];
                        const float w2 = rec[(f + 2) * rec_floats + 4 + j], w3 = rec[(f + 3) * rec_floats + 4 + j];
                        Y = fmaf(ckk[f], w0, Y), Z = fmaf(ckq[f], w0, Z);
                        Y1 = fmaf(ckk[f + 1], w1, Y1), Z1 = fmaf(ckq[f + 1], w1, Z1);
                        Y2 = fmaf(ckk[f + 2], w2, Y2), Z2 = fmaf(ckq[f + 2], w2, Z2);
                        Y3 = fmaf(ckk[f + 3], w3, Y3), Z3 = fmaf(ckq[f + 3], w3, Z3);
                    }
                    for (; f < cpr; ++f) {
                        const float wf = rec[f * rec_floats + 4 + j];
                        Y = fmaf(ckk[f], wf, Y), Z = fmaf(ckq[f], wf, Z);
                    }
                    Y += (Y1 + Y2) + Y3;
                    Z += (Z1 + Z2) + Z3;
                    const float vj = load_elem(head + p.off_wv, j, p.in_dtype);
                    const float ww = be * (vj - al * Y);
                    store_elem(p.out, ((int64_t)b * p.Hv + h) * p.dv + j, p.out_dtype, fmaf(cdiag, ww, Z));
                    p.ring_rec[(unit_ring + pos0 % L) * rec_floats + 4 + j] = ww;
                }
            }
        } else {
            const int passes = p.rows / C::RPP;
            for (int ps = 0; ps < passes; ++ps) {
                const int r = ps * C::RPP + rsub;
                const int j = c * p.rows + r;
                float s[C::E];
                load_row(r, s);
                if (T > 0) {
                    float y[TMAX], z[TMAX];
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        float dy = 0.f, dz = 0.f;
                        if (C::KW_REG) {
#pragma unroll
                            for (int e = 0; e < C::E; ++e)
                                dy = fmaf(s[e], kw[C::KW_REG ? t : 0][e], dy), dz = fmaf(s[e], qw[C::KW_REG ? t : 0][e], dz);
                        } else if (t < T) {
#pragma unroll
                            for (int cc = 0; cc < C::NC; ++cc) {
#pragma unroll
                                for (int u = 0; u < C::VEC; u += 4) {
                                    const float4 vk = win(kwp, t, cc, u), vq = win(qwp, t, cc, u);
                                    const int e0 = cc * C::VEC + u;
                                    dy = fmaf(s[e0], vk.x, dy), dy = fmaf(s[e0 + 1], vk.y, dy);
                                    dy = fmaf(s[e0 + 2], vk.z, dy), dy = fmaf(s[e0 + 3], vk.w, dy);
                                    dz = fmaf(s[e0], vq.x, dz), dz = fmaf(s[e0 + 1], vq.y, dz);
                                    dz = fmaf(s[e0 + 2], vq.z, dz), dz = fmaf(s[e0 + 3], vq.w, dz);
                                }
                            }
                        }
                        y[t] = t < T ? G1[t] * dy : 0.f;
                        z[t] = t < T ? G2[t] * dz : 0.f;
                    }
                    for (int f = pg; f < cpr; f += C::LPR) {
                        const float wf = rec[f * rec_floats + 4 + j];
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) {
                            if (t < T) {
                                y[t] = fmaf(ckk[t * LT + f], wf, y[t]);
                                z[t] = fmaf(ckq[t * LT + f], wf, z[t]);
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        y[t] = group_sum<C::LPR>(y[t]);
                        z[t] = group_sum<C::LPR>(z[t]);
                    }
                    float ww[TMAX];
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        if (t < T) {
                            float sk = y[t];
#pragma unroll
                            for (int x = 0; x < t; ++x) sk = fmaf(ckk[t * LT + cpr + x], ww[x], sk);
                            const float vj = load_elem(head + p.off_wv + t * p.dv * in_sz, j, p.in_dtype);
                            ww[t] = meta->beta[t] * (vj - meta->alpha[t] * sk);
                            float o = z[t];
#pragma unroll
                            for (int x = 0; x <= t; ++x) o = fmaf(ckq[t * LT + cpr + x], ww[x], o);
                            if (pg == 0) {
                                store_elem(p.out, (((int64_t)b * T + t) * p.Hv + h) * p.dv + j, p.out_dtype, o);
                                p.ring_rec[(unit_ring + (pos0 + t) % L) * rec_floats + 4 + j] = ww[t];
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            if (!(T > 0 && C::FAST)) mbar_arrive(&cempty[cs]);
            mbar_arrive(&sempty[ss]);
            mbar_arrive(&hempty[hs]);
        }
    }
    if (!ok && lane == 0) set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
}

}  // namespace gdn
