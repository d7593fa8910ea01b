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
// The ring keeps w_f (fp32) beside each entry's raw inputs, so one pass over
// S0 -- two dot products per state element per window token -- and O(count)
// vector work give every output; S_t itself is only materialised (in FP32
// registers) when the ring is folded: S0 <- round(G S0 + sum A k w^T).
//
// Kernel shape: persistent CTAs over (sequence, value head) units with four
// warp roles, so the per-unit scalar work never stalls the state stream:
//   warp 0       head producer: per-unit metadata (slot, pointers, gates)
//                for 32 units at a time, then bulk copies (TMA engine) of the
//                unit's window rows and buffered ring entries into a head ring;
//   warp 1       chunk producer: streams S0 in 16 KB chunks into a chunk ring;
//   NPW warps    prep: one warp prepares one whole unit -- normalised window
//                keys/queries, key-key / key-query dot products times decay
//                products (the coefficients above), fold coefficients -- into
//                a scratch slot, appends the window to the ring and moves the
//                pointers;
//   NRW warps    rows: stream S0 rows from the chunk ring, fold if required,
//                two dot products per element per window token, the w
//                recursion, and the outputs.
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
    int off_kw, off_qw, off_khat, off_coef;                   // inside a scratch slot
};

constexpr int REPLAY_META = 128;  // bytes of per-unit metadata at the start of a head stage

template <typename ST, int DK, int TMAX, int NPW, int NRW>
struct ReplayCfg {
    static constexpr int VEC = Store<ST>::VEC;
    static constexpr int E = TMAX <= 2 ? 16 : 8;  // state elements per lane per row
    static constexpr int NC = E / VEC;
    static constexpr int LPR = DK / E;
    static constexpr int RPP = 32 / LPR;  // rows per warp pass
    static constexpr int ROW_BYTES = DK * (int)sizeof(ST);
    static constexpr int PE = DK / 32;  // elements per lane when one warp handles a vector
    static constexpr int THREADS = (2 + NPW + NRW) * 32;
    static constexpr bool KW_REG = TMAX <= 4;  // window vectors held in registers by the row warps
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
    uint64_t* sfull = hempty + NH;
    uint64_t* sempty = sfull + NSC;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&cfull[s], 1), mbar_init(&cempty[s], NRW);
        for (int s = 0; s < NH; ++s) mbar_init(&hfull[s], 1), mbar_init(&hempty[s], NRW + 1);
        for (int s = 0; s < NSC; ++s) mbar_init(&sfull[s], 1), mbar_init(&sempty[s], NRW);
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
            if (!(ok = __all_sync(FULL_MASK, mbar_wait(&hfull[hs], (n / NH) & 1)))) break;
            const int slot = reinterpret_cast<const ReplayMeta*>(heads + hs * p.head_bytes)->slot;
            if (slot < 0) continue;
            const int h = unit % p.Hv;
            if (lane < p.nchunk) {
                const uint32_t mc = m + lane;
                const int cs = mc % NS;
                ok = mc < (uint32_t)NS || mbar_wait(&cempty[cs], ((mc / NS) + 1) & 1);
                if (ok) {
                    const char* src = static_cast<const char*>(p.ckpt) + ((int64_t)slot * p.Hv + h) * p.dv * C::ROW_BYTES +
                                      (int64_t)lane * cbytes;
                    mbar_arrive_expect_tx(&cfull[cs], cbytes);
                    bulk_load_hint(chunks + cs * CHUNK_BYTES, src, cbytes, &cfull[cs], pol);
                }
            }
            ok = __all_sync(FULL_MASK, ok);
            m += p.nchunk;
        }
        if (!ok && lane == 0) {
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
            if (!(ok = mbar_wait(&hfull[hs], (n / NH) & 1))) break;
            if (n >= NSC && !(ok = mbar_wait(&sempty[ss], ((n / NSC) + 1) & 1))) break;
            const unsigned char* head = heads + hs * p.head_bytes;
            const ReplayMeta* meta = reinterpret_cast<const ReplayMeta*>(head);
            const int slot = meta->slot;
            if (slot >= 0) {
                unsigned char* scr = smem + p.scratch_off + ss * p.scratch_bytes;
                float* kw = reinterpret_cast<float*>(scr + p.off_kw);      // [TMAX][DK] window keys
                float* qw = reinterpret_cast<float*>(scr + p.off_qw);      // [TMAX][DK] window queries
                float* khat = reinterpret_cast<float*>(scr + p.off_khat);  // [L][DK] ring keys (fold only)
                float* ckk = reinterpret_cast<float*>(scr + p.off_coef);   // [TMAX][LT]
                float* ckq = ckk + TMAX * LT;                              // [TMAX][LT]
                float* G1 = ckq + TMAX * LT;                               // [TMAX]
                float* G2 = G1 + TMAX;                                     // [TMAX]
                float* Gf = G2 + TMAX;                                     // [1]
                float* cf = Gf + 1;                                        // [L]
                const int count = meta->count, fold = meta->fold, pos0 = meta->pos0;
                const int cpr = fold ? 0 : count;  // ring entries in front of the window
                const float* rec = reinterpret_cast<const float*>(head + p.off_rec);
                const int b = unit / p.Hv, h = unit - b * p.Hv;
                const int64_t unit_ring = ((int64_t)slot * p.Hv + h) * L;

                // window keys and queries, normalised; lane holds elements lane + 32 m
                float kwr[TMAX][C::PE], qwr[TMAX][C::PE];
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                    float ssk = 0.f, ssq = 0.f;
#pragma unroll
                    for (int m = 0; m < C::PE; ++m) {
                        const int i = lane + 32 * m;
                        kwr[t][m] = t < T ? load_elem(head + p.off_wk + t * DK * in_sz, i, p.in_dtype) : 0.f;
                        qwr[t][m] = t < T ? load_elem(head + p.off_wq + t * DK * in_sz, i, p.in_dtype) : 0.f;
                        ssk = fmaf(kwr[t][m], kwr[t][m], ssk);
                        ssq = fmaf(qwr[t][m], qwr[t][m], ssq);
                    }
                    if (t < T) {
                        const float ik = rsqrtf(warp_sum(ssk) + 1e-6f);
                        const float iq = rsqrtf(warp_sum(ssq) + 1e-6f) * p.q_scale;
#pragma unroll
                        for (int m = 0; m < C::PE; ++m) {
                            kwr[t][m] *= ik, qwr[t][m] *= iq;
                            kw[t * DK + lane + 32 * m] = kwr[t][m];
                            qw[t * DK + lane + 32 * m] = qwr[t][m];
                        }
                    }
                }
                // window-window dots (entries cpr + s): k_s.k_t for s < t, k_s.q_t for s <= t
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
#pragma unroll
                    for (int s = 0; s <= t; ++s) {
                        if (t < T) {
                            float dkk = 0.f, dkq = 0.f;
#pragma unroll
                            for (int m = 0; m < C::PE; ++m)
                                dkk = fmaf(kwr[s][m], kwr[t][m], dkk), dkq = fmaf(kwr[s][m], qwr[t][m], dkq);
                            dkk = warp_sum(dkk);
                            dkq = warp_sum(dkq);
                            if (lane == 0) {
                                if (s < t) ckk[t * LT + cpr + s] = dkk;
                                ckq[t * LT + cpr + s] = dkq;
                            }
                        }
                    }
                }
                // buffered ring entries: norms, and dots with the window (or normalised keys for a fold)
                const unsigned char* rk = head + p.off_rk;
                for (int f = 0; f < count; ++f) {
                    float x[C::PE], ss2 = 0.f;
#pragma unroll
                    for (int m = 0; m < C::PE; ++m) {
                        x[m] = load_elem(rk + f * DK * in_sz, lane + 32 * m, p.in_dtype);
                        ss2 = fmaf(x[m], x[m], ss2);
                    }
                    const float ik = rsqrtf(warp_sum(ss2) + 1e-6f);
                    if (fold) {
#pragma unroll
                        for (int m = 0; m < C::PE; ++m) khat[f * DK + lane + 32 * m] = x[m] * ik;
                    } else {
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) {
                            if (t < T) {
                                float dkk = 0.f, dkq = 0.f;
#pragma unroll
                                for (int m = 0; m < C::PE; ++m)
                                    dkk = fmaf(x[m], kwr[t][m], dkk), dkq = fmaf(x[m], qwr[t][m], dkq);
                                dkk = warp_sum(dkk);
                                dkq = warp_sum(dkq);
                                if (lane == 0) ckk[t * LT + f] = dkk * ik, ckq[t * LT + f] = dkq * ik;
                            }
                        }
                    }
                }
                __syncwarp();
                // decay products. Entry e (post-fold numbering): e < cpr ring entry, else window
                // token e - cpr. Item f = -1 gives G(e); f >= 0 scales the dot products by A(f, .).
                const int etot = cpr + T;
                for (int f = lane - 1; f < etot; f += 32) {
                    float prod = 1.f;  // A(f, e - 1) at the top of iteration e
                    for (int e = f + 1; e < etot; ++e) {
                        const int t = e - cpr;
                        if (t >= 0) {
                            if (f >= 0)
                                ckk[t * LT + f] *= prod;
                            else
                                G1[t] = prod;
                        }
                        prod *= e < cpr ? rec[e * rec_floats] : meta->alpha[t];
                        if (t >= 0) {
                            if (f >= 0)
                                ckq[t * LT + f] *= prod;
                            else
                                G2[t] = prod;
                        }
                    }
                }
                if (fold) {  // fold coefficients over the pre-fold ring entries 0..count-1
                    for (int f = lane - 1; f < count; f += 32) {
                        float prod = 1.f;
                        for (int e = f + 1; e < count; ++e) prod *= rec[e * rec_floats];
                        if (f >= 0)
                            cf[f] = prod;
                        else
                            Gf[0] = prod;
                    }
                }
                // append the window's raw inputs and gates to the ring; move the pointers
                const int kvec = DK * in_sz / 16, vvec = p.dv * in_sz / 16;
                for (int t = 0; t < T; ++t) {
                    const int64_t ent = unit_ring + (pos0 + t) % L;
                    for (int x = lane; x < kvec; x += 32)
                        reinterpret_cast<uint4*>(static_cast<char*>(p.ring_k) + ent * DK * in_sz)[x] =
                            reinterpret_cast<const uint4*>(head + p.off_wk + t * DK * in_sz)[x];
                    for (int x = lane; x < vvec; x += 32)
                        reinterpret_cast<uint4*>(static_cast<char*>(p.ring_v) + ent * p.dv * in_sz)[x] =
                            reinterpret_cast<const uint4*>(head + p.off_wv + t * p.dv * in_sz)[x];
                    if (lane == 0)
                        *reinterpret_cast<float4*>(p.ring_rec + ent * rec_floats) =
                            make_float4(meta->alpha[t], meta->beta[t], 0.f, 0.f);
                }
                if (lane == 0) {
                    const int64_t idx = (int64_t)slot * p.Hv + h;
                    p.pos[idx] = pos0 + T;
                    if (fold) p.ckpt_pos[idx] = pos0;
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sfull[ss]);
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
    const int passes = p.rows / C::RPP;
    uint32_t m = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
        const int unit = blockIdx.x + n * gridDim.x;
        if (unit >= total) break;
        const int hs = n % NH, ss = n % NSC;
        if (!(ok = mbar_wait(&sfull[ss], (n / NSC) & 1) && mbar_wait(&hfull[hs], (n / NH) & 1))) break;
        const unsigned char* head = heads + hs * p.head_bytes;
        const ReplayMeta* meta = reinterpret_cast<const ReplayMeta*>(head);
        const int slot = meta->slot;
        const int b = unit / p.Hv, h = unit - b * p.Hv;
        if (slot >= 0) {
            const int count = meta->count, fold = meta->fold, pos0 = meta->pos0;
            const int cpr = fold ? 0 : count;
            const int64_t unit_ring = ((int64_t)slot * p.Hv + h) * L;
            const float* rec = reinterpret_cast<const float*>(head + p.off_rec);
            const unsigned char* scr = smem + p.scratch_off + ss * p.scratch_bytes;
            const float* kwp = reinterpret_cast<const float*>(scr + p.off_kw);
            const float* qwp = reinterpret_cast<const float*>(scr + p.off_qw);
            const float* khat = reinterpret_cast<const float*>(scr + p.off_khat);
            const float* ckk = reinterpret_cast<const float*>(scr + p.off_coef);
            const float* ckq = ckk + TMAX * LT;
            const float* G1 = ckq + TMAX * LT;
            const float* G2 = G1 + TMAX;
            const float gfold = fold ? G2[TMAX] : 1.f;  // Gf follows G2
            const float* cf = G2 + TMAX + 1;

            // window vectors at this lane's key positions
            auto win = [&](const float* base, int t, int c, int u) -> float4 {
                return *reinterpret_cast<const float4*>(base + t * DK + (c * C::LPR + pg) * C::VEC + u);
            };
            constexpr int KWN = C::KW_REG ? TMAX : 1;
            float kw[KWN][C::E], qw[KWN][C::E];
            if (C::KW_REG) {
#pragma unroll
                for (int t = 0; t < KWN; ++t) {
#pragma unroll
                    for (int c = 0; c < C::NC; ++c) {
#pragma unroll
                        for (int u = 0; u < C::VEC; u += 4) {
                            float4 vk = make_float4(0.f, 0.f, 0.f, 0.f), vq = vk;
                            if (t < T) vk = win(kwp, t, c, u), vq = win(qwp, t, c, u);
                            const int e0 = c * C::VEC + u;
                            kw[t][e0] = vk.x, kw[t][e0 + 1] = vk.y, kw[t][e0 + 2] = vk.z, kw[t][e0 + 3] = vk.w;
                            qw[t][e0] = vq.x, qw[t][e0 + 1] = vq.y, qw[t][e0 + 2] = vq.z, qw[t][e0 + 3] = vq.w;
                        }
                    }
                }
            }
            char* gck = static_cast<char*>(p.ckpt) + ((int64_t)slot * p.Hv + h) * p.dv * C::ROW_BYTES;
            for (int c = 0; c < p.nchunk; ++c, ++m) {
                const int cs = m % NS;
                if (!(ok = mbar_wait(&cfull[cs], (m / NS) & 1))) break;
                const unsigned char* tile = chunks + cs * CHUNK_BYTES;
                // passes of the unit spread over the row warps across chunks
                for (int ps = ((rw - c * passes) % NRW + NRW) % NRW; ps < passes; ps += NRW) {
                    const int r = ps * C::RPP + rsub;
                    const int j = c * p.rows + r;
                    float s[C::E];
#pragma unroll
                    for (int cc = 0; cc < C::NC; ++cc) {
                        const uint4 raw =
                            *reinterpret_cast<const uint4*>(tile + r * C::ROW_BYTES + (cc * C::LPR + pg) * 16);
                        Store<ST>::unpack(raw, s + cc * C::VEC);
                    }
                    if (fold) {
                        // S0 <- round(G S0 + sum_f A(f, count-1) k_f w_f^T), row j
#pragma unroll
                        for (int e = 0; e < C::E; ++e) s[e] *= gfold;
                        for (int f = 0; f < count; ++f) {
                            const float cwf = cf[f] * rec[f * rec_floats + 4 + j];
                            const float* kf = khat + f * DK;
#pragma unroll
                            for (int cc = 0; cc < C::NC; ++cc) {
#pragma unroll
                                for (int u = 0; u < C::VEC; u += 4) {
                                    const float4 kv =
                                        *reinterpret_cast<const float4*>(kf + (cc * C::LPR + pg) * C::VEC + u);
                                    const int e0 = cc * C::VEC + u;
                                    s[e0] = fmaf(kv.x, cwf, s[e0]), s[e0 + 1] = fmaf(kv.y, cwf, s[e0 + 1]);
                                    s[e0 + 2] = fmaf(kv.z, cwf, s[e0 + 2]), s[e0 + 3] = fmaf(kv.w, cwf, s[e0 + 3]);
                                }
                            }
                        }
                        char* dst = gck + (int64_t)j * C::ROW_BYTES;
#pragma unroll
                        for (int cc = 0; cc < C::NC; ++cc) {
                            const uint4 packed = Store<ST>::pack(s + cc * C::VEC);
                            *reinterpret_cast<uint4*>(dst + (cc * C::LPR + pg) * 16) = packed;
                            Store<ST>::unpack(packed, s + cc * C::VEC);  // continue from the stored values
                        }
                    }
                    if (T > 0) {
                        float y[TMAX], z[TMAX];
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) {
                            float dy = 0.f, dz = 0.f;
                            if (C::KW_REG) {
#pragma unroll
                                for (int e = 0; e < C::E; ++e)
                                    dy = fmaf(s[e], kw[C::KW_REG ? t : 0][e], dy),
                                    dz = fmaf(s[e], qw[C::KW_REG ? t : 0][e], dz);
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
                __syncwarp();
                if (lane == 0) mbar_arrive(&cempty[cs]);
            }
            if (!ok) break;
        } else if (slot == -1 && T > 0) {
            for (int x = rw * 32 + lane; x < T * p.dv; x += NRW * 32) {
                const int t = x / p.dv, j = x - t * p.dv;
                store_elem(p.out, (((int64_t)b * T + t) * p.Hv + h) * p.dv + j, p.out_dtype, 0.f);
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&sempty[ss]);
            mbar_arrive(&hempty[hs]);
        }
    }
    if (!ok && lane == 0) set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
}

}  // namespace gdn
