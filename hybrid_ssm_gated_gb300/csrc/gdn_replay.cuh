// gdn_replay.cuh -- ReplaySSM for the gated delta rule: standard decode step,
// speculative verify window, fold (flush) and rollback.
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
// Kernel shape: like the decode kernel -- persistent CTAs over (sequence,
// value head) units, a producer warp streaming the unit's ring entries,
// window rows and S0 chunks with bulk copies, NCW consumer warps. Per unit
// the consumers (1) normalise the ring and window keys/queries into a shared
// FP32 table, (2) build the per-unit coefficient tables (dot products times
// decay products), (3) stream the S0 rows: fold if required, then the window
// dot products, the w recursion and the outputs.
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
    int rows, nchunk, nstage;
    float q_scale;
    // shared-memory layout, bytes
    int head_bytes, off_wq, off_wk, off_wv, off_rk, off_rec;  // inside a head stage
    int heads_off, scratch_off, scratch_bytes, bars_off;      // inside the CTA's buffer
    int off_khat, off_qhat, off_coef;                         // inside a scratch buffer
};

constexpr int REPLAY_NH = 2;      // head stages
constexpr int REPLAY_META = 128;  // bytes of per-unit metadata at the start of a head stage

template <typename ST, int DK, int TMAX, int NCW>
struct ReplayCfg {
    static constexpr int VEC = Store<ST>::VEC;
    static constexpr int E = TMAX <= 2 ? 16 : 8;  // state elements per lane per row
    static constexpr int NC = E / VEC;
    static constexpr int LPR = DK / E;
    static constexpr int RPP = 32 / LPR;  // rows per warp pass == lane groups per warp
    static constexpr int ROW_BYTES = DK * (int)sizeof(ST);
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int NBARS = 2 * REPLAY_NH + 2;  // hfull/hempty per head stage, 2 consumer syncs
    static_assert(E % VEC == 0 && DK % E == 0 && LPR <= 32, "unsupported dk");
};

// Per-unit metadata written by the producer at the start of a head stage.
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

template <typename ST, int DK, int TMAX, int NCW>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) replay_kernel(const ReplayArgs p) {
    using C = ReplayCfg<ST, DK, TMAX, NCW>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* chunks = smem;
    unsigned char* heads = smem + p.heads_off;
    uint64_t* cfull = reinterpret_cast<uint64_t*>(smem + p.bars_off);
    uint64_t* cempty = cfull + p.nstage;
    uint64_t* hfull = cempty + p.nstage;
    uint64_t* hempty = hfull + REPLAY_NH;
    uint64_t* csync = hempty + REPLAY_NH;  // two consumer-wide barriers

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NS = p.nstage;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&cfull[s], 1), mbar_init(&cempty[s], NCW);
        for (int s = 0; s < REPLAY_NH; ++s) mbar_init(&hfull[s], 1), mbar_init(&hempty[s], NCW);
        mbar_init(&csync[0], NCW * 32);
        mbar_init(&csync[1], NCW * 32);
        fence_barrier_init();
    }
    __syncthreads();

    const int total = p.B * p.Hv;
    const int in_sz = dtype_size(p.in_dtype);
    const int group = p.Hv / p.Hk;
    const int T = p.T, L = p.L;
    const int rec_floats = 4 + p.dv;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        const uint64_t pol = policy_evict_first();
        const uint32_t qbytes = DK * in_sz, vbytes = p.dv * in_sz, recbytes = rec_floats * 4;
        const uint32_t cbytes = p.rows * C::ROW_BYTES;
        uint32_t m = 0, nh = 0;
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
                if (lane == 0) {
                    const int hs = n % REPLAY_NH;
                    if (n >= REPLAY_NH) ok = mbar_wait(&hempty[hs], ((n / REPLAY_NH) + 1) & 1);
                    if (ok) {
                        unsigned char* head = heads + hs * p.head_bytes;
                        ReplayMeta* meta = reinterpret_cast<ReplayMeta*>(head);
                        meta->slot = s_i, meta->count = c_i, meta->fold = f_i, meta->pos0 = p_i, meta->ckpt0 = k_i;
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) meta->alpha[t] = al_i[t], meta->beta[t] = be_i[t];
                        if (s_i >= 0) {
                            const int b = unit / p.Hv, h = unit - b * p.Hv, kh = h / group;
                            const int64_t unit_ring = ((int64_t)s_i * p.Hv + h) * L;
                            const int rbase = k_i % L;
                            const int n1 = min(c_i, L - rbase);
                            mbar_arrive_expect_tx(&hfull[hs], T * (2 * qbytes + vbytes) + c_i * (qbytes + recbytes));
                            for (int t = 0; t < T; ++t) {
                                const int64_t qrow = ((int64_t)b * T + t) * p.Hk + kh;
                                const int64_t vrow = ((int64_t)b * T + t) * p.Hv + h;
                                bulk_load(head + p.off_wq + t * qbytes, static_cast<const char*>(p.q) + qrow * qbytes,
                                          qbytes, &hfull[hs]);
                                bulk_load(head + p.off_wk + t * qbytes, static_cast<const char*>(p.k) + qrow * qbytes,
                                          qbytes, &hfull[hs]);
                                bulk_load(head + p.off_wv + t * vbytes, static_cast<const char*>(p.v) + vrow * vbytes,
                                          vbytes, &hfull[hs]);
                            }
                            if (n1 > 0) {
                                bulk_load(head + p.off_rk, static_cast<const char*>(p.ring_k) + (unit_ring + rbase) * qbytes,
                                          n1 * qbytes, &hfull[hs]);
                                bulk_load(head + p.off_rec, p.ring_rec + (unit_ring + rbase) * rec_floats, n1 * recbytes,
                                          &hfull[hs]);
                            }
                            if (c_i > n1) {
                                bulk_load(head + p.off_rk + n1 * qbytes, static_cast<const char*>(p.ring_k) + unit_ring * qbytes,
                                          (c_i - n1) * qbytes, &hfull[hs]);
                                bulk_load(head + p.off_rec + n1 * recbytes, p.ring_rec + unit_ring * rec_floats,
                                          (c_i - n1) * recbytes, &hfull[hs]);
                            }
                            const char* src = static_cast<const char*>(p.ckpt) + ((int64_t)s_i * p.Hv + h) * p.dv * C::ROW_BYTES;
                            for (int c = 0; c < p.nchunk; ++c, ++m) {
                                const int cs = m % NS;
                                if (m >= (uint32_t)NS && !(ok = mbar_wait(&cempty[cs], ((m / NS) + 1) & 1))) break;
                                mbar_arrive_expect_tx(&cfull[cs], cbytes);
                                bulk_load_hint(chunks + cs * CHUNK_BYTES, src + (int64_t)c * cbytes, cbytes, &cfull[cs], pol);
                            }
                        } else {
                            mbar_arrive(&hfull[hs]);
                        }
                        ++nh;
                    }
                }
                ok = __shfl_sync(FULL_MASK, ok, 0);
                if (!ok) break;
            }
        }
        if (!ok && lane == 0) {
            set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
            for (uint32_t s = 0; s < (uint32_t)NS && s < m; ++s) mbar_wait(&cfull[s], ((m - 1 - s) / NS) & 1);
            for (uint32_t s = 0; s < REPLAY_NH && s < nh; ++s) mbar_wait(&hfull[s], ((nh - 1 - s) / REPLAY_NH) & 1);
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int pg = lane % C::LPR;
    const int rsub = lane / C::LPR;
    const int passes = p.rows / C::RPP;
    const int LT = L + TMAX;  // row stride of the coefficient tables
    uint32_t m = 0, nsync = 0;
    bool ok = true;

    // consumer-wide barrier on an mbarrier (bounded wait)
    auto consumer_sync = [&](int which) {
        mbar_arrive(&csync[which]);
        ok = mbar_wait(&csync[which], (nsync >> 1) & 1) && ok;
        ++nsync;
    };

    for (int n = 0; ok; ++n) {
        const int unit = blockIdx.x + n * gridDim.x;
        if (unit >= total) break;
        const int hs = n % REPLAY_NH;
        if (!mbar_wait(&hfull[hs], (n / REPLAY_NH) & 1)) {
            ok = false;
            break;
        }
        const unsigned char* head = heads + hs * p.head_bytes;
        const ReplayMeta* meta = reinterpret_cast<const ReplayMeta*>(head);
        const int slot = meta->slot;
        const int b = unit / p.Hv, h = unit - b * p.Hv;
        if (slot < 0) {
            if (slot == -1 && T > 0) {
                for (int x = cw * 32 + lane; x < T * p.dv; x += NCW * 32) {
                    const int t = x / p.dv, j = x - t * p.dv;
                    store_elem(p.out, (((int64_t)b * T + t) * p.Hv + h) * p.dv + j, p.out_dtype, 0.f);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&hempty[hs]);
            continue;
        }
        const int count = meta->count, fold = meta->fold, pos0 = meta->pos0;
        const int cpr = fold ? 0 : count;  // entries left in front of the window
        const int64_t unit_ring = ((int64_t)slot * p.Hv + h) * L;
        const unsigned char* rk = head + p.off_rk;
        const float* rec = reinterpret_cast<const float*>(head + p.off_rec);
        unsigned char* scratch = smem + p.scratch_off + (n & 1) * p.scratch_bytes;
        float* khat = reinterpret_cast<float*>(scratch + p.off_khat);  // [L + TMAX][DK]: ring keys, window keys at L..
        float* qhat = reinterpret_cast<float*>(scratch + p.off_qhat);  // [TMAX][DK]
        float* coef = reinterpret_cast<float*>(scratch + p.off_coef);
        float* ckk = coef;                      // [TMAX][LT]
        float* ckq = coef + TMAX * LT;          // [TMAX][LT]
        float* G1 = coef + 2 * TMAX * LT;       // [TMAX]
        float* G2 = G1 + TMAX;                  // [TMAX]
        float* Gf = G2 + TMAX;                  // [1]
        float* cf = Gf + 1;                     // [L]

        // ---- phase A: normalise ring keys, window keys and queries.
        // Loops are warp-uniform (each warp takes RPP consecutive tasks per
        // round, one per lane group) because group_sum shuffles the full warp.
        const int nvec = count + 2 * T;
        for (int t0 = cw * C::RPP; t0 < nvec; t0 += NCW * C::RPP) {
            const int t = min(t0 + rsub, nvec - 1);
            const unsigned char* raw;
            float* dst;
            float scale = 1.f;
            if (t < count) {
                raw = rk + t * DK * in_sz, dst = khat + t * DK;
            } else if (t < count + T) {
                raw = head + p.off_wk + (t - count) * DK * in_sz, dst = khat + (L + t - count) * DK;
            } else {
                raw = head + p.off_wq + (t - count - T) * DK * in_sz, dst = qhat + (t - count - T) * DK;
                scale = p.q_scale;
            }
            float x[C::E];
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < C::NC; ++c) load_run<C::VEC>(raw, (c * C::LPR + pg) * C::VEC, p.in_dtype, x + c * C::VEC);
#pragma unroll
            for (int e = 0; e < C::E; ++e) ss = fmaf(x[e], x[e], ss);
            ss = group_sum<C::LPR>(ss);
            const float inv = rsqrtf(ss + 1e-6f) * scale;
            if (t0 + rsub < nvec) {
#pragma unroll
                for (int c = 0; c < C::NC; ++c) {
#pragma unroll
                    for (int u = 0; u < C::VEC; u += 4) {
                        const int e0 = c * C::VEC + u;
                        *reinterpret_cast<float4*>(dst + (c * C::LPR + pg) * C::VEC + u) =
                            make_float4(x[e0] * inv, x[e0 + 1] * inv, x[e0 + 2] * inv, x[e0 + 3] * inv);
                    }
                }
            }
        }
        if (cw == 0) {
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
        consumer_sync(0);
        if (!ok) break;

        // ---- phase B: coefficient tables
        // entry e (post-fold numbering): e < cpr ring entry e; e >= cpr window token e - cpr
        auto alpha_of = [&](int e) -> float { return e < cpr ? rec[e * rec_floats] : meta->alpha[e - cpr]; };
        auto krow = [&](int e) -> const float* { return khat + (e < cpr ? e : L + e - cpr) * DK; };
        {
            // task x enumerates, window token by window token, the e key-key
            // and e + 1 key-query dot products of token t (e = cpr + t)
            int ntasks = 0;
            for (int t = 0; t < T; ++t) ntasks += 2 * (cpr + t) + 1;
            for (int x0 = cw * C::RPP; x0 < ntasks; x0 += NCW * C::RPP) {
                int x = min(x0 + rsub, ntasks - 1), t = 0;
                while (x >= 2 * (cpr + t) + 1) x -= 2 * (cpr + t) + 1, ++t;
                const int e = cpr + t;
                const bool kk = x < e;
                const int f = kk ? x : x - e;
                const float* a_row = krow(f);
                const float* b_row = kk ? krow(e) : qhat + t * DK;
                float d = 0.f;
#pragma unroll
                for (int c = 0; c < C::NC; ++c) {
#pragma unroll
                    for (int u = 0; u < C::VEC; u += 4) {
                        const int off = (c * C::LPR + pg) * C::VEC + u;
                        const float4 va = *reinterpret_cast<const float4*>(a_row + off);
                        const float4 vb = *reinterpret_cast<const float4*>(b_row + off);
                        d = fmaf(va.x, vb.x, d), d = fmaf(va.y, vb.y, d);
                        d = fmaf(va.z, vb.z, d), d = fmaf(va.w, vb.w, d);
                    }
                }
                d = group_sum<C::LPR>(d);
                const int last = kk ? e - 1 : e;
                float decay = 1.f;
                for (int g = f + 1; g <= last; ++g) decay *= alpha_of(g);
                if (pg == 0 && x0 + rsub < ntasks) (kk ? ckk : ckq)[t * LT + f] = d * decay;
            }
        }
        if (cw == 0) {
            if (lane < T) {
                const int e = cpr + lane;
                float g = 1.f;
                for (int x = 0; x < e; ++x) g *= alpha_of(x);
                G1[lane] = g;
                G2[lane] = g * alpha_of(e);
            }
            if (fold) {  // fold coefficients over the pre-fold ring entries 0..count-1
                for (int f = lane; f < count; f += 32) {
                    float g = 1.f;
                    for (int x = f + 1; x < count; ++x) g *= rec[x * rec_floats];
                    cf[f] = g;
                }
                if (lane == 0) {
                    float g = 1.f;
                    for (int x = 0; x < count; ++x) g *= rec[x * rec_floats];
                    Gf[0] = g;
                }
            }
        }
        consumer_sync(1);
        if (!ok) break;

        // ---- phase C: stream S0 rows
        float kw[TMAX][C::E], qw[TMAX][C::E];
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
#pragma unroll
            for (int c = 0; c < C::NC; ++c) {
#pragma unroll
                for (int u = 0; u < C::VEC; u += 4) {
                    const int off = (c * C::LPR + pg) * C::VEC + u;
                    float4 vk = make_float4(0.f, 0.f, 0.f, 0.f), vq = vk;
                    if (t < T) {
                        vk = *reinterpret_cast<const float4*>(khat + (L + t) * DK + off);
                        vq = *reinterpret_cast<const float4*>(qhat + t * DK + off);
                    }
                    const int e0 = c * C::VEC + u;
                    kw[t][e0] = vk.x, kw[t][e0 + 1] = vk.y, kw[t][e0 + 2] = vk.z, kw[t][e0 + 3] = vk.w;
                    qw[t][e0] = vq.x, qw[t][e0 + 1] = vq.y, qw[t][e0 + 2] = vq.z, qw[t][e0 + 3] = vq.w;
                }
            }
        }
        const float gfold = fold ? Gf[0] : 1.f;
        char* gck = static_cast<char*>(p.ckpt) + ((int64_t)slot * p.Hv + h) * p.dv * C::ROW_BYTES;
        for (int c = 0; c < p.nchunk; ++c, ++m) {
            const int cs = m % NS;
            if (!mbar_wait(&cfull[cs], (m / NS) & 1)) {
                ok = false;
                break;
            }
            const unsigned char* tile = chunks + cs * CHUNK_BYTES;
            for (int ps = cw; ps < passes; ps += NCW) {
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
#pragma unroll
                        for (int e = 0; e < C::E; ++e) dy = fmaf(s[e], kw[t][e], dy), dz = fmaf(s[e], qw[t][e], dz);
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
                    float ww[TMAX];
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        y[t] = group_sum<C::LPR>(y[t]);
                        z[t] = group_sum<C::LPR>(z[t]);
                    }
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&hempty[hs]);
    }
    if (!ok && lane == 0) set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
}

}  // namespace gdn
