// gdn_replay_warp.cuh -- ReplaySSM with two checkpoints, one warp per
// (sequence, value head) unit: the standard decode step, the speculative
// verify window and the fold (flush).
//
// The mode and its arithmetic are in gdn_replay_common.cuh. This kernel serves
// the two-checkpoint mode where the producer kernel's layout (gdn_replay_producer.cuh)
// does not fit: long rings with wide heads.
//
// Kernel shape. Persistent CTAs of NW warps; the units c, c + grid, ... of CTA
// c are taken by its warps one at a time from a shared-memory counter, so a
// warp that meets a fold unit (several times the work of another) does not
// hold the CTA back. A warp runs its unit alone, with no barrier, producer or
// hand-off:
//  - lane t < T computes token t's gates; every lane loads its E positions of
//    the window's keys and queries and normalises them (a sum over the G lanes
//    of a row);
//  - the coefficients of the w terms, decays included, are dot products
//    of the buffered keys with the window's keys and queries: one entry per
//    G-lane row group, written to a per-warp table in shared memory;
//  - S0 streams through registers in batches of 32 rows with coalesced
//    16-byte loads, G lanes a row, E elements a lane (E = 16, 8, 4 for
//    windows of 1, <= 4, <= 8 tokens, so that the window's keys and queries
//    stay in registers). The 2T partial dot products of NSB rows are
//    reduce-scattered over the row's lanes into a per-warp tile of row sums;
//    then lane l finishes row l of the batch: the ring terms, the window's own
//    recursion, the outputs and the new w, all coalesced across the warp;
//  - a fold unit folds each row as it is loaded, stores it rounded, and goes on
//    from the stored value; the window is appended to the ring at the end.
// Two checkpoints (same article, its paragraph on precision): with a wider
// master type MT, a unit that does not fold reads the read copy (ST); one that
// folds reads the master, runs every buffered entry's raw inputs through the
// rule on it in FP32 (each row's prediction a dot product within the row),
// stores it and the copy rounded from it, and goes on from the copy's values.
// The kernel also takes the Mamba2 rule (RULE_MAMBA2: B, C and x for the key,
// query and value, no normalisation, no prediction, plus D x), for which the
// ABI offers no read copy.
#pragma once

#include <type_traits>

#include "gdn_replay_common.cuh"

namespace gdn {

// N consecutive state elements of type T at element `first` of a row, loaded
// through the streaming (evict-first) path: read once per call. 16-bit types
// take N = 4 (8 bytes) or a multiple of 8 (16-byte vectors); fp32 a multiple
// of 4.
template <typename T, int N>
__device__ __forceinline__ void ld_state(const unsigned char* row, int first, float* x) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int e = 0; e < N; e += 4) {
            const float4 f = __ldcs(reinterpret_cast<const float4*>(row + (first + e) * 4));
            x[e] = f.x, x[e + 1] = f.y, x[e + 2] = f.z, x[e + 3] = f.w;
        }
    } else if constexpr (N == 4) {
        const uint2 r = __ldcs(reinterpret_cast<const uint2*>(row + first * 2));
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            x[0] = bf16_lo(r.x), x[1] = bf16_hi(r.x), x[2] = bf16_lo(r.y), x[3] = bf16_hi(r.y);
        } else {
            float2 f = f16x2_to_f2(r.x);
            x[0] = f.x, x[1] = f.y;
            f = f16x2_to_f2(r.y);
            x[2] = f.x, x[3] = f.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < N; e += 8)
            Store<T>::unpack(__ldcs(reinterpret_cast<const uint4*>(row + (first + e) * 2)), x + e);
    }
}

template <typename ST, typename MT, int DK, int TMAX, int RULE>
struct WarpCfg {
    static constexpr int E = TMAX == 1 ? 16 : (TMAX <= 4 ? 8 : 4);  // state elements per lane per row
    static constexpr int G = DK / E;                                 // lanes per row
    static constexpr int RPS = 32 / G;                               // rows per warp-wide set
    static constexpr int NSET = G;                                   // sets per batch of 32 rows
    static constexpr int VEC = 16 / (int)sizeof(ST) < E ? 16 / (int)sizeof(ST) : E;  // elements per vector
    static constexpr int NVEC = E / VEC;                             // vectors per lane per row
    static constexpr int NK = RULE == RULE_GDN ? 2 : 1;              // dot products per window token
    static constexpr int VPR = NK * TMAX;                            // row sums per row
    // sets per sub-batch: the unit of the copy pipeline and of one reduce-scatter; enough for every
    // lane to end with a sum where that takes at most 32 state elements a lane
    static constexpr int NSB_FULL = G > VPR ? G / VPR : 1;
    static constexpr int NSB_CAP = 32 / E > 1 ? 32 / E : 1;
    static constexpr int NSB = NSB_FULL < NSB_CAP ? NSB_FULL : NSB_CAP;
    static constexpr int SPB = NSET / NSB;            // sub-batches per batch of 32 rows
    static constexpr int V = NSB * VPR;               // values per lane in one reduce-scatter
    static constexpr int HELD = V >= G ? V / G : 1;   // sums a lane holds after it
    static constexpr int DUP = V >= G ? 1 : G / V;    // lanes holding the same sum
    static constexpr int TILE = VPR + 1;              // floats per row of the row-sum tile
    static constexpr int CW = 2 * TMAX;               // floats per coefficient-table entry
    // copy pipeline: a stage holds one sub-batch of rows of the wider checkpoint type; NS stages keep
    // about 8 KB a warp in flight, and at most SPB + 1 so that a batch's staged ring columns
    // (double-buffered) are not overwritten before its last sub-batch reads them
    static constexpr int STAGE = NSB * 32 * E * (int)sizeof(MT);
    static constexpr int NS_WANT = 1 + (8192 + STAGE - 1) / STAGE;
    static constexpr int NS_CAP = SPB + 1 < 8 ? SPB + 1 : 8;
    static constexpr int NS = NS_WANT < 2 ? 2 : (NS_WANT > NS_CAP ? NS_CAP : NS_WANT);
    static_assert(DK % E == 0 && G >= 1 && G <= 32 && NSET % NSB == 0 && NS >= 2, "unsupported dk");
};

// One warp's shared memory, 16-byte aligned pieces: the copy stages; the staged ring columns of the
// current batch (w, and for two-checkpoint folds the raw values v; double-buffered by batch); the
// unit's buffered raw keys and record headers {alpha, beta, 1/|k|, n}; the row-sum tile; the
// coefficient table (ring entries, then window tokens).
struct WarpLayout {
    int stage, wcol, vcol, keys, hdr, tile, coef, bytes;
};

template <typename ST, typename MT, int DK, int TMAX, int RULE>
__host__ __device__ constexpr WarpLayout replay_warp_layout(int L, int in_sz) {
    using C = WarpCfg<ST, MT, DK, TMAX, RULE>;
    WarpLayout w{};
    w.stage = 0;
    w.wcol = w.stage + C::NS * C::STAGE;
    w.vcol = w.wcol + 2 * L * 32 * 4;
    w.keys = w.vcol + (std::is_same<ST, MT>::value ? 0 : 2 * L * 32 * 4);
    w.hdr = w.keys + L * DK * in_sz;
    w.tile = w.hdr + L * 16;
    w.coef = w.tile + 32 * C::TILE * 4;
    w.bytes = align_up(w.coef + (L + TMAX) * C::CW * 4, 16);
    return w;
}

// ST: the checkpoint that steps and windows read (the read copy in the two-checkpoint mode);
// MT: the checkpoint that folds read and write (ST itself with one checkpoint).
template <typename ST, int DK, int TMAX, int NW, typename MT = ST, int RULE = RULE_GDN, int IO = IO_ANY>
__global__ void __launch_bounds__(NW * 32, 1) replay_warp_kernel(const ReplayArgs p) {
    using C = WarpCfg<ST, MT, DK, TMAX, RULE>;
    constexpr bool MIXED = !std::is_same<ST, MT>::value;
    constexpr bool GDN = RULE == RULE_GDN;
    constexpr int E = C::E, G = C::G, VEC = C::VEC, NS = C::NS, NSB = C::NSB, SPB = C::SPB;
    constexpr int SROW = DK * (int)sizeof(ST), MROW = DK * (int)sizeof(MT);
    const int in_dt = io_in<IO>(p.in_dtype), out_dt = io_out<IO>(p.out_dtype);
    const int in_sz = dtype_size(in_dt);
    // dynamic shared memory: the unit counter, then one region per warp
    extern __shared__ __align__(128) unsigned char smem[];
    int* ctr = reinterpret_cast<int*>(smem);              // next list index; folds listed; others listed
    int4* lfold = reinterpret_cast<int4*>(smem + 16);     // {unit, slot, pos, ckpt_pos} of the fold units
    int4* lrest = lfold + REPLAY_ROUND;                   // ... and of the others
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane % G;   // lane's place in its row group
    const int rg = lane / G;  // row group within the warp
    const WarpLayout lay = replay_warp_layout<ST, MT, DK, TMAX, RULE>(p.L, in_sz);
    unsigned char* region = smem + REPLAY_SMEM_HEAD + warp * lay.bytes;
    unsigned char* stages = region + lay.stage;
    float* wcol = reinterpret_cast<float*>(region + lay.wcol);        // [2][L][32]: w of the batch's columns
    uint32_t* vcol = reinterpret_cast<uint32_t*>(region + lay.vcol);  // [2][L][32]: 4 bytes of raw v
    unsigned char* keys = region + lay.keys;                          // [L][DK] raw keys, entry order
    const float4* hdr = reinterpret_cast<const float4*>(region + lay.hdr);  // [L] {alpha, beta, 1/|k|, n}
    float* tile = reinterpret_cast<float*>(region + lay.tile);
    float* coef = reinterpret_cast<float*>(region + lay.coef);  // [entry][CW]: S^T k at [t], S^T q at [TMAX + t]

    const int total = p.B * p.Hv;
    const int T = p.T, L = p.L;
    const int group = p.Hv / p.Hk;
    const int rec_floats = 4 + p.dv;
    const int kbytes = DK * in_sz;           // a raw key row
    // array extents in bytes: every copy and store checks against them in bounds-checking builds
    const uint64_t cells = (uint64_t)p.num_slots * p.Hv;
    const uint64_t ext_m = cells * p.dv * MROW, ext_s = cells * p.dv * SROW, ext_rk = cells * p.L * kbytes;
    const uint64_t ext_rv = cells * p.L * p.dv * in_sz, ext_rec = cells * p.L * rec_floats * 4, ext_ptr = cells * 4;
    const uint64_t ext_out = (uint64_t)p.B * p.T * p.Hv * p.dv * dtype_size(out_dt);
    const void* sbase = MIXED ? p.ckpt_copy : p.ckpt;  // the checkpoint steps read
    auto out_ok = [&](int64_t i) { return in_bounds(static_cast<char*>(p.out) + i * dtype_size(out_dt),
                                                    dtype_size(out_dt), p.out, ext_out, p.dev_err); };
    const int Q = p.dv / 32 * SPB;           // sub-batches of a unit
    auto pos_of = [&](int c) { return (c * G + g) * VEC; };  // first element of the lane's c-th vector

    const int per_cta = (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    for (int r0 = 0; r0 < per_cta; r0 += REPLAY_ROUND) {
    const int nr = per_cta - r0 < REPLAY_ROUND ? per_cta - r0 : REPLAY_ROUND;
    replay_list_round(p, T, L, r0, nr, ctr, lfold, lrest);
    const int nf = ctr[1];
    for (;;) {
        int li = 0;
        if (lane == 0) li = atomicAdd(&ctr[0], 1);
        li = __shfl_sync(FULL_MASK, li, 0);
        if (li >= nr) break;
        const int4 ent = li < nf ? lfold[li] : lrest[li - nf];
        const int unit = ent.x, slot = ent.y, pos0 = ent.z, ck0 = ent.w;
        const int b = unit / p.Hv, h = unit - b * p.Hv, kh = h / group;

        // ------------------------------------------------ the window's raw inputs (independent of the slot)
        float kw[TMAX][E], qw[TMAX][E];
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
#pragma unroll
            for (int e = 0; e < E; ++e) kw[t][e] = 0.f, qw[t][e] = 0.f;
            if (t < T) {
                const int64_t qrow = ((int64_t)b * T + t) * p.Hk + kh;
                const unsigned char* kr = static_cast<const unsigned char*>(p.k) + qrow * kbytes;
                const unsigned char* qr = static_cast<const unsigned char*>(p.q) + qrow * kbytes;
#pragma unroll
                for (int c = 0; c < C::NVEC; ++c) {
                    load_run<VEC>(qr, pos_of(c), in_dt, qw[t] + c * VEC);
                    load_run<VEC>(kr, pos_of(c), in_dt, kw[t] + c * VEC);
                }
            }
        }
        float al_l = 1.f, be_l = 0.f;  // lane t < T: token t's gates
        if (lane < T) {
            const int64_t gi = ((int64_t)b * T + lane) * p.Hv + h;
            rule_gates<RULE>(p.A_log[h], p.dt_bias[h], p.a, p.b, gi, in_dt, al_l, be_l);
        }

        // ------------------------------------------------ pointers, fold decision
        int count = 0, fold = 0;
        bool zero = false, skip = false;
        if (slot >= p.num_slots) {
            if (lane == 0) set_error(p.dev_err, GDN_DEVERR_SLOT);
            zero = true;
        } else if (slot < 0) {
            zero = true;
        } else {
            count = pos0 - ck0;
            if (ck0 < 0 || count < 0 || count > L) {
                if (lane == 0) set_error(p.dev_err, GDN_DEVERR_RING);
                zero = true;
            } else if (T > 0) {
                fold = count + T > L;
            } else {
                fold = p.force ? count > 0 : count + 1 > L;
                skip = !fold;
            }
        }
        if (zero || skip) {
            for (int x = lane; zero && x < T * p.dv; x += 32) {
                const int t = x / p.dv, j = x - t * p.dv;
                const int64_t oi = (((int64_t)b * T + t) * p.Hv + h) * p.dv + j;
                if (out_ok(oi)) store_elem(p.out, oi, out_dt, 0.f);
            }
            continue;
        }
        const int cpr = fold ? 0 : count;  // ring entries in front of the window
        const int64_t uidx = (int64_t)slot * p.Hv + h;
        const int64_t unit_ring = uidx * L;
        float* rec = p.ring_rec + unit_ring * rec_floats;
        const int rbase = ck0 % L;
        auto ring_at = [&](int f) { const int r = rbase + f; return r >= L ? r - L : r; };  // ring index of entry f

        // ------------------------------------------------ the copy pipeline over S0
        // Sub-batch q holds rows q * NSB * RPS + u * RPS + rg (u < NSB) -- batch q / SPB of 32 rows. Its
        // stage keeps, per set u, the lane's pieces in the order of its elements, lanes interleaved per
        // piece. The first sub-batch of a batch also stages the batch's 32 columns of every buffered
        // entry's w (or, for a two-checkpoint fold, its raw v); the unit's first also stages the
        // buffered raw keys and record headers. A lane reads back only what it copied, except the
        // staged columns, keys and headers, which are read after a warp barrier.
        const bool fm = MIXED && fold;  // a two-checkpoint fold reads and writes the master
        const unsigned char* s0 = static_cast<const unsigned char*>(MIXED && !fold ? p.ckpt_copy : p.ckpt) +
                                  uidx * p.dv * (fm ? MROW : SROW) + (int64_t)rg * (fm ? MROW : SROW);
        auto issue = [&](int q) {
            if (q < Q) {
                unsigned char* st = stages + (q % NS) * C::STAGE;
                if (fm) {
                    constexpr int PS = VEC * 4 < 16 ? VEC * 4 : 16, PPV = VEC * 4 / PS, NP = C::NVEC * PPV;
                    const unsigned char* src = s0 + (int64_t)q * NSB * C::RPS * MROW;
#pragma unroll
                    for (int u = 0; u < NSB; ++u)
#pragma unroll
                        for (int k = 0; k < NP; ++k) {
                            const unsigned char* g_ = src + u * C::RPS * MROW + pos_of(k / PPV) * 4 + (k % PPV) * PS;
                            if (in_bounds(g_, PS, p.ckpt, ext_m, p.dev_err))
                                cp_async_piece<PS>(st + ((u * NP + k) * 32 + lane) * PS, g_);
                        }
                } else {
                    constexpr int SZ = (int)sizeof(ST);
                    constexpr int PS = VEC * SZ < 16 ? VEC * SZ : 16, PPV = VEC * SZ / PS, NP = C::NVEC * PPV;
                    const unsigned char* src = s0 + (int64_t)q * NSB * C::RPS * SROW;
#pragma unroll
                    for (int u = 0; u < NSB; ++u)
#pragma unroll
                        for (int k = 0; k < NP; ++k) {
                            const unsigned char* g_ = src + u * C::RPS * SROW + pos_of(k / PPV) * SZ + (k % PPV) * PS;
                            if (in_bounds(g_, PS, sbase, ext_s, p.dev_err))
                                cp_async_piece<PS>(st + ((u * NP + k) * 32 + lane) * PS, g_);
                        }
                }
                if (q == 0) {
                    for (int f = lane; f < count; f += 32) {
                        const float* g_ = rec + ring_at(f) * rec_floats;
                        if (in_bounds(g_, 16, p.ring_rec, ext_rec, p.dev_err)) cp_async_piece<16>(region + lay.hdr + f * 16, g_);
                    }
                    const int kp = kbytes / 16;
                    for (int i = lane; i < count * kp; i += 32) {
                        const int f = i / kp, k = i - f * kp;
                        const unsigned char* g_ =
                            static_cast<const unsigned char*>(p.ring_k) + (unit_ring + ring_at(f)) * kbytes + k * 16;
                        if (in_bounds(g_, 16, p.ring_k, ext_rk, p.dev_err)) cp_async_piece<16>(keys + f * kbytes + k * 16, g_);
                    }
                }
                if (q % SPB == 0) {
                    const int bq = q / SPB, buf = bq & 1;
                    const int col = bq * 32 + lane;
                    if (fm) {
                        // 4 bytes holding column col of every entry's raw v (and its pair's, 16-bit)
                        const int pair = in_sz == 4 ? col : (col & ~1);
                        for (int f = 0; f < count; ++f) {
                            const unsigned char* g_ = static_cast<const unsigned char*>(p.ring_v) +
                                                      ((unit_ring + ring_at(f)) * p.dv + pair) * in_sz;
                            if (in_bounds(g_, 4, p.ring_v, ext_rv, p.dev_err))
                                cp_async_piece<4>(vcol + (buf * L + f) * 32 + lane, g_);
                        }
                    } else {
                        for (int f = 0; f < count; ++f) {
                            const float* g_ = rec + ring_at(f) * rec_floats + 4 + col;
                            if (in_bounds(g_, 4, p.ring_rec, ext_rec, p.dev_err)) cp_async_piece<4>(wcol + (buf * L + f) * 32 + lane, g_);
                        }
                    }
                }
            }
            cp_async_commit();
        };
#pragma unroll
        for (int q = 0; q < NS - 1; ++q) issue(q);

        // ------------------------------------------------ window: gates, normalised keys and queries
        float aw[TMAX], bw[TMAX];  // every token's gates, in every lane
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
            aw[t] = __shfl_sync(FULL_MASK, al_l, t), bw[t] = __shfl_sync(FULL_MASK, be_l, t);
            if (t >= T) aw[t] = 1.f, bw[t] = 0.f;
        }
        float ik_l = 1.f;  // lane t < T: token t's inverse key norm
        if constexpr (GDN) {
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
                if (t < T) {
                    float ssk = 0.f, ssq = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) ssk = fmaf(kw[t][e], kw[t][e], ssk), ssq = fmaf(qw[t][e], qw[t][e], ssq);
                    const float ik = rsqrtf(group_sum<G>(ssk) + 1e-6f);
                    const float iq = rsqrtf(group_sum<G>(ssq) + 1e-6f) * p.q_scale;
                    if (lane == t) ik_l = ik;
#pragma unroll
                    for (int e = 0; e < E; ++e) kw[t][e] *= ik, qw[t][e] *= iq;
                }
            }
        }
        // prefix decays of the window: Pk[t] = prod_{y<t} alpha_y, Pq[t] = Pk[t] alpha_t
        float Pk[TMAX], Pq[TMAX];
        {
            float run = 1.f;
#pragma unroll
            for (int t = 0; t < TMAX; ++t) Pk[t] = run, run *= aw[t], Pq[t] = run;
        }

        // set on the first sub-batch, from the staged headers: R(f) = prod_{f<g<count} alpha_g for lane f
        // (entries 32 + f in the _hi values), the product of all ring alphas, and a fold's scale of
        // entry f's rank-one term, R(f) / |k_f|
        const bool ring_hi = L > 32;
        float R = 1.f, R_hi = 1.f, gring = 1.f, fsc = 0.f, fsc_hi = 0.f;
        // entry f's value of a lane pair (lo: entries 0..31, hi: 32..63); f warp-uniform
        auto entry_val = [&](float lo, float hv, int f) {
            return f < 32 ? __shfl_sync(FULL_MASK, lo, f) : __shfl_sync(FULL_MASK, hv, f - 32);
        };
        unsigned char* mck = static_cast<unsigned char*>(p.ckpt) + uidx * p.dv * MROW;
        unsigned char* cck = static_cast<unsigned char*>(MIXED ? p.ckpt_copy : p.ckpt) + uidx * p.dv * SROW;
        const int64_t out_b = ((int64_t)b * T * p.Hv + h) * p.dv;  // output (t = 0, j = 0)
        const int64_t out_t = (int64_t)p.Hv * p.dv;                // next token
        float vx_pre[TMAX];  // the window's values at the lane's column of the current batch

        for (int q = 0; q < Q; ++q) {
            __syncwarp();  // no lane still reads the columns the next copy may overwrite
            issue(q + NS - 1);
            cp_async_wait<NS - 1>();
            __syncwarp();  // every lane's staged columns, keys and headers
            const int bq = q / SPB, sb = q - bq * SPB, buf = bq & 1;
            const int j0 = bq * 32;
            if (q == 0) {
                // ring decays by suffix products over the staged alphas
                float suf = lane < count ? hdr[lane].x : 1.f;
                float suf_hi = ring_hi && lane + 32 < count ? hdr[lane + 32].x : 1.f;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_down_sync(FULL_MASK, suf, off);
                    if (lane + off < 32) suf *= o;
                    if (ring_hi) {
                        const float oh = __shfl_down_sync(FULL_MASK, suf_hi, off);
                        if (lane + off < 32) suf_hi *= oh;
                    }
                }
                const float ghi = ring_hi ? __shfl_sync(FULL_MASK, suf_hi, 0) : 1.f;  // entries 32..count-1
                suf *= ghi;
                gring = __shfl_sync(FULL_MASK, suf, 0);
                R = __shfl_down_sync(FULL_MASK, suf, 1);
                R_hi = ring_hi ? __shfl_down_sync(FULL_MASK, suf_hi, 1) : 1.f;
                if (lane == 31) R = ghi, R_hi = 1.f;
                fsc = lane < count ? R * hdr[lane].z : 0.f;
                fsc_hi = ring_hi && lane + 32 < count ? R_hi * hdr[lane + 32].z : 0.f;
            }
            if (sb == 0 && T > 0) {
#pragma unroll
                for (int x = 0; x < TMAX; ++x)
                    vx_pre[x] = x < T ? load_elem(p.v, (((int64_t)b * T + x) * p.Hv + h) * p.dv + j0 + lane, in_dt)
                                      : 0.f;
            }
            const unsigned char* stg = stages + (q % NS) * C::STAGE;
            float st[NSB][E];
            int jr[NSB];
#pragma unroll
            for (int u = 0; u < NSB; ++u) {
                jr[u] = q * NSB * C::RPS + u * C::RPS + rg;
                if (fm) {
                    constexpr int PS = VEC * 4 < 16 ? VEC * 4 : 16, PPV = VEC * 4 / PS, NP = C::NVEC * PPV;
#pragma unroll
                    for (int k = 0; k < NP; ++k) {
                        const unsigned char* src = stg + ((u * NP + k) * 32 + lane) * PS;
                        if constexpr (PS == 16) {
                            const float4 f = *reinterpret_cast<const float4*>(src);
                            st[u][k * 4] = f.x, st[u][k * 4 + 1] = f.y, st[u][k * 4 + 2] = f.z, st[u][k * 4 + 3] = f.w;
                        } else {
                            const float2 f = *reinterpret_cast<const float2*>(src);
                            st[u][k * 2] = f.x, st[u][k * 2 + 1] = f.y;
                        }
                    }
                } else {
                    constexpr int SZ = (int)sizeof(ST);
                    constexpr int PS = VEC * SZ < 16 ? VEC * SZ : 16, PPV = VEC * SZ / PS, NP = C::NVEC * PPV;
                    constexpr int EPP = PS / SZ;  // elements per piece
#pragma unroll
                    for (int k = 0; k < NP; ++k) {
                        const unsigned char* src = stg + ((u * NP + k) * 32 + lane) * PS;
                        if constexpr (SZ == 4) {
                            const float4 f = *reinterpret_cast<const float4*>(src);
                            st[u][k * 4] = f.x, st[u][k * 4 + 1] = f.y, st[u][k * 4 + 2] = f.z, st[u][k * 4 + 3] = f.w;
                        } else if constexpr (PS == 16) {
                            Store<ST>::unpack(*reinterpret_cast<const uint4*>(src), st[u] + k * EPP);
                        } else {
                            const uint2 r = *reinterpret_cast<const uint2*>(src);
                            if constexpr (std::is_same<ST, __nv_bfloat16>::value) {
                                st[u][k * 4] = bf16_lo(r.x), st[u][k * 4 + 1] = bf16_hi(r.x);
                                st[u][k * 4 + 2] = bf16_lo(r.y), st[u][k * 4 + 3] = bf16_hi(r.y);
                            } else {
                                float2 f = f16x2_to_f2(r.x);
                                st[u][k * 4] = f.x, st[u][k * 4 + 1] = f.y;
                                f = f16x2_to_f2(r.y);
                                st[u][k * 4 + 2] = f.x, st[u][k * 4 + 3] = f.y;
                            }
                        }
                    }
                }
            }
            if (fold) {
                if constexpr (MIXED) {
                    // the recurrence on the master: every buffered entry's raw inputs through the rule, in
                    // order; the raw key's inverse norm scales the dot product and the correction
                    for (int f = 0; f < count; ++f) {
                        const float4 hf = hdr[f];
                        const float alf = hf.x, bef = hf.y, ikf = hf.z;
                        float kf[E];
#pragma unroll
                        for (int c = 0; c < C::NVEC; ++c) load_run<VEC>(keys + f * kbytes, pos_of(c), in_dt, kf + c * VEC);
                        float u_[NSB];
#pragma unroll
                        for (int u = 0; u < NSB; ++u) {
                            float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
                            for (int e = 0; e < E / 2; ++e)
                                d2 = __ffma2_rn(make_float2(st[u][2 * e], st[u][2 * e + 1]),
                                                make_float2(kf[2 * e], kf[2 * e + 1]), d2);
                            u_[u] = d2.x + d2.y;
                        }
#pragma unroll
                        for (int u = 0; u < NSB; ++u) u_[u] = group_sum<G>(u_[u]) * ikf;
                        const float2 a2 = make_float2(alf, alf);
#pragma unroll
                        for (int u = 0; u < NSB; ++u) {
                            // the staged 4 bytes of column jr[u] - j0 hold its value (16-bit: and its pair's)
                            const int c = jr[u] - j0;
                            const uint32_t raw = vcol[(buf * L + f) * 32 + c];
                            const uint32_t hv = (c & 1) ? raw >> 16 : raw & 0xffffu;
                            const float vf = in_sz == 4          ? __uint_as_float(raw)
                                             : in_dt == GDN_BF16 ? __uint_as_float(hv << 16)
                                                                 : __half2float(__ushort_as_half((unsigned short)hv));
                            const float wk = bef * (vf - alf * u_[u]) * ikf;
                            const float2 w2 = make_float2(wk, wk);
#pragma unroll
                            for (int e = 0; e < E / 2; ++e) {
                                float2 t2 = __fmul2_rn(make_float2(st[u][2 * e], st[u][2 * e + 1]), a2);
                                t2 = __ffma2_rn(make_float2(kf[2 * e], kf[2 * e + 1]), w2, t2);
                                st[u][2 * e] = t2.x, st[u][2 * e + 1] = t2.y;
                            }
                        }
                    }
                } else {
                    // S0 <- G S0 + sum_f A(f) k_f w_f^T with the buffered w
#pragma unroll
                    for (int u = 0; u < NSB; ++u)
#pragma unroll
                        for (int e = 0; e < E; ++e) st[u][e] *= gring;
                    for (int f = 0; f < count; ++f) {
                        const float sc = entry_val(fsc, fsc_hi, f);
                        float kf[E];
#pragma unroll
                        for (int c = 0; c < C::NVEC; ++c) load_run<VEC>(keys + f * kbytes, pos_of(c), in_dt, kf + c * VEC);
#pragma unroll
                        for (int u = 0; u < NSB; ++u) {
                            const float wk = sc * wcol[(buf * L + f) * 32 + (jr[u] - j0)];
                            const float2 w2 = make_float2(wk, wk);
#pragma unroll
                            for (int e = 0; e < E / 2; ++e) {
                                const float2 t2 = __ffma2_rn(make_float2(kf[2 * e], kf[2 * e + 1]), w2,
                                                             make_float2(st[u][2 * e], st[u][2 * e + 1]));
                                st[u][2 * e] = t2.x, st[u][2 * e + 1] = t2.y;
                            }
                        }
                    }
                }
                // store the folded rows (the master and its rounded copy); go on from the stored values
#pragma unroll
                for (int u = 0; u < NSB; ++u)
#pragma unroll
                    for (int c = 0; c < C::NVEC; ++c) {
                        if (in_bounds(mck + jr[u] * MROW + pos_of(c) * (int)sizeof(MT), VEC * sizeof(MT), p.ckpt, ext_m,
                                      p.dev_err))
                            st_state<MT, VEC>(mck + jr[u] * MROW, pos_of(c), st[u] + c * VEC);
                        if constexpr (MIXED)
                            if (in_bounds(cck + jr[u] * SROW + pos_of(c) * (int)sizeof(ST), VEC * sizeof(ST), sbase, ext_s,
                                          p.dev_err))
                                st_state<ST, VEC>(cck + jr[u] * SROW, pos_of(c), st[u] + c * VEC);
                    }
            }
            if (T == 0) continue;
            // the row sums S0^T k_t (GDN) and S0^T q_t of the sub-batch's rows, reduce-scattered into the tile
            {
                float x[C::V];
#pragma unroll
                for (int u = 0; u < NSB; ++u)
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        float2 a2 = make_float2(0.f, 0.f), b2 = a2;
#pragma unroll
                        for (int e = 0; e < E / 2; ++e) {
                            const float2 s2 = make_float2(st[u][2 * e], st[u][2 * e + 1]);
                            if constexpr (GDN) a2 = __ffma2_rn(s2, make_float2(kw[t][2 * e], kw[t][2 * e + 1]), a2);
                            b2 = __ffma2_rn(s2, make_float2(qw[t][2 * e], qw[t][2 * e + 1]), b2);
                        }
                        if constexpr (GDN) {
                            x[u * C::VPR + t] = a2.x + a2.y;
                            x[u * C::VPR + TMAX + t] = b2.x + b2.y;
                        } else {
                            x[u * C::VPR + t] = b2.x + b2.y;
                        }
                    }
                reduce_scatter_values<C::V, G>(x, g);
                if (g % C::DUP == 0) {
#pragma unroll
                    for (int i = 0; i < C::HELD; ++i) {
                        const int idx = g / C::DUP * C::HELD + i, u = idx / C::VPR, vv = idx - u * C::VPR;
                        tile[((sb * NSB + u) * C::RPS + rg) * C::TILE + vv] = x[i];
                    }
                }
            }
            if (sb != SPB - 1) continue;
            if (q == SPB - 1) {
                // ------------------------------------ coefficient table, before the first batch's rows
                // entry x (ring entry f = x < cpr, else window token s = x - cpr) against every window
                // token t: coef[x][t] = (k_x.k_t) times the decay from x to token t's prediction,
                // coef[x][TMAX + t] = (k_x.q_t) times the decay from x to token t's output; zero where x
                // does not precede t
                const int J = cpr + T;
                for (int x0 = 0; x0 < J; x0 += C::RPS) {
                    const int x = x0 + rg;
                    const int xc = x < J ? x : J - 1;
                    const bool ring = xc < cpr;
                    const int sw = xc - cpr;
                    float kx[E];
                    if (ring) {
#pragma unroll
                        for (int c = 0; c < C::NVEC; ++c) load_run<VEC>(keys + xc * kbytes, pos_of(c), in_dt, kx + c * VEC);
                        const float ikf = hdr[xc].z;
#pragma unroll
                        for (int e = 0; e < E; ++e) kx[e] *= ikf;
                    } else {
#pragma unroll
                        for (int e = 0; e < E; ++e) kx[e] = kw[0][e];
#pragma unroll
                        for (int t = 1; t < TMAX; ++t)
                            if (t == sw) {
#pragma unroll
                                for (int e = 0; e < E; ++e) kx[e] = kw[t][e];
                            }
                    }
                    float v[C::VPR];
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        float2 a2 = make_float2(0.f, 0.f), b2 = a2;
#pragma unroll
                        for (int e = 0; e < E / 2; ++e) {
                            const float2 x2 = make_float2(kx[2 * e], kx[2 * e + 1]);
                            if constexpr (GDN) a2 = __ffma2_rn(x2, make_float2(kw[t][2 * e], kw[t][2 * e + 1]), a2);
                            b2 = __ffma2_rn(x2, make_float2(qw[t][2 * e], qw[t][2 * e + 1]), b2);
                        }
                        if constexpr (GDN) {
                            v[t] = a2.x + a2.y;
                            v[TMAX + t] = b2.x + b2.y;
                        } else {
                            v[t] = b2.x + b2.y;
                        }
                    }
                    reduce_scatter_values<C::VPR, G>(v, g);
                    const int rsrc = ring ? xc : 0;  // differs between the warp's row groups
                    float Rx = __shfl_sync(FULL_MASK, R, rsrc & 31);
                    if (ring_hi) {
                        const float rh = __shfl_sync(FULL_MASK, R_hi, rsrc & 31);
                        if (rsrc >= 32) Rx = rh;
                    }
                    constexpr int NVL = C::VPR >= G ? C::VPR / G : 1;   // sums a lane holds
                    constexpr int DUPC = C::VPR >= G ? 1 : G / C::VPR;  // lanes holding the same sum
                    if (x < J && g % DUPC == 0) {
#pragma unroll
                        for (int i = 0; i < NVL; ++i) {
                            const int idx = C::VPR >= G ? g * NVL + i : g / DUPC;
                            const bool kq = GDN ? idx >= TMAX : true;  // a q coefficient
                            const int t = GDN && kq ? idx - TMAX : idx;
                            const bool live = t < T && (ring || (kq ? t >= sw : t > sw));
                            // the window tokens' decays after the entry (all of them after a ring entry),
                            // up to token t's prediction (y < t) or output (y <= t)
                            float dec = ring ? Rx : 1.f;
#pragma unroll
                            for (int y = 0; y < TMAX; ++y)
                                if ((ring || y > sw) && (kq ? y <= t : y < t)) dec *= aw[y];
                            coef[x * C::CW + (kq ? TMAX + t : t)] = live ? v[i] * dec : 0.f;
                        }
                    }
                }
            }
            __syncwarp();
            // ---------------------------------------- lane l finishes row j0 + l
            {
                const int j = j0 + lane;
                const float G1 = fold ? 1.f : gring;  // decay of S0 to the window's first token
                const float* tr = tile + lane * C::TILE;
                float y[TMAX], z[TMAX];
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                    y[t] = GDN ? tr[t] * (G1 * Pk[t]) : 0.f;
                    z[t] = tr[(GDN ? TMAX : 0) + t] * (G1 * Pq[t]);
                }
                // the buffered entries' terms (their w staged with the batch)
                const float* wc = wcol + buf * L * 32 + lane;
                for (int f = 0; f < cpr; ++f) {
                    const float wf = wc[f * 32];
                    const float* cf = coef + f * C::CW;
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        if constexpr (GDN) y[t] = fmaf(cf[t], wf, y[t]);
                        z[t] = fmaf(cf[TMAX + t], wf, z[t]);
                    }
                }
                // the window: w_x, then its terms in the later sums of the row
                int ri = pos0 % L;
#pragma unroll
                for (int x = 0; x < TMAX; ++x) {
                    if (x < T) {
                        const float wx = GDN ? bw[x] * (vx_pre[x] - aw[x] * y[x]) : bw[x] * vx_pre[x];
                        if (in_bounds(rec + ri * rec_floats + 4 + j, 4, p.ring_rec, ext_rec, p.dev_err))
                            rec[ri * rec_floats + 4 + j] = wx;
                        ri = ri + 1 == L ? 0 : ri + 1;
                        const float* cx = coef + (cpr + x) * C::CW;
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) {
                            if constexpr (GDN) y[t] = fmaf(cx[t], wx, y[t]);
                            z[t] = fmaf(cx[TMAX + t], wx, z[t]);
                        }
                    }
                }
                const float dskip = RULE == RULE_MAMBA2 ? p.D[h] : 0.f;
#pragma unroll
                for (int t = 0; t < TMAX; ++t)
                    if (t < T) {
                        float o = z[t];
                        if constexpr (RULE == RULE_MAMBA2) o = fmaf(dskip, vx_pre[t], o);
                        if (out_ok(out_b + t * out_t + j)) store_elem(p.out, out_b + t * out_t + j, out_dt, o);
                    }
            }
            __syncwarp();  // the tile is free for the next batch
        }
        cp_async_wait<0>();  // no copy of this unit is left in flight (the trailing groups are empty)
        __syncwarp();        // every lane is done with the staged data before the next unit's copies

        // ------------------------------------------------ append the window; move the pointers
        // (after the pass: a fold reads the old entries' records until its last row)
        if (T > 0) {
            const int kvec = kbytes / 16, vvec = p.dv * in_sz / 16;
            for (int t = 0; t < T; ++t) {
                const int64_t ent = unit_ring + (pos0 + t) % L;
                const int64_t qrow = ((int64_t)b * T + t) * p.Hk + kh;
                const int64_t vrow = ((int64_t)b * T + t) * p.Hv + h;
                for (int x = lane; x < kvec + vvec; x += 32) {
                    if (x < kvec) {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(p.ring_k) + ent * kbytes) + x;
                        if (in_bounds(dst, 16, p.ring_k, ext_rk, p.dev_err))
                            *dst = reinterpret_cast<const uint4*>(static_cast<const char*>(p.k) + qrow * kbytes)[x];
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(p.ring_v) + ent * p.dv * in_sz) + x - kvec;
                        if (in_bounds(dst, 16, p.ring_v, ext_rv, p.dev_err))
                            *dst = reinterpret_cast<const uint4*>(static_cast<const char*>(p.v) + vrow * p.dv * in_sz)[x - kvec];
                    }
                }
            }
            if (lane < T) {
                const int64_t ent = unit_ring + (pos0 + lane) % L;
                // field 3: the call's window length on its first entry (what a rollback checks), else 0
                float4* dst = reinterpret_cast<float4*>(p.ring_rec + ent * rec_floats);
                if (in_bounds(dst, 16, p.ring_rec, ext_rec, p.dev_err))
                    *dst = make_float4(al_l, be_l, ik_l, lane == 0 ? (float)T : 0.f);
            }
        }
        if (lane == 0 && in_bounds(p.pos + uidx, 4, p.pos, ext_ptr, p.dev_err)) {
            p.pos[uidx] = pos0 + T;
            if (fold) p.ckpt_pos[uidx] = pos0;
        }
    }
    __syncthreads();  // the next round rewrites the lists
    }
}

}  // namespace gdn
