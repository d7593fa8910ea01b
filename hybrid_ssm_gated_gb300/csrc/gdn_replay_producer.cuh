// gdn_replay_producer.cuh -- ReplaySSM in the decode kernel's producer/consumer
// form (the mode and its arithmetic are in gdn_replay_common.cuh). It serves the
// two-checkpoint mode and one fp32 checkpoint's single tokens, where its deep
// chunk ring measured faster than the row kernel (gdn_replay_rows.cuh).
//
// Kernel shape: persistent CTAs over (sequence, value head) units, one
// producer warp and NCW consumer warps, as in the decode kernel.
//  - The producer warp fetches pointers and gates for 32 units at a time (one
//    lane per unit). Per unit it bulk-copies the window's q/k/v rows and the
//    buffered ring entries (keys, records) into an NH-deep head ring and S0 in
//    16 KB chunks into an NS-deep chunk ring, one copy per lane, in one
//    convergent copy instruction (a large unit sends its rows and ring ahead
//    in one, then the chunks): a thread
//    issues a bulk copy only every ~0.25 us, but the lanes of one instruction
//    issue together.
//  - Every consumer warp visits every unit in order. A unit's state rows are
//    split into items dealt round robin over the warps, continuing across
//    units (a fold unit's items are split further, so that its extra work
//    spreads over all warps). The dot products of the buffered entries with
//    the window -- the coefficients of the w_f terms, decays included --
//    are dealt to the "crew", the warps after those, one entry per lane group,
//    and written to a table in the unit's head stage; the first crew warp also
//    appends the window to the ring. The crew's last warp to finish arms a
//    per-stage barrier that publishes the table, so row warps wait only for
//    that unit's crew, never for warps busy with other units, and only after
//    their pass over S0.
//  - Window of one token: an item is LPR warp passes of partial dot products,
//    then one reduce-scatter across a row's lanes leaves every lane owning one
//    row, so the w recursion, the output and the w store run once per row.
//    Larger windows take one pass per item and scatter the 2T sums of a row
//    over its lanes; the window's own recursion then passes each w_t across
//    lanes.
// Two checkpoints (same article, its paragraph on precision): with a wider
// master type MT, every unit that does not fold streams the read copy (ST)
// and one that folds streams the master, folds it in FP32, stores it, and
// rewrites the copy from the stored rows; the call's tokens then continue
// from the copy's values, as if it had been read back. A master chunk holds
// fewer rows, so its items release the chunk with a larger weight.
// Mamba2 (RULE_MAMBA2, gdn_device.cuh) runs through the same kernel: keys,
// queries and values are B, C and x, nothing is normalised (the stored inverse
// key norm is 1), w_e = delta_e x_e needs no prediction, so the S^T k sums and
// their ring terms are skipped, and every output gains D x.
// Hand-offs. Every warp visits every head stage in order, so the head and
// table barriers' parity waits cannot alias. The head barrier takes two
// arrivals: one arms its copies, the other comes with the metadata once every
// S0 chunk of the unit is armed. A warp that has seen a unit's head complete
// therefore waits on that unit's chunk barriers directly, although it skips
// the chunks of other warps' items: the chunk's fill has been armed, so the
// previous fill of its stage has completed, and the next fill needs this
// warp's release first. Every wait is bounded (GDN_DEVERR_TIMEOUT, then
// return).
#pragma once

#include <type_traits>

#include "gdn_decode.cuh"
#include "gdn_replay_common.cuh"

namespace gdn {

constexpr int REPLAY_META = 128;  // bytes of per-unit metadata at the start of a head stage

#ifndef GDN_REPLAY_CREW_PASSES
#define GDN_REPLAY_CREW_PASSES 4
#endif
constexpr int REPLAY_CREW_PASSES = GDN_REPLAY_CREW_PASSES;  // coefficient passes per crew warp
#ifndef GDN_REPLAY_WIDE_FOLD_PASSES
#define GDN_REPLAY_WIDE_FOLD_PASSES 4
#endif
constexpr int REPLAY_WIDE_FOLD_PASSES = GDN_REPLAY_WIDE_FOLD_PASSES;  // passes of a fold sub-item, T > 1

template <typename ST, int DK, int TMAX, int NCW>
struct ReplayCfg {
    static constexpr int VEC = Store<ST>::VEC;
    static constexpr int E = TMAX == 1 ? 16 : 8;  // state elements per lane per row
    static constexpr int NC = E / VEC;
    static constexpr int LPR = DK / E;                  // lanes per row
    static constexpr int RPP = 32 / LPR;                // rows per warp pass
    // a consumer work item is LPR warp passes = 32 rows, after which every lane owns one row: for
    // one token through a reduce-scatter of the item's sums, for wider windows through a per-warp
    // shared-memory tile of the row sums
    static constexpr int PPI = LPR;
    static constexpr int ITEM = PPI * RPP;
    static constexpr int SUMS = TMAX == 1 ? 0 : 32 * (2 * TMAX + 1);  // floats of a warp's row-sum tile
    static constexpr int V = 2 * TMAX;                  // sums per row: S^T k_t and S^T q_t
    static constexpr int NVL = V >= LPR ? V / LPR : 1;  // sums a lane holds after the reduce-scatter
    static constexpr int DUP = V >= LPR ? 1 : LPR / V;  // lanes holding the same sum
    static constexpr int FP = 2;                        // rows a lane folds at once (key reuse)
    // a fold unit's items are split further (SUB sub-items of FPS passes), so that its extra work
    // spreads over all warps; chunk releases count in sub-items. Wider windows take four passes a
    // sub-item, so that their per-lane recursion runs on more rows at once.
    static constexpr int FPS = TMAX == 1 ? FP : (PPI < REPLAY_WIDE_FOLD_PASSES ? PPI : REPLAY_WIDE_FOLD_PASSES);
    static constexpr int SUB = PPI / FPS;
    static constexpr int ROW_BYTES = DK * (int)sizeof(ST);
    static constexpr int THREADS = (NCW + 1) * 32;
    static_assert(E % VEC == 0 && DK % E == 0 && LPR >= 2 && LPR <= 32, "unsupported dk");
    static_assert(PPI % FPS == 0 && FPS % FP == 0 && ITEM == 32, "item blocking");
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

// ST: the checkpoint that steps and windows read (the read copy in the two-checkpoint mode);
// MT: the checkpoint that folds read and write (ST itself with one checkpoint).
template <typename ST, int DK, int TMAX, int NCW, typename MT = ST, int RULE = RULE_GDN, int IO = IO_ANY>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) replay_producer_kernel(const ReplayArgs p) {
    using C = ReplayCfg<ST, DK, TMAX, NCW>;
    const int in_dt = io_in<IO>(p.in_dtype), out_dt = io_out<IO>(p.out_dtype);
    constexpr bool MIXED = !std::is_same<ST, MT>::value;
    constexpr int MROW_BYTES = DK * (int)sizeof(MT);  // a master row
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* chunks = smem;
    unsigned char* heads = smem + p.heads_off;
    const int NS = p.nstage, NH = p.nhead;
    uint64_t* cfull = reinterpret_cast<uint64_t*>(smem + p.bars_off);
    uint64_t* cempty = cfull + NS;
    uint64_t* hfull = cempty + NS;
    uint64_t* hempty = hfull + NH;
    uint64_t* cready = hempty + NH;                        // per head stage: its coefficient table is written
    int* crew_done = reinterpret_cast<int*>(cready + NH);  // per head stage: table writers finished

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ipu = p.dv / C::ITEM;    // items per unit
    const int ipc = p.rows / C::ITEM;  // items per chunk
    // a fold unit's master chunks hold fewer rows than the read copy's: their sub-items release
    // with weight fw, so that every chunk fill takes ipc * SUB releases
    const int fw = MIXED ? ipc / (p.mrows / C::ITEM) : 1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&cfull[s], 1), mbar_init(&cempty[s], ipc * C::SUB);
        for (int s = 0; s < NH; ++s)
            mbar_init(&hfull[s], 2), mbar_init(&hempty[s], NCW), mbar_init(&cready[s], 1), crew_done[s] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const int total = p.B * p.Hv;
    const int in_sz = dtype_size(in_dt);
    const int group = p.Hv / p.Hk;
    const int T = p.T, L = p.L;
    const int rec_floats = 4 + p.dv;
    // array extents in bytes: every copy and store checks against them in bounds-checking builds
    const int TW = T > 0 ? T : 1;
    const uint64_t cells = (uint64_t)p.num_slots * p.Hv;
    const uint64_t ext_m = cells * p.dv * MROW_BYTES, ext_s = cells * p.dv * C::ROW_BYTES;
    const uint64_t ext_rk = cells * L * DK * in_sz, ext_rv = cells * L * p.dv * in_sz;
    const uint64_t ext_rec = cells * L * rec_floats * 4, ext_ptr = cells * 4;
    const uint64_t ext_qk = (uint64_t)p.B * TW * p.Hk * DK * in_sz, ext_v = (uint64_t)p.B * TW * p.Hv * p.dv * in_sz;
    const uint64_t ext_out = (uint64_t)p.B * TW * p.Hv * p.dv * dtype_size(out_dt);
    auto out_ok = [&](int64_t i) {
        return in_bounds(static_cast<char*>(p.out) + i * dtype_size(out_dt), dtype_size(out_dt), p.out, ext_out,
                         p.dev_err);
    };
    auto rec_ok = [&](const float* r) { return in_bounds(r, 4, p.ring_rec, ext_rec, p.dev_err); };

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        const uint64_t pol_once = policy_evict_first();   // S0 chunks and window rows: read once
        const uint64_t pol_ring = policy_evict_normal();  // ring entries: read again by later steps
        const uint32_t qbytes = DK * in_sz, vbytes = p.dv * in_sz, recbytes = rec_floats * 4;
        const uint32_t cbytes = p.rows * C::ROW_BYTES;
        uint32_t m = 0;   // chunk fills issued
        uint32_t nh = 0;  // head fills issued
        int n = 0;
        int hs = 0;        // head stage of unit n
        uint32_t hph = 0;  // parity of that stage's current fill
        int ms = 0;        // chunk stage of the next chunk fill (m mod NS)
        uint32_t mph = 0;  // its fill parity
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
                        fold = count + T > L;
                        slot = s;
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) {
                            if (t < T) {
                                const int64_t gi = ((int64_t)b * T + t) * p.Hv + h;
                                rule_gates<RULE>(p.A_log[h], p.dt_bias[h], p.a, p.b, gi, in_dt, al[t], be[t]);
                            }
                        }
                    } else {
                        fold = p.force ? count > 0 : count + 1 > L;
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
                unsigned char* head = heads + hs * p.head_bytes;
                const int rbase = k_i % L;
                const int n1 = min(c_i, L - rbase);
                // The head barrier takes two arrivals: the first arms its copies; the second comes
                // with the metadata once every S0 chunk of the unit is armed, so a consumer that has
                // seen the head complete may wait on the unit's chunk barriers directly.
                // a two-checkpoint fold also takes the buffered raw values: it re-runs the entries on the master
                const bool fm = MIXED && f_i;
                if (lane == 0) {
                    if (n >= NH) ok = mbar_wait(&hempty[hs], hph ^ 1);
                    if (ok) {
                        if (s_i >= 0)
                            mbar_arrive_expect_tx(&hfull[hs], T * (2 * qbytes + vbytes) +
                                                                  c_i * (qbytes + recbytes + (fm ? vbytes : 0u)));
                        else
                            mbar_arrive(&hfull[hs]);
                        ++nh;
                    }
                }
                ok = __shfl_sync(FULL_MASK, ok, 0);
                if (!ok) break;
                auto publish = [&]() {  // the metadata and the second arrival, then on to the next stage
                    if (lane == 0) {
                        ReplayMeta* meta = reinterpret_cast<ReplayMeta*>(head);
                        meta->slot = s_i, meta->count = c_i, meta->fold = f_i, meta->pos0 = p_i, meta->ckpt0 = k_i;
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) meta->alpha[t] = al_i[t], meta->beta[t] = be_i[t];
                        mbar_arrive(&hfull[hs]);
                    }
                    if (++hs == NH) hs = 0, hph ^= 1;
                };
                if (s_i < 0) {
                    publish();
                    continue;
                }
                const int b = unit / p.Hv, h = unit - b * p.Hv, kh = h / group;
                const int64_t unit_ring = ((int64_t)s_i * p.Hv + h) * L;
                // a fold unit streams the master checkpoint, any other the one steps read
                const int nck = fm ? p.mnchunk : p.nchunk;
                const uint32_t ub = fm ? p.mrows * MROW_BYTES : cbytes;
                const void* s0_base = MIXED && !f_i ? p.ckpt_copy : p.ckpt;
                const uint64_t s0_ext = MIXED && !f_i ? ext_s : ext_m;
                const char* s0 = static_cast<const char*>(MIXED && !f_i ? p.ckpt_copy : p.ckpt) +
                                 ((int64_t)s_i * p.Hv + h) * p.dv * (fm ? MROW_BYTES : C::ROW_BYTES);
                // Copies: lanes 0..3T-1 the window's q/k/v rows, the next four (six) up to two ring ranges
                // (keys, records, and values for a two-checkpoint fold), the others S0 chunks, at most NS of them at a time so that no lane waits for a
                // stage another lane is about to fill. A unit of more than two chunks issues its rows and
                // ring first, then each chunk as soon as its stage is free: waiting for all of them would
                // hold the rows back by up to a unit's worth of consumption (T = 4 windows over fp32
                // 128 x 128 states: 11% faster, single tokens 2%). Otherwise every copy of the unit goes
                // out in one convergent bulk-copy instruction once its chunk stages are free (more rounds
                // only when the chunks do not fit). The split is compiled only where it can pay: in the
                // single-token kernels of small units, even untaken, it cost up to 17%.
                constexpr bool SPLIT = TMAX > 1 || (RULE == RULE_GDN && std::is_same<ST, float>::value && !MIXED);
                constexpr int NJ = MIXED ? 6 : 4;  // ring-range copy jobs
                const int hj = 3 * T + NJ;
                bool split = false;
                if constexpr (SPLIT) split = nck > 2;
                for (int c0 = 0, round = 0; ok && (round == 0 || c0 < nck); ++round) {
                    const int cl0 = split ? 32 : round == 0 ? hj : 0;  // first chunk lane of this round
                    const int per = min(NS, 32 - cl0);                 // chunk lanes of this round
                    const char* src = nullptr;
                    unsigned char* dst = nullptr;
                    uint32_t bytes = 0;
                    uint64_t* bar = &hfull[hs];
                    uint64_t pol = pol_ring;
                    const void* gbase = nullptr;  // the source's array and its extent
                    uint64_t gext = 0;
                    if (round == 0 && lane < 3 * T) {
                        const int t = lane / 3, kind = lane - 3 * t;
                        const int64_t qrow = ((int64_t)b * T + t) * p.Hk + kh;
                        const int64_t vrow = ((int64_t)b * T + t) * p.Hv + h;
                        src = kind == 0   ? static_cast<const char*>(p.q) + qrow * qbytes
                              : kind == 1 ? static_cast<const char*>(p.k) + qrow * qbytes
                                          : static_cast<const char*>(p.v) + vrow * vbytes;
                        dst = head + (kind == 0 ? p.off_wq + t * qbytes : kind == 1 ? p.off_wk + t * qbytes
                                                                                    : p.off_wv + t * vbytes);
                        bytes = kind == 2 ? vbytes : qbytes;
                        pol = pol_once;
                        gbase = kind == 0 ? p.q : kind == 1 ? p.k : p.v;
                        gext = kind == 2 ? ext_v : ext_qk;
                    } else if (round == 0 && lane < hj) {
                        // job bit 0: the first ring range or the wrapped one; job / 2: keys, records, values
                        const int job = lane - 3 * T, wrap = job & 1, kind = job >> 1;
                        const int first = wrap ? n1 : 0, cnt = wrap ? c_i - n1 : n1, ridx = wrap ? 0 : rbase;
                        if (cnt > 0) {
                            if (kind == 0) {
                                src = static_cast<const char*>(p.ring_k) + (unit_ring + ridx) * qbytes;
                                dst = head + p.off_rk + first * qbytes;
                                bytes = cnt * qbytes;
                                gbase = p.ring_k, gext = ext_rk;
                            } else if (kind == 1) {
                                src = reinterpret_cast<const char*>(p.ring_rec + (unit_ring + ridx) * rec_floats);
                                dst = head + p.off_rec + first * recbytes;
                                bytes = cnt * recbytes;
                                gbase = p.ring_rec, gext = ext_rec;
                            } else if (fm) {
                                src = static_cast<const char*>(p.ring_v) + (unit_ring + ridx) * vbytes;
                                dst = head + p.off_rv + first * vbytes;
                                bytes = cnt * vbytes;
                                gbase = p.ring_v, gext = ext_rv;
                            }
                        }
                    }
                    const int c = c0 + lane - cl0;
                    if (lane >= cl0 && lane - cl0 < per && c < nck) {
                        const uint32_t mc = m + c;
                        int cs = ms + c;  // stage and fill parity of chunk mc (c < 32, NS >= 2)
                        uint32_t cph = mph;
                        while (cs >= NS) cs -= NS, cph ^= 1;
                        ok = mc < (uint32_t)NS || mbar_wait(&cempty[cs], cph ^ 1);
                        if (ok) {
                            mbar_arrive_expect_tx(&cfull[cs], ub);
                            src = s0 + (int64_t)c * ub;
                            dst = chunks + cs * CHUNK_BYTES;
                            bytes = ub;
                            bar = &cfull[cs];
                            pol = pol_once;
                            gbase = s0_base, gext = s0_ext;
                        }
                    }
                    ok = __all_sync(FULL_MASK, ok);
                    if (ok && bytes) bulk_load_hint_checked(dst, src, bytes, bar, pol, gbase, gext, p.dev_err);
                    if (split) break;
                    c0 += per;
                }
                if (split) {
                    for (int c0 = 0; ok && c0 < nck; c0 += NS) {
                        const int c = c0 + lane;
                        if (lane < NS && c < nck) {
                            const uint32_t mc = m + c;
                            int cs = ms + c;  // stage and fill parity of chunk mc
                            uint32_t cph = mph;
                            while (cs >= NS) cs -= NS, cph ^= 1;
                            ok = mc < (uint32_t)NS || mbar_wait(&cempty[cs], cph ^ 1);
                            if (ok) {
                                mbar_arrive_expect_tx(&cfull[cs], ub);
                                bulk_load_hint_checked(chunks + cs * CHUNK_BYTES, s0 + (int64_t)c * ub, ub, &cfull[cs],
                                                       pol_once, s0_base, s0_ext, p.dev_err);
                            }
                        }
                        ok = __all_sync(FULL_MASK, ok);
                    }
                }
                m += nck;
                for (ms += nck; ms >= NS;) ms -= NS, mph ^= 1;
                publish();
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
    const int pg = lane % C::LPR;    // lane's position within its row group
    const int rsub = lane / C::LPR;  // row group within the warp
    float* sums = reinterpret_cast<float*>(smem + p.sums_off) + cw * C::SUMS;  // this warp's row-sum tile
    auto pos_of = [&](int cc) { return (cc * C::LPR + pg) * C::VEC; };
    // index of the i-th sum this lane holds after reduce_scatter_values
    auto held = [&](int i) { return C::V >= C::LPR ? pg * C::NVL + i : pg / C::DUP; };
    int ms = 0;        // chunk stage of the unit's first chunk
    uint32_t mph = 0;  // its fill parity
    int base = 0;      // warp of the unit's first item (items of earlier units, mod NCW)
    int hs = 0;        // head stage of unit n
    uint32_t hph = 0;  // its fill parity
    bool ok = true;
    for (int n = 0; ok; ++n, hs = hs + 1 == NH ? 0 : hs + 1, hph ^= hs == 0) {
        const int unit = blockIdx.x + n * gridDim.x;
        if (unit >= total) break;
        if (!(ok = mbar_wait(&hfull[hs], hph))) break;
        unsigned char* head = heads + hs * p.head_bytes;
        const ReplayMeta* meta = reinterpret_cast<const ReplayMeta*>(head);
        const int slot = meta->slot;
        if (slot < 0) {
            const int b = unit / p.Hv, h = unit - b * p.Hv;
            if (slot == -1) {
                for (int x = cw * 32 + lane; x < T * p.dv; x += NCW * 32) {
                    const int t = x / p.dv, j = x - t * p.dv;
                    const int64_t oi = (((int64_t)b * T + t) * p.Hv + h) * p.dv + j;
                    if (out_ok(oi)) store_elem(p.out, oi, out_dt, 0.f);
                }
            }
            __syncwarp();
            if (lane == 0) {
                if (cw == 0) mbar_arrive(&cready[hs]);  // keeps the table barrier's phases one per unit
                mbar_arrive(&hempty[hs]);
            }
            continue;
        }
        const int count = meta->count, fold = meta->fold, pos0 = meta->pos0;
        const int upc = MIXED && fold ? p.mrows / C::ITEM : ipc;  // items per chunk of this unit
        const int cpr = fold ? 0 : count;         // ring entries in front of the window
        const int J = T > 1 ? cpr + T : cpr;      // coefficient-table entries: ring, then window (T > 1)
        const int nitems = fold ? ipu * C::SUB : ipu;
        const int dbase = (base + nitems) % NCW;  // warp of the unit's first coefficient pass
        const int i0 = (cw - base + NCW) % NCW;   // this warp's first item
        const int d0 = (cw - dbase + NCW) % NCW;  // this warp's first coefficient pass
        // the crew: warps with coefficient passes (up to REPLAY_CREW_PASSES each, so that few warps
        // spend a window normalisation on them), at least the appender; its last warp to finish
        // arms the table barrier, so row warps never wait for warps busy with other units
        const int dpasses = (J + C::RPP - 1) / C::RPP;
        const int crew = max(1, min(NCW, (dpasses + REPLAY_CREW_PASSES - 1) / REPLAY_CREW_PASSES));
        const bool rows_here = i0 < nitems;
        const bool in_crew = d0 < crew;
        const bool dots_here = in_crew && J > 0;
        const bool appender = d0 == 0;
        if (rows_here || in_crew) {
            const int b = unit / p.Hv, h = unit - b * p.Hv;
            const int64_t unit_ring = ((int64_t)slot * p.Hv + h) * L;
            const float* rec = reinterpret_cast<const float*>(head + p.off_rec);
            float* coef = reinterpret_cast<float*>(head + p.off_coef);  // [J][V]
            const unsigned char* rk = head + p.off_rk;

            // window keys and queries, normalised, at this lane's key positions
            float2 kw2[TMAX][C::E / 2], qw2[TMAX][C::E / 2];
            float ikw[TMAX];
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
                float xk[C::E], xq[C::E];
#pragma unroll
                for (int e = 0; e < C::E; ++e) xk[e] = 0.f, xq[e] = 0.f;
                ikw[t] = 0.f;
                if (t < T) {
#pragma unroll
                    for (int cc = 0; cc < C::NC; ++cc) {
                        load_run<C::VEC>(head + p.off_wk + t * DK * in_sz, pos_of(cc), in_dt, xk + cc * C::VEC);
                        load_run<C::VEC>(head + p.off_wq + t * DK * in_sz, pos_of(cc), in_dt, xq + cc * C::VEC);
                    }
                    ikw[t] = 1.f;
                    if constexpr (RULE == RULE_GDN) {
                        float ssk = 0.f, ssq = 0.f;
#pragma unroll
                        for (int e = 0; e < C::E; ++e) ssk = fmaf(xk[e], xk[e], ssk), ssq = fmaf(xq[e], xq[e], ssq);
                        const float ik = rsqrtf(group_sum<C::LPR>(ssk) + 1e-6f);
                        const float iq = rsqrtf(group_sum<C::LPR>(ssq) + 1e-6f) * p.q_scale;
                        ikw[t] = ik;
#pragma unroll
                        for (int e = 0; e < C::E; ++e) xk[e] *= ik, xq[e] *= iq;
                    }
                }
#pragma unroll
                for (int e = 0; e < C::E / 2; ++e)
                    kw2[t][e] = make_float2(xk[2 * e], xk[2 * e + 1]), qw2[t][e] = make_float2(xq[2 * e], xq[2 * e + 1]);
            }
            // decays of the ring entries, lane f holding entries f and 32 + f:
            // R(f) = prod_{f<g<count} alpha_g by suffix scans (the upper half only when L > 32)
            float suf = lane < count ? rec[lane * rec_floats] : 1.f;
            float suf_hi = 1.f;
            const bool ring_hi = L > 32;
            if (ring_hi && lane + 32 < count) suf_hi = rec[(lane + 32) * rec_floats];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_down_sync(FULL_MASK, suf, off);
                if (lane + off < 32) suf *= o;
                if (ring_hi) {
                    const float oh = __shfl_down_sync(FULL_MASK, suf_hi, off);
                    if (lane + off < 32) suf_hi *= oh;
                }
            }
            const float ghi = ring_hi ? __shfl_sync(FULL_MASK, suf_hi, 0) : 1.f;  // product of entries 32..count-1
            suf *= ghi;
            const float gring = __shfl_sync(FULL_MASK, suf, 0);  // product of all ring alphas
            float R = __shfl_down_sync(FULL_MASK, suf, 1);
            float R_hi = ring_hi ? __shfl_down_sync(FULL_MASK, suf_hi, 1) : 1.f;
            if (lane == 31) R = ghi, R_hi = 1.f;
            // entry f's value of a per-lane pair (lo: entries 0..31, hi: 32..63); f warp-uniform
            auto entry_val = [&](float lo, float hv, int f) {
                return f < 32 ? __shfl_sync(FULL_MASK, lo, f) : __shfl_sync(FULL_MASK, hv, f - 32);
            };

            if (dots_here) {
                // entry x (ring entry f = x < cpr, else window token s = x - cpr) against every window
                // token t: coef[x][t] = (k_x.k_t) times the decay from x to token t's S^T k_t,
                // coef[x][TMAX + t] = (k_x.q_t) times the decay from x to token t's output; zero where
                // the entry does not precede the token
                for (int dp = d0; dp < dpasses; dp += crew) {
                    const int x = dp * C::RPP + rsub;
                    const int xc = min(x, J - 1);
                    const bool ring = xc < cpr;
                    const int s = xc - cpr;  // window token of a window entry
                    float2 kx[C::E / 2];
                    if (ring) {
                        float raw[C::E];
#pragma unroll
                        for (int cc = 0; cc < C::NC; ++cc)
                            load_run<C::VEC>(rk + xc * DK * in_sz, pos_of(cc), in_dt, raw + cc * C::VEC);
                        const float ikf = rec[xc * rec_floats + 2];
#pragma unroll
                        for (int e = 0; e < C::E / 2; ++e) kx[e] = make_float2(raw[2 * e] * ikf, raw[2 * e + 1] * ikf);
                    } else {
#pragma unroll
                        for (int e = 0; e < C::E / 2; ++e) kx[e] = kw2[0][e];
#pragma unroll
                        for (int t = 1; t < TMAX; ++t)
                            if (t == s) {
#pragma unroll
                                for (int e = 0; e < C::E / 2; ++e) kx[e] = kw2[t][e];
                            }
                    }
                    float v[C::V];
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        float2 a2 = make_float2(0.f, 0.f), b2 = a2;
#pragma unroll
                        for (int e = 0; e < C::E / 2; ++e)
                        {
                            if constexpr (RULE == RULE_GDN) a2 = __ffma2_rn(kx[e], kw2[t][e], a2);
                            b2 = __ffma2_rn(kx[e], qw2[t][e], b2);
                        }
                        v[t] = a2.x + a2.y;
                        v[TMAX + t] = b2.x + b2.y;
                    }
                    reduce_scatter_values<C::V, C::LPR>(v, pg);
                    const int rsrc = ring ? xc : 0;  // differs between the warp's row groups
                    float Rf = __shfl_sync(FULL_MASK, R, rsrc & 31);
                    if (ring_hi) {
                        const float rh = __shfl_sync(FULL_MASK, R_hi, rsrc & 31);
                        if (rsrc >= 32) Rf = rh;
                    }
                    if (x < J && pg % C::DUP == 0) {
#pragma unroll
                        for (int i = 0; i < C::NVL; ++i) {
                            const int idx = held(i);
                            const bool kq = idx >= TMAX;
                            const int t = idx - (kq ? TMAX : 0);
                            const int hi = t + (kq ? 1 : 0);  // decays of window tokens y < hi apply
                            const bool live = t < T && (ring || (kq ? t >= s : t > s));
                            float dec = ring ? Rf : 1.f;
#pragma unroll
                            for (int y = 0; y < TMAX; ++y)
                                if (y < hi && (ring || y > s)) dec *= meta->alpha[y];
                            coef[x * C::V + idx] = live ? v[i] * dec : 0.f;
                        }
                    }
                }
            }
            if (appender && T > 0) {
                // append the window's raw inputs, gates and key norms to the ring
                const int kvec = DK * in_sz / 16, vvec = p.dv * in_sz / 16;
                for (int t = 0; t < T; ++t) {
                    const int64_t ent = unit_ring + (pos0 + t) % L;
                    for (int x = lane; x < kvec; x += 32) {
                        uint4* d = reinterpret_cast<uint4*>(static_cast<char*>(p.ring_k) + ent * DK * in_sz) + x;
                        if (in_bounds(d, 16, p.ring_k, ext_rk, p.dev_err))
                            *d = reinterpret_cast<const uint4*>(head + p.off_wk + t * DK * in_sz)[x];
                    }
                    for (int x = lane; x < vvec; x += 32) {
                        uint4* d = reinterpret_cast<uint4*>(static_cast<char*>(p.ring_v) + ent * p.dv * in_sz) + x;
                        if (in_bounds(d, 16, p.ring_v, ext_rv, p.dev_err))
                            *d = reinterpret_cast<const uint4*>(head + p.off_wv + t * p.dv * in_sz)[x];
                    }
                }
                if (lane < T) {
                    float ikt = ikw[0];
#pragma unroll
                    for (int t = 1; t < TMAX; ++t)
                        if (lane == t) ikt = ikw[t];
                    const int64_t ent = unit_ring + (pos0 + lane) % L;
                    // field 3: the call's window length on its first entry (what a rollback checks), else 0
                    float4* d = reinterpret_cast<float4*>(p.ring_rec + ent * rec_floats);
                    if (in_bounds(d, 16, p.ring_rec, ext_rec, p.dev_err))
                        *d = make_float4(meta->alpha[lane], meta->beta[lane], ikt, lane == 0 ? (float)T : 0.f);
                }
            }
            if (appender && lane == 0) {
                const int64_t idx = (int64_t)slot * p.Hv + h;
                if (in_bounds(p.pos + idx, 4, p.pos, ext_ptr, p.dev_err)) {
                    p.pos[idx] = pos0 + T;
                    if (fold) p.ckpt_pos[idx] = pos0;
                }
            }
            __syncwarp();
            if (in_crew && lane == 0) {
                __threadfence_block();  // every lane's table entries before the count
                if (atomicAdd(crew_done + hs, 1) == crew - 1) {
                    crew_done[hs] = 0;  // next used for unit n + NH, after every warp has left this one
                    __threadfence_block();
                    mbar_arrive(&cready[hs]);
                }
            }

            if (rows_here) {
                // Mamba2's skip weight (a flush, T = 0, has no outputs and no D)
                const float dskip = RULE == RULE_MAMBA2 && T > 0 ? p.D[h] : 0.f;
                const float g1 = fold ? 1.f : gring;  // decay of S0 to the window's first token
                // fold: scale of entry f's rank-one term, R(f) / |k_f| (lane f, entries 32 + f in fsc_hi)
                const float fsc = lane < count ? R * rec[lane * rec_floats + 2] : 0.f;
                const float fsc_hi = ring_hi && lane + 32 < count ? R_hi * rec[(lane + 32) * rec_floats + 2] : 0.f;
                const float gfold = gring;
                unsigned char* gck =
                    static_cast<unsigned char*>(p.ckpt) + ((int64_t)slot * p.Hv + h) * p.dv * MROW_BYTES;
                bool have_coef = false;

                // S0 <- round(G S0 + sum_f A(f) k_f w_f^T) for NR rows s[r] (state rows j[r]) of this
                // lane: each buffered key is loaded once for all NR rows; the rows are stored to the
                // checkpoint and continue as the stored (rounded) values
                auto fold_rows = [&](auto& s, const auto& j) {
                    constexpr int NR = sizeof(j) / sizeof(j[0]);
                    if constexpr (MIXED) {
                        // Two checkpoints: the recurrence runs on the master. Every buffered entry's raw
                        // inputs go through the rule on the FP32 master rows, in order; a row's
                        // prediction S^T k_f is a dot product within the row, so rows never wait for
                        // one another. The raw key's inverse norm scales the dot product and the
                        // correction instead of the key.
                        for (int f = 0; f < count; ++f) {
                            const float* rf = rec + f * rec_floats;
                            const float alf = rf[0], bef = rf[1], ikf = rf[2];
                            float kr[C::E];
#pragma unroll
                            for (int cc = 0; cc < C::NC; ++cc)
                                load_run<C::VEC>(rk + f * DK * in_sz, pos_of(cc), in_dt, kr + cc * C::VEC);
                            float u[NR];
#pragma unroll
                            for (int r = 0; r < NR; ++r) {
                                float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
                                for (int e = 0; e < C::E / 2; ++e)
                                    d2 = __ffma2_rn(make_float2(s[r][2 * e], s[r][2 * e + 1]),
                                                    make_float2(kr[2 * e], kr[2 * e + 1]), d2);
                                u[r] = d2.x + d2.y;
                            }
#pragma unroll
                            for (int r = 0; r < NR; ++r) u[r] = group_sum<C::LPR>(u[r]) * ikf;
                            const float2 a2 = make_float2(alf, alf);
#pragma unroll
                            for (int r = 0; r < NR; ++r) {
                                const float vf = load_elem(head + p.off_rv + f * p.dv * in_sz, j[r], in_dt);
                                const float wk = bef * (vf - alf * u[r]) * ikf;
                                const float2 w2 = make_float2(wk, wk);
#pragma unroll
                                for (int e = 0; e < C::E / 2; ++e) {
                                    float2 t2 = __fmul2_rn(make_float2(s[r][2 * e], s[r][2 * e + 1]), a2);
                                    t2 = __ffma2_rn(make_float2(kr[2 * e], kr[2 * e + 1]), w2, t2);
                                    s[r][2 * e] = t2.x, s[r][2 * e + 1] = t2.y;
                                }
                            }
                        }
                    } else {
#pragma unroll
                    for (int r = 0; r < NR; ++r)
#pragma unroll
                        for (int e = 0; e < C::E; ++e) s[r][e] *= gfold;
                    // entries two at a time (keys and weights of both loaded first); each element still
                    // takes the entries in order
                    for (int f = 0; f < count; f += 2) {
                        const bool two = f + 1 < count;
                        const float sc0 = entry_val(fsc, fsc_hi, f);
                        const float sc1 = two ? entry_val(fsc, fsc_hi, f + 1) : 0.f;
                        float k0[C::E], k1[C::E];
#pragma unroll
                        for (int cc = 0; cc < C::NC; ++cc) {
                            load_run<C::VEC>(rk + f * DK * in_sz, pos_of(cc), in_dt, k0 + cc * C::VEC);
                            load_run<C::VEC>(rk + (two ? f + 1 : f) * DK * in_sz, pos_of(cc), in_dt, k1 + cc * C::VEC);
                        }
#pragma unroll
                        for (int r = 0; r < NR; ++r) {
                            const float w0 = sc0 * rec[f * rec_floats + 4 + j[r]];
                            const float w1 = two ? sc1 * rec[(f + 1) * rec_floats + 4 + j[r]] : 0.f;
                            const float2 a2 = make_float2(w0, w0), b2 = make_float2(w1, w1);
#pragma unroll
                            for (int e = 0; e < C::E / 2; ++e) {
                                float2 t2 = __ffma2_rn(make_float2(k0[2 * e], k0[2 * e + 1]), a2,
                                                       make_float2(s[r][2 * e], s[r][2 * e + 1]));
                                if (two) t2 = __ffma2_rn(make_float2(k1[2 * e], k1[2 * e + 1]), b2, t2);
                                s[r][2 * e] = t2.x, s[r][2 * e + 1] = t2.y;
                            }
                        }
                    }
                    }
#pragma unroll
                    for (int r = 0; r < NR; ++r) {
                        unsigned char* dst = gck + (int64_t)j[r] * MROW_BYTES;
#pragma unroll
                        for (int cc = 0; cc < C::NC; ++cc)
                            if (in_bounds(dst + pos_of(cc) * (int)sizeof(MT), C::VEC * sizeof(MT), p.ckpt, ext_m, p.dev_err))
                                store_row_run<MT, C::VEC>(dst, pos_of(cc), s[r] + cc * C::VEC);
                        if constexpr (MIXED) {  // the read copy: the stored master row, rounded to ST
                            unsigned char* cdst = static_cast<unsigned char*>(p.ckpt_copy) +
                                                  (((int64_t)slot * p.Hv + h) * p.dv + j[r]) * C::ROW_BYTES;
#pragma unroll
                            for (int cc = 0; cc < C::NC; ++cc)
                                if (in_bounds(cdst + pos_of(cc) * (int)sizeof(ST), C::VEC * sizeof(ST), p.ckpt_copy, ext_s,
                                              p.dev_err))
                                    store_row_run<ST, C::VEC>(cdst, pos_of(cc), s[r] + cc * C::VEC);
                        }
                    }
                };
                // row r of a chunk (a master chunk on a fold unit)
                auto load_state = [&](const unsigned char* tile, int r, float* s) {
                    if (MIXED && fold) {
#pragma unroll
                        for (int cc = 0; cc < C::NC; ++cc)
                            load_row_run<MT, C::VEC>(tile + r * MROW_BYTES, pos_of(cc), s + cc * C::VEC);
                    } else {
#pragma unroll
                        for (int cc = 0; cc < C::NC; ++cc)
                            load_row_run<ST, C::VEC>(tile + r * C::ROW_BYTES, pos_of(cc), s + cc * C::VEC);
                    }
                };

                // k.q, the window token's own term in its output (one token)
                float qk = 0.f;
                if (TMAX == 1 && T > 0) {
                    float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < C::E / 2; ++e) d2 = __ffma2_rn(kw2[0][e], qw2[0][e], d2);
                    qk = group_sum<C::LPR>(d2.x + d2.y);
                }
                for (int it = i0; it < nitems; it += NCW) {
                    const int bi = fold ? it / C::SUB : it;  // the item (of a fold sub-item)
                    const int c = bi / upc;
                    int cs = ms + c;  // stage and fill parity of the item's chunk
                    uint32_t cph = mph;
                    while (cs >= NS) cs -= NS, cph ^= 1;
                    // the unit's head completing means all its chunks are armed: no other fill of the
                    // stage can be taken for this one
                    if (!(ok = mbar_wait(&cfull[cs], cph))) break;
                    const unsigned char* tile = chunks + cs * CHUNK_BYTES;
                    const int r0 = (bi - c * upc) * C::ITEM;  // item's first row within the chunk
                    const int j0 = bi * C::ITEM;              // item's first row within the state

                    if constexpr (TMAX == 1) {
                        // PPI passes of partial dot products, then a reduce-scatter leaves lane (rsub, pg)
                        // with the sums of row pg * RPP + rsub of the item
                        if (fold) {
                            // sub-item: FP passes, folded, then dot products reduced per pass
                            const int ps0 = (it - bi * C::SUB) * C::FPS;
                            float s[C::FP][C::E];
                            int jr[C::FP];
#pragma unroll
                            for (int r = 0; r < C::FP; ++r) {
                                load_state(tile, r0 + (ps0 + r) * C::RPP + rsub, s[r]);
                                jr[r] = j0 + (ps0 + r) * C::RPP + rsub;
                            }
                            __syncwarp();
                            if (lane == 0) mbar_arrive_n(&cempty[cs], fw);
                            fold_rows(s, jr);
                            if (T > 0) {
                                const float al = meta->alpha[0], be = meta->beta[0];
#pragma unroll
                                for (int r = 0; r < C::FP; ++r) {
                                    float2 u2 = make_float2(0.f, 0.f), v2 = u2;
#pragma unroll
                                    for (int e = 0; e < C::E / 2; ++e) {
                                        const float2 s2 = make_float2(s[r][2 * e], s[r][2 * e + 1]);
                                        if constexpr (RULE == RULE_GDN) u2 = __ffma2_rn(s2, kw2[0][e], u2);
                                        v2 = __ffma2_rn(s2, qw2[0][e], v2);
                                    }
                                    // after a fold the window's first token follows S0 directly
                                    const float Y = group_sum<C::LPR>(u2.x + u2.y);
                                    const float Z = group_sum<C::LPR>(v2.x + v2.y) * al;
                                    const int j = jr[r];
                                    const float vj = load_elem(head + p.off_wv, j, in_dt);
                                    const float ww = RULE == RULE_GDN ? be * (vj - al * Y) : be * vj;
                                    if (pg == 0) {
                                        const int64_t oi = ((int64_t)b * p.Hv + h) * p.dv + j;
                                        if (out_ok(oi)) store_elem(p.out, oi, out_dt, fmaf(dskip, vj, fmaf(qk, ww, Z)));
                                        float* wd = p.ring_rec + (unit_ring + pos0 % L) * rec_floats + 4 + j;
                                        if (rec_ok(wd)) *wd = ww;
                                    }
                                }
                            }
                            continue;
                        }
                        float y[C::PPI], z[C::PPI];
                        {
                            // 16-byte vector cc of all passes first, then their math: 2*PPI independent chains
                            float2 u2[C::PPI], v2[C::PPI];
#pragma unroll
                            for (int ps = 0; ps < C::PPI; ++ps) u2[ps] = make_float2(0.f, 0.f), v2[ps] = u2[ps];
#pragma unroll
                            for (int cc = 0; cc < C::NC; ++cc) {
                                uint4 raw[C::PPI];
#pragma unroll
                                for (int ps = 0; ps < C::PPI; ++ps)
                                    raw[ps] = *reinterpret_cast<const uint4*>(
                                        tile + (r0 + ps * C::RPP + rsub) * C::ROW_BYTES + pos_of(cc) * (int)sizeof(ST));
#pragma unroll
                                for (int ps = 0; ps < C::PPI; ++ps) {
                                    float sv[C::VEC];
                                    Store<ST>::unpack(raw[ps], sv);
#pragma unroll
                                    for (int e = 0; e < C::VEC / 2; ++e) {
                                        const float2 s2 = make_float2(sv[2 * e], sv[2 * e + 1]);
                                        if constexpr (RULE == RULE_GDN)
                                            u2[ps] = __ffma2_rn(s2, kw2[0][cc * C::VEC / 2 + e], u2[ps]);
                                        v2[ps] = __ffma2_rn(s2, qw2[0][cc * C::VEC / 2 + e], v2[ps]);
                                    }
                                }
                            }
#pragma unroll
                            for (int ps = 0; ps < C::PPI; ++ps) y[ps] = u2[ps].x + u2[ps].y, z[ps] = v2[ps].x + v2[ps].y;
                        }
                        // the item's state rows are consumed: hand the stage back before the per-row tail
                        __syncwarp();
                        if (lane == 0) mbar_arrive_n(&cempty[cs], C::SUB);
                        if (T > 0) {
                            const float al = meta->alpha[0], be = meta->beta[0];
                            float Y = RULE == RULE_GDN ? reduce_scatter<C::PPI>(y, pg) * g1 : 0.f;
                            float Z = reduce_scatter<C::PPI>(z, pg) * (g1 * al);
                            const int j = j0 + pg * C::RPP + rsub;
                            if (cpr > 0) {
                                if (!have_coef && !(ok = mbar_wait(&cready[hs], hph))) break;
                                have_coef = true;
                                const float2* cf2 = reinterpret_cast<const float2*>(coef);
                                float Y1 = 0.f, Z1 = 0.f;
                                int f = 0;
                                for (; f + 2 <= cpr; f += 2) {
                                    const float2 c0 = cf2[f], c1 = cf2[f + 1];
                                    const float w0 = rec[f * rec_floats + 4 + j], w1 = rec[(f + 1) * rec_floats + 4 + j];
                                    Z = fmaf(c0.y, w0, Z), Z1 = fmaf(c1.y, w1, Z1);
                                    if constexpr (RULE == RULE_GDN) Y = fmaf(c0.x, w0, Y), Y1 = fmaf(c1.x, w1, Y1);
                                }
                                if (f < cpr) {
                                    const float2 c0 = cf2[f];
                                    const float w0 = rec[f * rec_floats + 4 + j];
                                    Z = fmaf(c0.y, w0, Z);
                                    if constexpr (RULE == RULE_GDN) Y = fmaf(c0.x, w0, Y);
                                }
                                Y += Y1, Z += Z1;
                            }
                            const float vj = load_elem(head + p.off_wv, j, in_dt);
                            const float ww = RULE == RULE_GDN ? be * (vj - al * Y) : be * vj;
                            const int64_t oi = ((int64_t)b * p.Hv + h) * p.dv + j;
                            if (out_ok(oi)) store_elem(p.out, oi, out_dt, fmaf(dskip, vj, fmaf(qk, ww, Z)));
                            float* wd = p.ring_rec + (unit_ring + pos0 % L) * rec_floats + 4 + j;
                            if (rec_ok(wd)) *wd = ww;
                        }
                    } else {
                        // Passes of RPP rows: the 2T sums of S0 with the window's keys and queries
                        // are reduce-scattered over a row's lanes and parked in this warp's tile, one
                        // tile row per state row; then one lane per row adds the buffered entries'
                        // terms, runs the window's recursion and stores the row's outputs. The
                        // coefficient table is needed only then.
                        const int np = fold ? C::FPS : C::PPI;                    // passes of this (sub-)item
                        const int ps0 = fold ? (it - bi * C::SUB) * C::FPS : 0;  // its first pass
                        // two passes at a time (np is even): their loads, FMA chains and shuffles interleave
                        for (int q = 0; q < np; q += 2) {
                            float s2[2][C::E];
                            int jr[2];
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                load_state(tile, r0 + (ps0 + q + r) * C::RPP + rsub, s2[r]);
                                jr[r] = j0 + (ps0 + q + r) * C::RPP + rsub;
                            }
                            if (fold) fold_rows(s2, jr);
                            float v[2][C::V];
                            float G1 = g1;  // decay of S0 to token t: g1 prod_{y<t} alpha_y
#pragma unroll
                            for (int t = 0; t < TMAX; ++t) {
                                const float G2 = t < T ? G1 * meta->alpha[t] : 0.f;
#pragma unroll
                                for (int r = 0; r < 2; ++r) {
                                    float2 a2 = make_float2(0.f, 0.f), b2 = a2;
#pragma unroll
                                    for (int e = 0; e < C::E / 2; ++e) {
                                        const float2 x2 = make_float2(s2[r][2 * e], s2[r][2 * e + 1]);
                                        if constexpr (RULE == RULE_GDN) a2 = __ffma2_rn(x2, kw2[t][e], a2);
                                        b2 = __ffma2_rn(x2, qw2[t][e], b2);
                                    }
                                    v[r][t] = (a2.x + a2.y) * G1;
                                    v[r][TMAX + t] = (b2.x + b2.y) * G2;
                                }
                                G1 = G2;
                            }
                            reduce_scatter_values<C::V, C::LPR>(v[0], pg);
                            reduce_scatter_values<C::V, C::LPR>(v[1], pg);
                            if (pg % C::DUP == 0) {
#pragma unroll
                                for (int r = 0; r < 2; ++r)
#pragma unroll
                                    for (int i = 0; i < C::NVL; ++i)
                                        sums[((q + r) * C::RPP + rsub) * (C::V + 1) + held(i)] = v[r][i];
                            }
                        }
                        if (!ok) break;
                        __syncwarp();
                        if (lane == 0) mbar_arrive_n(&cempty[cs], fold ? fw : C::SUB);
                        if (!have_coef && !(ok = mbar_wait(&cready[hs], hph))) break;  // the window's coefficients
                        have_coef = true;
                        if (lane < np * C::RPP) {
                            const int j = j0 + ps0 * C::RPP + lane;
                            float y[TMAX], z[TMAX];
#pragma unroll
                            for (int t = 0; t < TMAX; ++t)
                                y[t] = sums[lane * (C::V + 1) + t], z[t] = sums[lane * (C::V + 1) + TMAX + t];
                            // the buffered entries' terms (coefficients broadcast from the table)
                            for (int f = 0; f < cpr; ++f) {
                                const float wf = rec[f * rec_floats + 4 + j];
                                const float* cf = coef + f * C::V;
#pragma unroll
                                for (int t = 0; t < TMAX; ++t)
                                    y[t] = fmaf(cf[t], wf, y[t]), z[t] = fmaf(cf[TMAX + t], wf, z[t]);
                            }
                            // w_x, then its terms into the later sums of the row (the table holds
                            // zeros where an entry does not precede a token)
                            int ri = pos0 % L;  // ring index of window token x (advanced without a division)
                            float* wcol = p.ring_rec + unit_ring * rec_floats + 4 + j;
#pragma unroll
                            for (int x = 0; x < TMAX; ++x) {
                                if (x < T) {
                                    const float vx = load_elem(head + p.off_wv + x * p.dv * in_sz, j, in_dt);
                                    const float wx = RULE == RULE_GDN ? meta->beta[x] * (vx - meta->alpha[x] * y[x])
                                                                      : meta->beta[x] * vx;
                                    if (rec_ok(wcol + (int64_t)ri * rec_floats)) wcol[(int64_t)ri * rec_floats] = wx;
                                    if (++ri == L) ri = 0;
                                    const float* cx = coef + (cpr + x) * C::V;
#pragma unroll
                                    for (int t = 0; t < TMAX; ++t)
                                        y[t] = fmaf(cx[t], wx, y[t]), z[t] = fmaf(cx[TMAX + t], wx, z[t]);
                                }
                            }
                            const int64_t ob = ((int64_t)b * T * p.Hv + h) * p.dv + j;  // output (t = 0)
                            const int64_t ot = (int64_t)p.Hv * p.dv;                    // next token
#pragma unroll
                            for (int t = 0; t < TMAX; ++t)
                                if (t < T) {
                                    float o = z[t];
                                    if constexpr (RULE == RULE_MAMBA2)
                                        o = fmaf(dskip, load_elem(head + p.off_wv + t * p.dv * in_sz, j, in_dt), o);
                                    if (out_ok(ob + t * ot)) store_elem(p.out, ob + t * ot, out_dt, o);
                                }
                        }
                        __syncwarp();  // the tile is free for the next item
                    }
                }
                if (!ok) break;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hempty[hs]);
        base = (base + nitems) % NCW;
        for (ms += MIXED && fold ? p.mnchunk : p.nchunk; ms >= NS;) ms -= NS, mph ^= 1;
    }
    if (!ok && lane == 0) set_error(p.dev_err, GDN_DEVERR_TIMEOUT);
}

}  // namespace gdn
