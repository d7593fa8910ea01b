// gdn_replay_rows.cuh -- ReplaySSM with one checkpoint: the standard decode
// step, the speculative verify window and the fold (flush), one warp per
// (sequence, value head) unit and one state row per lane.
//
// The arithmetic is in gdn_replay_common.cuh (AREX article on ReplaySSM,
// section "缓存输入而非状态"): outputs from one pass over S0 plus the ring's w
// terms, the window's own recursion per row, the ring folded into S0 when
// full. The layout removes every cross-lane reduction from the pass over S0:
//  - a batch is 64 state rows, lane l owning rows l and 32 + l; the rows
//    stream through shared memory in 64-byte column chunks (64 rows x 64 B =
//    4 KB a stage, copied with cp.async by the whole warp, coalesced, into a
//    layout whose 16-byte pieces are XOR-swizzled by row so that the lanes'
//    row reads hit distinct banks), double-buffered: measured, more stages
//    (fewer warps) were slower, the kernel being bound by its warps' issue
//    rather than by the bytes in flight;
//  - the window's normalised keys and queries sit in shared memory and are
//    read as broadcasts, four elements at a time, shared by the lane's two
//    rows; each lane accumulates its rows' 2T dot products (T for Mamba2) in
//    registers over the chunks, so when a batch's last chunk is done every
//    lane holds whole row sums and runs the rows' tails at once. Windows of 4
//    and 8 tokens over a 16-bit checkpoint take these dot products on the
//    tensor cores instead (warp-level TF32 MMA, the checkpoint exact in TF32,
//    the vectors split hi + lo), and turn the fragments into row sums through
//    the stage at a batch's end (measured: bf16 windows of four 195 -> 185 us
//    at B = 256; an FP32 checkpoint, needing three products, was slower);
//  - a fold applies the buffered entries to each chunk as it arrives (raw
//    keys broadcast from shared memory, the entry's scale -- decay and 1/|k| --
//    and the row's w in registers), stores it rounded and goes on from the
//    stored value;
//  - a batch's 64 columns of every buffered entry's w are staged with its
//    first chunk; a lane reads only the columns of its own rows;
//  - units are taken from per-round lists, fold units first
//    (gdn_replay_common.cuh).
// The two-checkpoint mode runs in gdn_replay_producer.cuh: its fold runs the
// rule sequentially on whole master rows, which column chunks do not hold.
#pragma once

#include "gdn_replay_common.cuh"

namespace gdn {

template <typename ST, int DK, int TMAX, int RULE>
struct RowsCfg {
    static constexpr int SZ = (int)sizeof(ST);
    static constexpr int CB = 64;                   // bytes of a row chunk
    static constexpr int CE = CB / SZ;              // elements of a row chunk
    static constexpr int NCH = DK * SZ / CB;        // chunks of a row
    static constexpr int STAGE = 64 * CB;           // a stage: 64 rows x one chunk
    static constexpr int NS = 2;                    // stages: one in flight while the other is read
    static constexpr int NK = RULE == RULE_GDN ? 2 : 1;  // dot products per window token
    static constexpr int VPR = NK * TMAX;           // row sums per row
    static constexpr int CW = 2 * TMAX;             // floats per coefficient-table entry
    static_assert(DK * SZ % CB == 0 && CE % 4 == 0, "unsupported dk");
};

// One warp's shared memory: the copy stages; the window's normalised keys and queries [TMAX][DK]
// each; the buffered keys [L][DK] as stored (raw, in the activation dtype: their 1/|k| joins the
// scalars they are multiplied by), and record headers {alpha, beta, 1/|k|, n} [L]; the current
// batch's 64 columns of every buffered entry's w [L][64]; the coefficient table [L + TMAX][CW].
struct RowsLayout {
    int stage, kwin, qwin, keys, hdr, wcol, coef, bytes;
};

template <typename ST, int DK, int TMAX, int RULE>
__host__ __device__ constexpr RowsLayout replay_rows_layout(int L, int in_sz) {
    using C = RowsCfg<ST, DK, TMAX, RULE>;
    RowsLayout w{};
    w.stage = 0;
    w.kwin = C::NS * C::STAGE;
    w.qwin = w.kwin + TMAX * DK * 4;
    w.keys = w.qwin + TMAX * DK * 4;
    w.hdr = w.keys + L * DK * in_sz;
    w.wcol = w.hdr + L * 16;
    w.coef = w.wcol + L * 64 * 4;
    w.bytes = align_up(w.coef + (L + TMAX) * C::CW * 4, 16);
    return w;
}

// Swizzled position of 16-byte piece p (of 4) of row r in a stage: pieces of rows 2m and 2m + 1
// shift by m mod 4, so that the 8 lanes of a shared-memory phase, reading piece p of 8 consecutive
// rows, cover all 32 banks.
__device__ __forceinline__ int rows_piece(int r, int p) { return r * 64 + ((p ^ ((r >> 1) & 3)) << 4); }

// Four consecutive state elements of type T from 16-bit or fp32 storage at byte `src` (shared memory).
template <typename T>
__device__ __forceinline__ void ld4(const unsigned char* src, float* x) {
    if constexpr (sizeof(T) == 4) {
        const float4 f = *reinterpret_cast<const float4*>(src);
        x[0] = f.x, x[1] = f.y, x[2] = f.z, x[3] = f.w;
    } else {
        const uint2 r = *reinterpret_cast<const uint2*>(src);
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            x[0] = bf16_lo(r.x), x[1] = bf16_hi(r.x), x[2] = bf16_lo(r.y), x[3] = bf16_hi(r.y);
        } else {
            float2 f = f16x2_to_f2(r.x);
            x[0] = f.x, x[1] = f.y;
            f = f16x2_to_f2(r.y);
            x[2] = f.x, x[3] = f.y;
        }
    }
}

// x as a TF32 pair hi + lo, each rounded to nearest: hi keeps the top 11 significand bits, lo the next
// 11, so that hi b + lo b and hi b' products keep FP32-level accuracy.
__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    hi = tf32_rna(x);
    lo = tf32_rna(x - __uint_as_float(hi));
}

// d += a b on the tensor cores, one warp: a 16 x 8 (row fragment), b 8 x 8 (column fragment), d 16 x 8,
// TF32 operands, FP32 accumulation (PTX ISA, mma.m16n8k8 fragment layouts for .tf32).
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <typename ST, int DK, int TMAX, int NW, int RULE = RULE_GDN, int IO = IO_ANY>
__global__ void __launch_bounds__(NW * 32, 1) replay_rows_kernel(const ReplayArgs p) {
    using C = RowsCfg<ST, DK, TMAX, RULE>;
    constexpr bool GDN = RULE == RULE_GDN;
    constexpr int SZ = C::SZ, CE = C::CE, NCH = C::NCH, NS = C::NS;
    constexpr int SROW = DK * SZ;
    constexpr int EPL = DK / 32;  // key elements per lane in the warp-wide dot products
    // windows of 4 and 8 tokens over a 16-bit checkpoint take the pass's dot products on the tensor
    // cores (MMA_NT tiles of 8 window vectors); single tokens (2 sums a row, Mamba2 1) and FP32
    // checkpoints (whose TF32 split needs three products) measured faster on the FMA pipe
    constexpr bool MMA = TMAX >= 4 && sizeof(ST) == 2;
    constexpr int MMA_NT = (C::VPR + 7) / 8;
    constexpr int KS = CE / 8;  // k-steps of 8 in a chunk
    const int in_dt = io_in<IO>(p.in_dtype), out_dt = io_out<IO>(p.out_dtype);
    const int in_sz = dtype_size(in_dt);
    // dynamic shared memory: the round's counters and unit lists, then one region per warp
    extern __shared__ __align__(128) unsigned char smem[];
    int* ctr = reinterpret_cast<int*>(smem);              // next list index; folds listed; others listed
    int4* lfold = reinterpret_cast<int4*>(smem + 16);     // {unit, slot, pos, ckpt_pos} of the fold units
    int4* lrest = lfold + REPLAY_ROUND;                   // ... and of the others
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const RowsLayout lay = replay_rows_layout<ST, DK, TMAX, RULE>(p.L, in_sz);
    unsigned char* region = smem + REPLAY_SMEM_HEAD + warp * lay.bytes;
    unsigned char* stages = region + lay.stage;
    float* kwin = reinterpret_cast<float*>(region + lay.kwin);  // [TMAX][DK] normalised window keys
    float* qwin = reinterpret_cast<float*>(region + lay.qwin);  // [TMAX][DK] normalised, scaled queries
    unsigned char* keys = region + lay.keys;                    // [L][DK] buffered keys, raw
    const float4* hdr = reinterpret_cast<const float4*>(region + lay.hdr);
    float* wcol = reinterpret_cast<float*>(region + lay.wcol);  // [L][64] w of the batch's columns
    float* coef = reinterpret_cast<float*>(region + lay.coef);  // [entry][CW]: S^T k at [t], S^T q at [TMAX + t]

    const int total = p.B * p.Hv;
    const int T = p.T, L = p.L;
    const int group = p.Hv / p.Hk;
    const int rec_floats = 4 + p.dv;
    const int kbytes = DK * in_sz;
    // array extents in bytes: every copy and store checks against them in bounds-checking builds
    const uint64_t cells = (uint64_t)p.num_slots * p.Hv;
    const uint64_t ext_ckpt = cells * p.dv * DK * SZ, ext_rk = cells * p.L * kbytes;
    const uint64_t ext_rv = cells * p.L * p.dv * in_sz, ext_rec = cells * p.L * rec_floats * 4, ext_ptr = cells * 4;
    const uint64_t ext_out = (uint64_t)p.B * p.T * p.Hv * p.dv * dtype_size(out_dt);
    auto out_ok = [&](int64_t i) { return in_bounds(static_cast<char*>(p.out) + i * dtype_size(out_dt),
                                                    dtype_size(out_dt), p.out, ext_out, p.dev_err); };
    const int nbat = (p.dv + 63) / 64;  // batches of 64 rows (the last may have 32)
    const int Q = nbat * NCH;           // sub-batches (batch, chunk) of a unit
    int dso[8];                         // the lane's stage pieces: row (lane / 4) + 8 m, piece lane % 4
#pragma unroll
    for (int m = 0; m < 8; ++m) dso[m] = rows_piece((lane >> 2) + 8 * m, lane & 3);

    // the CTA's units, in rounds of listed units, fold units first (REPLAY_ROUND, gdn_replay_common.cuh)
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
        float kr[TMAX][EPL], qr[TMAX][EPL];  // lane's EPL consecutive elements of each token's key, query
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) kr[t][e] = 0.f, qr[t][e] = 0.f;
            if (t < T) {
                const int64_t row = (((int64_t)b * T + t) * p.Hk + kh) * DK + lane * EPL;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    kr[t][e] = load_elem(p.k, row + e, in_dt);
                    qr[t][e] = load_elem(p.q, row + e, in_dt);
                }
            }
        }
        float ga = 0.f, gb = 0.f;  // lane t < T: token t's raw gate inputs (a and b; Mamba2: dt)
        if (lane < T) {
            const int64_t gi = ((int64_t)b * T + lane) * p.Hv + h;
            ga = load_elem(p.a, gi, in_dt);
            if constexpr (GDN) gb = load_elem(p.b, gi, in_dt);
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
        unsigned char* s0 = static_cast<unsigned char*>(p.ckpt) + uidx * p.dv * SROW;

        // ------------------------------------------------ the copy pipeline
        // sub-batch q = (batch q / NCH, chunk q % NCH): rows 64 * batch .. + 63 (those below dv), bytes
        // [64 chunk, 64 chunk + 64) of each; lane l copies pieces l + 32 m, m < 8 (row (l + 32 m) / 4,
        // piece l % 4). The unit's first sub-batch also stages batch 0's 64 columns of every buffered
        // entry's w (later batches' go out after the previous batch's rows are done), and
        // stages the buffered raw keys and record headers. The columns, keys and headers are read by
        // every lane after a warp barrier.
        auto issue_w = [&](int bq) {
            const int npc = (p.dv - bq * 64 < 64 ? p.dv - bq * 64 : 64) / 4;  // 16-byte pieces of an entry
            for (int i = lane; i < count * npc; i += 32) {
                const int f = i / npc, pc = i - f * npc;
                const float* src = rec + ring_at(f) * rec_floats + 4 + bq * 64 + pc * 4;
                if (in_bounds(src, 16, p.ring_rec, ext_rec, p.dev_err)) cp_async_piece<16>(wcol + f * 64 + pc * 4, src);
            }
        };
        auto issue = [&](int q) {
            if (q < Q) {
                const int bq = q / NCH, ch = q - bq * NCH;
                unsigned char* st = stages + (q % NS) * C::STAGE;
                const int rows = p.dv - bq * 64 < 64 ? p.dv - bq * 64 : 64;
                const unsigned char* src = s0 + (int64_t)bq * 64 * SROW + ch * C::CB + (lane & 3) * 16;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int r = (lane >> 2) + 8 * m;
                    if (r < rows && in_bounds(src + (int64_t)r * SROW, 16, p.ckpt, ext_ckpt, p.dev_err))
                        cp_async_piece<16>(st + dso[m], src + (int64_t)r * SROW);
                }
                if (q == 0) {
                    for (int f = lane; f < count; f += 32) {
                        const float* src = rec + ring_at(f) * rec_floats;
                        if (in_bounds(src, 16, p.ring_rec, ext_rec, p.dev_err))
                            cp_async_piece<16>(region + lay.hdr + f * 16, src);
                    }
                    const int kp = kbytes / 16;
                    for (int i = lane; i < count * kp; i += 32) {
                        const int f = i / kp, k = i - f * kp;
                        const unsigned char* src =
                            static_cast<const unsigned char*>(p.ring_k) + (unit_ring + ring_at(f)) * kbytes + k * 16;
                        if (in_bounds(src, 16, p.ring_k, ext_rk, p.dev_err))
                            cp_async_piece<16>(keys + f * kbytes + k * 16, src);
                    }
                    issue_w(0);
                }
            }
            cp_async_commit();
        };
#pragma unroll
        for (int q = 0; q < NS - 1; ++q) issue(q);

        // ------------------------------------------------ window: gates, normalised keys and queries
        float al_l = 1.f, be_l = 0.f;  // lane t < T: token t's gates
        if (lane < T) {
            if constexpr (GDN) {
                gates(p.A_log[h], p.dt_bias[h], ga, gb, al_l, be_l);
            } else {
                const float x = ga + p.dt_bias[h];
                be_l = x > 20.f ? x : log1pf(expf(x));
                al_l = expf(-expf(p.A_log[h]) * be_l);
            }
        }
        float aw[TMAX], bw[TMAX];  // every token's gates, in every lane
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
            aw[t] = __shfl_sync(FULL_MASK, al_l, t), bw[t] = __shfl_sync(FULL_MASK, be_l, t);
            if (t >= T) aw[t] = 1.f, bw[t] = 0.f;
        }
        float ik_l = 1.f;  // lane t < T: token t's inverse key norm
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
            if constexpr (GDN) {
                float ssk = 0.f, ssq = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) ssk = fmaf(kr[t][e], kr[t][e], ssk), ssq = fmaf(qr[t][e], qr[t][e], ssq);
                const float ik = rsqrtf(group_sum<32>(ssk) + 1e-6f);
                const float iq = rsqrtf(group_sum<32>(ssq) + 1e-6f) * p.q_scale;
                if (lane == t) ik_l = ik;
#pragma unroll
                for (int e = 0; e < EPL; ++e) kr[t][e] *= ik, qr[t][e] *= iq;
            }
#pragma unroll
            for (int e = 0; e < EPL; ++e) kwin[t * DK + lane * EPL + e] = kr[t][e], qwin[t * DK + lane * EPL + e] = qr[t][e];
        }
        // prefix decays of the window: Pk[t] = prod_{y<t} alpha_y, Pq[t] = Pk[t] alpha_t
        float Pk[TMAX], Pq[TMAX];
        {
            float run = 1.f;
#pragma unroll
            for (int t = 0; t < TMAX; ++t) Pk[t] = run, run *= aw[t], Pq[t] = run;
        }

        const bool ring_hi = L > 32;
        float R = 1.f, R_hi = 1.f, gring = 1.f, fsc = 0.f, fsc_hi = 0.f;
        auto entry_val = [&](float lo, float hv, int f) {
            return f < 32 ? __shfl_sync(FULL_MASK, lo, f) : __shfl_sync(FULL_MASK, hv, f - 32);
        };
        const int64_t out_b = ((int64_t)b * T * p.Hv + h) * p.dv;  // output (t = 0, j = 0)
        const int64_t out_t = (int64_t)p.Hv * p.dv;                // next token
        float2 acc[2][C::VPR];  // the lane's two rows' partial sums: S0^T k_t at [t], S0^T q_t at [NK - 1 ...]
        float dm[4][MMA ? MMA_NT : 1][4];  // tensor-core sums: m-tile (16 rows), n-tile, fragment
        float vx_pre[2][TMAX];  // the window's values at the lane's two columns of the current batch

        // the unit's first stage, with the buffered keys and headers
        cp_async_wait<NS - 2>();
        __syncwarp();
        // ring decays by suffix products over the staged alphas: R(f) = prod_{f<g<count} alpha_g
        // (lane f; entries 32 + f in the _hi values), their product, and a fold's scale of the raw key
        // k_f, R(f) / |k_f|
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
        const float ghi = ring_hi ? __shfl_sync(FULL_MASK, suf_hi, 0) : 1.f;
        suf *= ghi;
        gring = __shfl_sync(FULL_MASK, suf, 0);
        R = __shfl_down_sync(FULL_MASK, suf, 1);
        R_hi = ring_hi ? __shfl_down_sync(FULL_MASK, suf_hi, 1) : 1.f;
        if (lane == 31) R = ghi, R_hi = 1.f;
        fsc = lane < count ? R * hdr[lane].z : 0.f;
        fsc_hi = ring_hi && lane + 32 < count ? R_hi * hdr[lane + 32].z : 0.f;
        if (T > 0) {
            // ------------------------------ coefficient table
            // entry x (ring entry f = x < cpr, else window token s = x - cpr) against every window
            // token t: coef[x][t] = (k_x.k_t) times the decay from x to token t's prediction,
            // coef[x][TMAX + t] = (k_x.q_t) times the decay from x to token t's output; zero where x
            // does not precede t. First the dot products, NE entries at a time (the lanes split the
            // key dimension; one reduce-scatter leaves lane i with value i of the NE * VPR), then the
            // decays, lane x scaling entry x.
            constexpr int NE = 32 / C::VPR > 0 ? 32 / C::VPR : 1;
            constexpr int VV = NE * C::VPR;
            constexpr int HV = VV >= 32 ? VV / 32 : 1;  // sums a lane holds
            constexpr int DV = VV >= 32 ? 1 : 32 / VV;  // lanes holding the same sum
            const int J = cpr + T;
            for (int x0 = 0; x0 < J; x0 += NE) {
                float v[VV];
#pragma unroll
                for (int i = 0; i < NE; ++i) {
                    const int x = x0 + i < J ? x0 + i : J - 1;
                    float kx[EPL];
                    if (x < cpr) {
                        // the raw key, normalised here
                        const float ik = hdr[x].z;
                        if constexpr (EPL % 4 == 0) {
#pragma unroll
                            for (int e = 0; e < EPL; e += 4) load_run<4>(keys + x * kbytes, lane * EPL + e, in_dt, kx + e);
                        } else {
#pragma unroll
                            for (int e = 0; e < EPL; ++e) kx[e] = load_elem(keys + x * kbytes, lane * EPL + e, in_dt);
                        }
#pragma unroll
                        for (int e = 0; e < EPL; ++e) kx[e] *= ik;
                    } else {
#pragma unroll
                        for (int e = 0; e < EPL; ++e) kx[e] = kwin[(x - cpr) * DK + lane * EPL + e];
                    }
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        float sk = 0.f, sq = 0.f;
#pragma unroll
                        for (int e = 0; e < EPL; ++e) {
                            if constexpr (GDN) sk = fmaf(kx[e], kr[t][e], sk);
                            sq = fmaf(kx[e], qr[t][e], sq);
                        }
                        if constexpr (GDN) {
                            v[i * C::VPR + t] = sk;
                            v[i * C::VPR + TMAX + t] = sq;
                        } else {
                            v[i * C::VPR + t] = sq;
                        }
                    }
                }
                reduce_scatter_values<VV, 32>(v, lane);
                if (lane % DV == 0) {
#pragma unroll
                    for (int hv = 0; hv < HV; ++hv) {
                        const int idx = lane / DV * HV + hv;  // entry x0 + idx / VPR, value idx % VPR
                        const int i = idx / C::VPR, vv = idx - i * C::VPR;
                        if (x0 + i < J) coef[(x0 + i) * C::CW + (GDN ? vv : TMAX + vv)] = v[hv];
                    }
                }
            }
            __syncwarp();
            for (int x = lane; x < J; x += 32) {
                const bool ring = x < cpr;
                const int sw = x - cpr;
                const float Rx = x < 32 ? R : R_hi;  // lane x: R(x); lane x - 32: R(x) for x >= 32
                float* cx = coef + x * C::CW;
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                    // the window tokens' decays after the entry (all of them after a ring entry), up to
                    // token t's prediction (y < t) or output (y <= t)
                    float dk = ring ? Rx : 1.f, dq = dk;
#pragma unroll
                    for (int y = 0; y < TMAX; ++y) {
                        if ((ring || y > sw) && y < t) dk *= aw[y];
                        if ((ring || y > sw) && y <= t) dq *= aw[y];
                    }
                    const bool live_k = t < T && (ring || t > sw), live_q = t < T && (ring || t >= sw);
                    if constexpr (GDN) cx[t] = live_k ? cx[t] * dk : 0.f;
                    cx[TMAX + t] = live_q ? cx[TMAX + t] * dq : 0.f;
                }
            }
            __syncwarp();
        }

        for (int q = 0; q < Q; ++q) {
            __syncwarp();
            issue(q + NS - 1);
            cp_async_wait<NS - 1>();
            const int bq = q / NCH, ch = q - bq * NCH;
            const int j0 = bq * 64;
            const bool row2 = j0 + 32 < p.dv;  // the batch has a second row per lane
            if (ch == 0) {
                // a new batch: zero the row sums; the window's values at the lane's columns
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int v = 0; v < C::VPR; ++v) acc[r][v] = make_float2(0.f, 0.f);
#pragma unroll
                for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                    for (int nt = 0; nt < (MMA ? MMA_NT : 1); ++nt)
#pragma unroll
                        for (int i = 0; i < 4; ++i) dm[mt][nt][i] = 0.f;
                if (T > 0) {
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int x = 0; x < TMAX; ++x) {
                            const int j = j0 + 32 * r + lane;
                            vx_pre[r][x] = x < T && (r == 0 || row2)
                                               ? load_elem(p.v, (((int64_t)b * T + x) * p.Hv + h) * p.dv + j, in_dt)
                                               : 0.f;
                        }
                }
            }
            const unsigned char* stg = stages + (q % NS) * C::STAGE;
            const int e0 = ch * CE;  // the chunk's first element
            // a batch's w columns go out after the previous batch's rows are done (one buffer), so a fold
            // (on its first chunk) and a one-chunk batch (on its rows) drain the pipeline to have them
            if (bq > 0 && ((fold && ch == 0) || (NCH == 1 && T > 0))) {
                cp_async_wait<0>();
                __syncwarp();
            }
            if (fold) {
                // S0 <- G S0 + sum_f A(f) k_f w_f^T on the lane's rows of this chunk (k_f normalised),
                // stored rounded; the dot products below then read the stored values
                float s[2][CE];
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int g4 = 0; g4 < CE / 4; ++g4)
                        ld4<ST>(stg + rows_piece(32 * r + lane, g4 * 4 * SZ / 16) + (g4 * 4 * SZ) % 16, s[r] + 4 * g4);
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int e = 0; e < CE; ++e) s[r][e] *= gring;
                for (int f = 0; f < count; ++f) {
                    const float sc = entry_val(fsc, fsc_hi, f);
                    const float2 w0 = make_float2(sc * wcol[f * 64 + lane], sc * wcol[f * 64 + lane]);
                    const float w1s = row2 ? sc * wcol[f * 64 + 32 + lane] : 0.f;
                    const float2 w1 = make_float2(w1s, w1s);
#pragma unroll
                    for (int g4 = 0; g4 < CE / 4; ++g4) {
                        float kf[4];  // the raw key's elements (its 1/|k| is in the scale)
                        load_run<4>(keys + f * kbytes, e0 + 4 * g4, in_dt, kf);
                        const float2 k01 = make_float2(kf[0], kf[1]), k23 = make_float2(kf[2], kf[3]);
                        float2 a = make_float2(s[0][4 * g4], s[0][4 * g4 + 1]), c = make_float2(s[0][4 * g4 + 2], s[0][4 * g4 + 3]);
                        a = __ffma2_rn(k01, w0, a), c = __ffma2_rn(k23, w0, c);
                        s[0][4 * g4] = a.x, s[0][4 * g4 + 1] = a.y, s[0][4 * g4 + 2] = c.x, s[0][4 * g4 + 3] = c.y;
                        a = make_float2(s[1][4 * g4], s[1][4 * g4 + 1]), c = make_float2(s[1][4 * g4 + 2], s[1][4 * g4 + 3]);
                        a = __ffma2_rn(k01, w1, a), c = __ffma2_rn(k23, w1, c);
                        s[1][4 * g4] = a.x, s[1][4 * g4 + 1] = a.y, s[1][4 * g4 + 2] = c.x, s[1][4 * g4 + 3] = c.y;
                    }
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (r == 1 && !row2) break;
                    unsigned char* dst = s0 + (int64_t)(j0 + 32 * r + lane) * SROW;
#pragma unroll
                    for (int v = 0; v < CE; v += 16 / SZ)
                        if (in_bounds(dst + (e0 + v) * SZ, 16, p.ckpt, ext_ckpt, p.dev_err))
                            st_state<ST, 16 / SZ>(dst, e0 + v, s[r] + v);
                }
                if (MMA && T > 0) {
                    // the stored (rounded) rows back into the stage, where the tensor-core pass reads them
                    unsigned char* st = stages + (q % NS) * C::STAGE;
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int pc = 0; pc < 4; ++pc)
                            *reinterpret_cast<uint4*>(st + rows_piece(32 * r + lane, pc)) =
                                Store<ST>::pack(s[r] + pc * (16 / SZ));
                } else if (T > 0) {
#pragma unroll
                    for (int g4 = 0; g4 < CE / 4; ++g4) {
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) {
                            const float4 qv = *reinterpret_cast<const float4*>(qwin + t * DK + e0 + 4 * g4);
                            const float2 q01 = make_float2(qv.x, qv.y), q23 = make_float2(qv.z, qv.w);
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const float2 s01 = make_float2(s[r][4 * g4], s[r][4 * g4 + 1]);
                                const float2 s23 = make_float2(s[r][4 * g4 + 2], s[r][4 * g4 + 3]);
                                float2& aq = acc[r][(GDN ? TMAX : 0) + t];
                                aq = __ffma2_rn(s01, q01, aq), aq = __ffma2_rn(s23, q23, aq);
                            }
                            if constexpr (GDN) {
                                const float4 kv = *reinterpret_cast<const float4*>(kwin + t * DK + e0 + 4 * g4);
                                const float2 k01 = make_float2(kv.x, kv.y), k23 = make_float2(kv.z, kv.w);
#pragma unroll
                                for (int r = 0; r < 2; ++r) {
                                    const float2 s01 = make_float2(s[r][4 * g4], s[r][4 * g4 + 1]);
                                    const float2 s23 = make_float2(s[r][4 * g4 + 2], s[r][4 * g4 + 3]);
                                    acc[r][t] = __ffma2_rn(s01, k01, acc[r][t]), acc[r][t] = __ffma2_rn(s23, k23, acc[r][t]);
                                }
                            }
                        }
                    }
                }
            } else if (!MMA && T > 0) {
                // the lane's rows' dot products with the window's keys and queries, four elements at a time
#pragma unroll
                for (int g4 = 0; g4 < CE / 4; ++g4) {
                    float s[2][4];
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        ld4<ST>(stg + rows_piece(32 * r + lane, g4 * 4 * SZ / 16) + (g4 * 4 * SZ) % 16, s[r]);
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        if (t < T) {
                            const float4 qv = *reinterpret_cast<const float4*>(qwin + t * DK + e0 + 4 * g4);
                            const float2 q01 = make_float2(qv.x, qv.y), q23 = make_float2(qv.z, qv.w);
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                float2& aq = acc[r][(GDN ? TMAX : 0) + t];
                                aq = __ffma2_rn(make_float2(s[r][0], s[r][1]), q01, aq);
                                aq = __ffma2_rn(make_float2(s[r][2], s[r][3]), q23, aq);
                            }
                            if constexpr (GDN) {
                                const float4 kv = *reinterpret_cast<const float4*>(kwin + t * DK + e0 + 4 * g4);
                                const float2 k01 = make_float2(kv.x, kv.y), k23 = make_float2(kv.z, kv.w);
#pragma unroll
                                for (int r = 0; r < 2; ++r) {
                                    acc[r][t] = __ffma2_rn(make_float2(s[r][0], s[r][1]), k01, acc[r][t]);
                                    acc[r][t] = __ffma2_rn(make_float2(s[r][2], s[r][3]), k23, acc[r][t]);
                                }
                            }
                        }
                    }
                }
            }
            if (MMA && T > 0) {
                // The chunk's rows against the window's vectors on the tensor cores: D[row][n] +=
                // S0[row][.] . vec_n[.], rows as M (4 tiles of 16), the chunk's CE columns as K, vector n
                // (GDN: keys of tokens 0..TMAX-1, then queries; Mamba2: queries) as N. The columns are
                // permuted within the chunk so that a lane's A and B elements are one 16-byte piece: lane
                // (g, c) takes columns (CE / 4) c + 2 s and + 1 as its k = c and c + 4 of k-step s.
                // 16-bit checkpoint values are exact in TF32; the vectors are split into TF32 hi + lo.
                if (fold) __syncwarp();  // every lane's folded rows are in the stage
                const int g = lane >> 2, c = lane & 3;
                const int rows = p.dv - j0 < 64 ? p.dv - j0 : 64;
                uint32_t bh[MMA ? MMA_NT : 1][2 * KS], bl[MMA ? MMA_NT : 1][2 * KS];
#pragma unroll
                for (int nt = 0; nt < (MMA ? MMA_NT : 1); ++nt) {
                    const int n = 8 * nt + g;
                    float bv[2 * KS];
#pragma unroll
                    for (int i = 0; i < 2 * KS; i += 4) {
                        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (n < C::VPR)
                            f = *reinterpret_cast<const float4*>((GDN ? kwin : qwin) + n * DK + e0 + (CE / 4) * c + i);
                        bv[i] = f.x, bv[i + 1] = f.y, bv[i + 2] = f.z, bv[i + 3] = f.w;
                    }
#pragma unroll
                    for (int i = 0; i < 2 * KS; ++i) split_tf32(bv[i], bh[nt][i], bl[nt][i]);
                }
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    if (16 * mt >= rows) break;
                    float a0[2 * KS], a1[2 * KS];  // rows 16 mt + g and + 8, the lane's piece
                    Store<ST>::unpack(*reinterpret_cast<const uint4*>(stg + rows_piece(16 * mt + g, c)), a0);
                    Store<ST>::unpack(*reinterpret_cast<const uint4*>(stg + rows_piece(16 * mt + g + 8, c)), a1);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const uint32_t x0 = __float_as_uint(a0[2 * ks]), x1 = __float_as_uint(a1[2 * ks]);
                        const uint32_t x2 = __float_as_uint(a0[2 * ks + 1]), x3 = __float_as_uint(a1[2 * ks + 1]);
#pragma unroll
                        for (int nt = 0; nt < (MMA ? MMA_NT : 1); ++nt) {
                            mma_tf32(dm[mt][nt], x0, x1, x2, x3, bl[nt][2 * ks], bl[nt][2 * ks + 1]);
                            mma_tf32(dm[mt][nt], x0, x1, x2, x3, bh[nt][2 * ks], bh[nt][2 * ks + 1]);
                        }
                    }
                }
                if (ch == NCH - 1) {
                    // the batch's sums from the fragments (lane (g, c): rows g and g + 8 of each m-tile,
                    // vectors 2c and 2c + 1 of each n-tile) to the row layout (lane l: rows l and 32 + l,
                    // every vector) through the stage, which the pass no longer reads
                    __syncwarp();
                    unsigned char* scr = stages + (q % NS) * C::STAGE;
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt) {
                        if (16 * mt >= rows) break;
#pragma unroll
                        for (int nt = 0; nt < (MMA ? MMA_NT : 1); ++nt)
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const int n = 8 * nt + 2 * c;
                                *reinterpret_cast<float2*>(scr + rows_piece(16 * mt + g + 8 * hh, n >> 2) + (n & 3) * 4) =
                                    make_float2(dm[mt][nt][2 * hh], dm[mt][nt][2 * hh + 1]);
                            }
                    }
                    __syncwarp();
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int pc = 0; pc < (C::VPR + 3) / 4; ++pc) {
                            const float4 f = *reinterpret_cast<const float4*>(scr + rows_piece(32 * r + lane, pc));
                            const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                if (4 * pc + i < C::VPR) acc[r][4 * pc + i] = make_float2(fv[i], 0.f);
                        }
                }
            }
            if (ch != NCH - 1) continue;
            // ---------------------------------------- the batch's last chunk: lane l finishes rows j0 + l, j0 + 32 + l
            __syncwarp();  // every lane's copies of the batch's columns have landed
            if (T > 0) {
                const float G1 = fold ? 1.f : gring;  // decay of S0 to the window's first token
                const float dskip = RULE == RULE_MAMBA2 ? p.D[h] : 0.f;
                // both rows at once, so that each coefficient is loaded once (a batch of 32 rows leaves
                // the second row's values unused)
                float y[2][TMAX], z[2][TMAX];
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        y[r][t] = GDN ? (acc[r][t].x + acc[r][t].y) * (G1 * Pk[t]) : 0.f;
                        const float2 aq = acc[r][(GDN ? TMAX : 0) + t];
                        z[r][t] = (aq.x + aq.y) * (G1 * Pq[t]);
                    }
                // the buffered entries' terms (their w staged with the batch)
                for (int f = 0; f < cpr; ++f) {
                    const float w0 = wcol[f * 64 + lane], w1 = wcol[f * 64 + 32 + lane];
                    const float* cf = coef + f * C::CW;
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) {
                        if constexpr (GDN) {
                            const float ck = cf[t];
                            y[0][t] = fmaf(ck, w0, y[0][t]), y[1][t] = fmaf(ck, w1, y[1][t]);
                        }
                        const float cq = cf[TMAX + t];
                        z[0][t] = fmaf(cq, w0, z[0][t]), z[1][t] = fmaf(cq, w1, z[1][t]);
                    }
                }
                // the window: w_x, then its terms in the later sums of the rows
                int ri = pos0 % L;
#pragma unroll
                for (int x = 0; x < TMAX; ++x) {
                    if (x < T) {
                        float wx[2];
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            wx[r] = GDN ? bw[x] * (vx_pre[r][x] - aw[x] * y[r][x]) : bw[x] * vx_pre[r][x];
                            float* dst = rec + ri * rec_floats + 4 + j0 + 32 * r + lane;
                            if ((r == 0 || row2) && in_bounds(dst, 4, p.ring_rec, ext_rec, p.dev_err)) *dst = wx[r];
                        }
                        ri = ri + 1 == L ? 0 : ri + 1;
                        const float* cx = coef + (cpr + x) * C::CW;
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) {
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                if constexpr (GDN) y[r][t] = fmaf(cx[t], wx[r], y[r][t]);
                                z[r][t] = fmaf(cx[TMAX + t], wx[r], z[r][t]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (r == 1 && !row2) break;
                    const int j = j0 + 32 * r + lane;
#pragma unroll
                    for (int t = 0; t < TMAX; ++t)
                        if (t < T) {
                            float o = z[r][t];
                            if constexpr (RULE == RULE_MAMBA2) o = fmaf(dskip, vx_pre[r][t], o);
                            if (out_ok(out_b + t * out_t + j)) store_elem(p.out, out_b + t * out_t + j, out_dt, o);
                        }
                }
            }
            // the next batch's w columns, once every lane is done with this batch's
            if (bq + 1 < nbat) {
                __syncwarp();
                issue_w(bq + 1);
                cp_async_commit();
            }
        }
        cp_async_wait<0>();
        __syncwarp();  // every lane is done with the staged keys and headers before the next unit's copies

        // ------------------------------------------------ append the window; move the pointers
        // (after the pass: a fold reads the old entries' records until its last chunk)
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
