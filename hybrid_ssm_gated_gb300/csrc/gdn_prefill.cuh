// gdn_prefill.cuh -- prefill of the gated delta rule with a rounded state
// write-back per chunk (gdn_prefill), token by token on the FP32 pipe: the
// kernel for FP32 states (exact FP32 arithmetic) and for shapes the chunked
// tensor-core kernel (gdn_prefill_tc.cuh: 16-bit states, dk = 128, dv a
// multiple of 128) does not take.
//
// Semantics (vLLM PR #52191 summary, section 实现拆解 items 3-4: the chunked
// kernel works on an FP32 copy of the state within a chunk and writes it back,
// rounded to the state dtype, at the end of each chunk): the tokens of a
// sequence run through the rule in order; the state is rounded to its storage
// dtype after every `interval` tokens and after the last one, and only the
// final state is stored. Outputs come from the unrounded FP32 state.
//
// Kernel shape. One CTA per (sequence, value head, block of 128 state rows);
// each of its 8 warps keeps 16 rows of S in FP32 registers for the whole
// sequence, so the state is read once and written once. Tokens are staged in
// chunks of PF_TC through shared memory with 16-byte asynchronous copies,
// double buffered: while a chunk is processed the next one is in flight.
// Per chunk, the warps first normalise its keys and queries and convert its
// values (one token per warp at a time) into FP32 tables, so the row loop only
// reads them; then every warp runs the chunk's tokens over its rows: two dot
// products per row, whose 2 x PASSES partial sums over the LPR lanes of a row
// group are finished by one reduce-scatter (lane g of the group then owns one
// sum), the correction and output of one row per lane pair, the corrections
// broadcast back, and the rank-one update. A lane keeps the row of pass
// p ^ (g >> 1) in its register slot p: partners in the reduce-scatter's pass
// levels then hold each other's values in the same slots, so those levels
// need no per-lane selects. Outputs go to a shared-memory tile
// and leave, coalesced and in the output dtype, once per chunk. Rows are
// independent given the token, so warps never wait for one another inside a
// chunk. The step is bound by FP32 arithmetic (7 dk dv flops per token and
// head), not by memory.
// The decay is applied lazily: the registers hold S / sigma, sigma being the
// product of the decays since the last rescale (uniform over the CTA), so a
// token's update is one fused multiply-add per element, S/sigma' += k
// (delta / sigma'), instead of a multiply and an add. The registers are
// rescaled when sigma falls below 2^-32 (or a decay underflows), at every
// write-back (where the rounding happens on sigma S) and at the end.
#pragma once

#include "gdn_device.cuh"
#include "gdn_io.cuh"

namespace gdn {

struct PrefillArgs {
    void* pool;
    const int32_t* slots;
    const int32_t* cu_seqlens;  // [B + 1] token offsets
    const void* q;              // [total][Hk][dk]
    const void* k;
    const void* v;  // [total][Hv][dv]
    const void* a;  // [total][Hv]
    const void* b;
    const float* A_log;
    const float* dt_bias;
    void* out;  // [total][Hv][dv]
    int32_t* dev_err;
    int64_t num_slots;
    int B, Hk, Hv, dv, total, interval;
    int in_dtype, out_dtype;
    int row_blocks;  // ceil(dv / PF_ROWS)
    float q_scale;
    // dynamic shared memory layout, bytes
    int raw_bytes;  // one staged chunk: q, k [TC][dk] and v [TC][PF_ROWS] in the input dtype
    int off_kqn, off_qk, off_vf, off_of, off_gates;
};

#ifndef GDN_PREFILL_WARPS
#define GDN_PREFILL_WARPS 8  // a CTA covers 128 state rows: the per-chunk staging and normalisation serve more rows
#endif
constexpr int PF_WARPS = GDN_PREFILL_WARPS;
constexpr int PF_ROWS = 16 * PF_WARPS;  // state rows per CTA, 16 per warp
#ifndef GDN_PREFILL_TOKENS
#define GDN_PREFILL_TOKENS 16
#endif
constexpr int PF_TC = GDN_PREFILL_TOKENS;  // tokens per staged chunk
#ifndef GDN_PREFILL_MIN_BLOCKS
#define GDN_PREFILL_MIN_BLOCKS 2  // CTAs per SM the register budget must allow (128 registers a thread)
#endif

template <typename ST, int DK>
struct PrefillCfg {
    static constexpr int VEC = Store<ST>::VEC;  // state elements per 16 bytes
    static constexpr int E = 16;                // state elements per lane per row
    static constexpr int NC = E / VEC;
    static constexpr int LPR = DK / E;       // lanes per row
    static constexpr int RPP = 32 / LPR;     // rows per warp pass
    static constexpr int PASSES = 16 / RPP;  // passes covering a warp's 16 rows
    static constexpr int ROW_BYTES = DK * (int)sizeof(ST);
    static_assert(DK % E == 0 && 16 % RPP == 0 && 2 * PASSES == LPR, "unsupported dk");
};

template <typename ST, int DK, int IO = IO_ANY>
__global__ void __launch_bounds__(PF_WARPS * 32, GDN_PREFILL_MIN_BLOCKS) prefill_kernel(const PrefillArgs p) {
    using C = PrefillCfg<ST, DK>;
    const int in_dt = io_in<IO>(p.in_dtype), out_dt = io_out<IO>(p.out_dtype);
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = blockIdx.x % p.row_blocks;
    const int unit = blockIdx.x / p.row_blocks;
    const int bseq = unit / p.Hv, h = unit - bseq * p.Hv, kh = h / (p.Hv / p.Hk);
    const int slot = p.slots[bseq];
    const int t0 = p.cu_seqlens[bseq], t1 = p.cu_seqlens[bseq + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.total) {
        if (threadIdx.x == 0 && rb == 0 && h == 0) set_error(p.dev_err, GDN_DEVERR_SEQLEN);
        return;
    }
    const int T = t1 - t0;
    // array extents in bytes, for the bounds-checking build
    const int osz = dtype_size(out_dt);
    const uint64_t ext_out = (uint64_t)p.total * p.Hv * p.dv * osz;
    const uint64_t ext_state = (uint64_t)p.num_slots * p.Hv * p.dv * C::ROW_BYTES;
    const uint64_t ext_qk = (uint64_t)p.total * p.Hk * DK * dtype_size(in_dt);
    const uint64_t ext_v = (uint64_t)p.total * p.Hv * p.dv * dtype_size(in_dt);
    const int row0 = rb * PF_ROWS;
    const int nrows = min(PF_ROWS, p.dv - row0);  // a multiple of 16
    if (slot < 0 || slot >= p.num_slots) {
        if (slot >= p.num_slots && threadIdx.x == 0 && rb == 0) set_error(p.dev_err, GDN_DEVERR_SLOT);
        for (int i = threadIdx.x; i < T * nrows; i += blockDim.x) {
            const int t = i / nrows, r = i - t * nrows;
            const int64_t oi = ((int64_t)(t0 + t) * p.Hv + h) * p.dv + row0 + r;
            if (in_bounds(static_cast<char*>(p.out) + oi * osz, osz, p.out, ext_out, p.dev_err))
                store_elem(p.out, oi, out_dt, 0.f);
        }
        return;
    }
    if (T == 0) return;

    const int isz = dtype_size(in_dt);
    auto raw = [&](int c) { return smem + (c & 1) * p.raw_bytes; };  // staged chunk c
    // [TC][2][DK] normalised k, q, each row in lane order: the 4-element piece e4 of a lane's run cc sits at
    // ((cc * VEC / 4 + e4) * LPR + pg) * 4, so the row loop's 16-byte reads are consecutive across lanes
    float* kqn = reinterpret_cast<float*>(smem + p.off_kqn);
    float* qkb = reinterpret_cast<float*>(smem + p.off_qk);      // [TC] q.k
    float* vf = reinterpret_cast<float*>(smem + p.off_vf);       // [TC][PF_ROWS] v in FP32
    float* of = reinterpret_cast<float*>(smem + p.off_of);       // [TC][PF_ROWS] outputs
    float4* gts = reinterpret_cast<float4*>(smem + p.off_gates);  // [2][TC] (alpha, beta, 1 / alpha, 0)
    const int qbytes = DK * isz, vbytes = nrows * isz;
    const int nchunks = (T + PF_TC - 1) / PF_TC;

    // stage chunk c (its q, k rows and this block's slice of v) into buffer c & 1
    auto stage = [&](int c) {
        unsigned char* dst = raw(c);
        const int n = min(PF_TC, T - c * PF_TC);
        const int per_tok = 2 * (qbytes / 16) + vbytes / 16;  // 16-byte pieces per token
        for (int i = threadIdx.x; i < n * per_tok; i += blockDim.x) {
            const int t = i / per_tok, x = i - t * per_tok;
            const int64_t tok = t0 + c * PF_TC + t;
            const char* src;
            unsigned char* d;
            bool ok_;
            if (x < 2 * (qbytes / 16)) {
                const int which = x / (qbytes / 16), piece = x - which * (qbytes / 16);
                src = static_cast<const char*>(which ? p.k : p.q) + (tok * p.Hk + kh) * qbytes + piece * 16;
                d = dst + (which * PF_TC + t) * qbytes + piece * 16;
                ok_ = in_bounds(src, 16, which ? p.k : p.q, ext_qk, p.dev_err);
            } else {
                const int piece = x - 2 * (qbytes / 16);
                src = static_cast<const char*>(p.v) + ((tok * p.Hv + h) * p.dv + row0) * isz + piece * 16;
                d = dst + 2 * PF_TC * qbytes + t * PF_ROWS * isz + piece * 16;
                ok_ = in_bounds(src, 16, p.v, ext_v, p.dev_err);
            }
            if (ok_) cp_async16(d, src);
        }
        cp_async_commit();
    };
    // gates of chunk c, one thread per token
    auto gate = [&](int c, float& al, float& be) {  // and 1 / alpha, below
        const int t = c * PF_TC + threadIdx.x;
        al = 0.f, be = 0.f;
        if (threadIdx.x < PF_TC && t < T) {
            const int64_t gi = (int64_t)(t0 + t) * p.Hv + h;
            gates(p.A_log[h], p.dt_bias[h], load_elem(p.a, gi, in_dt), load_elem(p.b, gi, in_dt), al, be);
        }
    };

    // this lane's rows and element positions
    const int pg = lane % C::LPR, rsub = lane / C::LPR;
    const int pq_bits = pg >> 1;  // register slot s holds the row of pass s ^ pq_bits
    const int wrow = warp * 16;               // the warp's first row within the block
    const bool wvalid = wrow < nrows;         // whole warps are valid or not (nrows % 16 == 0)
    auto pos_of = [&](int cc) { return (cc * C::LPR + pg) * C::VEC; };
    unsigned char* gstate =
        static_cast<unsigned char*>(p.pool) + (((int64_t)slot * p.Hv + h) * p.dv + row0) * C::ROW_BYTES;

    stage(0);
    {
        float al, be;
        gate(0, al, be);
        if (threadIdx.x < PF_TC) gts[threadIdx.x] = make_float4(al, be, 1.f / al, 0.f);
    }
    float S[C::PASSES][C::E];  // the state divided by sig
    float sig = 1.f, isig = 1.f;  // sig and 1 / sig (a product of the decays' reciprocals, re-taken per chunk)
    int until_wb = p.interval;  // tokens until the next write-back
    if (wvalid) {
#pragma unroll
        for (int ps = 0; ps < C::PASSES; ++ps) {
            const int r = wrow + (ps ^ pq_bits) * C::RPP + rsub;
#pragma unroll
            for (int cc = 0; cc < C::NC; ++cc)
                load_row_run<ST, C::VEC>(gstate + (int64_t)r * C::ROW_BYTES, pos_of(cc), S[ps] + cc * C::VEC);
        }
    }

    for (int c = 0; c < nchunks; ++c) {
        const int n = min(PF_TC, T - c * PF_TC);
        float nal = 0.f, nbe = 0.f;
        if (c + 1 < nchunks) {
            stage(c + 1);
            gate(c + 1, nal, nbe);
            cp_async_wait<1>();  // chunk c has landed (this thread's copies)
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // every thread's copies of chunk c are visible

        // normalised keys and queries of the chunk, one token per warp at a time
        const unsigned char* src = raw(c);
        for (int t = warp; t < n; t += PF_WARPS) {
            float kx[DK / 32], qx[DK / 32];
            float ssk = 0.f, ssq = 0.f;
#pragma unroll
            for (int e = 0; e < DK / 32; ++e) {
                kx[e] = load_elem(src + (PF_TC + t) * qbytes, lane + 32 * e, in_dt);
                qx[e] = load_elem(src + t * qbytes, lane + 32 * e, in_dt);
                ssk = fmaf(kx[e], kx[e], ssk), ssq = fmaf(qx[e], qx[e], ssq);
            }
            const float ik = rsqrtf(group_sum<32>(ssk) + 1e-6f);
            const float iq = rsqrtf(group_sum<32>(ssq) + 1e-6f) * p.q_scale;
            float kq = 0.f;
#pragma unroll
            for (int e = 0; e < DK / 32; ++e) {
                kx[e] *= ik, qx[e] *= iq;
                kq = fmaf(kx[e], qx[e], kq);
                const int i = lane + 32 * e, run = i / C::VEC, within = i - run * C::VEC;
                const int slot = (((run / C::LPR) * (C::VEC / 4) + within / 4) * C::LPR + run % C::LPR) * 4 + within % 4;
                kqn[(t * 2) * DK + slot] = kx[e];
                kqn[(t * 2 + 1) * DK + slot] = qx[e];
            }
            kq = group_sum<32>(kq);
            if (lane == 0) qkb[t] = kq;
            for (int r = lane; r < nrows; r += 32)
                vf[t * PF_ROWS + r] = load_elem(src + 2 * PF_TC * qbytes + t * PF_ROWS * isz, r, in_dt);
        }
        __syncthreads();  // the table is complete

        if (wvalid) {
            const float4* g = gts + (c & 1) * PF_TC;
            isig = __frcp_rn(sig);  // re-taken once per chunk, so the products drift by at most 16 roundings
            for (int t = 0; t < n; ++t) {
                float2 k2[C::E / 2], q2[C::E / 2];
#pragma unroll
                for (int cc = 0; cc < C::NC; ++cc) {
#pragma unroll
                    for (int e = 0; e < C::VEC; e += 4) {
                        const int slot = ((cc * (C::VEC / 4) + e / 4) * C::LPR + pg) * 4;
                        const float4 kv = *reinterpret_cast<const float4*>(kqn + (t * 2) * DK + slot);
                        const float4 qv = *reinterpret_cast<const float4*>(kqn + (t * 2 + 1) * DK + slot);
                        const int i = (cc * C::VEC + e) / 2;
                        k2[i] = make_float2(kv.x, kv.y), k2[i + 1] = make_float2(kv.z, kv.w);
                        q2[i] = make_float2(qv.x, qv.y), q2[i + 1] = make_float2(qv.z, qv.w);
                    }
                }
                const float4 gab = g[t];
                const float al = gab.x, be = gab.y, ial = gab.z, qk = qkb[t];
                // partial sums: x[2 s] = S[:, row in slot s] . k, x[2 s + 1] = . q
                float x[2 * C::PASSES];
#pragma unroll
                for (int ps = 0; ps < C::PASSES; ++ps) {
                    float2 u2 = make_float2(0.f, 0.f), p2 = u2;
#pragma unroll
                    for (int e = 0; e < C::E / 2; ++e) {
                        const float2 s2 = make_float2(S[ps][2 * e], S[ps][2 * e + 1]);
                        u2 = __ffma2_rn(s2, k2[e], u2);
                        p2 = __ffma2_rn(s2, q2[e], p2);
                    }
                    x[2 * ps] = u2.x + u2.y, x[2 * ps + 1] = p2.x + p2.y;
                }
                // Reduce-scatter over the row group. Slot s of lane g holds pass s ^ (g >> 1), so across a
                // pass level (lane bit h >= 2) partner g ^ h keeps in slot i + h what this lane keeps in
                // slot i: every lane sends its upper half and adds into its lower half. The last level
                // (the k/q bit) is the usual one. Lane pg then owns (pass pg / 2, k or q); a lane pair
                // finishes the row of its pass.
                float mine;
                {
#pragma unroll
                    for (int half = C::PASSES; half >= 2; half >>= 1)
#pragma unroll
                        for (int i = 0; i < half; ++i) x[i] += __shfl_xor_sync(FULL_MASK, x[i + half], half);
                    const bool odd = (pg & 1) != 0;
                    mine = (odd ? x[1] : x[0]) + __shfl_xor_sync(FULL_MASK, odd ? x[0] : x[1], 1);
                }
                const float other = __shfl_xor_sync(FULL_MASK, mine, 1);
                const float u = sig * ((pg & 1) ? other : mine), pq = sig * ((pg & 1) ? mine : other);
                const int rme = wrow + (pg >> 1) * C::RPP + rsub;
                const float delta_me = be * (vf[t * PF_ROWS + rme] - al * u);
                if ((pg & 1) == 0) of[t * PF_ROWS + rme] = fmaf(al, pq, qk * delta_me);
                // S_t = alpha S_{t-1} + k delta^T with S_{t-1} = sig S: the registers keep S_t / (sig alpha)
                float sn = sig * al, inv = isig * ial;
                if (sn < 0x1p-32f) {  // uniform over the CTA: fold the decay into the registers
#pragma unroll
                    for (int ps = 0; ps < C::PASSES; ++ps)
#pragma unroll
                        for (int e = 0; e < C::E; ++e) S[ps][e] *= sn;
                    sn = 1.f, inv = 1.f;
                }
#pragma unroll
                for (int ps = 0; ps < C::PASSES; ++ps) {
                    const float delta = __shfl_sync(FULL_MASK, delta_me, 2 * (ps ^ pq_bits), C::LPR) * inv;
                    const float2 d2 = make_float2(delta, delta);
#pragma unroll
                    for (int e = 0; e < C::E / 2; ++e) {
                        const float2 r2 = __ffma2_rn(k2[e], d2, make_float2(S[ps][2 * e], S[ps][2 * e + 1]));
                        S[ps][2 * e] = r2.x, S[ps][2 * e + 1] = r2.y;
                    }
                }
                sig = sn, isig = inv;
                // chunk write-back: the state continues as stored (sig S rounded), except after the last
                // token, which is stored below
                if (--until_wb == 0) {
                    until_wb = p.interval;
                    if (c * PF_TC + t + 1 < T) {  // the registers become the stored state exactly
#pragma unroll
                        for (int ps = 0; ps < C::PASSES; ++ps)
#pragma unroll
                            for (int cc = 0; cc < C::NC; ++cc) {
                                float* x = S[ps] + cc * C::VEC;
#pragma unroll
                                for (int e = 0; e < C::VEC; ++e) x[e] *= sig;
                                if constexpr (!std::is_same<ST, float>::value) Store<ST>::unpack(Store<ST>::pack(x), x);
                            }
                        sig = 1.f, isig = 1.f;
                    }
                }
            }
        }
        if (c + 1 < nchunks && threadIdx.x < PF_TC)
            gts[((c + 1) & 1) * PF_TC + threadIdx.x] = make_float4(nal, nbe, 1.f / nal, 0.f);
        __syncthreads();  // buffer c & 1 and the tables are free again; the output tile is complete
        // the chunk's outputs, coalesced along the rows of each token, four at a time
        const int q4 = nrows / 4;
        for (int i = threadIdx.x; i < n * q4; i += blockDim.x) {
            const int t = i / q4, r = (i - t * q4) * 4;
            const float4 o = *reinterpret_cast<const float4*>(of + t * PF_ROWS + r);
            const int64_t oi = ((int64_t)(t0 + c * PF_TC + t) * p.Hv + h) * p.dv + row0 + r;
            if (!in_bounds(static_cast<char*>(p.out) + oi * osz, 4 * osz, p.out, ext_out, p.dev_err)) continue;
            if (out_dt == GDN_F32) {
                *reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi) = o;
            } else {
                const float ov[4] = {o.x, o.y, o.z, o.w};
                uint32_t w[2];
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    w[e] = out_dt == GDN_BF16 ? pack_bf16x2(ov[2 * e], ov[2 * e + 1])
                                                   : pack_f16x2(ov[2 * e], ov[2 * e + 1]);
                *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + oi) = make_uint2(w[0], w[1]);
            }
        }
    }

    if (wvalid) {
#pragma unroll
        for (int ps = 0; ps < C::PASSES; ++ps) {
            const int r = wrow + (ps ^ pq_bits) * C::RPP + rsub;
#pragma unroll
            for (int cc = 0; cc < C::NC; ++cc) {
#pragma unroll
                for (int e = 0; e < C::VEC; ++e) S[ps][cc * C::VEC + e] *= sig;
                if (in_bounds(gstate + (int64_t)r * C::ROW_BYTES + pos_of(cc) * (int)sizeof(ST), C::VEC * sizeof(ST),
                              p.pool, ext_state, p.dev_err))
                    store_row_run<ST, C::VEC>(gstate + (int64_t)r * C::ROW_BYTES, pos_of(cc), S[ps] + cc * C::VEC);
            }
        }
    }
}

}  // namespace gdn
