/*
 * gdn_oracle.c -- CPU oracle for the GDN recurrent-state decode step and its
 * ReplaySSM mode.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the package smoke check and
 * the benchmark's CPU-baseline leg, never by the product path. It shares no
 * code, header, table or helper with the CUDA library.
 *
 * What it computes, and where that comes from
 *   - The decode rule is the standard gated delta rule. The vLLM PR #52191
 *     summary ("CPU AMX GDN state FP16/BF16 persistence", section 实现拆解,
 *     items 3-4) names the fused sigmoid-gating delta-rule update kernel and
 *     states its numeric contract -- compute in FP32 (here: fp64), keep the
 *     state in a narrow type, round once per write-back -- but not the rule
 *     itself, so the rule is written out as it is usually defined:
 *         alpha = exp(-exp(A_log) * softplus(a + dt_bias)),  beta = sigmoid(b)
 *         k <- k / sqrt(|k|^2 + 1e-6),   q <- q / sqrt(|q|^2 + 1e-6) / sqrt(dk)
 *         S_t = alpha S_{t-1} + beta k (v - alpha S_{t-1}^T k)^T,   o_t = S_t^T q
 *     with value head h reading key head h / (Hv / Hk).
 *   - ReplaySSM (AREX article on ReplaySSM, section "缓存输入而非状态：
 *     checkpoint 每 L 步才更新一次"): keep a checkpoint S0 and the
 *     state-building inputs (k, v, alpha, beta) of the tokens since it; an
 *     output is the readout of the state rebuilt from S0 through those
 *     inputs; the buffer is folded into S0 (the only state write, rounded to
 *     the checkpoint dtype) when it is full; rejected draft tokens are dropped
 *     by moving the buffer pointer back.
 *
 * Everything is fp64, in the order the rule is stated, with no blocking,
 * fusion or algebraic rewriting. The replay functions deliberately rebuild
 * the state from S0 for every output instead of keeping it.
 */
#include "gdn_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ formats */

int orc_dtype_size(int dtype) {
    switch (dtype) {
        case ORC_F32: return 4;
        case ORC_BF16: return 2;
        case ORC_F16: return 2;
        case ORC_F64: return 8;
        default: return 0;
    }
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double f16_bits_to_double(uint16_t h) {
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return s ? -v : v;
}

/* Round x to a binary format with `mbits` fraction bits, minimum normal
 * exponent `emin` and largest finite value `maxfin`, ties to even. Below
 * 2^emin the spacing stays 2^(emin - mbits) (gradual underflow). */
static double round_to_format(double x, int mbits, int emin, double maxfin) {
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    double ax = fabs(x);
    int e = ilogb(ax); /* floor(log2(ax)) */
    if (e < emin) e = emin;
    double quantum = ldexp(1.0, e - mbits);
    double r = nearbyint(ax / quantum) * quantum; /* default mode: ties to even */
    if (r > maxfin) r = INFINITY;
    return copysign(r, x);
}

double orc_round(double x, int dtype) {
    switch (dtype) {
        case ORC_F32: return round_to_format(x, 23, -126, 3.4028234663852886e38);
        case ORC_BF16: return round_to_format(x, 7, -126, 3.3895313892515355e38);
        case ORC_F16: return round_to_format(x, 10, -14, 65504.0);
        default: return x;
    }
}

static uint16_t f16_bits_of(double r) { /* r already on the binary16 grid */
    uint16_t s = signbit(r) ? 0x8000u : 0u;
    double a = fabs(r);
    if (isnan(r)) return 0x7E00u;
    if (isinf(a)) return (uint16_t)(s | 0x7C00u);
    if (a == 0.0) return s;
    int e = ilogb(a);
    if (e < -14) return (uint16_t)(s | (uint16_t)(a / ldexp(1.0, -24)));
    uint16_t frac = (uint16_t)(a / ldexp(1.0, e - 10) - 1024.0);
    return (uint16_t)(s | (uint16_t)((e + 15) << 10) | frac);
}

double orc_load(const void* base, int64_t idx, int dtype) {
    switch (dtype) {
        case ORC_F32: return (double)((const float*)base)[idx];
        case ORC_BF16: return bf16_bits_to_double(((const uint16_t*)base)[idx]);
        case ORC_F16: return f16_bits_to_double(((const uint16_t*)base)[idx]);
        case ORC_F64: return ((const double*)base)[idx];
        default: return NAN;
    }
}

void orc_store(void* base, int64_t idx, int dtype, double x) {
    double r = orc_round(x, dtype);
    switch (dtype) {
        case ORC_F32: ((float*)base)[idx] = (float)r; break; /* exact: r is on the grid */
        case ORC_BF16: {
            float f = (float)r;
            uint32_t u;
            memcpy(&u, &f, 4);
            ((uint16_t*)base)[idx] = isnan(r) ? (uint16_t)0x7FC0u : (uint16_t)(u >> 16);
            break;
        }
        case ORC_F16: ((uint16_t*)base)[idx] = f16_bits_of(r); break;
        case ORC_F64: ((double*)base)[idx] = x; break;
        default: break;
    }
}

void orc_round_array(const double* x, int64_t n, int dtype, void* out) {
    for (int64_t i = 0; i < n; ++i) orc_store(out, i, dtype, x[i]);
}

void orc_load_array(const void* in, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_load(in, i, dtype);
}

static const void* elem_ptr(const void* base, int64_t idx, int dtype) {
    return (const char*)base + idx * orc_dtype_size(dtype);
}

static void load_vec(const void* base, int64_t first, int n, int dtype, double* out) {
    for (int i = 0; i < n; ++i) out[i] = orc_load(base, first + i, dtype);
}

/* ------------------------------------------------------------------ gating */

/* softplus with beta = 1 and the usual linear cut-over above 20. */
static double softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }

void orc_gating(double A_log, double dt_bias, double a, double b, double* alpha, double* beta) {
    *alpha = exp(-exp(A_log) * softplus(a + dt_bias));
    *beta = 1.0 / (1.0 + exp(-b));
}

void orc_l2norm(int n, const double* x, double scale, double* y) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss + 1e-6);
    for (int i = 0; i < n; ++i) y[i] = x[i] * inv * scale;
}

/* ------------------------------------------------------------------ the rule */

/* One gated delta-rule step on an fp64 state S (dk x dv, column j at j*dk).
 * kn is the normalised key. Column by column:
 *   u_j = sum_i S_ij k_i                (S^T k)
 *   S'_ij = alpha S_ij + beta k_i (v_j - alpha u_j) */
static void rule_step(int dk, int dv, double* S, const double* kn, const double* v, double alpha,
                      double beta) {
    for (int j = 0; j < dv; ++j) {
        double* col = S + (int64_t)j * dk;
        double u = 0.0;
        for (int i = 0; i < dk; ++i) u += col[i] * kn[i];
        for (int i = 0; i < dk; ++i) col[i] = alpha * col[i] + beta * kn[i] * (v[j] - alpha * u);
    }
}

/* o_j = sum_i S_ij q_i   (S^T q) */
static void readout(int dk, int dv, const double* S, const double* qn, double* o) {
    for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += S[(int64_t)j * dk + i] * qn[i];
        o[j] = acc;
    }
}

void orc_decode_head(int dk, int dv, void* S, int sdt, const void* q, const void* k, const void* v,
                     int idt, double alpha, double beta, double* out) {
    int64_t n = (int64_t)dk * dv;
    double* Sd = (double*)malloc(sizeof(double) * (size_t)n);
    double* buf = (double*)malloc(sizeof(double) * (size_t)(4 * dk + dv));
    double *kr = buf, *qr = buf + dk, *kn = buf + 2 * dk, *qn = buf + 3 * dk, *vv = buf + 4 * dk;
    load_vec(S, 0, (int)n, sdt, Sd);
    load_vec(k, 0, dk, idt, kr);
    load_vec(q, 0, dk, idt, qr);
    load_vec(v, 0, dv, idt, vv);
    orc_l2norm(dk, kr, 1.0, kn);
    orc_l2norm(dk, qr, 1.0 / sqrt((double)dk), qn);
    rule_step(dk, dv, Sd, kn, vv, alpha, beta);
    readout(dk, dv, Sd, qn, out);
    for (int64_t i = 0; i < n; ++i) orc_store(S, i, sdt, Sd[i]);
    free(buf);
    free(Sd);
}

int orc_decode_step(int B, int Hk, int Hv, int dk, int dv, int64_t num_slots, void* pool, int sdt,
                    const int32_t* slots, const void* q, const void* k, const void* v, const void* a,
                    const void* b, int idt, const float* A_log, const float* dt_bias, double* out,
                    int nthreads) {
    int bad = 0;
    int group = Hv / Hk;
    int64_t units = (int64_t)B * Hv;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 4) reduction(+ : bad) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int bi = (int)(u / Hv), h = (int)(u % Hv), kh = h / group;
        double* o = out + u * dv;
        int32_t slot = slots[bi];
        if (slot < 0 || slot >= num_slots) {
            if (slot >= num_slots) bad += 1;
            for (int j = 0; j < dv; ++j) o[j] = 0.0;
            continue;
        }
        double alpha, beta;
        orc_gating(A_log[h], dt_bias[h], orc_load(a, u, idt), orc_load(b, u, idt), &alpha, &beta);
        void* S = (char*)pool + ((int64_t)slot * Hv + h) * (int64_t)dv * dk * orc_dtype_size(sdt);
        orc_decode_head(dk, dv, S, sdt, elem_ptr(q, ((int64_t)bi * Hk + kh) * dk, idt),
                        elem_ptr(k, ((int64_t)bi * Hk + kh) * dk, idt), elem_ptr(v, u * dv, idt), idt,
                        alpha, beta, o);
    }
    return bad;
}

/* ------------------------------------------------------------------ speculative step */

/* The window's tokens applied in order to the state, each a plain decode step;
 * the copy after token t is the state rounded once, while the recursion goes on
 * from the unrounded state. */
void orc_spec_head(int dk, int dv, int T, const void* S_in, int sdt, void* S_out, const int32_t* write,
                   const void* q, const void* k, const void* v, int idt, const double* alpha,
                   const double* beta, double* out) {
    int64_t n = (int64_t)dk * dv;
    double* Sd = (double*)malloc(sizeof(double) * (size_t)n);
    double* buf = (double*)malloc(sizeof(double) * (size_t)(4 * dk + dv));
    double *kr = buf, *qr = buf + dk, *kn = buf + 2 * dk, *qn = buf + 3 * dk, *vv = buf + 4 * dk;
    load_vec(S_in, 0, (int)n, sdt, Sd);
    for (int t = 0; t < T; ++t) {
        load_vec(k, (int64_t)t * dk, dk, idt, kr);
        load_vec(q, (int64_t)t * dk, dk, idt, qr);
        load_vec(v, (int64_t)t * dv, dv, idt, vv);
        orc_l2norm(dk, kr, 1.0, kn);
        orc_l2norm(dk, qr, 1.0 / sqrt((double)dk), qn);
        rule_step(dk, dv, Sd, kn, vv, alpha[t], beta[t]);
        readout(dk, dv, Sd, qn, out + (int64_t)t * dv);
        if (write[t])
            for (int64_t i = 0; i < n; ++i) orc_store(S_out, (int64_t)t * n + i, sdt, Sd[i]);
    }
    free(buf);
    free(Sd);
}

int orc_spec_step(int B, int T, int Hk, int Hv, int dk, int dv, int64_t num_slots, void* pool, int sdt,
                  const int32_t* src_slots, const int32_t* dst_slots, const void* q, const void* k,
                  const void* v, const void* a, const void* b, int idt, const float* A_log,
                  const float* dt_bias, double* out, int nthreads) {
    int bad = 0;
    int group = Hv / Hk;
    int64_t units = (int64_t)B * Hv, n = (int64_t)dk * dv;
    int esz = orc_dtype_size(sdt);
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 4) reduction(+ : bad) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int bi = (int)(u / Hv), h = (int)(u % Hv), kh = h / group;
        int32_t src = src_slots[bi];
        int ok = src >= 0 && src < num_slots;
        for (int t = 0; t < T; ++t) {
            int32_t d = dst_slots[(int64_t)bi * T + t];
            if (d >= num_slots) ok = 0;
        }
        if (!ok) {
            if (src >= 0) bad += 1; /* the source or a destination out of range */
            for (int t = 0; t < T; ++t)
                for (int j = 0; j < dv; ++j) out[(((int64_t)bi * T + t) * Hv + h) * dv + j] = 0.0;
            continue;
        }
        double* al = (double*)malloc(sizeof(double) * (size_t)(2 * T));
        double* be = al + T;
        int32_t* wr = (int32_t*)malloc(sizeof(int32_t) * (size_t)T);
        double* o = (double*)malloc(sizeof(double) * (size_t)(T * dv));
        char* qs = (char*)malloc((size_t)(2 * T * dk + T * dv) * (size_t)orc_dtype_size(idt));
        char *ks = qs + (size_t)T * dk * orc_dtype_size(idt), *vs = ks + (size_t)T * dk * orc_dtype_size(idt);
        void* copies = malloc((size_t)(T * n) * (size_t)esz);
        int isz = orc_dtype_size(idt);
        for (int t = 0; t < T; ++t) {
            int64_t g = ((int64_t)bi * T + t) * Hv + h;
            orc_gating(A_log[h], dt_bias[h], orc_load(a, g, idt), orc_load(b, g, idt), &al[t], &be[t]);
            wr[t] = dst_slots[(int64_t)bi * T + t] >= 0;
            memcpy(qs + (size_t)t * dk * isz, elem_ptr(q, (((int64_t)bi * T + t) * Hk + kh) * dk, idt), (size_t)dk * isz);
            memcpy(ks + (size_t)t * dk * isz, elem_ptr(k, (((int64_t)bi * T + t) * Hk + kh) * dk, idt), (size_t)dk * isz);
            memcpy(vs + (size_t)t * dv * isz, elem_ptr(v, g * dv, idt), (size_t)dv * isz);
        }
        orc_spec_head(dk, dv, T, (const char*)pool + ((int64_t)src * Hv + h) * n * esz, sdt, copies, wr, qs, ks,
                      vs, idt, al, be, o);
        for (int t = 0; t < T; ++t) {
            for (int j = 0; j < dv; ++j) out[(((int64_t)bi * T + t) * Hv + h) * dv + j] = o[(int64_t)t * dv + j];
            if (wr[t])
                memcpy((char*)pool + ((int64_t)dst_slots[(int64_t)bi * T + t] * Hv + h) * n * esz,
                       (const char*)copies + (size_t)t * n * esz, (size_t)n * esz);
        }
        free(copies);
        free(qs);
        free(o);
        free(wr);
        free(al);
    }
    return bad;
}

/* ------------------------------------------------------------------ prefill */

/* The tokens one decode step at a time (vLLM PR #52191 summary, 实现拆解 items
 * 3-4: the chunked kernel keeps the state in an FP32 buffer within a chunk and
 * writes it back, rounded to the state dtype, at the end of every chunk). */
void orc_prefill_head(int dk, int dv, int T, void* S, int sdt, const void* q, const void* k, const void* v, int idt,
                      const double* alpha, const double* beta, int interval, double* out) {
    int64_t n = (int64_t)dk * dv;
    double* Sd = (double*)malloc(sizeof(double) * (size_t)n);
    double* buf = (double*)malloc(sizeof(double) * (size_t)(4 * dk + dv));
    double *kr = buf, *qr = buf + dk, *kn = buf + 2 * dk, *qn = buf + 3 * dk, *vv = buf + 4 * dk;
    load_vec(S, 0, (int)n, sdt, Sd);
    for (int t = 0; t < T; ++t) {
        load_vec(k, (int64_t)t * dk, dk, idt, kr);
        load_vec(q, (int64_t)t * dk, dk, idt, qr);
        load_vec(v, (int64_t)t * dv, dv, idt, vv);
        orc_l2norm(dk, kr, 1.0, kn);
        orc_l2norm(dk, qr, 1.0 / sqrt((double)dk), qn);
        rule_step(dk, dv, Sd, kn, vv, alpha[t], beta[t]);
        readout(dk, dv, Sd, qn, out + (int64_t)t * dv);
        if ((t + 1) % interval == 0 || t == T - 1) { /* chunk write-back: round, continue from the stored state */
            for (int64_t i = 0; i < n; ++i) orc_store(S, i, sdt, Sd[i]);
            load_vec(S, 0, (int)n, sdt, Sd);
        }
    }
    free(buf);
    free(Sd);
}

int orc_prefill(int B, int Hk, int Hv, int dk, int dv, int64_t num_slots, void* pool, int sdt,
                const int32_t* slots, const int32_t* cu_seqlens, const void* q, const void* k, const void* v,
                const void* a, const void* b, int idt, const float* A_log, const float* dt_bias, int interval,
                double* out, int nthreads) {
    int bad = 0;
    int group = Hv / Hk;
    int64_t units = (int64_t)B * Hv;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int bi = (int)(u / Hv), h = (int)(u % Hv), kh = h / group;
        int t0 = cu_seqlens[bi], T = cu_seqlens[bi + 1] - t0;
        int32_t slot = slots[bi];
        if (slot < 0 || slot >= num_slots) {
            if (slot >= num_slots) bad += 1;
            for (int t = 0; t < T; ++t)
                for (int j = 0; j < dv; ++j) out[((int64_t)(t0 + t) * Hv + h) * dv + j] = 0.0;
            continue;
        }
        if (T <= 0) continue;
        double* al = (double*)malloc(sizeof(double) * (size_t)(2 * T));
        double* be = al + T;
        double* o = (double*)malloc(sizeof(double) * (size_t)T * dv);
        char* qs = (char*)malloc((size_t)T * dk * orc_dtype_size(idt));
        char* ks = (char*)malloc((size_t)T * dk * orc_dtype_size(idt));
        char* vs = (char*)malloc((size_t)T * dv * orc_dtype_size(idt));
        int isz = orc_dtype_size(idt);
        for (int t = 0; t < T; ++t) { /* gather this head's rows of the sequence */
            int64_t tok = t0 + t;
            memcpy(qs + (size_t)t * dk * isz, elem_ptr(q, (tok * Hk + kh) * dk, idt), (size_t)dk * isz);
            memcpy(ks + (size_t)t * dk * isz, elem_ptr(k, (tok * Hk + kh) * dk, idt), (size_t)dk * isz);
            memcpy(vs + (size_t)t * dv * isz, elem_ptr(v, (tok * Hv + h) * dv, idt), (size_t)dv * isz);
            orc_gating(A_log[h], dt_bias[h], orc_load(a, tok * Hv + h, idt), orc_load(b, tok * Hv + h, idt), &al[t],
                       &be[t]);
        }
        void* S = (char*)pool + ((int64_t)slot * Hv + h) * (int64_t)dv * dk * orc_dtype_size(sdt);
        orc_prefill_head(dk, dv, T, S, sdt, qs, ks, vs, idt, al, be, interval, o);
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < dv; ++j) out[((int64_t)(t0 + t) * Hv + h) * dv + j] = o[(int64_t)t * dv + j];
        free(vs);
        free(ks);
        free(qs);
        free(o);
        free(al);
    }
    return bad;
}

/* ------------------------------------------------------------------ ReplaySSM */

/* The fp64 state after the first n buffered entries, rebuilt from S0 by
 * applying the rule once per entry, in arrival order. */
static void rebuild(int dk, int dv, const void* S0, int sdt, int n, const void* ek, const void* ev,
                    int idt, const double* ea, const double* eb, double* S) {
    double* tmp = (double*)malloc(sizeof(double) * (size_t)(2 * dk + dv));
    double *kr = tmp, *kn = tmp + dk, *vv = tmp + 2 * dk;
    load_vec(S0, 0, dk * dv, sdt, S);
    for (int e = 0; e < n; ++e) {
        load_vec(ek, (int64_t)e * dk, dk, idt, kr);
        load_vec(ev, (int64_t)e * dv, dv, idt, vv);
        orc_l2norm(dk, kr, 1.0, kn);
        rule_step(dk, dv, S, kn, vv, ea[e], eb[e]);
    }
    free(tmp);
}

/* Fold every buffered entry into the checkpoint: S0 <- round(S_pos-1). */
static void fold(int dk, int dv, void* S0, int sdt, const void* ek, const void* ev, int idt,
                 const double* ea, const double* eb, int32_t* meta) {
    int64_t n = (int64_t)dk * dv;
    double* S = (double*)malloc(sizeof(double) * (size_t)n);
    rebuild(dk, dv, S0, sdt, meta[0], ek, ev, idt, ea, eb, S);
    for (int64_t i = 0; i < n; ++i) orc_store(S0, i, sdt, S[i]);
    free(S);
    meta[0] = 0;       /* count */
    meta[2] = meta[1]; /* ckpt_pos = pos */
}

int orc_replay_window(int dk, int dv, int L, void* S0, int sdt, void* ek, void* ev, int idt,
                      double* ealpha, double* ebeta, int32_t* meta, int T, const void* q,
                      const void* k, const void* v, const double* a, const double* b, double A_log,
                      double dt_bias, double* out) {
    if (T < 1 || T > L) return -1;
    if (meta[0] < 0 || meta[0] > L || meta[1] - meta[2] != meta[0]) return -2;
    /* The ring has room for L entries: fold first when T more would not fit. */
    if (meta[0] + T > L) fold(dk, dv, S0, sdt, ek, ev, idt, ealpha, ebeta, meta);
    int c = meta[0];
    int isz = orc_dtype_size(idt);
    for (int t = 0; t < T; ++t) { /* append the window's inputs */
        memcpy((char*)ek + (int64_t)(c + t) * dk * isz, (const char*)k + (int64_t)t * dk * isz,
               (size_t)dk * isz);
        memcpy((char*)ev + (int64_t)(c + t) * dv * isz, (const char*)v + (int64_t)t * dv * isz,
               (size_t)dv * isz);
        orc_gating(A_log, dt_bias, a[t], b[t], &ealpha[c + t], &ebeta[c + t]);
    }
    int64_t n = (int64_t)dk * dv;
    double* S = (double*)malloc(sizeof(double) * (size_t)n);
    double* qv = (double*)malloc(sizeof(double) * (size_t)(2 * dk));
    for (int t = 0; t < T; ++t) { /* output t reads the state after window token t */
        rebuild(dk, dv, S0, sdt, c + t + 1, ek, ev, idt, ealpha, ebeta, S);
        load_vec(q, (int64_t)t * dk, dk, idt, qv);
        orc_l2norm(dk, qv, 1.0 / sqrt((double)dk), qv + dk);
        readout(dk, dv, S, qv + dk, out + (int64_t)t * dv);
    }
    free(qv);
    free(S);
    meta[0] = c + T;
    meta[1] += T;
    return 0;
}

/* ------------------------------------------------------------------ ReplaySSM, two checkpoints */

/* A high-precision checkpoint M for the recurrence and a low-precision copy Rd
 * for reading (AREX ReplaySSM article, section "缓存输入而非状态", its
 * paragraph on precision: the recurrence runs on the high-precision
 * checkpoint, reads go to the low-precision copy). Folding re-runs every
 * buffered entry's raw inputs (k, v, alpha, beta) through the rule starting
 * from M -- each prediction S^T k comes from the master's own state -- rounds
 * the result to mdt and stores it; then Rd is rewritten as that stored master
 * rounded to rdt. The read copy plays no part in a fold: the master evolves as
 * a single-checkpoint replay in mdt would. */
static void fold2(int dk, int dv, void* M, int mdt, void* Rd, int rdt, const void* ek, const void* ev, int idt,
                  const double* ea, const double* eb, int32_t* meta) {
    int64_t n = (int64_t)dk * dv;
    double* Sm = (double*)malloc(sizeof(double) * (size_t)n);
    rebuild(dk, dv, M, mdt, meta[0], ek, ev, idt, ea, eb, Sm);
    for (int64_t i = 0; i < n; ++i) {
        double m = orc_round(Sm[i], mdt);
        orc_store(M, i, mdt, m);
        orc_store(Rd, i, rdt, m);
    }
    free(Sm);
    meta[0] = 0;
    meta[2] = meta[1];
}

int orc_replay2_window(int dk, int dv, int L, void* M, int mdt, void* Rd, int rdt, void* ek, void* ev, int idt,
                       double* ealpha, double* ebeta, int32_t* meta, int T, const void* q, const void* k,
                       const void* v, const double* a, const double* b, double A_log, double dt_bias, double* out) {
    if (T < 1 || T > L) return -1;
    if (meta[0] < 0 || meta[0] > L || meta[1] - meta[2] != meta[0]) return -2;
    if (meta[0] + T > L) fold2(dk, dv, M, mdt, Rd, rdt, ek, ev, idt, ealpha, ebeta, meta);
    /* outputs read the copy: the single-checkpoint window on Rd, which it never folds */
    return orc_replay_window(dk, dv, L, Rd, rdt, ek, ev, idt, ealpha, ebeta, meta, T, q, k, v, a, b, A_log,
                             dt_bias, out);
}

int orc_replay2_flush(int dk, int dv, int L, void* M, int mdt, void* Rd, int rdt, const void* ek, const void* ev,
                      int idt, const double* ealpha, const double* ebeta, int32_t* meta, int force) {
    if (meta[0] < 0 || meta[0] > L || meta[1] - meta[2] != meta[0]) return -2;
    if (force ? meta[0] > 0 : meta[0] == L) fold2(dk, dv, M, mdt, Rd, rdt, ek, ev, idt, ealpha, ebeta, meta);
    return 0;
}

int orc_replay_flush(int dk, int dv, int L, void* S0, int sdt, const void* ek, const void* ev,
                     int idt, const double* ealpha, const double* ebeta, int32_t* meta, int force) {
    if (meta[0] < 0 || meta[0] > L || meta[1] - meta[2] != meta[0]) return -2;
    if (force ? meta[0] > 0 : meta[0] == L) fold(dk, dv, S0, sdt, ek, ev, idt, ealpha, ebeta, meta);
    return 0;
}

int orc_replay_rollback(int32_t* meta, int T, int accepted) {
    if (accepted < 0 || accepted > T - 1) return -3;
    int r = T - 1 - accepted; /* rejected drafts */
    if (meta[0] - r < 0) return -2;
    meta[0] -= r;
    meta[1] -= r;
    return 0;
}
