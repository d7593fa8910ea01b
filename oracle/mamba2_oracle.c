/*
 * mamba2_oracle.c -- CPU oracle for the Mamba2 selective-state decode step and
 * its ReplaySSM mode.
 *
 * TEST INFRASTRUCTURE ONLY (see mamba2_oracle.h). It uses the storage-format
 * routines of gdn_oracle.c (rounding and loading of fp32/bf16/fp16/fp64
 * values) and nothing of the CUDA library.
 *
 * What it computes
 *   - The decode step is the Mamba2 recurrence as it is usually written for
 *     one decode token (dt passed through softplus with a per-head bias, a
 *     scalar decay per head, a rank-one input term delta x B^T, readout by C
 *     and the skip term D x). The AREX article on ReplaySSM (section
 *     "每步写回完整循环状态") gives only its state shape (nheads, d, n) and
 *     the readout vector C; the rule is the standard one.
 *   - ReplaySSM (same article, section "缓存输入而非状态：checkpoint 每 L
 *     步才更新一次"): the ring keeps the state-building inputs (B, x and the
 *     gates); C is read from the current activations only. An output is the
 *     readout of the state rebuilt from S0 through every buffered input; the
 *     ring is folded into S0 when it is full.
 * Everything is fp64, in the order the rule is stated. The replay functions
 * rebuild the state from S0 for every output instead of keeping it.
 */
#include "mamba2_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "gdn_oracle.h"

static void load_n(const void* base, int64_t first, int n, int dtype, double* out) {
    for (int i = 0; i < n; ++i) out[i] = orc_load(base, first + i, dtype);
}

static const void* at(const void* base, int64_t idx, int dtype) {
    return (const char*)base + idx * orc_dtype_size(dtype);
}

static double softplus_m2(double x) { return x > 20.0 ? x : log1p(exp(x)); }

void orc_m2_gating(double A_log, double dt_bias, double dt, double* alpha, double* delta) {
    *delta = softplus_m2(dt + dt_bias);
    *alpha = exp(-exp(A_log) * *delta);
}

/* S[p][i] <- alpha S[p][i] + delta x[p] B[i] */
static void m2_update(int N, int P, double* S, const double* Bv, const double* x, double alpha, double delta) {
    for (int p = 0; p < P; ++p)
        for (int i = 0; i < N; ++i) S[(int64_t)p * N + i] = alpha * S[(int64_t)p * N + i] + delta * x[p] * Bv[i];
}

/* y[p] = sum_i S[p][i] C[i] + D x[p] */
static void m2_readout(int N, int P, const double* S, const double* Cv, const double* x, double D, double* y) {
    for (int p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int i = 0; i < N; ++i) acc += S[(int64_t)p * N + i] * Cv[i];
        y[p] = acc + D * x[p];
    }
}

void orc_m2_decode_head(int N, int P, void* S, int sdt, const void* x, const void* Bv, const void* Cv, int idt,
                        double alpha, double delta, double D, double* out) {
    int64_t n = (int64_t)N * P;
    double* Sd = (double*)malloc(sizeof(double) * (size_t)n);
    double* buf = (double*)malloc(sizeof(double) * (size_t)(2 * N + P));
    double *bv = buf, *cv = buf + N, *xv = buf + 2 * N;
    load_n(S, 0, (int)n, sdt, Sd);
    load_n(Bv, 0, N, idt, bv);
    load_n(Cv, 0, N, idt, cv);
    load_n(x, 0, P, idt, xv);
    m2_update(N, P, Sd, bv, xv, alpha, delta);
    m2_readout(N, P, Sd, cv, xv, D, out);
    for (int64_t i = 0; i < n; ++i) orc_store(S, i, sdt, Sd[i]);
    free(buf);
    free(Sd);
}

int orc_m2_decode_step(int B, int G, int H, int N, int P, int64_t num_slots, void* pool, int sdt,
                       const int32_t* slots, const void* x, const void* dt, const void* Bm, const void* Cm, int idt,
                       const float* A_log, const float* dt_bias, const float* D, double* out, int nthreads) {
    int bad = 0;
    int per_group = H / G;
    int64_t units = (int64_t)B * H;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 4) reduction(+ : bad) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int bi = (int)(u / H), h = (int)(u % H), g = h / per_group;
        double* o = out + u * P;
        int32_t slot = slots[bi];
        if (slot < 0 || slot >= num_slots) {
            if (slot >= num_slots) bad += 1;
            for (int p = 0; p < P; ++p) o[p] = 0.0;
            continue;
        }
        double alpha, delta;
        orc_m2_gating(A_log[h], dt_bias[h], orc_load(dt, u, idt), &alpha, &delta);
        void* S = (char*)pool + ((int64_t)slot * H + h) * (int64_t)P * N * orc_dtype_size(sdt);
        orc_m2_decode_head(N, P, S, sdt, at(x, u * P, idt), at(Bm, ((int64_t)bi * G + g) * N, idt),
                           at(Cm, ((int64_t)bi * G + g) * N, idt), idt, alpha, delta, D[h], o);
    }
    return bad;
}

/* ------------------------------------------------------------------ ReplaySSM */

/* The fp64 state after the first n buffered entries, rebuilt from S0. */
static void m2_rebuild(int N, int P, const void* S0, int sdt, int n, const void* eB, const void* ex, int idt,
                       const double* ea, const double* ed, double* S) {
    double* tmp = (double*)malloc(sizeof(double) * (size_t)(N + P));
    double *bv = tmp, *xv = tmp + N;
    load_n(S0, 0, N * P, sdt, S);
    for (int e = 0; e < n; ++e) {
        load_n(eB, (int64_t)e * N, N, idt, bv);
        load_n(ex, (int64_t)e * P, P, idt, xv);
        m2_update(N, P, S, bv, xv, ea[e], ed[e]);
    }
    free(tmp);
}

/* S0 <- round(state after every buffered entry); the ring is emptied. */
static void m2_fold(int N, int P, void* S0, int sdt, const void* eB, const void* ex, int idt, const double* ea,
                    const double* ed, int32_t* meta) {
    int64_t n = (int64_t)N * P;
    double* S = (double*)malloc(sizeof(double) * (size_t)n);
    m2_rebuild(N, P, S0, sdt, meta[0], eB, ex, idt, ea, ed, S);
    for (int64_t i = 0; i < n; ++i) orc_store(S0, i, sdt, S[i]);
    free(S);
    meta[0] = 0;
    meta[2] = meta[1];
}

int orc_m2_replay_window(int N, int P, int L, void* S0, int sdt, void* eB, void* ex, int idt, double* ealpha,
                         double* edelta, int32_t* meta, int T, const void* Cw, const void* Bw, const void* xw,
                         const double* dt, double A_log, double dt_bias, double D, double* out) {
    if (T < 1 || T > L) return -1;
    if (meta[0] < 0 || meta[0] > L || meta[1] - meta[2] != meta[0]) return -2;
    if (meta[0] + T > L) m2_fold(N, P, S0, sdt, eB, ex, idt, ealpha, edelta, meta);
    int c = meta[0];
    int isz = orc_dtype_size(idt);
    for (int t = 0; t < T; ++t) { /* append the window's inputs and gates */
        memcpy((char*)eB + (int64_t)(c + t) * N * isz, (const char*)Bw + (int64_t)t * N * isz, (size_t)N * isz);
        memcpy((char*)ex + (int64_t)(c + t) * P * isz, (const char*)xw + (int64_t)t * P * isz, (size_t)P * isz);
        orc_m2_gating(A_log, dt_bias, dt[t], &ealpha[c + t], &edelta[c + t]);
    }
    int64_t n = (int64_t)N * P;
    double* S = (double*)malloc(sizeof(double) * (size_t)n);
    double* buf = (double*)malloc(sizeof(double) * (size_t)(N + P));
    double *cv = buf, *xv = buf + N;
    for (int t = 0; t < T; ++t) { /* output t reads the state after window token t */
        m2_rebuild(N, P, S0, sdt, c + t + 1, eB, ex, idt, ealpha, edelta, S);
        load_n(Cw, (int64_t)t * N, N, idt, cv);
        load_n(xw, (int64_t)t * P, P, idt, xv);
        m2_readout(N, P, S, cv, xv, D, out + (int64_t)t * P);
    }
    free(buf);
    free(S);
    meta[0] = c + T;
    meta[1] += T;
    return 0;
}

int orc_m2_replay_flush(int N, int P, int L, void* S0, int sdt, const void* eB, const void* ex, int idt,
                        const double* ealpha, const double* edelta, int32_t* meta, int force) {
    if (meta[0] < 0 || meta[0] > L || meta[1] - meta[2] != meta[0]) return -2;
    if (meta[0] == L || (force && meta[0] > 0)) m2_fold(N, P, S0, sdt, eB, ex, idt, ealpha, edelta, meta);
    return 0;
}
