/*
 * mamba2_oracle.h -- CPU oracle for the Mamba2 selective-state decode step and
 * its ReplaySSM mode.
 *
 * TEST INFRASTRUCTURE ONLY, like gdn_oracle.h, and built into the same
 * library: the tests, the package smoke check and the benchmark's
 * CPU-baseline leg may load it; the CUDA library shares no code with it.
 *
 * The rule (the standard Mamba2 decode recurrence; the AREX article on
 * ReplaySSM, section "每步写回完整循环状态", names the state (nheads, d, n)
 * and the readout vector C). Per head h, with group g = h / (H / G):
 *   delta = softplus(dt + dt_bias[h]),   alpha = exp(-exp(A_log[h]) * delta)
 *   S_t[p][i] = alpha S_{t-1}[p][i] + delta x_t[p] B_t[g][i]
 *   y_t[p]    = sum_i S_t[p][i] C_t[g][i] + D[h] x_t[p]
 * Conventions
 *   - A head state is stored as P (head dim) rows of N (state dim) contiguous
 *     elements: element (i, p) at p*N + i. A pool is [num_slots][H][P][N].
 *   - Activations: x [B][H][P], dt [B][H], Bm, Cm [B][G][N], in the input
 *     dtype; A_log, dt_bias, D fp32 [H]. Outputs fp64.
 *   - fp64 arithmetic; a state is rounded to its storage dtype only when it
 *     is written back. Dtype codes as gdn_oracle.h.
 */
#ifndef MAMBA2_ORACLE_H
#define MAMBA2_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* delta = softplus(dt + dt_bias), alpha = exp(-exp(A_log) delta). */
void orc_m2_gating(double A_log, double dt_bias, double dt, double* alpha, double* delta);

/* One decode step of one head: S (P*N elements of sdt) updated in place and
 * rounded; out[P] = y from the unrounded S_t. */
void orc_m2_decode_head(int N, int P, void* S, int sdt, const void* x, const void* Bv, const void* Cv, int idt,
                        double alpha, double delta, double D, double* out);

/* One decode step of a batch through slot indices; slot < 0 is padding and
 * slot >= num_slots is refused (both: output zero, nothing written). Returns
 * the number of refused (sequence, head) units. */
int orc_m2_decode_step(int B, int G, int H, int N, int P, int64_t num_slots, void* pool, int sdt,
                       const int32_t* slots, const void* x, const void* dt, const void* Bm, const void* Cm, int idt,
                       const float* A_log, const float* dt_bias, const float* D, double* out, int nthreads);

/* ReplaySSM for one (sequence, head): checkpoint S0 (P*N of sdt), the
 * entries buffered since it in arrival order -- raw B [L][N] and x [L][P]
 * in idt, alpha and delta [L] -- and meta = {count, pos, ckpt_pos}. A window
 * of T tokens (Cw, Bw [T][N], xw [T][P], dt [T]) folds first when the ring
 * lacks room for T more entries, appends them, and gives out[t][P] from the
 * state after token t, rebuilt from S0. Return 0, or -1 bad T, -2 bad count. */
int orc_m2_replay_window(int N, int P, int L, void* S0, int sdt, void* eB, void* ex, int idt, double* ealpha,
                         double* edelta, int32_t* meta, int T, const void* Cw, const void* Bw, const void* xw,
                         const double* dt, double A_log, double dt_bias, double D, double* out);
/* Fold the ring into S0 when it is full, or whenever it is not empty with
 * force. */
int orc_m2_replay_flush(int N, int P, int L, void* S0, int sdt, const void* eB, const void* ex, int idt,
                        const double* ealpha, const double* edelta, int32_t* meta, int force);

#ifdef __cplusplus
}
#endif
#endif
