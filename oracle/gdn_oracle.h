/*
 * gdn_oracle.h -- CPU oracle for the GDN (Gated DeltaNet) recurrent-state
 * decode step and its ReplaySSM mode.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library; the product path
 * (the CUDA library and its binding) never does, and shares no code with it.
 *
 * Conventions
 *   - Storage dtype codes: 0 = fp32, 1 = bf16, 2 = fp16, 3 = fp64 (fp64 is an
 *     oracle-only "no rounding" storage used for drift references).
 *   - A head state S is dk x dv; it is stored column by column: element
 *     (i, j) -- key index i, value index j -- sits at j*dk + i. A state pool
 *     is [num_slots][Hv][dv][dk].
 *   - Activations: q, k [B][Hk][dk]; v [B][Hv][dv]; a, b [B][Hv]; all in the
 *     input dtype. A_log, dt_bias are fp32 [Hv]. Outputs are fp64.
 *   - All arithmetic is fp64. A state is rounded (round-to-nearest-even) to
 *     its storage dtype only when it is written back.
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2, ORC_F64 = 3 };

/* Storage formats. */
int orc_dtype_size(int dtype);
double orc_round(double x, int dtype);
double orc_load(const void* base, int64_t idx, int dtype);
void orc_store(void* base, int64_t idx, int dtype, double x);
void orc_round_array(const double* x, int64_t n, int dtype, void* out);
void orc_load_array(const void* in, int64_t n, int dtype, double* out);

/* Gating and normalisation. */
void orc_gating(double A_log, double dt_bias, double a, double b, double* alpha, double* beta);
void orc_l2norm(int n, const double* x, double scale, double* y);

/* One decode step of one (sequence, value head). S is updated in place
 * (rounded to sdt); out[dv] receives o = S_t^T q from the unrounded S_t. */
void orc_decode_head(int dk, int dv, void* S, int sdt, const void* q, const void* k, const void* v,
                     int idt, double alpha, double beta, double* out);

/* One decode step of a batch through slot indices. Returns the number of
 * (sequence, head) units whose slot was >= num_slots (skipped, output zero);
 * slot < 0 is padding (skipped, output zero). */
int orc_decode_step(int B, int Hk, int Hv, int dk, int dv, int64_t num_slots, void* pool, int sdt,
                    const int32_t* slots, const void* q, const void* k, const void* v, const void* a,
                    const void* b, int idt, const float* A_log, const float* dt_bias, double* out,
                    int nthreads);

/* Speculative step with one state copy per window token -- the baseline a
 * ReplaySSM verify window replaces. One (sequence, value head): the fp64
 * state loaded from S_in (dv*dk elements of sdt) takes the T window tokens in
 * order (q, k [T][dk], v [T][dv] in idt; gates alpha, beta [T]); after token
 * t the state is rounded into S_out + t*dv*dk when write[t] != 0, and the
 * recursion continues from the unrounded state; out[t*dv + j] = o_t. */
void orc_spec_head(int dk, int dv, int T, const void* S_in, int sdt, void* S_out, const int32_t* write,
                   const void* q, const void* k, const void* v, int idt, const double* alpha,
                   const double* beta, double* out);

/* The same for a batch through slot indices: sequence b starts from
 * pool[src_slots[b]] and writes its state after window token t to
 * pool[dst_slots[b*T + t]] (skipped when < 0). Activations are q, k
 * [B][T][Hk][dk], v [B][T][Hv][dv], a, b [B][T][Hv]; out [B][T][Hv][dv]. Every
 * source is read before any copy is written. src < 0 is padding (outputs zero,
 * nothing written). Returns the number of units with a slot >= num_slots. */
int orc_spec_step(int B, int T, int Hk, int Hv, int dk, int dv, int64_t num_slots, void* pool, int sdt,
                  const int32_t* src_slots, const int32_t* dst_slots, const void* q, const void* k,
                  const void* v, const void* a, const void* b, int idt, const float* A_log,
                  const float* dt_bias, double* out, int nthreads);

/* ReplaySSM, one (sequence, value head). The replay state is the checkpoint
 * S0 (dv*dk elements of sdt), the inputs of the entries buffered since the
 * checkpoint in arrival order -- raw k [L][dk] and v [L][dv] in idt, gates
 * alpha/beta [L] -- and meta = {count, pos, ckpt_pos}.
 * Return 0, or a negative code: -1 bad T, -2 bad count, -3 bad accepted. */
int orc_replay_window(int dk, int dv, int L, void* S0, int sdt, void* ek, void* ev, int idt,
                      double* ealpha, double* ebeta, int32_t* meta, int T, const void* q,
                      const void* k, const void* v, const double* a, const double* b, double A_log,
                      double dt_bias, double* out);
int orc_replay_flush(int dk, int dv, int L, void* S0, int sdt, const void* ek, const void* ev,
                     int idt, const double* ealpha, const double* ebeta, int32_t* meta, int force);
int orc_replay_rollback(int32_t* meta, int T, int accepted);

/* ReplaySSM with a high-precision checkpoint M (mdt) for the recurrence and a
 * low-precision copy Rd (rdt, dv*dk elements) for reading. Outputs, and every
 * entry's prediction S^T k, come from the state rebuilt from Rd. A fold
 * applies each entry's update, taken from that Rd-based rebuild, to M as
 * well; then it stores M rounded to mdt and Rd as the stored M rounded to
 * rdt. The window never folds Rd by itself. Codes as orc_replay_window. */
int orc_replay2_window(int dk, int dv, int L, void* M, int mdt, void* Rd, int rdt, void* ek, void* ev, int idt,
                       double* ealpha, double* ebeta, int32_t* meta, int T, const void* q, const void* k,
                       const void* v, const double* a, const double* b, double A_log, double dt_bias, double* out);
int orc_replay2_flush(int dk, int dv, int L, void* M, int mdt, void* Rd, int rdt, const void* ek, const void* ev,
                      int idt, const double* ealpha, const double* ebeta, int32_t* meta, int force);

/* Prefill of one (sequence, value head): T tokens in order from the state S
 * (dv*dk elements of sdt), each a plain decode step in fp64. The state is
 * rounded to sdt after every `interval` tokens (a chunk write-back: the next
 * chunk starts from the rounded state) and after the last token, which is the
 * state left in S. out[t*dv + j] = o_t from the unrounded S_t. q, k [T][dk],
 * v [T][dv] in idt; gates alpha, beta [T]. interval >= 1. */
void orc_prefill_head(int dk, int dv, int T, void* S, int sdt, const void* q, const void* k, const void* v, int idt,
                      const double* alpha, const double* beta, int interval, double* out);

/* Prefill of a batch of variable-length sequences: sequence b owns tokens
 * cu_seqlens[b] .. cu_seqlens[b+1]-1 of q, k [total][Hk][dk], v [total][Hv][dv],
 * a, b [total][Hv]; out [total][Hv][dv]. Its state is pool[slots[b]]; slot < 0
 * is padding and slot >= num_slots is refused (outputs zero, nothing written).
 * Returns the number of refused (sequence, head) units. */
int orc_prefill(int B, int Hk, int Hv, int dk, int dv, int64_t num_slots, void* pool, int sdt,
                const int32_t* slots, const int32_t* cu_seqlens, const void* q, const void* k, const void* v,
                const void* a, const void* b, int idt, const float* A_log, const float* dt_bias, int interval,
                double* out, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
