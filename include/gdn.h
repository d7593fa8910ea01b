/*
 * gdn.h -- C ABI of the GB300 (sm_103a) GDN recurrent-state decode library.
 *
 * The library runs one data-parallel hot path: the recurrent-state decode
 * step of a Gated DeltaNet (GDN) linear-attention layer -- the gated delta
 * rule that vLLM's fused sigmoid-gating delta-rule update kernel runs -- and
 * its ReplaySSM mode.
 *
 * Sources. The vLLM PR #52191 summary on prhub ("CPU AMX GDN state FP16/BF16
 * persistence, prefix caching +35%") names the decode kernel and its numeric
 * contract in section 实现拆解, items 3-4: arithmetic in FP32, the state kept
 * in fp32/bf16/fp16 and rounded once per write-back. It does not write out the
 * rule, so the standard gated delta rule is used. Per sequence b and value
 * head h, with key head kh = h / (Hv / Hk):
 *     alpha = exp(-exp(A_log[h]) * softplus(a[b,h] + dt_bias[h]))
 *     beta  = sigmoid(b[b,h])
 *     k = k[b,kh] / sqrt(|k[b,kh]|^2 + 1e-6)
 *     q = q[b,kh] / sqrt(|q[b,kh]|^2 + 1e-6) / sqrt(dk)
 *     S_t = alpha S_{t-1} + beta k (v[b,h] - alpha S_{t-1}^T k)^T    (S: dk x dv)
 *     o_t = S_t^T q
 * softplus(x) = x for x > 20, else log(1 + e^x). The ReplaySSM mode is the
 * one the AREX article on ReplaySSM describes in its section "缓存输入而非
 * 状态：checkpoint 每 L 步才更新一次": a checkpoint S0 plus a buffer of the
 * last tokens' state-building inputs; outputs are computed from S0 and the
 * buffer without writing the state; the buffer is folded into S0 when full;
 * rejected draft tokens are dropped by moving the buffer pointer.
 *
 * Conventions for every entry point
 *   - Asynchronous: work is enqueued on `stream` (a cudaStream_t, NULL = the
 *     legacy default stream). Nothing synchronises, allocates or logs.
 *   - The caller owns all memory. Every pointer is a device pointer unless
 *     noted, aligned to 16 bytes, to C-contiguous data with the layout given.
 *   - Return value: GDN_OK, or a negative GDN_ERR_* code when the arguments
 *     are rejected on the host (nothing is launched then) or a launch fails;
 *     gdn_last_error_string() describes the last failure on this thread.
 *   - Problems only visible on the device (a slot index >= num_slots, a
 *     replay pointer pair out of range, an accepted count out of range, a
 *     pipeline wait that timed out) set bits GDN_DEVERR_* in *dev_err with
 *     atomicOr; the affected (sequence, head) is skipped and, where it has an
 *     output, its output is zero-filled. Nothing traps. dev_err is required;
 *     the caller clears it and reads it back when convenient.
 *   - Slot indices are int32; a negative slot is padding: no state is read
 *     or written and the output rows are zero. Slots within one call must be
 *     distinct (not checked; duplicates race).
 *   - Shapes: dk in {32, 64, 128}; dv a multiple of 16 in [16, 256] (of 32
 *     for the ReplaySSM entry points); Hv a multiple of Hk; B >= 0 (B == 0
 *     launches nothing).
 *
 * The same kernels also run the Mamba2 decode recurrence (entry points
 * mamba2_*, at the end of this header), the other state-space layer the
 * ReplaySSM article covers (section "每步写回完整循环状态": a state of shape
 * (nheads, d, n) read through the vector C).
 */
#ifndef GDN_H
#define GDN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 4

/* Host-side return codes. */
#define GDN_OK 0
#define GDN_ERR_NULL (-1)    /* a required pointer is NULL */
#define GDN_ERR_DTYPE (-2)   /* unsupported dtype or dtype mismatch */
#define GDN_ERR_SHAPE (-3)   /* unsupported dk/dv, Hv % Hk != 0, negative sizes */
#define GDN_ERR_WINDOW (-4)  /* T < 1, T > 8, T > L, L < 1 or L > 64 */
#define GDN_ERR_ALIGN (-5)   /* a pointer is not 16-byte aligned */
#define GDN_ERR_LAUNCH (-6)  /* CUDA reported an error at launch */

/* Device-side error bits (set in *dev_err). */
#define GDN_DEVERR_SLOT 1    /* slot index >= num_slots */
#define GDN_DEVERR_RING 2    /* replay count pos - ckpt_pos outside [0, L], or a rollback below ckpt_pos */
#define GDN_DEVERR_ACCEPT 4  /* accepted count outside [0, T-1], or a rollback that does not undo a T-token window */
#define GDN_DEVERR_TIMEOUT 8 /* an internal pipeline wait gave up (should never happen) */
#define GDN_DEVERR_SEQLEN 16 /* prefill token offsets decreasing or beyond total_tokens */
#define GDN_DEVERR_BOUNDS 32 /* bounds-checking builds only (GDN_DEBUG_BOUNDS): a copy or store fell
                                outside its array and was skipped */

/* Element types of states, activations and outputs; mirrors the fp32 /
 * bf16 / fp16 choice of a mamba SSM cache dtype. */
enum gdn_dtype { GDN_F32 = 0, GDN_BF16 = 1, GDN_F16 = 2 };

/* Problem sizes. B: sequences in the call; Hk / Hv: key / value heads;
 * dk / dv: key / value head dimensions; num_slots: slots in the state pool. */
typedef struct gdn_dims {
    int32_t B, Hk, Hv, dk, dv;
    int64_t num_slots;
} gdn_dims;

/*
 * gdn_decode_step -- one gated delta-rule decode step for a batch of
 * sequences whose states live in a paged pool (vLLM PR #52191 summary,
 * 实现拆解 3-4: state_t storage, FP32 arithmetic, one rounding per
 * write-back).
 *
 * state_pool  [num_slots][Hv][dv][dk] of state_dtype. Element (i, j) of the
 *             dk x dv state of (slot, h) -- key index i, value index j -- is
 *             at ((slot*Hv + h)*dv + j)*dk + i. Read, updated, rounded
 *             (round-to-nearest-even) and written back in place.
 * slots       [B] int32, slot of each sequence (< 0: padding).
 * q, k        [B][Hk][dk] of in_dtype.   v: [B][Hv][dv];  a, b: [B][Hv].
 * A_log, dt_bias  [Hv] fp32.
 * out         [B][Hv][dv] of out_dtype: o_t, computed from the unrounded S_t.
 * dev_err     int32 error word (see GDN_DEVERR_*).
 */
int gdn_decode_step(const gdn_dims* dims, void* state_pool, int32_t state_dtype,
                    const int32_t* slots, const void* q, const void* k, const void* v,
                    const void* a, const void* b, int32_t in_dtype, const float* A_log,
                    const float* dt_bias, void* out, int32_t out_dtype, int32_t* dev_err,
                    void* stream);

/*
 * gdn_spec_step -- speculative step with one state copy per window token: the
 * baseline that the ReplaySSM verify window replaces (AREX ReplaySSM article,
 * section "每步写回完整循环状态：SSM 解码的两个瓶颈": to roll back rejected
 * drafts, the existing implementation keeps a recurrent state per draft token,
 * about (1 + num_spec) times the state memory).
 * Sequence b takes a window of T tokens (the last verified token and T-1
 * drafts, 1 <= T <= 8) from the state in state_pool[src_slots[b]]. After
 * window token t its state is rounded (round-to-nearest-even) into
 * state_pool[dst_slots[b*T + t]]; the recursion continues from the unrounded
 * FP32 state. Output t is o_t = S_t^T q_t. After verification the state of
 * the last accepted token is the copy in its destination slot.
 * state_pool  as for gdn_decode_step.
 * src_slots   [B] int32 (< 0: padding; outputs zero, nothing written).
 * dst_slots   [B][T] int32 (< 0: that token's copy is not written).
 *             Preconditions (not checked): no slot appears twice in a call,
 *             except that a sequence's destinations may include its own
 *             source slot. A source or destination >= num_slots sets
 *             GDN_DEVERR_SLOT; that sequence's outputs are zeroed and nothing
 *             of it is written.
 * q, k  [B][T][Hk][dk];  v [B][T][Hv][dv];  a, b [B][T][Hv];  out [B][T][Hv][dv].
 * Errors as gdn_decode_step; T outside [1, 8] gives GDN_ERR_WINDOW.
 */
int gdn_spec_step(const gdn_dims* dims, void* state_pool, int32_t state_dtype, const int32_t* src_slots,
                  const int32_t* dst_slots, int32_t T, const void* q, const void* k, const void* v,
                  const void* a, const void* b, int32_t in_dtype, const float* A_log,
                  const float* dt_bias, void* out, int32_t out_dtype, int32_t* dev_err, void* stream);

/*
 * ReplaySSM cache (AREX ReplaySSM article, "缓存输入而非状态"). Everything is
 * indexed by slot and value head; each (slot, h) is an independent unit with
 * its own checkpoint, L-entry ring and pointers.
 *
 * ckpt      [num_slots][Hv][dv][dk] of ckpt_dtype: the checkpoint S0, same
 *           layout as a decode state pool. Written only when folded.
 * ring_k    [num_slots][Hv][L][dk] of ring_dtype: raw (unnormalised) keys.
 * ring_v    [num_slots][Hv][L][dv] of ring_dtype: raw values.
 * ring_rec  [num_slots][Hv][L][4 + dv] fp32: per entry {alpha, beta,
 *           1/|k|, n, w[0..dv)}, where alpha and beta are the entry's gates,
 *           1/|k| = 1/sqrt(|k|^2 + 1e-6) its key's inverse norm,
 *           n the length T of the call that appended it on that call's
 *           first entry (0 on the others; gdn_rollback checks and clears
 *           it), and w = beta (v - alpha S_prev^T k) its correction vector
 *           (S_prev: the state just before the entry, as the outputs read
 *           it). 1/|k| and w are derived data the kernels keep so that an
 *           output needs one pass over S0, not one per buffered entry; w
 *           stays valid until the entry is folded. The ring is written only
 *           by these entry points; zero-filled is a valid initial ring.
 * pos       [num_slots][Hv] int32: absolute position of the next token.
 * ckpt_pos  [num_slots][Hv] int32: position the checkpoint corresponds to.
 *           count = pos - ckpt_pos entries are buffered, 0 <= count <= L;
 *           entry for absolute position t sits at ring index t mod L.
 * L         ring length, 1 <= L <= 64.
 *
 * A fresh sequence: ckpt = its initial state, pos = ckpt_pos (any value >= 0).
 * A fold -- ckpt <- round(S after all buffered entries), ckpt_pos <- pos --
 * happens exactly when appending the call's tokens would overflow the ring
 * (count + T > L), before they are appended, or on gdn_replay_flush.
 *
 * ckpt_read  NULL, or a low-precision read copy [num_slots][Hv][dv][dk] of
 *            read_dtype (bf16 or fp16; ckpt_dtype must then be fp32): the
 *            high-precision checkpoint for the recurrence and the
 *            low-precision copy for reading of the AREX ReplaySSM article
 *            (section "缓存输入而非状态", its precision paragraph). Every
 *            output, and every prediction S^T k between folds, then reads
 *            ckpt_read; only a fold reads ckpt: it runs the buffered entries'
 *            raw inputs through the rule on ckpt in FP32 -- every prediction
 *            of the recurrence comes from the fp32 checkpoint itself --
 *            stores it, and rewrites ckpt_read as the stored value rounded
 *            to read_dtype. ckpt therefore evolves exactly as a
 *            single-checkpoint replay with an fp32 checkpoint would. A fresh
 *            sequence: ckpt_read = ckpt rounded. One launch per call: units
 *            that fold stream the fp32 checkpoint and the buffered values,
 *            the others the read copy; the tokens of a call that folds run
 *            from the rewritten copy. Both arrays are 16-byte aligned and do
 *            not overlap.
 */
typedef struct gdn_replay_cache {
    void* ckpt;
    int32_t ckpt_dtype;
    void* ring_k;
    void* ring_v;
    int32_t ring_dtype;
    float* ring_rec;
    int32_t* pos;
    int32_t* ckpt_pos;
    int32_t L;
    void* ckpt_read;
    int32_t read_dtype;
} gdn_replay_cache;

/*
 * gdn_replay_step -- one ReplaySSM standard-decode step: o_t = S_t^T q_t with
 * S_t rebuilt in FP32 from S0 and the ring, the token's inputs appended, and
 * no state written unless the ring was full (then it is folded first).
 * Arguments as gdn_decode_step; in_dtype must equal cache->ring_dtype.
 * Equivalent to gdn_verify_window with T = 1.
 */
int gdn_replay_step(const gdn_dims* dims, const gdn_replay_cache* cache, const int32_t* slots,
                    const void* q, const void* k, const void* v, const void* a, const void* b,
                    int32_t in_dtype, const float* A_log, const float* dt_bias, void* out,
                    int32_t out_dtype, int32_t* dev_err, void* stream);

/*
 * gdn_verify_window -- ReplaySSM speculative verify (AREX ReplaySSM article,
 * "缓存输入而非状态": the draft window is checked in one pass from the cache).
 * T tokens per sequence (the last verified token plus T-1 drafts), 1 <= T <=
 * min(L, 8). Output j reads the state after window tokens 0..j. All T
 * tokens are appended (pos += T); none of them is ever folded by this call.
 * q, k  [B][T][Hk][dk];  v [B][T][Hv][dv];  a, b [B][T][Hv];
 * out   [B][T][Hv][dv].
 */
int gdn_verify_window(const gdn_dims* dims, const gdn_replay_cache* cache, const int32_t* slots,
                      int32_t T, const void* q, const void* k, const void* v, const void* a,
                      const void* b, int32_t in_dtype, const float* A_log, const float* dt_bias,
                      void* out, int32_t out_dtype, int32_t* dev_err, void* stream);

/*
 * gdn_replay_flush -- fold the ring into the checkpoint for the given slots:
 * every (slot, h) with count == L, or with count > 0 when force != 0.
 */
int gdn_replay_flush(const gdn_dims* dims, const gdn_replay_cache* cache, const int32_t* slots,
                     int32_t force, int32_t* dev_err, void* stream);

/*
 * gdn_rollback -- after a T-token verify, keep 1 + accepted[b] tokens of
 * sequence b: pos[slot][h] -= T - 1 - accepted[b] for every head. A pointer
 * move (AREX ReplaySSM article: rollback becomes moving the buffer pointer);
 * no state, ring key, value, gate or w is touched.
 * accepted  [B] int32 device array, each in [0, T-1].
 * T         must be the T of the gdn_verify_window call it undoes, with no
 *           other replay call on those slots in between. Each (slot, h)
 *           checks this against the window-length field of the window's
 *           first ring record and clears that field, so a second rollback
 *           of the same window is refused too: a mismatch sets
 *           GDN_DEVERR_ACCEPT and leaves pos unchanged. A rollback below
 *           ckpt_pos sets GDN_DEVERR_RING.
 */
int gdn_rollback(const gdn_dims* dims, const gdn_replay_cache* cache, const int32_t* slots,
                 const int32_t* accepted, int32_t T, int32_t* dev_err, void* stream);

/*
 * gdn_prefill -- prefill of variable-length sequences with the state written
 * back once per chunk (vLLM PR #52191 summary, section 实现拆解 items 3-4:
 * the chunked kernel updates an FP32 copy of the state and writes it back,
 * rounded to the state dtype, at the end of every chunk).
 * Sequence b owns tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 and the state
 * pool[slots[b]]; its tokens run through the rule in order, the state being
 * rounded to state_dtype after every state_write_interval tokens (the next
 * chunk continues from the rounded state) and after the last token, which is
 * what is stored. Outputs come from the unrounded FP32 state.
 * Arithmetic: FP32 for fp32 states. For bf16/fp16 states with dk = 128 and
 * dv a multiple of 128 the chunked form runs on the tensor cores: the state,
 * accumulation and rounding points stay FP32, the matrix products take TF32
 * operands (within the 16-bit state's own rounding).
 * cu_seqlens   [B + 1] int32 device array, 0 <= cu_seqlens[b] <= cu_seqlens[b+1]
 *              <= total_tokens (otherwise GDN_DEVERR_SEQLEN and the sequence
 *              is skipped).
 * q, k         [total_tokens][Hk][dk];  v [total_tokens][Hv][dv];
 * a, b         [total_tokens][Hv];      out [total_tokens][Hv][dv].
 * state_write_interval >= 1 (GDN_ERR_WINDOW otherwise). A padding slot zeroes
 * its sequence's outputs; an out-of-range slot also sets GDN_DEVERR_SLOT. An
 * empty sequence leaves its state untouched.
 */
int gdn_prefill(const gdn_dims* dims, void* state_pool, int32_t state_dtype, const int32_t* slots,
                const int32_t* cu_seqlens, int32_t total_tokens, const void* q, const void* k, const void* v,
                const void* a, const void* b, int32_t in_dtype, const float* A_log, const float* dt_bias,
                int32_t state_write_interval, void* out, int32_t out_dtype, int32_t* dev_err, void* stream);

/*
 * ---------------------------------------------------------------- Mamba2
 *
 * The Mamba2 decode recurrence (the standard one; the ReplaySSM article names
 * its state shape (nheads, d, n) and its readout vector C, section "每步写回
 * 完整循环状态"). Per sequence b and head h, group g = h / (H / G):
 *     delta = softplus(dt[b,h] + dt_bias[h]),  alpha = exp(-exp(A_log[h]) delta)
 *     S_t[p][i] = alpha S_{t-1}[p][i] + delta x[b,h][p] B[b,g][i]
 *     y_t[p]    = sum_i S_t[p][i] C[b,g][i] + D[h] x[b,h][p]
 * A head state is P rows of N contiguous elements, a pool [num_slots][H][P][N]
 * -- the layout of a GDN pool with dk = N and dv = P. Activations: x [B][H][P],
 * dt [B][H], Bm, Cm [B][G][N] in in_dtype; A_log, dt_bias, D fp32 [H]
 * (A = -exp(A_log) is Mamba2's per-head decay rate). Shapes: N in
 * {32, 64, 128}; P a multiple of 16 in [16, 256] (of 32 for replay); H a
 * multiple of G. Conventions otherwise as above.
 */
typedef struct mamba2_dims {
    int32_t B;          /* sequences in the batch */
    int32_t G;          /* groups (rows of B and C per sequence) */
    int32_t H;          /* heads */
    int32_t N;          /* state dim (d_state) */
    int32_t P;          /* head dim */
    int64_t num_slots;  /* slots in the state pool / replay cache */
} mamba2_dims;

/* mamba2_decode_step -- one decode step: reads and writes pool[slots[b]]
 * (rounded once to state_dtype), out [B][H][P] in out_dtype. */
int mamba2_decode_step(const mamba2_dims* dims, void* state_pool, int32_t state_dtype, const int32_t* slots,
                       const void* x, const void* dt, const void* Bm, const void* Cm, int32_t in_dtype,
                       const float* A_log, const float* dt_bias, const float* D, void* out, int32_t out_dtype,
                       int32_t* dev_err, void* stream);

/*
 * Mamba2 ReplaySSM, on a gdn_replay_cache read as: ckpt [num_slots][H][P][N];
 * ring_k [num_slots][H][L][N] the raw B rows; ring_v [num_slots][H][L][P] the
 * raw x rows; ring_rec [num_slots][H][L][4 + P] fp32 = {alpha, delta, 1, 0,
 * w[P] = delta x}; pos, ckpt_pos [num_slots][H]. C is never buffered (the
 * ReplaySSM article: the readout vector comes from the current activations).
 * Folding, windows and rollback follow the gdn_replay_* rules exactly; the
 * read copy (ckpt_read) is not supported here (GDN_ERR_DTYPE).
 *   mamba2_replay_step    one token: out [B][H][P].
 *   mamba2_verify_window  T tokens, 1 <= T <= min(L, 8), L <= 64: x [B][T][H][P],
 *                         dt [B][T][H], Bm, Cm [B][T][G][N], out [B][T][H][P].
 *   mamba2_replay_flush   fold full rings (or non-empty ones with force).
 *   mamba2_rollback       keep 1 + accepted[b] of the last window's T tokens.
 */
int mamba2_replay_step(const mamba2_dims* dims, const gdn_replay_cache* cache, const int32_t* slots, const void* x,
                       const void* dt, const void* Bm, const void* Cm, int32_t in_dtype, const float* A_log,
                       const float* dt_bias, const float* D, void* out, int32_t out_dtype, int32_t* dev_err,
                       void* stream);
int mamba2_verify_window(const mamba2_dims* dims, const gdn_replay_cache* cache, const int32_t* slots, int32_t T,
                         const void* x, const void* dt, const void* Bm, const void* Cm, int32_t in_dtype,
                         const float* A_log, const float* dt_bias, const float* D, void* out, int32_t out_dtype,
                         int32_t* dev_err, void* stream);
int mamba2_replay_flush(const mamba2_dims* dims, const gdn_replay_cache* cache, const int32_t* slots,
                        int32_t force, int32_t* dev_err, void* stream);
int mamba2_rollback(const mamba2_dims* dims, const gdn_replay_cache* cache, const int32_t* slots,
                    const int32_t* accepted, int32_t T, int32_t* dev_err, void* stream);

/* Text of the last host-side failure on the calling thread ("" if none). */
const char* gdn_last_error_string(void);

/* GDN_ABI_VERSION of the loaded library. */
int32_t gdn_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif
