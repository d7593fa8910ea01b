// gdn_abi.cu -- the extern "C" entry points declared in include/gdn.h:
// argument validation on the host, then one kernel launch on the caller's
// stream. Nothing here allocates, synchronises or logs.
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <string>

#include "../../include/gdn.h"
#include "gdn_dispatch.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int launched(cudaError_t e, const char* what) {
    if (e == cudaSuccess) {
        g_last_error.clear();
        return GDN_OK;
    }
    if (e == cudaErrorNotSupported) return fail(GDN_ERR_SHAPE, "%s: no kernel for this dtype/dk", what);
    return fail(GDN_ERR_LAUNCH, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void* p, int n) { return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)n) == 0; }
bool dtype_ok(int32_t d) { return d == GDN_F32 || d == GDN_BF16 || d == GDN_F16; }

int check_dims(const gdn_dims* d, const char* fn) {
    if (!d) return fail(GDN_ERR_NULL, "%s: dims is NULL", fn);
    if (d->B < 0 || d->Hk <= 0 || d->Hv <= 0 || d->num_slots < 0)
        return fail(GDN_ERR_SHAPE, "%s: negative or zero sizes (B=%d Hk=%d Hv=%d num_slots=%lld)", fn, d->B, d->Hk,
                    d->Hv, (long long)d->num_slots);
    if (d->Hv % d->Hk != 0) return fail(GDN_ERR_SHAPE, "%s: Hv=%d is not a multiple of Hk=%d", fn, d->Hv, d->Hk);
    if (d->dk != 32 && d->dk != 64 && d->dk != 128)
        return fail(GDN_ERR_SHAPE, "%s: dk=%d not in {32, 64, 128}", fn, d->dk);
    if (d->dv < 16 || d->dv > gdn::DV_MAX || d->dv % 16 != 0)
        return fail(GDN_ERR_SHAPE, "%s: dv=%d must be a multiple of 16 in [16, 256]", fn, d->dv);
    if ((int64_t)d->B * d->Hv > (int64_t)INT32_MAX / 8)
        return fail(GDN_ERR_SHAPE, "%s: B*Hv=%lld too large", fn, (long long)d->B * d->Hv);
    return GDN_OK;
}

// Rows of a state per 16 KB chunk: the largest power-of-two divisor of dv
// that keeps a chunk within CHUNK_BYTES.
void chunking(int dk, int dv, int state_bytes, int& rows, int& nchunk) {
    rows = gdn::CHUNK_BYTES / (dk * state_bytes);
    if (rows > dv) rows = dv;
    while (dv % rows != 0) rows /= 2;
    nchunk = dv / rows;
}

int check_activations(const char* fn, const void* q, const void* k, const void* v, const void* a, const void* b,
                      int32_t in_dtype, const float* A_log, const float* dt_bias, const void* out,
                      int32_t out_dtype) {
    if (!q || !k || !v || !a || !b || !A_log || !dt_bias || !out)
        return fail(GDN_ERR_NULL, "%s: an activation / parameter / output pointer is NULL", fn);
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype))
        return fail(GDN_ERR_DTYPE, "%s: unsupported dtype (in=%d out=%d)", fn, in_dtype, out_dtype);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v))
        return fail(GDN_ERR_ALIGN, "%s: q, k and v must be 16-byte aligned", fn);
    const int isz = gdn::dtype_size(in_dtype), osz = gdn::dtype_size(out_dtype);
    if (!aligned_to(a, isz) || !aligned_to(b, isz) || !aligned_to(out, osz) || !aligned_to(A_log, 4) ||
        !aligned_to(dt_bias, 4))
        return fail(GDN_ERR_ALIGN, "%s: a, b, A_log, dt_bias or out misaligned for its dtype", fn);
    return GDN_OK;
}

// The replay entry points of both recurrences. Mamba2 passes (C, B, x, dt) as (q, k, v, a), no b, and
// its skip weights D.
int replay_common(const char* fn, int rule, const gdn_dims* dims, const gdn_replay_cache* c, const int32_t* slots,
                  int32_t T, int32_t force, const void* q, const void* k, const void* v, const void* a, const void* b,
                  int32_t in_dtype, const float* A_log, const float* dt_bias, const float* D, void* out,
                  int32_t out_dtype, int32_t* dev_err, void* stream) {
    int rc = check_dims(dims, fn);
    if (rc) return rc;
    if (!c) return fail(GDN_ERR_NULL, "%s: cache is NULL", fn);
    if (dims->B == 0) return GDN_OK;
    if (!c->ckpt || !c->ring_k || !c->ring_v || !c->ring_rec || !c->pos || !c->ckpt_pos || !slots || !dev_err)
        return fail(GDN_ERR_NULL, "%s: a cache, slots or dev_err pointer is NULL", fn);
    if (!dtype_ok(c->ckpt_dtype) || !dtype_ok(c->ring_dtype))
        return fail(GDN_ERR_DTYPE, "%s: unsupported cache dtype (ckpt=%d ring=%d)", fn, c->ckpt_dtype, c->ring_dtype);
    if (c->L < 1 || c->L > gdn::L_MAX) return fail(GDN_ERR_WINDOW, "%s: L=%d not in [1, 64]", fn, c->L);
    if (dims->dv % 32 != 0) return fail(GDN_ERR_SHAPE, "%s: dv=%d must be a multiple of 32", fn, dims->dv);
    if (T > 0) {
        if (T > c->L || T > gdn::WINDOW_MAX)
            return fail(GDN_ERR_WINDOW, "%s: window T=%d exceeds min(L=%d, 8)", fn, T, c->L);
        rc = check_activations(fn, q, k, v, a, rule == gdn::RULE_GDN ? b : a, in_dtype, A_log, dt_bias, out,
                               out_dtype);
        if (rc) return rc;
        if (rule == gdn::RULE_MAMBA2 && (!D || !aligned_to(D, 4)))
            return fail(D ? GDN_ERR_ALIGN : GDN_ERR_NULL, "%s: D is NULL or misaligned", fn);
        if (in_dtype != c->ring_dtype)
            return fail(GDN_ERR_DTYPE, "%s: in_dtype=%d differs from the ring dtype %d", fn, in_dtype, c->ring_dtype);
    } else if (T < 0) {
        return fail(GDN_ERR_WINDOW, "%s: negative window", fn);
    }
    if (!aligned16(c->ckpt) || !aligned16(c->ring_k) || !aligned16(c->ring_v) || !aligned16(c->ring_rec) ||
        !aligned_to(c->pos, 4) || !aligned_to(c->ckpt_pos, 4) || !aligned_to(slots, 4) || !aligned_to(dev_err, 4))
        return fail(GDN_ERR_ALIGN, "%s: cache arrays must be 16-byte aligned", fn);

    if (c->ckpt_read) {
        if (rule != gdn::RULE_GDN) return fail(GDN_ERR_DTYPE, "%s: a read copy is not supported for Mamba2", fn);
        if (c->ckpt_dtype != GDN_F32 || (c->read_dtype != GDN_BF16 && c->read_dtype != GDN_F16))
            return fail(GDN_ERR_DTYPE, "%s: a read copy needs an fp32 checkpoint and a bf16/fp16 copy (ckpt=%d read=%d)", fn,
                        c->ckpt_dtype, c->read_dtype);
        if (!aligned16(c->ckpt_read)) return fail(GDN_ERR_ALIGN, "%s: ckpt_read must be 16-byte aligned", fn);
    }

    gdn::ReplayArgs p{};
    p.ckpt = c->ckpt, p.ring_k = c->ring_k, p.ring_v = c->ring_v, p.ring_rec = c->ring_rec;
    p.pos = c->pos, p.ckpt_pos = c->ckpt_pos, p.slots = slots;
    p.q = q, p.k = k, p.v = v, p.a = a, p.b = b, p.A_log = A_log, p.dt_bias = dt_bias, p.D = D;
    p.out = out, p.dev_err = dev_err;
    p.num_slots = dims->num_slots;
    p.B = dims->B, p.Hk = dims->Hk, p.Hv = dims->Hv, p.dv = dims->dv, p.L = c->L, p.T = T, p.force = force != 0;
    p.in_dtype = c->ring_dtype, p.out_dtype = T > 0 ? out_dtype : GDN_F32;
    p.q_scale = (float)(1.0 / sqrt((double)dims->dk));
    // the producer kernel's 16 KB chunks of the read type, and of the master (whose chunk holds a
    // whole number of the read type's items)
    if (c->ckpt_read) {
        chunking(dims->dk, dims->dv, gdn::dtype_size(c->read_dtype), p.rows, p.nchunk);
        chunking(dims->dk, p.rows, 4, p.mrows, p.mnchunk);
        p.mnchunk = dims->dv / p.mrows;
    } else {
        chunking(dims->dk, dims->dv, gdn::dtype_size(c->ckpt_dtype), p.rows, p.nchunk);
        p.mrows = p.rows, p.mnchunk = p.nchunk;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int tmax = T <= 1 ? 1 : (T <= 4 ? 4 : 8);
    bool too_big = false;
    cudaError_t e;
    if (c->ckpt_read) {
        // Two checkpoints, one launch: steps read the copy; folds stream the fp32 master, run the
        // rule on it, store it and rewrite the copy.
        p.ckpt_copy = c->ckpt_read;
        e = c->read_dtype == GDN_BF16 ? gdn::dispatch_replay_f32_bf16(dims->dk, tmax, p, s, too_big)
                                      : gdn::dispatch_replay_f32_f16(dims->dk, tmax, p, s, too_big);
    } else if (rule == gdn::RULE_MAMBA2) {
        if (c->ckpt_dtype == GDN_F32)
            e = gdn::dispatch_mamba2_replay_f32(dims->dk, tmax, p, s, too_big);
        else if (c->ckpt_dtype == GDN_BF16)
            e = gdn::dispatch_mamba2_replay_bf16(dims->dk, tmax, p, s, too_big);
        else
            e = gdn::dispatch_mamba2_replay_f16(dims->dk, tmax, p, s, too_big);
    } else {
        if (c->ckpt_dtype == GDN_F32)
            e = gdn::dispatch_replay_f32(dims->dk, tmax, p, s, too_big);
        else if (c->ckpt_dtype == GDN_BF16)
            e = gdn::dispatch_replay_bf16(dims->dk, tmax, p, s, too_big);
        else
            e = gdn::dispatch_replay_f16(dims->dk, tmax, p, s, too_big);
    }
    if (too_big) return fail(GDN_ERR_SHAPE, "%s: L=%d, T=%d, dv=%d do not fit in shared memory", fn, c->L, T, dims->dv);
    return launched(e, fn);
}

}  // namespace

extern "C" {

int gdn_decode_step(const gdn_dims* dims, void* state_pool, int32_t state_dtype, const int32_t* slots, const void* q,
                    const void* k, const void* v, const void* a, const void* b, int32_t in_dtype, const float* A_log,
                    const float* dt_bias, void* out, int32_t out_dtype, int32_t* dev_err, void* stream) {
    const char* fn = "gdn_decode_step";
    int rc = check_dims(dims, fn);
    if (rc) return rc;
    if (dims->B == 0) return GDN_OK;
    if (!state_pool || !slots || !dev_err) return fail(GDN_ERR_NULL, "%s: state_pool, slots or dev_err is NULL", fn);
    if (!dtype_ok(state_dtype)) return fail(GDN_ERR_DTYPE, "%s: unsupported state dtype %d", fn, state_dtype);
    rc = check_activations(fn, q, k, v, a, b, in_dtype, A_log, dt_bias, out, out_dtype);
    if (rc) return rc;
    if (!aligned16(state_pool) || !aligned_to(slots, 4) || !aligned_to(dev_err, 4))
        return fail(GDN_ERR_ALIGN, "%s: state_pool must be 16-byte aligned", fn);
    gdn::DecodeArgs p{};
    p.pool = state_pool, p.slots = slots, p.q = q, p.k = k, p.v = v, p.a = a, p.b = b;
    p.A_log = A_log, p.dt_bias = dt_bias, p.out = out, p.dev_err = dev_err;
    p.num_slots = dims->num_slots;
    p.B = dims->B, p.Hk = dims->Hk, p.Hv = dims->Hv, p.dv = dims->dv;
    p.in_dtype = in_dtype, p.out_dtype = out_dtype;
    p.q_scale = (float)(1.0 / sqrt((double)dims->dk));
    chunking(dims->dk, dims->dv, gdn::dtype_size(state_dtype), p.rows, p.nchunk);
    return launched(gdn::dispatch_decode(state_dtype, dims->dk, p, static_cast<cudaStream_t>(stream)), fn);
}

int gdn_spec_step(const gdn_dims* dims, void* state_pool, int32_t state_dtype, const int32_t* src_slots,
                  const int32_t* dst_slots, int32_t T, const void* q, const void* k, const void* v, const void* a,
                  const void* b, int32_t in_dtype, const float* A_log, const float* dt_bias, void* out,
                  int32_t out_dtype, int32_t* dev_err, void* stream) {
    const char* fn = "gdn_spec_step";
    int rc = check_dims(dims, fn);
    if (rc) return rc;
    if (T < 1 || T > gdn::SPEC_WINDOW_MAX) return fail(GDN_ERR_WINDOW, "%s: T=%d not in [1, 8]", fn, T);
    if (dims->B == 0) return GDN_OK;
    if (!state_pool || !src_slots || !dst_slots || !dev_err)
        return fail(GDN_ERR_NULL, "%s: state_pool, src_slots, dst_slots or dev_err is NULL", fn);
    if (!dtype_ok(state_dtype)) return fail(GDN_ERR_DTYPE, "%s: unsupported state dtype %d", fn, state_dtype);
    rc = check_activations(fn, q, k, v, a, b, in_dtype, A_log, dt_bias, out, out_dtype);
    if (rc) return rc;
    if (!aligned16(state_pool) || !aligned_to(src_slots, 4) || !aligned_to(dst_slots, 4) || !aligned_to(dev_err, 4))
        return fail(GDN_ERR_ALIGN, "%s: state_pool must be 16-byte aligned", fn);
    gdn::SpecArgs p{};
    p.pool = state_pool, p.src_slots = src_slots, p.dst_slots = dst_slots;
    p.q = q, p.k = k, p.v = v, p.a = a, p.b = b, p.A_log = A_log, p.dt_bias = dt_bias;
    p.out = out, p.dev_err = dev_err;
    p.num_slots = dims->num_slots;
    p.B = dims->B, p.Hk = dims->Hk, p.Hv = dims->Hv, p.dv = dims->dv, p.T = T;
    p.in_dtype = in_dtype, p.out_dtype = out_dtype;
    p.q_scale = (float)(1.0 / sqrt((double)dims->dk));
    chunking(dims->dk, dims->dv, gdn::dtype_size(state_dtype), p.rows, p.nchunk);
    const int tmax = T <= 4 ? 4 : 8;
    bool too_big = false;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (state_dtype == GDN_F32)
        e = gdn::dispatch_spec_f32(dims->dk, tmax, p, s, too_big);
    else if (state_dtype == GDN_BF16)
        e = gdn::dispatch_spec_bf16(dims->dk, tmax, p, s, too_big);
    else
        e = gdn::dispatch_spec_f16(dims->dk, tmax, p, s, too_big);
    if (too_big) return fail(GDN_ERR_SHAPE, "%s: T=%d, dv=%d do not fit in shared memory", fn, T, dims->dv);
    return launched(e, fn);
}

int gdn_prefill(const gdn_dims* dims, void* state_pool, int32_t state_dtype, const int32_t* slots,
                const int32_t* cu_seqlens, int32_t total_tokens, const void* q, const void* k, const void* v,
                const void* a, const void* b, int32_t in_dtype, const float* A_log, const float* dt_bias,
                int32_t state_write_interval, void* out, int32_t out_dtype, int32_t* dev_err, void* stream) {
    const char* fn = "gdn_prefill";
    int rc = check_dims(dims, fn);
    if (rc) return rc;
    if (state_write_interval < 1) return fail(GDN_ERR_WINDOW, "%s: state_write_interval=%d < 1", fn, state_write_interval);
    if (total_tokens < 0) return fail(GDN_ERR_SHAPE, "%s: total_tokens=%d < 0", fn, total_tokens);
    if ((int64_t)total_tokens * dims->Hv > (int64_t)INT32_MAX / 8)
        return fail(GDN_ERR_SHAPE, "%s: total_tokens*Hv too large", fn);
    if (dims->B == 0) return GDN_OK;
    if (!state_pool || !slots || !cu_seqlens || !dev_err)
        return fail(GDN_ERR_NULL, "%s: state_pool, slots, cu_seqlens or dev_err is NULL", fn);
    if (!dtype_ok(state_dtype)) return fail(GDN_ERR_DTYPE, "%s: unsupported state dtype %d", fn, state_dtype);
    rc = check_activations(fn, q, k, v, a, b, in_dtype, A_log, dt_bias, out, out_dtype);
    if (rc) return rc;
    if (!aligned16(state_pool) || !aligned16(out) || !aligned_to(slots, 4) || !aligned_to(cu_seqlens, 4) ||
        !aligned_to(dev_err, 4))
        return fail(GDN_ERR_ALIGN, "%s: state_pool and out must be 16-byte aligned", fn);
    gdn::PrefillArgs p{};
    p.pool = state_pool, p.slots = slots, p.cu_seqlens = cu_seqlens;
    p.q = q, p.k = k, p.v = v, p.a = a, p.b = b, p.A_log = A_log, p.dt_bias = dt_bias;
    p.out = out, p.dev_err = dev_err;
    p.num_slots = dims->num_slots;
    p.B = dims->B, p.Hk = dims->Hk, p.Hv = dims->Hv, p.dv = dims->dv, p.total = total_tokens;
    p.interval = state_write_interval;
    p.in_dtype = in_dtype, p.out_dtype = out_dtype;
    p.row_blocks = (dims->dv + gdn::PF_ROWS - 1) / gdn::PF_ROWS;
    p.q_scale = (float)(1.0 / sqrt((double)dims->dk));
    return launched(gdn::dispatch_prefill(state_dtype, dims->dk, p, static_cast<cudaStream_t>(stream)), fn);
}

int gdn_replay_step(const gdn_dims* dims, const gdn_replay_cache* cache, const int32_t* slots, const void* q,
                    const void* k, const void* v, const void* a, const void* b, int32_t in_dtype, const float* A_log,
                    const float* dt_bias, void* out, int32_t out_dtype, int32_t* dev_err, void* stream) {
    return replay_common("gdn_replay_step", gdn::RULE_GDN, dims, cache, slots, 1, 0, q, k, v, a, b, in_dtype, A_log,
                         dt_bias, nullptr, out, out_dtype, dev_err, stream);
}

int gdn_verify_window(const gdn_dims* dims, const gdn_replay_cache* cache, const int32_t* slots, int32_t T,
                      const void* q, const void* k, const void* v, const void* a, const void* b, int32_t in_dtype,
                      const float* A_log, const float* dt_bias, void* out, int32_t out_dtype, int32_t* dev_err,
                      void* stream) {
    if (T < 1) return fail(GDN_ERR_WINDOW, "gdn_verify_window: T=%d must be >= 1", T);
    return replay_common("gdn_verify_window", gdn::RULE_GDN, dims, cache, slots, T, 0, q, k, v, a, b, in_dtype,
                         A_log, dt_bias, nullptr, out, out_dtype, dev_err, stream);
}

int gdn_replay_flush(const gdn_dims* dims, const gdn_replay_cache* cache, const int32_t* slots, int32_t force,
                     int32_t* dev_err, void* stream) {
    return replay_common("gdn_replay_flush", gdn::RULE_GDN, dims, cache, slots, 0, force, nullptr, nullptr, nullptr,
                         nullptr, nullptr, cache ? cache->ring_dtype : GDN_F32, nullptr, nullptr, nullptr, nullptr,
                         GDN_F32, dev_err, stream);
}

int gdn_rollback(const gdn_dims* dims, const gdn_replay_cache* cache, const int32_t* slots, const int32_t* accepted,
                 int32_t T, int32_t* dev_err, void* stream) {
    const char* fn = "gdn_rollback";
    int rc = check_dims(dims, fn);
    if (rc) return rc;
    if (!cache) return fail(GDN_ERR_NULL, "%s: cache is NULL", fn);
    if (dims->B == 0) return GDN_OK;
    if (!cache->pos || !cache->ckpt_pos || !cache->ring_rec || !slots || !accepted || !dev_err)
        return fail(GDN_ERR_NULL, "%s: pos, ckpt_pos, ring_rec, slots, accepted or dev_err is NULL", fn);
    if (cache->L < 1 || cache->L > gdn::L_MAX) return fail(GDN_ERR_WINDOW, "%s: L=%d not in [1, 64]", fn, cache->L);
    if (T < 1 || T > cache->L || T > gdn::WINDOW_MAX)
        return fail(GDN_ERR_WINDOW, "%s: T=%d not in [1, min(L, 8)]", fn, T);
    if (!aligned_to(cache->pos, 4) || !aligned_to(cache->ckpt_pos, 4) || !aligned16(cache->ring_rec))
        return fail(GDN_ERR_ALIGN, "%s: pos, ckpt_pos or ring_rec misaligned", fn);
    return launched(gdn::launch_rollback(cache->pos, cache->ckpt_pos, cache->ring_rec, slots, accepted, dims->B,
                                         dims->Hv, T, cache->L, dims->dv, dims->num_slots, dev_err,
                                         static_cast<cudaStream_t>(stream)),
                    fn);
}

// ---------------------------------------------------------------- Mamba2

}  // extern "C"

namespace {

int m2_dims(const mamba2_dims* m, gdn_dims& d, const char* fn) {
    if (!m) return fail(GDN_ERR_NULL, "%s: dims is NULL", fn);
    d.B = m->B, d.Hk = m->G, d.Hv = m->H, d.dk = m->N, d.dv = m->P, d.num_slots = m->num_slots;
    return check_dims(&d, fn);
}

}  // namespace

extern "C" {

int mamba2_decode_step(const mamba2_dims* dims, void* state_pool, int32_t state_dtype, const int32_t* slots,
                       const void* x, const void* dt, const void* Bm, const void* Cm, int32_t in_dtype,
                       const float* A_log, const float* dt_bias, const float* D, void* out, int32_t out_dtype,
                       int32_t* dev_err, void* stream) {
    const char* fn = "mamba2_decode_step";
    gdn_dims d;
    int rc = m2_dims(dims, d, fn);
    if (rc) return rc;
    if (d.B == 0) return GDN_OK;
    if (!state_pool || !slots || !dev_err) return fail(GDN_ERR_NULL, "%s: state_pool, slots or dev_err is NULL", fn);
    if (!dtype_ok(state_dtype)) return fail(GDN_ERR_DTYPE, "%s: unsupported state dtype %d", fn, state_dtype);
    rc = check_activations(fn, Cm, Bm, x, dt, dt, in_dtype, A_log, dt_bias, out, out_dtype);
    if (rc) return rc;
    if (!D) return fail(GDN_ERR_NULL, "%s: D is NULL", fn);
    if (!aligned16(state_pool) || !aligned_to(slots, 4) || !aligned_to(dev_err, 4) || !aligned_to(D, 4))
        return fail(GDN_ERR_ALIGN, "%s: state_pool must be 16-byte aligned", fn);
    gdn::DecodeArgs p{};
    p.pool = state_pool, p.slots = slots, p.q = Cm, p.k = Bm, p.v = x, p.a = dt, p.b = nullptr;
    p.A_log = A_log, p.dt_bias = dt_bias, p.D = D, p.out = out, p.dev_err = dev_err;
    p.num_slots = d.num_slots;
    p.B = d.B, p.Hk = d.Hk, p.Hv = d.Hv, p.dv = d.dv;
    p.in_dtype = in_dtype, p.out_dtype = out_dtype;
    p.q_scale = 1.f;
    chunking(d.dk, d.dv, gdn::dtype_size(state_dtype), p.rows, p.nchunk);
    return launched(gdn::dispatch_mamba2_decode(state_dtype, d.dk, p, static_cast<cudaStream_t>(stream)), fn);
}

int mamba2_verify_window(const mamba2_dims* dims, const gdn_replay_cache* cache, const int32_t* slots, int32_t T,
                         const void* x, const void* dt, const void* Bm, const void* Cm, int32_t in_dtype,
                         const float* A_log, const float* dt_bias, const float* D, void* out, int32_t out_dtype,
                         int32_t* dev_err, void* stream) {
    const char* fn = T == 1 ? "mamba2_replay_step" : "mamba2_verify_window";
    if (T < 1) return fail(GDN_ERR_WINDOW, "%s: T=%d must be >= 1", fn, T);
    gdn_dims d;
    int rc = m2_dims(dims, d, fn);
    if (rc) return rc;
    return replay_common(fn, gdn::RULE_MAMBA2, &d, cache, slots, T, 0, Cm, Bm, x, dt, nullptr, in_dtype, A_log,
                         dt_bias, D, out, out_dtype, dev_err, stream);
}

int mamba2_replay_step(const mamba2_dims* dims, const gdn_replay_cache* cache, const int32_t* slots, const void* x,
                       const void* dt, const void* Bm, const void* Cm, int32_t in_dtype, const float* A_log,
                       const float* dt_bias, const float* D, void* out, int32_t out_dtype, int32_t* dev_err,
                       void* stream) {
    return mamba2_verify_window(dims, cache, slots, 1, x, dt, Bm, Cm, in_dtype, A_log, dt_bias, D, out, out_dtype,
                                dev_err, stream);
}

int mamba2_replay_flush(const mamba2_dims* dims, const gdn_replay_cache* cache, const int32_t* slots, int32_t force,
                        int32_t* dev_err, void* stream) {
    const char* fn = "mamba2_replay_flush";
    gdn_dims d;
    int rc = m2_dims(dims, d, fn);
    if (rc) return rc;
    return replay_common(fn, gdn::RULE_MAMBA2, &d, cache, slots, 0, force, nullptr, nullptr, nullptr, nullptr,
                         nullptr, cache ? cache->ring_dtype : GDN_F32, nullptr, nullptr, nullptr, nullptr, GDN_F32,
                         dev_err, stream);
}

int mamba2_rollback(const mamba2_dims* dims, const gdn_replay_cache* cache, const int32_t* slots,
                    const int32_t* accepted, int32_t T, int32_t* dev_err, void* stream) {
    gdn_dims d;
    int rc = m2_dims(dims, d, "mamba2_rollback");
    if (rc) return rc;
    return gdn_rollback(&d, cache, slots, accepted, T, dev_err, stream);
}

const char* gdn_last_error_string(void) { return g_last_error.c_str(); }

int32_t gdn_abi_version(void) { return GDN_ABI_VERSION; }

}  // extern "C"
