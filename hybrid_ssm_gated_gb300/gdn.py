"""Thin ctypes binding of the C ABI in include/gdn.h.

Functions carry the C entry points' names and only marshal arguments: they
read shapes and dtypes off torch tensors, pass raw device pointers and the
current CUDA stream, and raise GdnError on a non-zero return code. Every step
of the computation runs in libgdn.so; there is no fallback of any kind: if the
library is missing or a tensor is not a contiguous CUDA tensor, the call fails.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# GDN_LIBRARY may point at another build of the same library (e.g. a tuning variant)
LIB_PATH = os.environ.get("GDN_LIBRARY") or os.path.join(HERE, "lib", "libgdn.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "gdn.h")

GDN_F32, GDN_BF16, GDN_F16 = 0, 1, 2
DTYPE_CODE = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16, torch.float16: GDN_F16}
DEVERR_SLOT, DEVERR_RING, DEVERR_ACCEPT, DEVERR_TIMEOUT, DEVERR_SEQLEN, DEVERR_BOUNDS = 1, 2, 4, 8, 16, 32


class GdnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class gdn_dims(C.Structure):
    _fields_ = [("B", C.c_int32), ("Hk", C.c_int32), ("Hv", C.c_int32), ("dk", C.c_int32), ("dv", C.c_int32),
                ("num_slots", C.c_int64)]


class gdn_replay_cache(C.Structure):
    _fields_ = [("ckpt", C.c_void_p), ("ckpt_dtype", C.c_int32), ("ring_k", C.c_void_p), ("ring_v", C.c_void_p),
                ("ring_dtype", C.c_int32), ("ring_rec", C.c_void_p), ("pos", C.c_void_p),
                ("ckpt_pos", C.c_void_p), ("L", C.c_int32), ("ckpt_read", C.c_void_p), ("read_dtype", C.c_int32)]


class mamba2_dims(C.Structure):
    _fields_ = [("B", C.c_int32), ("G", C.c_int32), ("H", C.c_int32), ("N", C.c_int32), ("P", C.c_int32),
                ("num_slots", C.c_int64)]


_lib = None
_P = C.c_void_p
_I = C.c_int32
_SIGS = {
    "gdn_decode_step": [C.POINTER(gdn_dims), _P, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P],
    "gdn_prefill": [C.POINTER(gdn_dims), _P, _I, _P, _P, _I, _P, _P, _P, _P, _P, _I, _P, _P, _I, _P, _I, _P, _P],
    "gdn_spec_step": [C.POINTER(gdn_dims), _P, _I, _P, _P, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P],
    "gdn_replay_step": [C.POINTER(gdn_dims), C.POINTER(gdn_replay_cache), _P, _P, _P, _P, _P, _P, _I, _P, _P, _P,
                        _I, _P, _P],
    "gdn_verify_window": [C.POINTER(gdn_dims), C.POINTER(gdn_replay_cache), _P, _I, _P, _P, _P, _P, _P, _I, _P, _P,
                          _P, _I, _P, _P],
    "gdn_replay_flush": [C.POINTER(gdn_dims), C.POINTER(gdn_replay_cache), _P, _I, _P, _P],
    "gdn_rollback": [C.POINTER(gdn_dims), C.POINTER(gdn_replay_cache), _P, _P, _I, _P, _P],
    "mamba2_decode_step": [C.POINTER(mamba2_dims), _P, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _P, _P],
    "mamba2_replay_step": [C.POINTER(mamba2_dims), C.POINTER(gdn_replay_cache), _P, _P, _P, _P, _P, _I, _P, _P, _P,
                           _P, _I, _P, _P],
    "mamba2_verify_window": [C.POINTER(mamba2_dims), C.POINTER(gdn_replay_cache), _P, _I, _P, _P, _P, _P, _I, _P,
                             _P, _P, _P, _I, _P, _P],
    "mamba2_replay_flush": [C.POINTER(mamba2_dims), C.POINTER(gdn_replay_cache), _P, _I, _P, _P],
    "mamba2_rollback": [C.POINTER(mamba2_dims), C.POINTER(gdn_replay_cache), _P, _P, _I, _P, _P],
}


def lib() -> C.CDLL:
    """The loaded libgdn.so (built by hybrid_ssm_gated_gb300.build.build()). The environment variable
    GDN_LIBRARY names another build of it to load instead, such as the bounds-checking one
    (build.build(debug=True))."""
    global _lib
    if _lib is None:
        path = LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with hybrid_ssm_gated_gb300.build.build()")
        lib_ = C.CDLL(path)
        for name, args in _SIGS.items():
            fn = getattr(lib_, name)
            fn.argtypes = args
            fn.restype = C.c_int
        lib_.gdn_last_error_string.restype = C.c_char_p
        lib_.gdn_last_error_string.argtypes = []
        lib_.gdn_abi_version.restype = C.c_int32
        _lib = lib_
    return _lib


def declared_symbols() -> list[str]:
    """Names of the functions include/gdn.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*((?:gdn|mamba2)_[a-z_0-9]+)\s*\(", text,
                                 re.M)))


def gdn_last_error_string() -> str:
    return lib().gdn_last_error_string().decode()


def gdn_abi_version() -> int:
    return int(lib().gdn_abi_version())


def _check(rc: int) -> None:
    if rc != 0:
        raise GdnError(rc, gdn_last_error_string())


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("gdn: every tensor argument must be a contiguous CUDA tensor")
    return t.data_ptr()


def _code(t: torch.Tensor) -> int:
    try:
        return DTYPE_CODE[t.dtype]
    except KeyError:
        raise ValueError(f"gdn: unsupported dtype {t.dtype}") from None


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_dims(B: int, Hk: int, Hv: int, dk: int, dv: int, num_slots: int) -> gdn_dims:
    return gdn_dims(B, Hk, Hv, dk, dv, num_slots)


def gdn_decode_step(state_pool, slots, q, k, v, a, b, A_log, dt_bias, out, dev_err, stream=None) -> None:
    """state_pool [num_slots, Hv, dv, dk]; slots [B] int32; q, k [B, Hk, dk];
    v [B, Hv, dv]; a, b [B, Hv]; A_log, dt_bias [Hv] fp32; out [B, Hv, dv];
    dev_err [1] int32. Enqueued on `stream` (default: the current stream)."""
    num_slots, Hv, dv, dk = state_pool.shape
    B = slots.shape[0]
    d = make_dims(B, q.shape[-2], Hv, dk, dv, num_slots)
    _check(lib().gdn_decode_step(C.byref(d), _ptr(state_pool), _code(state_pool), _ptr(slots), _ptr(q), _ptr(k),
                                 _ptr(v), _ptr(a), _ptr(b), _code(q), _ptr(A_log), _ptr(dt_bias), _ptr(out),
                                 _code(out), _ptr(dev_err), _stream(stream)))


def gdn_spec_step(state_pool, src_slots, dst_slots, q, k, v, a, b, A_log, dt_bias, out, dev_err,
                  stream=None) -> None:
    """Speculative step with one state copy per window token: state_pool [num_slots, Hv, dv, dk];
    src_slots [B] int32; dst_slots [B, T] int32; q, k [B, T, Hk, dk]; v [B, T, Hv, dv];
    a, b [B, T, Hv]; A_log, dt_bias [Hv] fp32; out [B, T, Hv, dv]; dev_err [1] int32."""
    num_slots, Hv, dv, dk = state_pool.shape
    B, T = dst_slots.shape
    d = make_dims(B, q.shape[-2], Hv, dk, dv, num_slots)
    _check(lib().gdn_spec_step(C.byref(d), _ptr(state_pool), _code(state_pool), _ptr(src_slots), _ptr(dst_slots),
                               int(T), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _code(q), _ptr(A_log),
                               _ptr(dt_bias), _ptr(out), _code(out), _ptr(dev_err), _stream(stream)))


def gdn_prefill(state_pool, slots, cu_seqlens, q, k, v, a, b, A_log, dt_bias, out, dev_err, state_write_interval: int,
                stream=None) -> None:
    """Prefill of variable-length sequences: state_pool [num_slots, Hv, dv, dk]; slots [B] int32;
    cu_seqlens [B + 1] int32 (device); q, k [total, Hk, dk]; v [total, Hv, dv]; a, b [total, Hv];
    out [total, Hv, dv]; the state rounded to its dtype every state_write_interval tokens."""
    num_slots, Hv, dv, dk = state_pool.shape
    total = q.shape[0]
    d = make_dims(slots.shape[0], q.shape[-2], Hv, dk, dv, num_slots)
    _check(lib().gdn_prefill(C.byref(d), _ptr(state_pool), _code(state_pool), _ptr(slots), _ptr(cu_seqlens),
                             int(total), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _code(q), _ptr(A_log),
                             _ptr(dt_bias), int(state_write_interval), _ptr(out), _code(out), _ptr(dev_err),
                             _stream(stream)))


class ReplayCache:
    """Device tensors of a ReplaySSM cache (layouts as in include/gdn.h).

    ckpt [num_slots, Hv, dv, dk]; ring_k [num_slots, Hv, L, dk];
    ring_v [num_slots, Hv, L, dv]; ring_rec [num_slots, Hv, L, 4 + dv] fp32;
    pos, ckpt_pos [num_slots, Hv] int32; ckpt_read: None, or the low-precision read copy
    [num_slots, Hv, dv, dk] (bf16/fp16) of an fp32 ckpt.
    """

    def __init__(self, ckpt, ring_k, ring_v, ring_rec, pos, ckpt_pos, L: int, ckpt_read=None):
        self.ckpt, self.ring_k, self.ring_v, self.ring_rec = ckpt, ring_k, ring_v, ring_rec
        self.pos, self.ckpt_pos, self.L = pos, ckpt_pos, int(L)
        self.ckpt_read = ckpt_read

    @classmethod
    def allocate(cls, num_slots, Hv, dk, dv, L, ckpt_dtype=torch.float32, ring_dtype=torch.bfloat16,
                 device="cuda", read_dtype=None) -> "ReplayCache":
        """Zero-initialised cache; the caller then writes checkpoints (and the read copy, the
        checkpoint rounded, when read_dtype is given) and pointers."""
        z = lambda shape, dt: torch.zeros(shape, dtype=dt, device=device)
        read = None if read_dtype is None else z((num_slots, Hv, dv, dk), read_dtype)
        return cls(z((num_slots, Hv, dv, dk), ckpt_dtype), z((num_slots, Hv, L, dk), ring_dtype),
                   z((num_slots, Hv, L, dv), ring_dtype), z((num_slots, Hv, L, 4 + dv), torch.float32),
                   z((num_slots, Hv), torch.int32), z((num_slots, Hv), torch.int32), L, read)

    @property
    def shape(self):
        return self.ckpt.shape  # num_slots, Hv, dv, dk

    def c_struct(self) -> gdn_replay_cache:
        read = self.ckpt_read
        return gdn_replay_cache(_ptr(self.ckpt), _code(self.ckpt), _ptr(self.ring_k), _ptr(self.ring_v),
                                _code(self.ring_k), _ptr(self.ring_rec), _ptr(self.pos), _ptr(self.ckpt_pos),
                                self.L, None if read is None else _ptr(read), 0 if read is None else _code(read))


def _replay_dims(cache: ReplayCache, slots, q) -> gdn_dims:
    num_slots, Hv, dv, dk = cache.shape
    Hk = q.shape[-2] if q is not None else Hv
    return make_dims(slots.shape[0], Hk, Hv, dk, dv, num_slots)


def gdn_replay_step(cache: ReplayCache, slots, q, k, v, a, b, A_log, dt_bias, out, dev_err, stream=None) -> None:
    """One ReplaySSM decode step; arguments shaped as for gdn_decode_step."""
    d = _replay_dims(cache, slots, q)
    cs = cache.c_struct()
    _check(lib().gdn_replay_step(C.byref(d), C.byref(cs), _ptr(slots), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                 _code(q), _ptr(A_log), _ptr(dt_bias), _ptr(out), _code(out), _ptr(dev_err),
                                 _stream(stream)))


def gdn_verify_window(cache: ReplayCache, slots, q, k, v, a, b, A_log, dt_bias, out, dev_err, stream=None) -> None:
    """Verify a T-token window: q, k [B, T, Hk, dk]; v [B, T, Hv, dv]; a, b [B, T, Hv];
    out [B, T, Hv, dv]."""
    T = q.shape[1]
    d = _replay_dims(cache, slots, q)
    cs = cache.c_struct()
    _check(lib().gdn_verify_window(C.byref(d), C.byref(cs), _ptr(slots), T, _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                   _ptr(b), _code(q), _ptr(A_log), _ptr(dt_bias), _ptr(out), _code(out),
                                   _ptr(dev_err), _stream(stream)))


def gdn_replay_flush(cache: ReplayCache, slots, force: bool, dev_err, Hk: int | None = None, stream=None) -> None:
    """Fold the ring into the checkpoint (every full ring, or every non-empty one when force)."""
    d = _replay_dims(cache, slots, None)
    if Hk is not None:
        d.Hk = Hk
    cs = cache.c_struct()
    _check(lib().gdn_replay_flush(C.byref(d), C.byref(cs), _ptr(slots), int(bool(force)), _ptr(dev_err),
                                  _stream(stream)))


def gdn_rollback(cache: ReplayCache, slots, accepted, T: int, dev_err, stream=None) -> None:
    """Keep 1 + accepted[b] of the last verify window's T tokens (pointer move only)."""
    d = _replay_dims(cache, slots, None)
    cs = cache.c_struct()
    _check(lib().gdn_rollback(C.byref(d), C.byref(cs), _ptr(slots), _ptr(accepted), int(T), _ptr(dev_err),
                              _stream(stream)))


# ---------------------------------------------------------------- Mamba2


def _m2_dims(num_slots: int, H: int, P: int, N: int, B: int, G: int) -> mamba2_dims:
    return mamba2_dims(B, G, H, N, P, num_slots)


def mamba2_decode_step(state_pool, slots, x, dt, Bm, Cm, A_log, dt_bias, D, out, dev_err, stream=None) -> None:
    """Mamba2 decode step: state_pool [num_slots, H, P, N]; slots [B] int32; x [B, H, P]; dt [B, H];
    Bm, Cm [B, G, N]; A_log, dt_bias, D [H] fp32; out [B, H, P]; dev_err [1] int32."""
    num_slots, H, P, N = state_pool.shape
    d = _m2_dims(num_slots, H, P, N, slots.shape[0], Bm.shape[-2])
    _check(lib().mamba2_decode_step(C.byref(d), _ptr(state_pool), _code(state_pool), _ptr(slots), _ptr(x), _ptr(dt),
                                    _ptr(Bm), _ptr(Cm), _code(x), _ptr(A_log), _ptr(dt_bias), _ptr(D), _ptr(out),
                                    _code(out), _ptr(dev_err), _stream(stream)))


def _m2_replay_dims(cache: ReplayCache, slots, Bm) -> mamba2_dims:
    num_slots, H, P, N = cache.shape
    return _m2_dims(num_slots, H, P, N, slots.shape[0], Bm.shape[-2] if Bm is not None else H)


def mamba2_replay_step(cache: ReplayCache, slots, x, dt, Bm, Cm, A_log, dt_bias, D, out, dev_err,
                       stream=None) -> None:
    """One Mamba2 ReplaySSM step; arguments shaped as for mamba2_decode_step."""
    d = _m2_replay_dims(cache, slots, Bm)
    cs = cache.c_struct()
    _check(lib().mamba2_replay_step(C.byref(d), C.byref(cs), _ptr(slots), _ptr(x), _ptr(dt), _ptr(Bm), _ptr(Cm),
                                    _code(x), _ptr(A_log), _ptr(dt_bias), _ptr(D), _ptr(out), _code(out),
                                    _ptr(dev_err), _stream(stream)))


def mamba2_verify_window(cache: ReplayCache, slots, x, dt, Bm, Cm, A_log, dt_bias, D, out, dev_err,
                         stream=None) -> None:
    """A T-token Mamba2 verify window: x [B, T, H, P]; dt [B, T, H]; Bm, Cm [B, T, G, N];
    out [B, T, H, P]."""
    T = x.shape[1]
    d = _m2_replay_dims(cache, slots, Bm)
    cs = cache.c_struct()
    _check(lib().mamba2_verify_window(C.byref(d), C.byref(cs), _ptr(slots), T, _ptr(x), _ptr(dt), _ptr(Bm),
                                      _ptr(Cm), _code(x), _ptr(A_log), _ptr(dt_bias), _ptr(D), _ptr(out),
                                      _code(out), _ptr(dev_err), _stream(stream)))


def mamba2_replay_flush(cache: ReplayCache, slots, force: bool, dev_err, stream=None) -> None:
    """Fold Mamba2 rings into their checkpoints (full ones, or every non-empty one when force)."""
    d = _m2_replay_dims(cache, slots, None)
    cs = cache.c_struct()
    _check(lib().mamba2_replay_flush(C.byref(d), C.byref(cs), _ptr(slots), int(bool(force)), _ptr(dev_err),
                                     _stream(stream)))


def mamba2_rollback(cache: ReplayCache, slots, accepted, T: int, dev_err, stream=None) -> None:
    """Keep 1 + accepted[b] of the last Mamba2 verify window's T tokens (pointer move only)."""
    d = _m2_replay_dims(cache, slots, None)
    cs = cache.c_struct()
    _check(lib().mamba2_rollback(C.byref(d), C.byref(cs), _ptr(slots), _ptr(accepted), int(T), _ptr(dev_err),
                                 _stream(stream)))
