"""CPU oracle for the GDN and Mamba2 decode steps and their ReplaySSM mode
(ctypes wrapper).

TEST INFRASTRUCTURE ONLY. Only tests/, the package smoke check and the
benchmark's CPU-baseline leg may import this package. It shares no code with
the CUDA library: the arithmetic lives in gdn_oracle.c and mamba2_oracle.c
(plain C, fp64).

Storage arrays follow hybrid_ssm_gated_gb300.workload: fp32 as float32, fp16 as
float16, bf16 as uint16 bit patterns, and the oracle-only fp64 as float64.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .build import build

F32, BF16, F16, F64 = 0, 1, 2, 3
CODE = {"f32": F32, "bf16": BF16, "f16": F16, "f64": F64}
NPTYPE = {F32: np.float32, BF16: np.uint16, F16: np.float16, F64: np.float64}

_lib = None


def lib() -> C.CDLL:
    """The oracle library: this package's build, or the one ORACLE_LIBRARY names (the planted-mistake
    tests point it at altered copies)."""
    global _lib
    if _lib is None:
        _lib = C.CDLL(os.environ.get("ORACLE_LIBRARY") or build())
        P, I, I64, D = C.c_void_p, C.c_int, C.c_int64, C.c_double
        sig = {
            "orc_round": (D, [D, I]),
            "orc_round_array": (None, [P, I64, I, P]),
            "orc_load_array": (None, [P, I64, I, P]),
            "orc_gating": (None, [D, D, D, D, P, P]),
            "orc_l2norm": (None, [I, P, D, P]),
            "orc_decode_head": (None, [I, I, P, I, P, P, P, I, D, D, P]),
            "orc_decode_step": (I, [I, I, I, I, I, I64, P, I, P, P, P, P, P, P, I, P, P, P, I]),
            "orc_spec_head": (None, [I, I, I, P, I, P, P, P, P, P, I, P, P, P]),
            "orc_spec_step": (I, [I, I, I, I, I, I, I64, P, I, P, P, P, P, P, P, P, I, P, P, P, I]),
            "orc_replay_window": (I, [I, I, I, P, I, P, P, I, P, P, P, I, P, P, P, P, P, D, D, P]),
            "orc_replay_flush": (I, [I, I, I, P, I, P, P, I, P, P, P, I]),
            "orc_replay_rollback": (I, [P, I, I]),
            "orc_replay2_window": (I, [I, I, I, P, I, P, I, P, P, I, P, P, P, I, P, P, P, P, P, D, D, P]),
            "orc_replay2_flush": (I, [I, I, I, P, I, P, I, P, P, I, P, P, P, I]),
            "orc_prefill_head": (None, [I, I, I, P, I, P, P, P, I, P, P, I, P]),
            "orc_prefill": (I, [I, I, I, I, I, I64, P, I, P, P, P, P, P, P, P, I, P, P, I, P, I]),
            "orc_m2_gating": (None, [D, D, D, P, P]),
            "orc_m2_decode_head": (None, [I, I, P, I, P, P, P, I, D, D, D, P]),
            "orc_m2_decode_step": (I, [I, I, I, I, I, I64, P, I, P, P, P, P, P, I, P, P, P, P, I]),
            "orc_m2_replay_window": (I, [I, I, I, P, I, P, P, I, P, P, P, I, P, P, P, P, D, D, D, P]),
            "orc_m2_replay_flush": (I, [I, I, I, P, I, P, P, I, P, P, P, I]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(_lib, name)
            fn.restype = res
            fn.argtypes = args
    return _lib


def _code(dt) -> int:
    return CODE[dt] if isinstance(dt, str) else int(dt)


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _arr(x, dt) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=NPTYPE[_code(dt)])


# ---------------------------------------------------------------- formats


def round_to(x: np.ndarray, dtype) -> np.ndarray:
    """Round fp64 values to a storage dtype; returns the storage array."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=NPTYPE[_code(dtype)])
    lib().orc_round_array(_ptr(x), x.size, _code(dtype), _ptr(out))
    return out


def load(arr: np.ndarray, dtype) -> np.ndarray:
    """Exact fp64 values of a storage array."""
    arr = _arr(arr, dtype)
    out = np.empty(arr.shape, dtype=np.float64)
    lib().orc_load_array(_ptr(arr), arr.size, _code(dtype), _ptr(out))
    return out


def gating(A_log: float, dt_bias: float, a: float, b: float) -> tuple[float, float]:
    al, be = C.c_double(), C.c_double()
    lib().orc_gating(float(A_log), float(dt_bias), float(a), float(b), C.addressof(al), C.addressof(be))
    return al.value, be.value


def l2norm(x: np.ndarray, scale: float = 1.0) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib().orc_l2norm(x.size, _ptr(x), float(scale), _ptr(y))
    return y


# ---------------------------------------------------------------- decode


def decode_head(S: np.ndarray, sdt, q, k, v, idt, alpha: float, beta: float) -> np.ndarray:
    """One decode step of one head; S ([dv, dk] storage array) is updated in place."""
    assert S.dtype == NPTYPE[_code(sdt)] and S.flags["C_CONTIGUOUS"]
    dv, dk = S.shape
    q, k, v = _arr(q, idt), _arr(k, idt), _arr(v, idt)
    out = np.empty(dv, dtype=np.float64)
    lib().orc_decode_head(dk, dv, _ptr(S), _code(sdt), _ptr(q), _ptr(k), _ptr(v), _code(idt),
                          float(alpha), float(beta), _ptr(out))
    return out


def decode_step(pool: np.ndarray, sdt, slots, q, k, v, a, b, idt, A_log, dt_bias,
                nthreads: int = 1) -> tuple[np.ndarray, int]:
    """One decode step of a batch; pool [num_slots, Hv, dv, dk] is updated in place.

    Returns (out [B, Hv, dv] fp64, number of (sequence, head) units whose slot
    was out of range).
    """
    assert pool.dtype == NPTYPE[_code(sdt)] and pool.flags["C_CONTIGUOUS"]
    num_slots, Hv, dv, dk = pool.shape
    q, k, v, a, b = (_arr(x, idt) for x in (q, k, v, a, b))
    B = int(np.asarray(slots).shape[0])
    Hk = q.size // (B * dk)
    slots = np.ascontiguousarray(slots, dtype=np.int32)
    A_log = np.ascontiguousarray(A_log, dtype=np.float32)
    dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float32)
    out = np.empty((B, Hv, dv), dtype=np.float64)
    bad = lib().orc_decode_step(B, Hk, Hv, dk, dv, num_slots, _ptr(pool), _code(sdt), _ptr(slots),
                                _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _code(idt),
                                _ptr(A_log), _ptr(dt_bias), _ptr(out), int(nthreads))
    return out, bad


# ---------------------------------------------------------------- speculative step


def spec_head(S: np.ndarray, sdt, q, k, v, idt, alpha, beta, write=None) -> tuple[np.ndarray, np.ndarray]:
    """One head's speculative step over a T-token window from the state S ([dv, dk] storage array,
    not modified): q, k [T, dk] and v [T, dv] in idt, gates alpha, beta [T]. Returns (out [T, dv]
    fp64, copies [T, dv, dk] in sdt: the state after each token, rounded once; rows where write is
    False are left zero)."""
    assert S.dtype == NPTYPE[_code(sdt)] and S.flags["C_CONTIGUOUS"]
    dv, dk = S.shape
    q, k, v = _arr(q, idt), _arr(k, idt), _arr(v, idt)
    T = q.shape[0]
    alpha = np.ascontiguousarray(alpha, dtype=np.float64)
    beta = np.ascontiguousarray(beta, dtype=np.float64)
    write = np.ones(T, np.int32) if write is None else np.ascontiguousarray(write, dtype=np.int32)
    out = np.empty((T, dv), dtype=np.float64)
    copies = np.zeros((T, dv, dk), dtype=S.dtype)
    lib().orc_spec_head(dk, dv, T, _ptr(S), _code(sdt), _ptr(copies), _ptr(write), _ptr(q), _ptr(k), _ptr(v),
                        _code(idt), _ptr(alpha), _ptr(beta), _ptr(out))
    return out, copies


def spec_step(pool: np.ndarray, sdt, src_slots, dst_slots, q, k, v, a, b, idt, A_log, dt_bias,
              nthreads: int = 1) -> tuple[np.ndarray, int]:
    """Speculative step of a batch with one state copy per window token: pool [num_slots, Hv, dv,
    dk] is updated in place; src_slots [B], dst_slots [B, T] (< 0: no copy); q, k [B, T, Hk, dk],
    v [B, T, Hv, dv], a, b [B, T, Hv]. Returns (out [B, T, Hv, dv] fp64, number of units with an
    out-of-range slot)."""
    assert pool.dtype == NPTYPE[_code(sdt)] and pool.flags["C_CONTIGUOUS"]
    num_slots, Hv, dv, dk = pool.shape
    q, k, v, a, b = (_arr(x, idt) for x in (q, k, v, a, b))
    src_slots = np.ascontiguousarray(src_slots, dtype=np.int32)
    dst_slots = np.ascontiguousarray(dst_slots, dtype=np.int32)
    B, T = dst_slots.shape
    Hk = q.size // (B * T * dk)
    A_log = np.ascontiguousarray(A_log, dtype=np.float32)
    dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float32)
    out = np.empty((B, T, Hv, dv), dtype=np.float64)
    bad = lib().orc_spec_step(B, T, Hk, Hv, dk, dv, num_slots, _ptr(pool), _code(sdt), _ptr(src_slots),
                              _ptr(dst_slots), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _code(idt),
                              _ptr(A_log), _ptr(dt_bias), _ptr(out), int(nthreads))
    return out, bad


# ---------------------------------------------------------------- prefill


def prefill_head(S: np.ndarray, sdt, q, k, v, idt, alpha, beta, interval: int) -> np.ndarray:
    """Prefill of one head: T tokens from S ([dv, dk] storage array, updated in place), the state
    rounded to sdt after every `interval` tokens and after the last. Returns out [T, dv] fp64."""
    assert S.dtype == NPTYPE[_code(sdt)] and S.flags["C_CONTIGUOUS"]
    dv, dk = S.shape
    q, k, v = _arr(q, idt), _arr(k, idt), _arr(v, idt)
    T = q.shape[0]
    alpha = np.ascontiguousarray(alpha, dtype=np.float64)
    beta = np.ascontiguousarray(beta, dtype=np.float64)
    out = np.empty((T, dv), dtype=np.float64)
    lib().orc_prefill_head(dk, dv, T, _ptr(S), _code(sdt), _ptr(q), _ptr(k), _ptr(v), _code(idt), _ptr(alpha),
                           _ptr(beta), int(interval), _ptr(out))
    return out


def prefill(pool: np.ndarray, sdt, slots, cu_seqlens, q, k, v, a, b, idt, A_log, dt_bias, interval: int,
            nthreads: int = 1) -> tuple[np.ndarray, int]:
    """Prefill of variable-length sequences: sequence i owns tokens cu_seqlens[i]:cu_seqlens[i+1] of
    q, k [total, Hk, dk], v [total, Hv, dv], a, b [total, Hv]; pool [num_slots, Hv, dv, dk] updated
    in place. Returns (out [total, Hv, dv] fp64, number of refused units)."""
    assert pool.dtype == NPTYPE[_code(sdt)] and pool.flags["C_CONTIGUOUS"]
    num_slots, Hv, dv, dk = pool.shape
    q, k, v, a, b = (_arr(x, idt) for x in (q, k, v, a, b))
    slots = np.ascontiguousarray(slots, dtype=np.int32)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    B = slots.shape[0]
    total = int(cu[-1])
    Hk = q.size // max(1, total * dk) if total else 1
    A_log = np.ascontiguousarray(A_log, dtype=np.float32)
    dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float32)
    out = np.empty((total, Hv, dv), dtype=np.float64)
    bad = lib().orc_prefill(B, Hk, Hv, dk, dv, num_slots, _ptr(pool), _code(sdt), _ptr(slots), _ptr(cu), _ptr(q),
                            _ptr(k), _ptr(v), _ptr(a), _ptr(b), _code(idt), _ptr(A_log), _ptr(dt_bias), int(interval),
                            _ptr(out), int(nthreads))
    return out, bad


# ---------------------------------------------------------------- ReplaySSM


class ReplayHead:
    """ReplaySSM state of one (sequence, value head), as the oracle defines it.

    S0: the checkpoint (storage dtype). Entries buffered since the checkpoint
    are kept in arrival order (entry e is the e-th token after ckpt_pos):
    raw k [L, dk] and v [L, dv] in the input dtype, alpha/beta [L] fp64.
    meta = [count, pos, ckpt_pos].

    With read_dtype, S0 is a high-precision checkpoint used only for folding and
    Sr, its copy rounded to read_dtype, is what outputs read (orc_replay2_*).
    """

    def __init__(self, S0: np.ndarray, sdt, idt, L: int, pos: int = 0, read_dtype=None):
        self.sdt, self.idt, self.L = _code(sdt), _code(idt), int(L)
        self.S0 = np.ascontiguousarray(S0, dtype=NPTYPE[self.sdt]).copy()
        self.rdt = None if read_dtype is None else _code(read_dtype)
        self.Sr = None if self.rdt is None else round_to(load(self.S0, self.sdt), self.rdt)
        self.dv, self.dk = self.S0.shape
        self.ek = np.zeros((L, self.dk), dtype=NPTYPE[self.idt])
        self.ev = np.zeros((L, self.dv), dtype=NPTYPE[self.idt])
        self.ea = np.zeros(L, dtype=np.float64)
        self.eb = np.zeros(L, dtype=np.float64)
        self.meta = np.array([0, pos, pos], dtype=np.int32)

    @property
    def count(self) -> int:
        return int(self.meta[0])

    @property
    def pos(self) -> int:
        return int(self.meta[1])

    @property
    def ckpt_pos(self) -> int:
        return int(self.meta[2])

    def window(self, q, k, v, a, b, A_log: float, dt_bias: float) -> np.ndarray:
        """Process T tokens (T = q.shape[0]); returns out [T, dv] fp64."""
        q, k, v = _arr(q, self.idt), _arr(k, self.idt), _arr(v, self.idt)
        T = q.shape[0]
        a = np.ascontiguousarray(a, dtype=np.float64).reshape(T)
        b = np.ascontiguousarray(b, dtype=np.float64).reshape(T)
        out = np.empty((T, self.dv), dtype=np.float64)
        if self.rdt is None:
            rc = lib().orc_replay_window(self.dk, self.dv, self.L, _ptr(self.S0), self.sdt, _ptr(self.ek),
                                         _ptr(self.ev), self.idt, _ptr(self.ea), _ptr(self.eb),
                                         _ptr(self.meta), T, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                         float(A_log), float(dt_bias), _ptr(out))
        else:
            rc = lib().orc_replay2_window(self.dk, self.dv, self.L, _ptr(self.S0), self.sdt, _ptr(self.Sr), self.rdt,
                                          _ptr(self.ek), _ptr(self.ev), self.idt, _ptr(self.ea), _ptr(self.eb),
                                          _ptr(self.meta), T, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                          float(A_log), float(dt_bias), _ptr(out))
        if rc != 0:
            raise ValueError(f"oracle replay window rejected its input (code {rc})")
        return out

    def flush(self, force: bool = True) -> None:
        if self.rdt is None:
            rc = lib().orc_replay_flush(self.dk, self.dv, self.L, _ptr(self.S0), self.sdt, _ptr(self.ek),
                                        _ptr(self.ev), self.idt, _ptr(self.ea), _ptr(self.eb),
                                        _ptr(self.meta), int(bool(force)))
        else:
            rc = lib().orc_replay2_flush(self.dk, self.dv, self.L, _ptr(self.S0), self.sdt, _ptr(self.Sr), self.rdt,
                                         _ptr(self.ek), _ptr(self.ev), self.idt, _ptr(self.ea), _ptr(self.eb),
                                         _ptr(self.meta), int(bool(force)))
        if rc != 0:
            raise ValueError(f"oracle replay flush rejected its state (code {rc})")

    def rollback(self, T: int, accepted: int) -> None:
        rc = lib().orc_replay_rollback(_ptr(self.meta), int(T), int(accepted))
        if rc != 0:
            raise ValueError(f"oracle rollback rejected its input (code {rc})")


# ---------------------------------------------------------------- Mamba2


def m2_gating(A_log: float, dt_bias: float, dt: float) -> tuple[float, float]:
    """(alpha, delta) of one Mamba2 head: delta = softplus(dt + dt_bias), alpha = exp(-exp(A_log) delta)."""
    al, de = C.c_double(), C.c_double()
    lib().orc_m2_gating(float(A_log), float(dt_bias), float(dt), C.addressof(al), C.addressof(de))
    return al.value, de.value


def m2_decode_head(S: np.ndarray, sdt, x, Bv, Cv, idt, alpha: float, delta: float, D: float) -> np.ndarray:
    """One Mamba2 decode step of one head; S ([P, N] storage array) is updated in place."""
    assert S.dtype == NPTYPE[_code(sdt)] and S.flags["C_CONTIGUOUS"]
    P, N = S.shape
    x, Bv, Cv = _arr(x, idt), _arr(Bv, idt), _arr(Cv, idt)
    out = np.empty(P, dtype=np.float64)
    lib().orc_m2_decode_head(N, P, _ptr(S), _code(sdt), _ptr(x), _ptr(Bv), _ptr(Cv), _code(idt), float(alpha),
                             float(delta), float(D), _ptr(out))
    return out


def m2_decode_step(pool: np.ndarray, sdt, slots, x, dt, Bm, Cm, idt, A_log, dt_bias, D,
                   nthreads: int = 1) -> tuple[np.ndarray, int]:
    """One Mamba2 decode step of a batch; pool [num_slots, H, P, N] is updated in place; x [B, H, P],
    dt [B, H], Bm and Cm [B, G, N]. Returns (out [B, H, P] fp64, number of refused units)."""
    assert pool.dtype == NPTYPE[_code(sdt)] and pool.flags["C_CONTIGUOUS"]
    num_slots, H, P, N = pool.shape
    x, dt, Bm, Cm = (_arr(a, idt) for a in (x, dt, Bm, Cm))
    B = int(np.asarray(slots).shape[0])
    G = Bm.size // (B * N)
    slots = np.ascontiguousarray(slots, dtype=np.int32)
    A_log, dt_bias, D = (np.ascontiguousarray(a, dtype=np.float32) for a in (A_log, dt_bias, D))
    out = np.empty((B, H, P), dtype=np.float64)
    bad = lib().orc_m2_decode_step(B, G, H, N, P, num_slots, _ptr(pool), _code(sdt), _ptr(slots), _ptr(x),
                                   _ptr(dt), _ptr(Bm), _ptr(Cm), _code(idt), _ptr(A_log), _ptr(dt_bias), _ptr(D),
                                   _ptr(out), int(nthreads))
    return out, bad


class Mamba2ReplayHead:
    """ReplaySSM state of one Mamba2 (sequence, head): checkpoint S0 ([P, N] storage array), the
    buffered entries in arrival order (raw B [L, N] and x [L, P] in the input dtype, alpha and
    delta [L] fp64) and meta = [count, pos, ckpt_pos]. Rollback is the pointer move of
    ReplayHead.rollback."""

    def __init__(self, S0: np.ndarray, sdt, idt, L: int, pos: int = 0):
        self.sdt, self.idt, self.L = _code(sdt), _code(idt), int(L)
        self.S0 = np.ascontiguousarray(S0, dtype=NPTYPE[self.sdt]).copy()
        self.P, self.N = self.S0.shape
        self.eB = np.zeros((L, self.N), dtype=NPTYPE[self.idt])
        self.ex = np.zeros((L, self.P), dtype=NPTYPE[self.idt])
        self.ea = np.zeros(L, dtype=np.float64)
        self.ed = np.zeros(L, dtype=np.float64)
        self.meta = np.array([0, pos, pos], dtype=np.int32)

    @property
    def count(self) -> int:
        return int(self.meta[0])

    @property
    def pos(self) -> int:
        return int(self.meta[1])

    @property
    def ckpt_pos(self) -> int:
        return int(self.meta[2])

    def window(self, Cw, Bw, xw, dt, A_log: float, dt_bias: float, D: float) -> np.ndarray:
        """Process T tokens (Cw, Bw [T, N], xw [T, P], dt [T]); returns out [T, P] fp64."""
        Cw, Bw, xw = _arr(Cw, self.idt), _arr(Bw, self.idt), _arr(xw, self.idt)
        T = Cw.shape[0]
        dt = np.ascontiguousarray(dt, dtype=np.float64).reshape(T)
        out = np.empty((T, self.P), dtype=np.float64)
        rc = lib().orc_m2_replay_window(self.N, self.P, self.L, _ptr(self.S0), self.sdt, _ptr(self.eB),
                                        _ptr(self.ex), self.idt, _ptr(self.ea), _ptr(self.ed), _ptr(self.meta), T,
                                        _ptr(Cw), _ptr(Bw), _ptr(xw), _ptr(dt), float(A_log), float(dt_bias),
                                        float(D), _ptr(out))
        if rc != 0:
            raise ValueError(f"oracle Mamba2 replay window rejected its input (code {rc})")
        return out

    def flush(self, force: bool = True) -> None:
        rc = lib().orc_m2_replay_flush(self.N, self.P, self.L, _ptr(self.S0), self.sdt, _ptr(self.eB), _ptr(self.ex),
                                       self.idt, _ptr(self.ea), _ptr(self.ed), _ptr(self.meta), int(bool(force)))
        if rc != 0:
            raise ValueError(f"oracle Mamba2 replay flush rejected its state (code {rc})")

    def rollback(self, T: int, accepted: int) -> None:
        rc = lib().orc_replay_rollback(_ptr(self.meta), int(T), int(accepted))
        if rc != 0:
            raise ValueError(f"oracle rollback rejected its input (code {rc})")
