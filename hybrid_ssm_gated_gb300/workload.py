"""Seeded synthetic workloads for the GDN decode step and its ReplaySSM mode.

This module draws random numbers and casts them to storage dtypes. It holds
no step of the gated delta rule, so the CUDA path and the CPU oracle can both
take their inputs from here without sharing any of the method's arithmetic.

Every array is reproducible from (workload, seed) alone, and every per-step
or per-slot draw has its own seed, so a test can regenerate the inputs of one
step or the initial state of one slot without drawing the rest.

Shapes and distributions follow the synthetic decode workloads of this
library (Qwen3-Next-shaped GDN layers: Hk=16 key heads, Hv=32 value heads,
dk=dv=128): q/k/v/a/b ~ N(0,1) in the input dtype, A_log ~ U(0,2),
dt_bias ~ U(-1,1), initial states ~ N(0, 0.1) rounded to the state dtype.

Mamba2 workloads reuse the same fields with Hk = groups G, Hv = heads H,
dk = state dim N and dv = head dim P: x, dt, B, C ~ N(0,1) in the input dtype;
A_log = ln U(1, 16), dt_bias = the softplus inverse of a step size drawn
log-uniform in [0.001, 0.1], D ~ U(0.5, 1.5) (the ranges Mamba2 layers are
initialised in).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

# Storage dtype codes; the same integers are used by the C ABI and the oracle.
F32, BF16, F16 = 0, 1, 2
DTYPE_CODE = {"f32": F32, "bf16": BF16, "f16": F16}
DTYPE_BYTES = {"f32": 4, "bf16": 2, "f16": 2}

# Seed-stream tags: each kind of draw has its own stream.
(_TAG_PARAMS, _TAG_STATE, _TAG_STEP, _TAG_SLOTS, _TAG_OFFSETS, _TAG_ACCEPT, _TAG_M2_PARAMS, _TAG_M2_STEP,
 _TAG_PREFILL) = range(9)


@dataclass(frozen=True)
class Workload:
    """One synthetic configuration.

    steps counts decode steps (or verify rounds when T > 1). L > 0 marks a
    ReplaySSM workload with an L-entry ring; max_offset bounds the seeded
    number of entries already buffered per sequence at the start.
    """

    name: str
    B: int
    Hk: int
    Hv: int
    dk: int
    dv: int
    steps: int
    state_dtype: str = "f32"
    in_dtype: str = "bf16"
    num_slots: int = 0
    slot_mode: str = "perm"  # "identity" or "perm"
    seed: int = 0
    state_std: float = 0.1
    L: int = 0
    T: int = 1
    max_offset: int = 0
    prefill_len: int = 0  # tokens per sequence of a prefill workload

    def __post_init__(self):
        if self.num_slots == 0:
            object.__setattr__(self, "num_slots", 2 * self.B if self.slot_mode == "perm" else self.B)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # Small case the oracle finishes in well under a second.
    "tiny": Workload("tiny", B=2, Hk=2, Hv=4, dk=32, dv=32, steps=8, state_dtype="f32",
                     in_dtype="f32", num_slots=2, slot_mode="identity"),
    # Qwen3-Next-shaped decode, fp32 state pool of 2B slots, permuted slots.
    "qwen3next_b64": Workload("qwen3next_b64", B=64, Hk=16, Hv=32, dk=128, dv=128, steps=100),
    # The headline decode shape: B=256, fp32 state pool of 512 slots.
    "decode_b256_f32": Workload("decode_b256_f32", B=256, Hk=16, Hv=32, dk=128, dv=128, steps=200),
    # Low-precision state pools at B=256.
    "decode_b256_bf16": Workload("decode_b256_bf16", B=256, Hk=16, Hv=32, dk=128, dv=128, steps=200,
                                 state_dtype="bf16"),
    "decode_b256_f16": Workload("decode_b256_f16", B=256, Hk=16, Hv=32, dk=128, dv=128, steps=200,
                                state_dtype="f16"),
    # ReplaySSM standard decode: L=16 ring, start offsets in [0, 15], 64 steps.
    "replay_b256_f32": Workload("replay_b256_f32", B=256, Hk=16, Hv=32, dk=128, dv=128, steps=64,
                                L=16, max_offset=15),
    "replay_b256_bf16": Workload("replay_b256_bf16", B=256, Hk=16, Hv=32, dk=128, dv=128, steps=64,
                                 state_dtype="bf16", L=16, max_offset=15),
    # ReplaySSM speculative verify: T=4 window, accepted drafts in {0..3}, 32 rounds.
    "verify_b256_f32": Workload("verify_b256_f32", B=256, Hk=16, Hv=32, dk=128, dv=128, steps=32,
                                L=16, T=4),
    "verify_b256_bf16": Workload("verify_b256_bf16", B=256, Hk=16, Hv=32, dk=128, dv=128, steps=32,
                                 state_dtype="bf16", L=16, T=4),
    # Prefill of 19 sequences of 2048 tokens, state written back every 64 tokens.
    "prefill_b19_f32": Workload("prefill_b19_f32", B=19, Hk=16, Hv=32, dk=128, dv=128, steps=1, prefill_len=2048),
    # Mamba2 layer of 128 heads, head dim 64, state dim 128, 8 groups (Hk = G, Hv = H, dk = N, dv = P).
    "mamba2_b256_f32": Workload("mamba2_b256_f32", B=256, Hk=8, Hv=128, dk=128, dv=64, steps=64),
    "mamba2_b256_bf16": Workload("mamba2_b256_bf16", B=256, Hk=8, Hv=128, dk=128, dv=64, steps=64,
                                 state_dtype="bf16"),
    "mamba2_replay_b256_f32": Workload("mamba2_replay_b256_f32", B=256, Hk=8, Hv=128, dk=128, dv=64, steps=64,
                                       L=16, max_offset=15),
    "mamba2_replay_b256_bf16": Workload("mamba2_replay_b256_bf16", B=256, Hk=8, Hv=128, dk=128, dv=64, steps=64,
                                        state_dtype="bf16", L=16, max_offset=15),
}


def _rng(w: Workload, tag: int, *idx: int) -> np.random.Generator:
    return np.random.default_rng([w.seed, tag, *idx])


# ---------------------------------------------------------------- dtype casts


def quantize(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to a storage dtype (round-to-nearest-even).

    Returns float32 for "f32", float16 for "f16" and the raw uint16 bit
    patterns for "bf16" (numpy has no bfloat16); the rounding is done by
    numpy / torch library casts.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        import torch

        t = torch.from_numpy(x).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(dtype)


def values(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of a storage array returned by quantize()."""
    if dtype == "bf16":
        bits = arr.astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    return arr.astype(np.float64)


def to_torch(arr: np.ndarray, dtype: str):
    """Host torch tensor with the storage dtype (bf16 reinterpreted from bits)."""
    import torch

    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr))


# ---------------------------------------------------------------- draws


def head_params(w: Workload) -> tuple[np.ndarray, np.ndarray]:
    """A_log ~ U(0,2) and dt_bias ~ U(-1,1), float32 [Hv]."""
    r = _rng(w, _TAG_PARAMS)
    A_log = r.uniform(0.0, 2.0, size=w.Hv).astype(np.float32)
    dt_bias = r.uniform(-1.0, 1.0, size=w.Hv).astype(np.float32)
    return A_log, dt_bias


def slots(w: Workload) -> np.ndarray:
    """int32 [B] slot indices: identity, or a seeded permutation's first B."""
    if w.slot_mode == "identity":
        return np.arange(w.B, dtype=np.int32)
    return _rng(w, _TAG_SLOTS).permutation(w.num_slots)[: w.B].astype(np.int32)


def slot_state(w: Workload, slot: int) -> np.ndarray:
    """Initial state of one slot, [Hv, dv, dk] ~ N(0, state_std), in the state dtype."""
    x = _rng(w, _TAG_STATE, slot).standard_normal((w.Hv, w.dv, w.dk), dtype=np.float32)
    return quantize(x * np.float32(w.state_std), w.state_dtype)


def initial_pool(w: Workload) -> np.ndarray:
    """The whole state pool [num_slots, Hv, dv, dk] in the state dtype."""
    first = slot_state(w, 0)
    pool = np.empty((w.num_slots,) + first.shape, dtype=first.dtype)
    pool[0] = first
    for s in range(1, w.num_slots):
        pool[s] = slot_state(w, s)
    return pool


def step_inputs(w: Workload, step: int) -> dict[str, np.ndarray]:
    """Activations of one decode step (or one verify window of T tokens).

    q, k: [B, T, Hk, dk]; v: [B, T, Hv, dv]; a, b: [B, T, Hv]; all ~ N(0,1)
    in the input dtype. For T == 1 the memory layout equals [B, Hk, dk] etc.
    """
    r = _rng(w, _TAG_STEP, step)
    T = w.T
    out = {}
    for name, shape in (("q", (w.B, T, w.Hk, w.dk)), ("k", (w.B, T, w.Hk, w.dk)),
                        ("v", (w.B, T, w.Hv, w.dv)), ("a", (w.B, T, w.Hv)), ("b", (w.B, T, w.Hv))):
        out[name] = quantize(r.standard_normal(shape, dtype=np.float32), w.in_dtype)
    return out


def start_offsets(w: Workload) -> np.ndarray:
    """Entries already buffered per sequence at the start, uniform in [0, max_offset]."""
    return _rng(w, _TAG_OFFSETS).integers(0, w.max_offset + 1, size=w.B).astype(np.int32)


def accepted(w: Workload, round_: int) -> np.ndarray:
    """Accepted draft tokens per sequence for one verify round, uniform in {0..T-1}."""
    return _rng(w, _TAG_ACCEPT, round_).integers(0, w.T, size=w.B).astype(np.int32)


# ---------------------------------------------------------------- Mamba2 draws


def mamba2_params(w: Workload) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """A_log = ln U(1, 16), dt_bias = softplus^-1(step) with step log-uniform in [0.001, 0.1],
    D ~ U(0.5, 1.5); float32 [H]."""
    r = _rng(w, _TAG_M2_PARAMS)
    A_log = np.log(r.uniform(1.0, 16.0, size=w.Hv)).astype(np.float32)
    step = np.exp(r.uniform(np.log(1e-3), np.log(1e-1), size=w.Hv))
    dt_bias = (step + np.log(-np.expm1(-step))).astype(np.float32)
    D = r.uniform(0.5, 1.5, size=w.Hv).astype(np.float32)
    return A_log, dt_bias, D


def mamba2_step_inputs(w: Workload, step: int) -> dict[str, np.ndarray]:
    """Activations of one Mamba2 decode step (or a window of T tokens): x [B, T, H, P], dt [B, T, H],
    Bm, Cm [B, T, G, N]; all ~ N(0,1) in the input dtype."""
    r = _rng(w, _TAG_M2_STEP, step)
    T = w.T
    out = {}
    for name, shape in (("x", (w.B, T, w.Hv, w.dv)), ("dt", (w.B, T, w.Hv)), ("Bm", (w.B, T, w.Hk, w.dk)),
                        ("Cm", (w.B, T, w.Hk, w.dk))):
        out[name] = quantize(r.standard_normal(shape, dtype=np.float32), w.in_dtype)
    return out


# ---------------------------------------------------------------- prefill draws


def prefill_inputs(w: Workload, total: int, call: int = 0) -> dict[str, np.ndarray]:
    """Activations of `total` prefill tokens: q, k [total, Hk, dk]; v [total, Hv, dv]; a, b [total, Hv];
    ~ N(0,1) in the input dtype."""
    r = _rng(w, _TAG_PREFILL, call)
    out = {}
    for name, shape in (("q", (total, w.Hk, w.dk)), ("k", (total, w.Hk, w.dk)), ("v", (total, w.Hv, w.dv)),
                        ("a", (total, w.Hv)), ("b", (total, w.Hv))):
        out[name] = quantize(r.standard_normal(shape, dtype=np.float32), w.in_dtype)
    return out
