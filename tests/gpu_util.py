"""Shared helpers for the GPU parity tests (inputs to device, oracle on units)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from hybrid_ssm_gated_gb300 import gdn
from hybrid_ssm_gated_gb300 import workload as wl

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
# Tolerances of the parity bar: max-abs 1e-4 with an fp32 state, atol 1e-2 with a
# bf16/fp16 state (the atol the vLLM PR #52191 summary's decode tests use).
TOL = {"f32": 1e-4, "bf16": 1e-2, "f16": 1e-2}


def dev(arr: np.ndarray, dt: str) -> torch.Tensor:
    return wl.to_torch(arr, dt).cuda()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def host_values(arr: np.ndarray, dt: str) -> np.ndarray:
    return wl.values(arr, dt)


def step_to_device(x: dict, dt: str) -> dict:
    return {k: dev(v, dt) for k, v in x.items()}


def dev_err() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def decode_oracle_unit(S: np.ndarray, sdt: str, x: dict, idt: str, b: int, h: int, Hv: int, Hk: int,
                       A_log, dt_bias) -> np.ndarray:
    """One oracle decode step of unit (b, h) on its state S (updated in place)."""
    kh = h // (Hv // Hk)
    al, be = oracle.gating(A_log[h], dt_bias[h], wl.values(x["a"][b, 0, h], idt), wl.values(x["b"][b, 0, h], idt))
    return oracle.decode_head(S, sdt, x["q"][b, 0, kh], x["k"][b, 0, kh], x["v"][b, 0, h], idt, al, be)


def sample_units(B: int, Hv: int, n: int, seed: int = 123) -> list[tuple[int, int]]:
    """n (sequence, head) units for a full-size parity run: the first and the last unit, three units of
    the persistent grid's ragged last round, the rest at random. Every kernel runs one CTA per SM and
    CTA c takes units c, c + SMs, ...; the units past the last whole round go to only some CTAs, so
    that round ends the launch unevenly and is where a wrong tail bound would show."""
    r = np.random.default_rng(seed)
    total = B * Hv
    picks = {(0, 0), (B - 1, Hv - 1)}
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tail0 = total // sms * sms  # first unit of the ragged round
    if sms < total and tail0 < total:
        for u in r.integers(tail0, total, size=3):
            picks.add(divmod(int(u), Hv))
    while len(picks) < min(n, total):
        picks.add((int(r.integers(B)), int(r.integers(Hv))))
    return sorted(picks)


def maxabs(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


GUARD = 256  # bytes of poisoned canary before and after a guarded array
POISON = 0xA5


def guarded(shape, dtype, keep: list) -> torch.Tensor:
    """A zeroed CUDA tensor with GUARD poisoned bytes before and after it in the same allocation (its
    storage is appended to `keep`, for canaries_intact)."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((n + 2 * GUARD,), POISON, dtype=torch.uint8, device="cuda")
    t = raw[GUARD:GUARD + n].view(dtype).view(shape)
    t.zero_()
    keep.append(raw)
    return t


def canaries_intact(keep: list) -> bool:
    """Every guarded tensor's poisoned bytes are unchanged: no kernel wrote just outside an array."""
    torch.cuda.synchronize()
    return all(bool((r[:GUARD] == POISON).all()) and bool((r[-GUARD:] == POISON).all()) for r in keep)


class GpuReplay:
    """A ReplaySSM cache on the GPU built from a workload's initial pool; every array of it sits
    between poisoned canary bytes (check with canaries_intact(self.guards))."""

    def __init__(self, w: wl.Workload, pool_host: np.ndarray, read_dtype=None):
        num_slots = pool_host.shape[0]
        self.guards = []
        g = lambda shape, dt: guarded(shape, dt, self.guards)
        sdt, idt = TORCH_DT[w.state_dtype], TORCH_DT[w.in_dtype]
        S = (num_slots, w.Hv)
        self.cache = gdn.ReplayCache(g(S + (w.dv, w.dk), sdt), g(S + (w.L, w.dk), idt), g(S + (w.L, w.dv), idt),
                                     g(S + (w.L, 4 + w.dv), torch.float32), g(S, torch.int32), g(S, torch.int32), w.L,
                                     None if read_dtype is None else g(S + (w.dv, w.dk), TORCH_DT[read_dtype]))
        self.cache.ckpt.copy_(dev(pool_host, w.state_dtype))
        if read_dtype is not None:  # a fresh sequence's read copy is its checkpoint rounded
            self.cache.ckpt_read.copy_(dev(oracle.round_to(oracle.load(pool_host, w.state_dtype), read_dtype),
                                           read_dtype))
        self.w = w


def replay_oracle_heads(w: wl.Workload, pool_host: np.ndarray, slots: np.ndarray, units, read_dtype=None) -> dict:
    return {(b, h): oracle.ReplayHead(pool_host[slots[b], h], w.state_dtype, w.in_dtype, w.L, read_dtype=read_dtype)
            for b, h in units}


def oracle_window(head: oracle.ReplayHead, x: dict, w: wl.Workload, b: int, h: int, A_log, dt_bias) -> np.ndarray:
    kh = h // (w.Hv // w.Hk)
    return head.window(q=x["q"][b, :, kh], k=x["k"][b, :, kh], v=x["v"][b, :, h],
                       a=wl.values(x["a"][b, :, h], w.in_dtype), b=wl.values(x["b"][b, :, h], w.in_dtype),
                       A_log=float(A_log[h]), dt_bias=float(dt_bias[h]))
