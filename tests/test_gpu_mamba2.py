"""GPU parity of the Mamba2 entry points (mamba2_decode_step, mamba2_replay_step,
mamba2_verify_window, mamba2_replay_flush, mamba2_rollback) against the CPU
oracle.

Small cases (several persistent rounds, ragged tails, padding, folds) compare
every output, every state element, the ring pointers and the raw ring entries
(bit-exact); the full-size Mamba2 layer (B = 256, 128 heads of dim 64, state
dim 128, 8 groups) compares sampled (sequence, head) units, which the oracle
recomputes through every step.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_ssm_gated_gb300 import build, gdn
from hybrid_ssm_gated_gb300 import workload as wl
from tests.gpu_util import (TOL, TORCH_DT, GpuReplay, canaries_intact, dev, dev_err, guarded, maxabs, sample_units,
                            step_to_device, to_f64)

pytestmark = pytest.mark.gpu

PREFILL = 100000


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gdn.lib()


def _params(w):
    A_log, dt_bias, D = wl.mamba2_params(w)
    return (A_log, dt_bias, D), tuple(torch.from_numpy(a).cuda() for a in (A_log, dt_bias, D))


def _decode_all(w: wl.Workload, slots=None, out_dtype="f32"):
    pool = wl.initial_pool(w)
    pool_gpu = dev(pool, w.state_dtype)
    slots = wl.slots(w) if slots is None else np.asarray(slots, np.int32)
    (A_log, dt_bias, D), (A_d, dt_d, D_d) = _params(w)
    s_d = torch.from_numpy(slots).cuda()
    err = dev_err()
    for t in range(w.steps):
        x = wl.mamba2_step_inputs(w, t)
        xd = step_to_device(x, w.in_dtype)
        out = torch.empty((len(slots), w.Hv, w.dv), dtype=TORCH_DT[out_dtype], device="cuda")
        gdn.mamba2_decode_step(pool_gpu, s_d, xd["x"], xd["dt"], xd["Bm"], xd["Cm"], A_d, dt_d, D_d, out, err)
        ref, bad = oracle.m2_decode_step(pool, w.state_dtype, slots, x["x"], x["dt"], x["Bm"], x["Cm"], w.in_dtype,
                                         A_log, dt_bias, D, nthreads=8)
        got = to_f64(out)
        ulp = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}[out_dtype]
        tol = TOL[w.state_dtype] + ulp * np.abs(ref)
        assert np.all(np.abs(got - ref) <= tol), f"step {t}: max |diff| {maxabs(got, ref):.3e}"
        for bi in np.flatnonzero((slots < 0) | (slots >= w.num_slots)):
            assert np.all(got[bi] == 0.0)
    torch.cuda.synchronize()
    final = to_f64(pool_gpu)
    assert maxabs(final, oracle.load(pool, w.state_dtype)) <= TOL[w.state_dtype]
    return int(err.item())


@pytest.mark.parametrize("sdt,idt", [("f32", "f32"), ("f32", "bf16"), ("bf16", "bf16"), ("f16", "f16")])
def test_decode_small_all_elements(sdt, idt):
    # 20 x 16 = 320 units over at most 152 persistent CTAs: several rounds and a ragged tail
    w = wl.Workload("m2d", B=20, Hk=2, Hv=16, dk=128, dv=64, steps=4, state_dtype=sdt, in_dtype=idt, seed=51)
    assert _decode_all(w) == 0


@pytest.mark.parametrize("N,P,G,H", [(32, 32, 1, 2), (64, 96, 2, 4), (128, 128, 1, 4), (32, 256, 2, 2),
                                     (64, 16, 4, 8)])
@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_decode_other_shapes(N, P, G, H, sdt):
    w = wl.Workload("m2s", B=7, Hk=G, Hv=H, dk=N, dv=P, steps=3, state_dtype=sdt, in_dtype="bf16", seed=52)
    assert _decode_all(w) == 0


def test_decode_padding_out_of_range_and_narrow_output():
    w = wl.Workload("m2p", B=6, Hk=2, Hv=4, dk=64, dv=64, steps=2, state_dtype="f32", in_dtype="bf16",
                    num_slots=8, seed=53)
    slots = np.array([3, -1, 0, 11, 7, -2], np.int32)
    assert _decode_all(w, slots=slots, out_dtype="bf16") == gdn.DEVERR_SLOT


def test_decode_padding_bf16_over_several_batches():
    """48 x 128 = 6,144 units, so CTAs take a second batch; padding and out-of-range sequences shift each
    unit's chunk fills, which the two producer warps of a 16-bit state count."""
    w = wl.Workload("m2pb", B=48, Hk=2, Hv=128, dk=64, dv=64, steps=2, state_dtype="bf16", in_dtype="bf16",
                    num_slots=120, seed=54)
    slots = wl.slots(w).copy()
    slots[::3] = -1
    slots[1::7] = w.num_slots + 3
    assert _decode_all(w, slots=slots) == gdn.DEVERR_SLOT


class M2Harness:
    """A Mamba2 replay cache on the GPU next to one oracle head per (sequence, head) unit."""

    def __init__(self, w: wl.Workload, units=None):
        self.w = w
        self.pool = wl.initial_pool(w)
        self.slots = wl.slots(w)
        (self.A_log, self.dt_bias, self.D), (self.A_d, self.dt_d, self.D_d) = _params(w)
        self.g = GpuReplay(w, self.pool)
        self.units = units if units is not None else [(b, h) for b in range(w.B) for h in range(w.Hv)]
        self.heads = {(b, h): oracle.Mamba2ReplayHead(self.pool[self.slots[b], h], w.state_dtype, w.in_dtype, w.L)
                      for b, h in self.units}
        self.err = dev_err()

    def window(self, x: dict, slots: np.ndarray, T: int, label: str):
        w = self.w
        xd = step_to_device(x, w.in_dtype)
        og = []  # the output's canaries, checked after the call
        out = guarded((w.B, T, w.Hv, w.dv), torch.float32, og)
        out.fill_(3.0)
        s_d = torch.from_numpy(slots).cuda()
        if T == 1:
            gdn.mamba2_replay_step(self.g.cache, s_d, xd["x"], xd["dt"], xd["Bm"], xd["Cm"], self.A_d, self.dt_d,
                                   self.D_d, out, self.err)
        else:
            gdn.mamba2_verify_window(self.g.cache, s_d, xd["x"], xd["dt"], xd["Bm"], xd["Cm"], self.A_d, self.dt_d,
                                     self.D_d, out, self.err)
        got = to_f64(out)
        assert canaries_intact(og), f"{label}: a kernel wrote outside the output"
        per = w.Hv // w.Hk
        for (b, h) in self.units:
            if slots[b] < 0:
                assert np.all(got[b, :, h] == 0.0)
                continue
            g = h // per
            ref = self.heads[(b, h)].window(x["Cm"][b, :, g], x["Bm"][b, :, g], x["x"][b, :, h],
                                            wl.values(x["dt"][b, :, h], w.in_dtype), float(self.A_log[h]),
                                            float(self.dt_bias[h]), float(self.D[h]))
            d = maxabs(got[b, :, h], ref)
            assert d <= TOL[w.state_dtype], f"{label} unit {(b, h)}: max |diff| {d:.3e}"

    def rollback(self, accepted: np.ndarray, T: int):
        gdn.mamba2_rollback(self.g.cache, torch.from_numpy(self.slots).cuda(), torch.from_numpy(accepted).cuda(), T,
                            self.err)
        for u in self.units:
            self.heads[u].rollback(T, int(accepted[u[0]]))

    def flush(self, force: bool):
        gdn.mamba2_replay_flush(self.g.cache, torch.from_numpy(self.slots).cuda(), force, self.err)
        for u in self.units:
            self.heads[u].flush(force)

    def prefill(self, offsets: np.ndarray):
        for s in range(int(offsets.max(initial=0))):
            x = wl.mamba2_step_inputs(self.w.with_(T=1), PREFILL + s)
            self.window(x, np.where(offsets > s, self.slots, -1).astype(np.int32), 1, f"prefill {s}")

    def check_state(self):
        """Checkpoints within tolerance; pointers and raw ring entries bit-exact; gates within 1e-5
        relative; the stored inverse key norm is exactly 1 (B is not normalised)."""
        w, c = self.w, self.g.cache
        torch.cuda.synchronize()
        pos, ck = c.pos.cpu().numpy(), c.ckpt_pos.cpu().numpy()
        raw = lambda t: t.view(torch.int16).cpu().numpy() if w.in_dtype != "f32" else t.cpu().numpy()
        rk, rv, rec = raw(c.ring_k), raw(c.ring_v), c.ring_rec.cpu().numpy()
        for (b, h) in self.units:
            hd, s = self.heads[(b, h)], self.slots[b]
            assert (pos[s, h], ck[s, h]) == (hd.pos, hd.ckpt_pos), f"pointers of {(b, h)}"
            d = maxabs(to_f64(c.ckpt[s, h]), oracle.load(hd.S0, w.state_dtype))
            assert d <= TOL[w.state_dtype], f"checkpoint of {(b, h)}: {d:.3e}"
            for e in range(hd.count):
                i = (hd.ckpt_pos + e) % w.L
                assert np.array_equal(rk[s, h, i].view(np.uint8), hd.eB[e].view(np.uint8)), f"ring B {(b, h, e)}"
                assert np.array_equal(rv[s, h, i].view(np.uint8), hd.ex[e].view(np.uint8)), f"ring x {(b, h, e)}"
                assert rec[s, h, i, 0] == pytest.approx(hd.ea[e], rel=1e-5, abs=1e-30)
                assert rec[s, h, i, 1] == pytest.approx(hd.ed[e], rel=1e-5, abs=1e-30)
                assert rec[s, h, i, 2] == 1.0
        assert int(self.err.item()) == 0
        assert canaries_intact(self.g.guards), "a kernel wrote outside a cache array"


@pytest.mark.parametrize("sdt,idt", [("f32", "f32"), ("bf16", "bf16"), ("f16", "bf16")])
@pytest.mark.parametrize("L", [1, 4])
def test_replay_steps_small_all_units(sdt, idt, L):
    w = wl.Workload("m2r", B=3, Hk=1, Hv=4, dk=64, dv=32, steps=3 * L + 5, state_dtype=sdt, in_dtype=idt, L=L,
                    seed=54)
    H = M2Harness(w)
    for t in range(w.steps):
        H.window(wl.mamba2_step_inputs(w, t), H.slots, 1, f"step {t}")
    H.check_state()


@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_replay_multi_round_with_offsets_and_flush(sdt):
    # 20 x 16 = 320 units over at most 152 persistent CTAs
    w = wl.Workload("m2m", B=20, Hk=2, Hv=16, dk=128, dv=64, steps=20, state_dtype=sdt, in_dtype="bf16", L=16,
                    max_offset=15, seed=55)
    H = M2Harness(w)
    H.prefill(wl.start_offsets(w))
    for t in range(w.steps):
        H.window(wl.mamba2_step_inputs(w, t), H.slots, 1, f"step {t}")
    H.check_state()
    H.flush(False)
    H.check_state()
    H.flush(True)
    H.check_state()
    H.window(wl.mamba2_step_inputs(w, 999), H.slots, 1, "after flush")
    H.check_state()


@pytest.mark.parametrize("N,P", [(32, 64), (128, 128), (64, 96)])
def test_replay_other_shapes(N, P):
    w = wl.Workload("m2h", B=5, Hk=2, Hv=4, dk=N, dv=P, steps=9, state_dtype="f32", in_dtype="bf16", L=4, seed=56)
    H = M2Harness(w)
    for t in range(w.steps):
        H.window(wl.mamba2_step_inputs(w, t), H.slots, 1, f"step {t}")
    H.check_state()


@pytest.mark.parametrize("T,L", [(2, 4), (4, 4), (4, 16), (8, 8), (3, 12)])
@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_verify_and_rollback_small(T, L, sdt):
    w = wl.Workload("m2v", B=4, Hk=2, Hv=4, dk=64, dv=64, steps=8, state_dtype=sdt, in_dtype="bf16", L=L, T=T,
                    seed=57)
    H = M2Harness(w)
    for r in range(w.steps):
        H.window(wl.mamba2_step_inputs(w, r), H.slots, T, f"round {r}")
        H.rollback(wl.accepted(w, r), T)
        if r % 3 == 2:
            H.window(wl.mamba2_step_inputs(w.with_(T=1), 500 + r), H.slots, 1, f"step after {r}")
    H.check_state()


@pytest.mark.parametrize("sdt,L,P", [("f32", 32, 256), ("bf16", 64, 256), ("f32", 64, 128)])
def test_verify_at_the_largest_ring_window_and_head(sdt, L, P):
    # 20 rounds of T = 8 keep 1..8 tokens each: counts pass 32 and every ring folds
    w = wl.Workload("m2x", B=3, Hk=1, Hv=2, dk=128, dv=P, steps=20, state_dtype=sdt, in_dtype="bf16", L=L, T=8,
                    seed=59)
    H = M2Harness(w)
    for r in range(w.steps):
        H.window(wl.mamba2_step_inputs(w, r), H.slots, 8, f"round {r}")
        H.rollback(wl.accepted(w, r), 8)
    H.window(wl.mamba2_step_inputs(w.with_(T=1), 700), H.slots, 1, "step")
    H.check_state()
    assert all(hd.ckpt_pos > 0 for hd in H.heads.values())


def test_single_steps_at_the_largest_ring():
    # 64-entry rings folded by single steps: every fold takes all 64 entries
    w = wl.Workload("m2l", B=3, Hk=1, Hv=2, dk=64, dv=32, steps=140, state_dtype="bf16", in_dtype="bf16", L=64,
                    seed=60)
    H = M2Harness(w)
    for t in range(w.steps):
        H.window(wl.mamba2_step_inputs(w, t), H.slots, 1, f"step {t}")
    H.check_state()


def test_padding_in_replay():
    w = wl.Workload("m2q", B=6, Hk=1, Hv=2, dk=32, dv=32, steps=6, state_dtype="f32", in_dtype="f32", L=4, seed=58)
    H = M2Harness(w)
    pad = H.slots.copy()
    pad[[1, 4]] = -1
    for t in range(w.steps):
        H.window(wl.mamba2_step_inputs(w, t), pad if t % 2 else H.slots, 1, f"step {t}")
    H.check_state()


def _decode_sampled(name: str, n_units: int):
    w = wl.WORKLOADS[name]
    pool = wl.initial_pool(w)
    slots = wl.slots(w)
    units = sample_units(w.B, w.Hv, n_units, seed=9)
    states = {u: pool[slots[u[0]], u[1]].copy() for u in units}
    pool_gpu = dev(pool, w.state_dtype)
    (A_log, dt_bias, D), (A_d, dt_d, D_d) = _params(w)
    s_d = torch.from_numpy(slots).cuda()
    err = dev_err()
    out = torch.empty((w.B, w.Hv, w.dv), device="cuda")
    per = w.Hv // w.Hk
    for t in range(w.steps):
        x = wl.mamba2_step_inputs(w, t)
        xd = step_to_device(x, w.in_dtype)
        gdn.mamba2_decode_step(pool_gpu, s_d, xd["x"], xd["dt"], xd["Bm"], xd["Cm"], A_d, dt_d, D_d, out, err)
        got = to_f64(out)
        for (b, h), S in states.items():
            al, de = oracle.m2_gating(A_log[h], dt_bias[h], wl.values(x["dt"][b, 0, h], w.in_dtype))
            ref = oracle.m2_decode_head(S, w.state_dtype, x["x"][b, 0, h], x["Bm"][b, 0, h // per],
                                        x["Cm"][b, 0, h // per], w.in_dtype, al, de, D[h])
            assert maxabs(got[b, h], ref) <= TOL[w.state_dtype], (t, b, h)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for (b, h), S in states.items():
        assert maxabs(to_f64(pool_gpu[slots[b], h]), oracle.load(S, w.state_dtype)) <= TOL[w.state_dtype]


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mamba2_b256_f32", "mamba2_b256_bf16"])
def test_decode_b256_sampled(name):
    _decode_sampled(name, 16)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mamba2_replay_b256_f32", "mamba2_replay_b256_bf16"])
def test_replay_b256_sampled(name):
    w = wl.WORKLOADS[name]
    H = M2Harness(w, sample_units(w.B, w.Hv, 16, seed=10))
    H.prefill(wl.start_offsets(w))
    for t in range(w.steps):
        H.window(wl.mamba2_step_inputs(w, t), H.slots, 1, f"{name} step {t}")
    H.check_state()
