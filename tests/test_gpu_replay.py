"""GPU parity of the ReplaySSM entry points (gdn_replay_step, gdn_verify_window,
gdn_replay_flush, gdn_rollback) against the CPU oracle.

The oracle keeps, per (sequence, head), the checkpoint and the raw inputs
buffered since it and rebuilds the state for every output; the kernels use a
ring with derived correction vectors. Outputs and checkpoints are compared
within the parity tolerances; the ring pointers and the raw k/v ring entries
are compared bit-exactly; the stored gates within 1e-5 relative (they come
from expf/log1pf in FP32 on the GPU and fp64 libm in the oracle, and the
composition exp(-exp(A) softplus(x)) amplifies the relative error of its
argument by |exp(A) softplus(x)| <= ~20).
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_ssm_gated_gb300 import build, gdn
from hybrid_ssm_gated_gb300 import workload as wl
from tests.gpu_util import (TOL, TORCH_DT, GpuReplay, canaries_intact, dev, dev_err, guarded, maxabs, oracle_window,
                            replay_oracle_heads, sample_units, step_to_device, to_f64)

pytestmark = pytest.mark.gpu

PREFILL = 100000  # step-seed offset of the pre-fill tokens


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gdn.lib()


class Harness:
    def __init__(self, w: wl.Workload, units=None, read_dtype=None):
        self.w = w
        self.rdt = read_dtype
        self.pool = wl.initial_pool(w)
        self.slots = wl.slots(w)
        self.A_log, self.dt_bias = wl.head_params(w)
        self.g = GpuReplay(w, self.pool, read_dtype)
        self.units = units if units is not None else [(b, h) for b in range(w.B) for h in range(w.Hv)]
        self.heads = replay_oracle_heads(w, self.pool, self.slots, self.units, read_dtype)
        self.A_d = torch.from_numpy(self.A_log).cuda()
        self.dt_d = torch.from_numpy(self.dt_bias).cuda()
        self.err = dev_err()
        self.worst = 0.0

    def window(self, x: dict, slots: np.ndarray, T: int, label: str):
        w = self.w
        xd = step_to_device(x, w.in_dtype)
        og = []  # the output's canaries, checked after the call
        out = guarded((w.B, T, w.Hv, w.dv), torch.float32, og)
        out.fill_(3.0)
        s_d = torch.from_numpy(slots).cuda()
        if T == 1:
            gdn.gdn_replay_step(self.g.cache, s_d, xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], self.A_d, self.dt_d,
                                out, self.err)
        else:
            gdn.gdn_verify_window(self.g.cache, s_d, xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], self.A_d, self.dt_d,
                                  out, self.err)
        got = to_f64(out)
        assert canaries_intact(og), f"{label}: a kernel wrote outside the output"
        for (b, h) in self.units:
            if slots[b] < 0:
                assert np.all(got[b, :, h] == 0.0)
                continue
            ref = oracle_window(self.heads[(b, h)], x, w, b, h, self.A_log, self.dt_bias)
            d = maxabs(got[b, :, h], ref)
            assert d <= TOL[w.state_dtype], f"{label} unit {(b, h)}: max |diff| {d:.3e}"
            self.worst = max(self.worst, d)

    def rollback(self, accepted: np.ndarray, T: int):
        gdn.gdn_rollback(self.g.cache, torch.from_numpy(self.slots).cuda(), torch.from_numpy(accepted).cuda(), T,
                         self.err)
        for (b, h) in self.units:
            self.heads[(b, h)].rollback(T, int(accepted[b]))

    def prefill(self, offsets: np.ndarray):
        for s in range(int(offsets.max(initial=0))):
            x = wl.step_inputs(self.w.with_(T=1), PREFILL + s)
            self.window(x, np.where(offsets > s, self.slots, -1).astype(np.int32), 1, f"prefill {s}")

    def check_state(self):
        """Checkpoints within tolerance; pointers and raw ring entries bit-exact."""
        w, c = self.w, self.g.cache
        torch.cuda.synchronize()
        pos, ck = c.pos.cpu().numpy(), c.ckpt_pos.cpu().numpy()
        rk = c.ring_k.view(torch.int16).cpu().numpy() if w.in_dtype != "f32" else c.ring_k.cpu().numpy()
        rv = c.ring_v.view(torch.int16).cpu().numpy() if w.in_dtype != "f32" else c.ring_v.cpu().numpy()
        rec = c.ring_rec.cpu().numpy()
        for (b, h) in self.units:
            hd, s = self.heads[(b, h)], self.slots[b]
            assert (pos[s, h], ck[s, h]) == (hd.pos, hd.ckpt_pos), f"pointers of {(b, h)}"
            S0 = to_f64(c.ckpt[s, h])
            d = maxabs(S0, oracle.load(hd.S0, w.state_dtype))
            assert d <= TOL[w.state_dtype], f"checkpoint of {(b, h)}: {d:.3e}"
            if self.rdt is not None:
                # the read copy: the stored checkpoint rounded, bit-exactly, and near the oracle's copy
                rd = c.ckpt_read[s, h].float().double().cpu().numpy()
                assert np.array_equal(rd, oracle.load(oracle.round_to(S0, self.rdt), self.rdt)), f"copy of {(b, h)}"
                d = maxabs(rd, oracle.load(hd.Sr, self.rdt))
                assert d <= TOL[self.rdt], f"read copy of {(b, h)}: {d:.3e}"
            for e in range(hd.count):
                i = (hd.ckpt_pos + e) % w.L
                assert np.array_equal(rk[s, h, i].view(np.uint8), hd.ek[e].view(np.uint8)), f"ring k {(b, h, e)}"
                assert np.array_equal(rv[s, h, i].view(np.uint8), hd.ev[e].view(np.uint8)), f"ring v {(b, h, e)}"
                assert rec[s, h, i, 0] == pytest.approx(hd.ea[e], rel=1e-5, abs=1e-30)
                assert rec[s, h, i, 1] == pytest.approx(hd.eb[e], rel=1e-5, abs=1e-30)
        assert int(self.err.item()) == 0
        assert canaries_intact(self.g.guards), "a kernel wrote outside a cache array or an output"


@pytest.mark.parametrize("sdt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("L", [1, 4, 64])
def test_replay_steps_small_all_units(sdt, L):
    w = wl.Workload("rs", B=3, Hk=1, Hv=2, dk=32, dv=32, steps=3 * L + 5, state_dtype=sdt, in_dtype="f32", L=L,
                    seed=21)
    H = Harness(w)
    for t in range(w.steps):
        H.window(wl.step_inputs(w, t), H.slots, 1, f"step {t}")
    H.check_state()


@pytest.mark.parametrize("sdt,idt", [("f32", "bf16"), ("bf16", "bf16"), ("f32", "f16")])
def test_replay_multi_round_with_offsets(sdt, idt):
    # 20 x 8 = 160 units over 152 persistent CTAs: a ragged second round
    w = wl.Workload("rm", B=20, Hk=2, Hv=8, dk=128, dv=128, steps=24, state_dtype=sdt, in_dtype=idt, L=16,
                    max_offset=15, seed=22)
    H = Harness(w)
    H.prefill(wl.start_offsets(w))
    for t in range(w.steps):
        H.window(wl.step_inputs(w, t), H.slots, 1, f"step {t}")
    H.check_state()


@pytest.mark.parametrize("dk,dv", [(64, 32), (128, 256), (32, 96), (64, 64)])
def test_replay_other_head_shapes(dk, dv):
    w = wl.Workload("rh", B=5, Hk=2, Hv=4, dk=dk, dv=dv, steps=9, state_dtype="f32", in_dtype="bf16", L=4, seed=23)
    H = Harness(w)
    for t in range(w.steps):
        H.window(wl.step_inputs(w, t), H.slots, 1, f"step {t}")
    H.check_state()


@pytest.mark.parametrize("T,L", [(2, 4), (3, 4), (4, 4), (4, 16), (8, 8), (5, 12)])
@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_verify_and_rollback_small(T, L, sdt):
    w = wl.Workload("vs", B=4, Hk=2, Hv=4, dk=64, dv=64, steps=10, state_dtype=sdt, in_dtype="bf16", L=L, T=T,
                    seed=24)
    H = Harness(w)
    for r in range(w.steps):
        H.window(wl.step_inputs(w, r), H.slots, T, f"round {r}")
        H.rollback(wl.accepted(w, r), T)
        if r % 3 == 2:  # interleave plain replay steps
            H.window(wl.step_inputs(w.with_(T=1), 500 + r), H.slots, 1, f"step after {r}")
    H.check_state()


@pytest.mark.parametrize("sdt,L,dv,rdt", [("f32", 64, 256, None), ("bf16", 64, 256, None), ("f32", 32, 256, None),
                                          ("f32", 64, 256, "bf16")])
def test_maximum_ring_window_and_head(sdt, L, dv, rdt):
    # the largest ring (L = 64) and window (T = 8) with the largest head (dk = 128, dv = 256); 20 rounds
    # keep 1..8 tokens each, so counts pass 32 and every ring folds
    w = wl.Workload("mx", B=3, Hk=1, Hv=2, dk=128, dv=dv, steps=20, state_dtype=sdt, in_dtype="bf16", L=L, T=8,
                    seed=27)
    H = Harness(w, read_dtype=rdt)
    most = 0
    for r in range(w.steps):
        most = max(most, max(hd.count for hd in H.heads.values()))
        H.window(wl.step_inputs(w, r), H.slots, 8, f"round {r}")
        H.rollback(wl.accepted(w, r), 8)
    H.window(wl.step_inputs(w.with_(T=1), 700), H.slots, 1, "step")
    H.check_state()
    assert most > L - 16 and all(hd.ckpt_pos > 0 for hd in H.heads.values())


def test_rollback_must_undo_the_last_window():
    """gdn_rollback's T must be that of the window just verified. A mismatch, a second rollback of the
    same window or a rollback after a plain step is refused -- GDN_DEVERR_ACCEPT, or GDN_DEVERR_RING
    where the move would pass the checkpoint -- and moves no pointer."""
    w = wl.Workload("rb", B=3, Hk=1, Hv=2, dk=32, dv=32, steps=3, state_dtype="f32", in_dtype="bf16", L=16, T=4,
                    seed=29)
    H = Harness(w)
    c, s_d = H.g.cache, torch.from_numpy(H.slots).cuda()
    acc0 = torch.from_numpy(wl.accepted(w, 0)).cuda()

    def refused(T, bits=gdn.DEVERR_ACCEPT | gdn.DEVERR_RING):
        before, err = c.pos.clone(), dev_err()
        gdn.gdn_rollback(c, s_d, acc0, T, err)
        torch.cuda.synchronize()
        e = int(err.item())
        assert e != 0 and e & ~bits == 0, e
        assert torch.equal(c.pos, before)

    H.window(wl.step_inputs(w, 0), H.slots, 4, "round 0")
    refused(3, gdn.DEVERR_ACCEPT)  # the window had 4 tokens
    H.rollback(wl.accepted(w, 0), 4)
    refused(4)  # already rolled back
    H.window(wl.step_inputs(w.with_(T=1), 900), H.slots, 1, "step")
    refused(4)  # the last call was a single step
    H.window(wl.step_inputs(w, 1), H.slots, 4, "round 1")
    H.rollback(wl.accepted(w, 1), 4)
    H.check_state()


@pytest.mark.parametrize("dk,dv", [(32, 96), (128, 32), (64, 256), (32, 32)])
@pytest.mark.parametrize("T", [3, 8])
def test_verify_other_head_shapes(dk, dv, T):
    w = wl.Workload("vh", B=5, Hk=2, Hv=4, dk=dk, dv=dv, steps=6, state_dtype="f32", in_dtype="bf16", L=16, T=T,
                    seed=28)
    H = Harness(w)
    for r in range(w.steps):
        H.window(wl.step_inputs(w, r), H.slots, T, f"round {r}")
        H.rollback(wl.accepted(w, r), T)
    H.check_state()


@pytest.mark.parametrize("force", [True, False])
def test_flush(force):
    w = wl.Workload("fl", B=6, Hk=1, Hv=2, dk=128, dv=64, steps=1, state_dtype="bf16", in_dtype="bf16", L=8,
                    max_offset=8, seed=25)
    H = Harness(w)
    H.prefill(wl.start_offsets(w))  # counts 0..8, some rings full
    gdn.gdn_replay_flush(H.g.cache, torch.from_numpy(H.slots).cuda(), force, H.err)
    for u in H.units:
        H.heads[u].flush(force)
    H.check_state()
    H.window(wl.step_inputs(w, 0), H.slots, 1, "after flush")
    H.check_state()


def test_replay_ring_errors_are_reported_not_fatal():
    w = wl.Workload("re", B=3, Hk=1, Hv=2, dk=32, dv=32, steps=1, state_dtype="f32", in_dtype="f32", L=4, seed=26)
    H = Harness(w)
    c = H.g.cache
    c.pos[H.slots[1]] = 9  # count 9 > L
    ck0 = c.ckpt.clone()
    x = step_to_device(wl.step_inputs(w, 0), "f32")
    out = torch.full((3, 1, 2, 32), 5.0, device="cuda")
    gdn.gdn_replay_step(c, torch.from_numpy(H.slots).cuda(), x["q"], x["k"], x["v"], x["a"], x["b"], H.A_d, H.dt_d,
                        out, H.err)
    torch.cuda.synchronize()
    assert int(H.err.item()) == gdn.DEVERR_RING
    assert torch.all(out[1] == 0) and torch.all(out[0] != 5.0) and torch.all(out[2] != 5.0)
    assert torch.equal(c.ckpt[H.slots[1]], ck0[H.slots[1]]) and int(c.pos[H.slots[1], 0]) == 9
    # an accepted count outside [0, T-1] is refused without moving the pointer
    err = dev_err()
    acc = torch.tensor([0, 5, 1], dtype=torch.int32, device="cuda")
    before = c.pos.clone()
    gdn.gdn_rollback(c, torch.from_numpy(H.slots).cuda(), acc, 4, err)
    torch.cuda.synchronize()
    assert int(err.item()) & gdn.DEVERR_ACCEPT
    assert torch.equal(c.pos[H.slots[1]], before[H.slots[1]])


def _sampled(name: str, n_units: int):
    w = wl.WORKLOADS[name]
    units = sample_units(w.B, w.Hv, n_units, seed=5)
    H = Harness(w, units)
    if w.max_offset:
        H.prefill(wl.start_offsets(w))
    for r in range(w.steps):
        H.window(wl.step_inputs(w, r), H.slots, w.T, f"{name} round {r}")
        if w.T > 1:
            H.rollback(wl.accepted(w, r), w.T)
    H.check_state()
    return H.worst


@pytest.mark.slow
@pytest.mark.parametrize("name", ["replay_b256_f32", "replay_b256_bf16"])
def test_replay_b256_sampled(name):
    _sampled(name, 16)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["verify_b256_f32", "verify_b256_bf16"])
def test_verify_b256_sampled(name):
    _sampled(name, 16)


@pytest.mark.parametrize("rdt", ["bf16", "f16"])
@pytest.mark.parametrize("T,L", [(1, 4), (3, 8)])
def test_read_copy_small_all_units(rdt, T, L):
    # fp32 checkpoint for the recurrence, bf16/fp16 copy for reading; 3 x 4 folds at least
    w = wl.Workload("rc", B=20, Hk=2, Hv=8, dk=64, dv=64, steps=12, state_dtype="f32", in_dtype="bf16", L=L, T=T,
                    seed=41)
    H = Harness(w, read_dtype=rdt)
    for r in range(w.steps):
        H.window(wl.step_inputs(w, r), H.slots, T, f"round {r}")
        if T > 1:
            H.rollback(wl.accepted(w, r), T)
    H.check_state()
    gdn.gdn_replay_flush(H.g.cache, torch.from_numpy(H.slots).cuda(), True, H.err)
    for u in H.units:
        H.heads[u].flush(True)
    H.check_state()


@pytest.mark.parametrize("T", [1, 4])
def test_read_copy_large_head(T):
    # 128 x 256 heads: a fold unit streams 8 master chunks, twice a copy unit's
    w = wl.Workload("rcl", B=3, Hk=1, Hv=2, dk=128, dv=256, steps=8, state_dtype="f32", in_dtype="bf16", L=8, T=T,
                    seed=42)
    H = Harness(w, read_dtype="bf16")
    for r in range(w.steps):
        H.window(wl.step_inputs(w, r), H.slots, T, f"round {r}")
        if T > 1:
            H.rollback(wl.accepted(w, r), T)
    H.check_state()


@pytest.mark.slow
def test_read_copy_b256_sampled():
    w = wl.WORKLOADS["replay_b256_f32"]
    H = Harness(w, sample_units(w.B, w.Hv, 16, seed=6), read_dtype="bf16")
    H.prefill(wl.start_offsets(w))
    for r in range(w.steps):
        H.window(wl.step_inputs(w, r), H.slots, 1, f"round {r}")
    H.check_state()
