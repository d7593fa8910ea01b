"""Slot gather and scatter above 4 GiB: decode, ReplaySSM and prefill on an fp32
pool of 2100 slots of 32 heads x 128 x 128 (4.1 GiB), the batch naming slots
near the end of it, so every state offset needs 64-bit arithmetic. Only the
named slots are initialised and compared (per unit, against the oracle);
outputs are written in bf16 to cover narrow outputs on these paths too."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_ssm_gated_gb300 import build, gdn
from hybrid_ssm_gated_gb300 import workload as wl
from tests.gpu_util import TOL, dev, dev_err, maxabs, step_to_device, to_f64

pytestmark = pytest.mark.gpu

NUM_SLOTS = 2100
SLOTS = np.array([2099, 3, 1500, 2048], np.int32)
OUT_TOL = TOL["f32"] + 2.0 ** -8  # bf16 outputs: half an output ulp of |o| <= ~1 on top


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gdn.lib()


def _w(**kw):
    return wl.Workload("big", B=len(SLOTS), Hk=16, Hv=32, dk=128, dv=128, steps=1, state_dtype="f32",
                       in_dtype="bf16", num_slots=NUM_SLOTS, seed=71, **kw)


def _pool(w):
    pool = torch.empty((NUM_SLOTS, w.Hv, w.dv, w.dk), dtype=torch.float32, device="cuda")
    host = {int(s): wl.slot_state(w, int(s)) for s in SLOTS}
    for s, st in host.items():
        pool[s].copy_(torch.from_numpy(st))
    return pool, host


def test_decode_above_4gib():
    w = _w()
    pool, host = _pool(w)
    A_log, dt_bias = wl.head_params(w)
    err = dev_err()
    for t in range(3):
        x = wl.step_inputs(w, t)
        xd = step_to_device(x, "bf16")
        out = torch.empty((w.B, w.Hv, w.dv), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_step(pool, torch.from_numpy(SLOTS).cuda(), xd["q"], xd["k"], xd["v"], xd["a"], xd["b"],
                            torch.from_numpy(A_log).cuda(), torch.from_numpy(dt_bias).cuda(), out, err)
        got = to_f64(out)
        for b, s in enumerate(SLOTS):
            ref, _ = oracle.decode_step(host[int(s)][None], "f32", np.array([0], np.int32), x["q"][b:b + 1],
                                        x["k"][b:b + 1], x["v"][b:b + 1], x["a"][b:b + 1], x["b"][b:b + 1], "bf16",
                                        A_log, dt_bias)
            assert maxabs(got[b], ref[0]) <= OUT_TOL, (t, b)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for s in SLOTS:
        assert maxabs(to_f64(pool[int(s)]), host[int(s)].astype(np.float64)) <= TOL["f32"]


def test_replay_above_4gib():
    w = _w(L=4)
    cache = gdn.ReplayCache.allocate(NUM_SLOTS, w.Hv, w.dk, w.dv, w.L, torch.float32, torch.bfloat16)
    heads = {}
    for s in SLOTS:
        st = wl.slot_state(w, int(s))
        cache.ckpt[int(s)].copy_(torch.from_numpy(st))
        for h in range(w.Hv):
            heads[(int(s), h)] = oracle.ReplayHead(st[h], "f32", "bf16", w.L)
    A_log, dt_bias = wl.head_params(w)
    err = dev_err()
    kh_of = lambda h: h // (w.Hv // w.Hk)
    for t in range(6):  # through a fold
        x = wl.step_inputs(w, t)
        xd = step_to_device(x, "bf16")
        out = torch.empty((w.B, 1, w.Hv, w.dv), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_replay_step(cache, torch.from_numpy(SLOTS).cuda(), xd["q"], xd["k"], xd["v"], xd["a"], xd["b"],
                            torch.from_numpy(A_log).cuda(), torch.from_numpy(dt_bias).cuda(), out, err)
        got = to_f64(out)
        for b, s in enumerate(SLOTS):
            for h in range(0, w.Hv, 7):
                ref = heads[(int(s), h)].window(x["q"][b, :, kh_of(h)], x["k"][b, :, kh_of(h)], x["v"][b, :, h],
                                                wl.values(x["a"][b, :, h], "bf16"), wl.values(x["b"][b, :, h], "bf16"),
                                                float(A_log[h]), float(dt_bias[h]))
                assert maxabs(got[b, :, h], ref) <= OUT_TOL, (t, b, h)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for s in SLOTS:
        for h in range(0, w.Hv, 7):
            assert maxabs(to_f64(cache.ckpt[int(s), h]), heads[(int(s), h)].S0.astype(np.float64)) <= TOL["f32"]


def test_prefill_above_4gib():
    w = _w()
    pool, host = _pool(w)
    lens = np.array([40, 17, 0, 33], np.int32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = wl.prefill_inputs(w, int(cu[-1]))
    xd = step_to_device(x, "bf16")
    A_log, dt_bias = wl.head_params(w)
    out = torch.empty((int(cu[-1]), w.Hv, w.dv), dtype=torch.bfloat16, device="cuda")
    err = dev_err()
    gdn.gdn_prefill(pool, torch.from_numpy(SLOTS).cuda(), torch.from_numpy(cu).cuda(), xd["q"], xd["k"], xd["v"],
                    xd["a"], xd["b"], torch.from_numpy(A_log).cuda(), torch.from_numpy(dt_bias).cuda(), out, err, 16)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = to_f64(out)
    for b, s in enumerate(SLOTS):
        sub = {k: v[cu[b]:cu[b + 1]] for k, v in x.items()}
        p1 = host[int(s)][None].copy()
        ref, _ = oracle.prefill(p1, "f32", np.array([0], np.int32), np.array([0, lens[b]], np.int32), sub["q"],
                                sub["k"], sub["v"], sub["a"], sub["b"], "bf16", A_log, dt_bias, 16)
        assert maxabs(got[cu[b]:cu[b + 1]], ref) <= OUT_TOL, b
        assert maxabs(to_f64(pool[int(s)]), p1[0].astype(np.float64)) <= TOL["f32"], b
