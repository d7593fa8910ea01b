"""GPU parity of gdn_decode_step against the CPU oracle.

Small cases (several persistent rounds, ragged tails, padding) compare every
output and every state element; the full-size workloads compare sampled
(sequence, head) units, which the oracle recomputes through every step, plus
properties that hold at any size (untouched slots bit-exact, slot-permutation
invariance bit-exact).
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_ssm_gated_gb300 import build, gdn
from hybrid_ssm_gated_gb300 import workload as wl
from tests.gpu_util import (TOL, TORCH_DT, decode_oracle_unit, dev, dev_err, maxabs, sample_units,
                            step_to_device, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gdn.lib()


def _run_full(w: wl.Workload, slots=None, out_dtype="f32"):
    """Run w.steps decode steps on GPU and in the oracle over the whole batch."""
    pool = wl.initial_pool(w)
    pool_gpu = dev(pool, w.state_dtype)
    slots = wl.slots(w) if slots is None else np.asarray(slots, np.int32)
    A_log, dt_bias = wl.head_params(w)
    s_d, A_d, dt_d = torch.from_numpy(slots).cuda(), torch.from_numpy(A_log).cuda(), torch.from_numpy(dt_bias).cuda()
    err = dev_err()
    worst = 0.0
    for t in range(w.steps):
        x = wl.step_inputs(w, t)
        xd = step_to_device(x, w.in_dtype)
        out = torch.empty((len(slots), w.Hv, w.dv), dtype=TORCH_DT[out_dtype], device="cuda")
        gdn.gdn_decode_step(pool_gpu, s_d, xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], A_d, dt_d, out, err)
        ref, bad = oracle.decode_step(pool, w.state_dtype, slots, x["q"], x["k"], x["v"], x["a"], x["b"], w.in_dtype,
                                      A_log, dt_bias, nthreads=8)
        got = to_f64(out)
        # a bf16/fp16 output is the fp32 result rounded once: allow half an ulp of the output type
        ulp = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}[out_dtype]
        tol = TOL[w.state_dtype] + ulp * np.abs(ref)
        assert np.all(np.abs(got - ref) <= tol), f"step {t}: max |diff| {maxabs(got, ref):.3e}"
        worst = max(worst, maxabs(got, ref))
    torch.cuda.synchronize()
    final = to_f64(pool_gpu)
    ref_pool = oracle.load(pool, w.state_dtype)
    assert maxabs(final, ref_pool) <= TOL[w.state_dtype], f"final state {maxabs(final, ref_pool):.3e}"
    return int(err.item()), final, ref_pool, worst


def test_tiny_workload_all_elements():
    w = wl.WORKLOADS["tiny"]
    err, final, ref, worst = _run_full(w)
    assert err == 0
    assert worst < 1e-5


@pytest.mark.parametrize("sdt,idt", [("f32", "bf16"), ("bf16", "bf16"), ("f16", "bf16"), ("f32", "f32"),
                                     ("bf16", "f16"), ("f16", "f32")])
def test_multi_round_ragged(sdt, idt):
    # 40 x 8 = 320 units over at most 152 persistent CTAs: several rounds and a ragged tail
    w = wl.Workload("ragged", B=40, Hk=4, Hv=8, dk=128, dv=128, steps=3, state_dtype=sdt, in_dtype=idt,
                    num_slots=50, seed=7)
    err, *_ = _run_full(w)
    assert err == 0


@pytest.mark.parametrize("dk,dv,Hk,Hv", [(64, 48, 2, 2), (32, 96, 1, 4), (32, 256, 2, 4), (64, 64, 3, 6),
                                         (128, 16, 2, 8), (128, 256, 1, 2)])
@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_other_head_shapes(dk, dv, Hk, Hv, sdt):
    w = wl.Workload("shape", B=9, Hk=Hk, Hv=Hv, dk=dk, dv=dv, steps=3, state_dtype=sdt, in_dtype="bf16", seed=11)
    err, *_ = _run_full(w)
    assert err == 0


@pytest.mark.parametrize("out_dtype", ["bf16", "f16"])
def test_narrow_output(out_dtype):
    w = wl.Workload("out", B=6, Hk=2, Hv=4, dk=128, dv=128, steps=2, seed=3)
    err, *_ = _run_full(w, out_dtype=out_dtype)
    assert err == 0


def test_padding_and_out_of_range_slots():
    w = wl.Workload("pad", B=6, Hk=2, Hv=4, dk=128, dv=64, steps=2, num_slots=8, seed=5)
    slots = np.array([3, -1, 9, 0, -5, 7], dtype=np.int32)  # 9 >= num_slots
    pool0 = wl.initial_pool(w)
    pool = pool0.copy()
    pool_gpu = dev(pool, "f32")
    A_log, dt_bias = wl.head_params(w)
    err = dev_err()
    out = torch.full((6, w.Hv, w.dv), 7.0, device="cuda")
    x = step_to_device(wl.step_inputs(w, 0), w.in_dtype)
    gdn.gdn_decode_step(pool_gpu, torch.from_numpy(slots).cuda(), x["q"], x["k"], x["v"], x["a"], x["b"],
                        torch.from_numpy(A_log).cuda(), torch.from_numpy(dt_bias).cuda(), out, err)
    o = out.cpu().numpy()
    assert int(err.item()) == gdn.DEVERR_SLOT
    assert np.all(o[[1, 2, 4]] == 0.0) and np.all(o[[0, 3, 5]] != 7.0)
    p = pool_gpu.cpu().numpy()
    for s in range(8):
        same = np.array_equal(p[s], pool0[s])
        assert same == (s not in (3, 0, 7)), f"slot {s}"


@pytest.mark.parametrize("sdt", ["bf16", "f16"])
def test_padding_over_several_batches(sdt):
    """160 x 32 = 5,120 units: more than 32 per CTA of a 152-CTA grid, so CTAs take a second batch of units.
    A third of the sequences are padding and a seventh out of range, so the valid units before a unit differ
    from its position: with 16-bit states two producer warps count them to place each unit's chunk fills."""
    w = wl.Workload("padb", B=160, Hk=2, Hv=32, dk=64, dv=64, steps=2, state_dtype=sdt, in_dtype="bf16",
                    num_slots=400, seed=7)
    slots = wl.slots(w).copy()
    slots[::3] = -1
    slots[1::7] = w.num_slots + 5
    err, *_ = _run_full(w, slots=slots)
    assert err == gdn.DEVERR_SLOT


def test_empty_batch():
    pool = torch.zeros((2, 2, 32, 32), device="cuda")
    z = torch.zeros(0, device="cuda")
    gdn.gdn_decode_step(pool, torch.zeros(0, dtype=torch.int32, device="cuda"), z.reshape(0, 2, 32),
                        z.reshape(0, 2, 32), z.reshape(0, 2, 32), z.reshape(0, 2), z.reshape(0, 2),
                        torch.zeros(2, device="cuda"), torch.zeros(2, device="cuda"), z.reshape(0, 2, 32), dev_err())
    torch.cuda.synchronize()
    assert torch.count_nonzero(pool) == 0


def test_slot_permutation_is_bit_exact():
    """Permuting batch rows together with their slots permutes the outputs
    bit-exactly and leaves an identical pool."""
    w = wl.WORKLOADS["qwen3next_b64"].with_(B=16, num_slots=24, steps=1)
    pool = dev(wl.initial_pool(w), "f32")
    slots = wl.slots(w)
    perm = np.random.default_rng(1).permutation(w.B)
    A_log, dt_bias = (torch.from_numpy(t).cuda() for t in wl.head_params(w))
    x = step_to_device(wl.step_inputs(w, 0), w.in_dtype)
    outs, pools = [], []
    for order in (np.arange(w.B), perm):
        p = pool.clone()
        o = torch.empty((w.B, w.Hv, w.dv), device="cuda")
        oi = torch.from_numpy(order).cuda()
        gdn.gdn_decode_step(p, torch.from_numpy(slots[order]).cuda(), x["q"][oi].contiguous(),
                            x["k"][oi].contiguous(), x["v"][oi].contiguous(), x["a"][oi].contiguous(),
                            x["b"][oi].contiguous(), A_log, dt_bias, o, dev_err())
        outs.append(o)
        pools.append(p)
    inv = np.argsort(perm)
    assert torch.equal(outs[1][torch.from_numpy(inv).cuda()], outs[0])
    assert torch.equal(pools[0], pools[1])


def _run_sampled(w: wl.Workload, n_units: int):
    """Full-size run on the GPU; the oracle follows sampled units through every step."""
    pool = wl.initial_pool(w)
    pool_gpu = dev(pool, w.state_dtype)
    slots = wl.slots(w)
    A_log, dt_bias = wl.head_params(w)
    s_d, A_d, dt_d = torch.from_numpy(slots).cuda(), torch.from_numpy(A_log).cuda(), torch.from_numpy(dt_bias).cuda()
    units = sample_units(w.B, w.Hv, n_units)
    S = {u: pool[slots[u[0]], u[1]].copy() for u in units}
    S_exact = {u: oracle.load(pool[slots[u[0]], u[1]], w.state_dtype).copy() for u in units}  # no rounding
    bi = torch.tensor([b for b, _ in units], device="cuda")
    hi = torch.tensor([h for _, h in units], device="cuda")
    err = dev_err()
    out = torch.empty((w.B, w.Hv, w.dv), device="cuda")
    worst, drift = 0.0, 0.0
    for t in range(w.steps):
        x = wl.step_inputs(w, t)
        xd = step_to_device(x, w.in_dtype)
        gdn.gdn_decode_step(pool_gpu, s_d, xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], A_d, dt_d, out, err)
        got = to_f64(out[bi, hi])
        for i, (b, h) in enumerate(units):
            ref = decode_oracle_unit(S[(b, h)], w.state_dtype, x, w.in_dtype, b, h, w.Hv, w.Hk, A_log, dt_bias)
            exact = decode_oracle_unit(S_exact[(b, h)], "f64", x, w.in_dtype, b, h, w.Hv, w.Hk, A_log, dt_bias)
            d = maxabs(got[i], ref)
            assert d <= TOL[w.state_dtype], f"step {t} unit {(b, h)}: {d:.3e}"
            worst = max(worst, d)
            drift = max(drift, maxabs(got[i], exact))
    final = pool_gpu[torch.from_numpy(slots).cuda()[bi], hi]
    for i, u in enumerate(units):
        d = maxabs(to_f64(final[i]), oracle.load(S[u], w.state_dtype))
        assert d <= TOL[w.state_dtype], f"final state of {u}: {d:.3e}"
    untouched = np.setdiff1d(np.arange(w.num_slots), slots)[:8]
    for s in untouched:
        assert torch.equal(pool_gpu[int(s)].cpu(), wl.to_torch(pool[s], w.state_dtype)), f"slot {s} modified"
    assert int(err.item()) == 0
    return worst, drift


@pytest.mark.slow
def test_qwen3next_b64_100_steps_sampled():
    worst, drift = _run_sampled(wl.WORKLOADS["qwen3next_b64"], 12)
    assert worst < 1e-4


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode_b256_bf16", "decode_b256_f16"])
def test_b256_low_precision_200_steps_sampled(name):
    worst, drift = _run_sampled(wl.WORKLOADS[name], 16)
    print(f"{name}: max |gpu - oracle(rounded)| = {worst:.3e}; drift vs unrounded fp64 = {drift:.3e}")
    assert worst <= 1e-2


@pytest.mark.slow
def test_b256_fp32_sampled():
    worst, _ = _run_sampled(wl.WORKLOADS["decode_b256_f32"].with_(steps=20), 16)
    assert worst < 1e-4
