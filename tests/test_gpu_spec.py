"""GPU parity of gdn_spec_step (speculative step with one state copy per window
token) against the CPU oracle.

Small cases compare every output and every slot of the pool after several
chained rounds (the next round starts from the copy of the last accepted token,
as a speculative decoder would); the full-size case compares sampled (sequence,
head) units, which the oracle recomputes from the source state.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_ssm_gated_gb300 import build, gdn
from hybrid_ssm_gated_gb300 import workload as wl
from tests.gpu_util import TOL, dev, dev_err, maxabs, sample_units, step_to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gdn.lib()


def _plan(B, T, seed, pad=False, skip=False, in_place=False):
    """Source slots [B] and destination slots [B, T] in a pool of B * (T + 1) slots."""
    r = np.random.default_rng(seed)
    perm = r.permutation(B * (T + 1)).astype(np.int32)
    src, dst = perm[:B].copy(), perm[B:].reshape(B, T).copy()
    if pad:
        src[r.random(B) < 0.25] = -1
    if skip:
        dst[r.random((B, T)) < 0.25] = -1
    if in_place:
        last = r.random(B) < 0.5
        dst[last, T - 1] = src[last]
    return src, dst


def _run(w: wl.Workload, rounds: int, seed: int, **plan):
    B, T = w.B, w.T
    src, dst = _plan(B, T, seed, **plan)
    num_slots = B * (T + 1)
    pool = wl.initial_pool(w.with_(num_slots=num_slots))
    pool_gpu = dev(pool, w.state_dtype)
    A_log, dt_bias = wl.head_params(w)
    A_d, dt_d = torch.from_numpy(A_log).cuda(), torch.from_numpy(dt_bias).cuda()
    err = dev_err()
    r = np.random.default_rng(seed + 1)
    for rd in range(rounds):
        x = wl.step_inputs(w, rd)
        xd = step_to_device(x, w.in_dtype)
        out = torch.full((B, T, w.Hv, w.dv), 7.0, device="cuda")
        gdn.gdn_spec_step(pool_gpu, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), xd["q"], xd["k"],
                          xd["v"], xd["a"], xd["b"], A_d, dt_d, out, err)
        ref, bad = oracle.spec_step(pool, w.state_dtype, src, dst, x["q"], x["k"], x["v"], x["a"], x["b"],
                                    w.in_dtype, A_log, dt_bias, nthreads=8)
        assert bad == 0
        got = to_f64(out)
        assert maxabs(got, ref) <= TOL[w.state_dtype], f"round {rd}: outputs {maxabs(got, ref):.3e}"
        for bi in np.flatnonzero(src < 0):
            assert np.all(got[bi] == 0.0)
        # the next round starts from the copy of a random accepted token (one that was written)
        acc = r.integers(0, T, B)
        nxt = np.array([dst[bi, acc[bi]] for bi in range(B)], np.int32)
        keep = (nxt >= 0) & (src >= 0)
        free = np.setdiff1d(np.arange(num_slots, dtype=np.int32), nxt[keep])
        new_src = np.where(keep, nxt, src)
        # fresh destinations for the next round among the slots nobody starts from
        cand = np.setdiff1d(free, new_src[new_src >= 0])
        r.shuffle(cand)
        new_dst = cand[: B * T].reshape(B, T).astype(np.int32)
        new_dst[dst < 0] = -1
        src, dst = new_src.astype(np.int32), new_dst
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    final = to_f64(pool_gpu)
    ref_pool = oracle.load(pool, w.state_dtype)
    assert maxabs(final, ref_pool) <= TOL[w.state_dtype], f"pool {maxabs(final, ref_pool):.3e}"


@pytest.mark.parametrize("sdt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("T", [1, 3, 4, 8])
def test_spec_small_all_units(sdt, T):
    w = wl.Workload("sp", B=3, Hk=1, Hv=2, dk=32, dv=32, steps=1, state_dtype=sdt, in_dtype="f32", T=T, seed=31)
    _run(w, rounds=3, seed=T)


@pytest.mark.parametrize("sdt,idt", [("f32", "bf16"), ("bf16", "bf16"), ("f16", "f16")])
def test_spec_multi_round_padding_and_in_place(sdt, idt):
    # 20 x 8 = 160 units over 152 persistent CTAs: a ragged second round
    w = wl.Workload("spm", B=20, Hk=2, Hv=8, dk=128, dv=128, steps=1, state_dtype=sdt, in_dtype=idt, T=4, seed=32)
    _run(w, rounds=3, seed=5, pad=True, skip=True, in_place=True)


@pytest.mark.parametrize("dk,dv,T", [(64, 32, 2), (128, 256, 5), (32, 96, 8), (64, 48, 4)])
def test_spec_other_head_shapes(dk, dv, T):
    w = wl.Workload("sph", B=5, Hk=2, Hv=4, dk=dk, dv=dv, steps=1, state_dtype="f32", in_dtype="bf16", T=T,
                    seed=33)
    _run(w, rounds=2, seed=dk + dv, skip=True)


def test_spec_out_of_range_destination_is_refused():
    w = wl.Workload("spe", B=3, Hk=1, Hv=2, dk=32, dv=32, steps=1, state_dtype="f32", in_dtype="f32", T=2, seed=34)
    src, dst = _plan(3, 2, 9)
    num_slots = 9
    dst[1, 1] = num_slots + 3
    pool = wl.initial_pool(w.with_(num_slots=num_slots))
    pool_gpu = dev(pool, "f32")
    before = pool_gpu.clone()
    A_log, dt_bias = wl.head_params(w)
    x = step_to_device(wl.step_inputs(w, 0), "f32")
    out = torch.full((3, 2, 2, 32), 7.0, device="cuda")
    err = dev_err()
    gdn.gdn_spec_step(pool_gpu, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), x["q"], x["k"], x["v"],
                      x["a"], x["b"], torch.from_numpy(A_log).cuda(), torch.from_numpy(dt_bias).cuda(), out, err)
    torch.cuda.synchronize()
    assert int(err.item()) == gdn.DEVERR_SLOT
    assert torch.all(out[1] == 0) and torch.all(out[0] != 7.0) and torch.all(out[2] != 7.0)
    assert torch.equal(pool_gpu[dst[1, 0]], before[dst[1, 0]])  # nothing of sequence 1 is written


@pytest.mark.slow
@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_spec_b256_sampled(sdt):
    w = wl.Workload("spec_b256", B=256, Hk=16, Hv=32, dk=128, dv=128, steps=1, state_dtype=sdt, in_dtype="bf16",
                    T=4, seed=35)
    B, T = w.B, w.T
    src, dst = _plan(B, T, 11, in_place=True)
    num_slots = B * (T + 1)
    pool = wl.initial_pool(w.with_(num_slots=num_slots))
    pool_gpu = dev(pool, sdt)
    A_log, dt_bias = wl.head_params(w)
    x = wl.step_inputs(w, 0)
    xd = step_to_device(x, w.in_dtype)
    out = torch.empty((B, T, w.Hv, w.dv), device="cuda")
    err = dev_err()
    gdn.gdn_spec_step(pool_gpu, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), xd["q"], xd["k"],
                      xd["v"], xd["a"], xd["b"], torch.from_numpy(A_log).cuda(), torch.from_numpy(dt_bias).cuda(),
                      out, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = to_f64(out)
    kh_of = lambda h: h // (w.Hv // w.Hk)
    for b, h in sample_units(B, w.Hv, 12, seed=7):
        al = np.empty(T)
        be = np.empty(T)
        for t in range(T):
            av = wl.values(x["a"][b, t, h], w.in_dtype)
            bv = wl.values(x["b"][b, t, h], w.in_dtype)
            al[t], be[t] = oracle.gating(float(A_log[h]), float(dt_bias[h]), float(av), float(bv))
        o, copies = oracle.spec_head(pool[src[b], h], sdt, x["q"][b, :, kh_of(h)], x["k"][b, :, kh_of(h)],
                                     x["v"][b, :, h], w.in_dtype, al, be)
        assert maxabs(got[b, :, h], o) <= TOL[sdt], (b, h)
        for t in range(T):
            copy = to_f64(pool_gpu[dst[b, t], h])
            assert maxabs(copy, oracle.load(copies[t], sdt)) <= TOL[sdt], (b, h, t)
