"""GPU parity of gdn_prefill (variable-length prefill with a rounded state
write-back per chunk) against the CPU oracle.

Small cases compare every output token and every slot of the pool, over
lengths that end inside, at and just past the kernel's 16-token staging
chunks and over several write-back intervals; a split of a sequence at a
chunk boundary into two calls must give bit-identical results; the full-size
workload (19 sequences of 2048 tokens, Qwen3-Next head shapes) compares
sampled (sequence, head) units, which the oracle recomputes from the initial
state.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_ssm_gated_gb300 import build, gdn
from hybrid_ssm_gated_gb300 import workload as wl
from tests.gpu_util import TOL, TORCH_DT, dev, dev_err, maxabs, sample_units, step_to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gdn.lib()


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def _gpu_prefill(pool_gpu, slots, cu, x, w, interval, out_dtype="f32", params=None):
    xd = step_to_device(x, w.in_dtype)
    total = int(cu[-1])
    out = torch.full((total, w.Hv, w.dv), 7.0, dtype=TORCH_DT[out_dtype], device="cuda")
    A_log, dt_bias = wl.head_params(w) if params is None else params
    err = dev_err()
    gdn.gdn_prefill(pool_gpu, torch.from_numpy(np.asarray(slots, np.int32)).cuda(), torch.from_numpy(cu).cuda(),
                    xd["q"], xd["k"], xd["v"], xd["a"], xd["b"], torch.from_numpy(A_log).cuda(),
                    torch.from_numpy(dt_bias).cuda(), out, err, interval)
    torch.cuda.synchronize()
    return out, int(err.item())


def _check_all(w, lens, slots, interval, out_dtype="f32", expect_err=0, params=None):
    cu = _cu(lens)
    pool = wl.initial_pool(w)
    pool_gpu = dev(pool, w.state_dtype)
    x = wl.prefill_inputs(w, int(cu[-1]))
    out, err = _gpu_prefill(pool_gpu, slots, cu, x, w, interval, out_dtype, params)
    assert err == expect_err
    A_log, dt_bias = wl.head_params(w) if params is None else params
    ref, bad = oracle.prefill(pool, w.state_dtype, slots, cu, x["q"], x["k"], x["v"], x["a"], x["b"], w.in_dtype,
                              A_log, dt_bias, interval, nthreads=8)
    got = to_f64(out)
    ulp = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}[out_dtype]
    tol = TOL[w.state_dtype] + ulp * np.abs(ref)
    assert np.all(np.abs(got - ref) <= tol), f"outputs: max |diff| {maxabs(got, ref):.3e}"
    final = to_f64(pool_gpu)
    assert maxabs(final, oracle.load(pool, w.state_dtype)) <= TOL[w.state_dtype]
    untouched = np.setdiff1d(np.arange(w.num_slots), np.asarray(slots)[np.asarray(lens) > 0])
    for s in untouched:  # slots no sequence with tokens names keep their bits
        assert np.array_equal(to_f64(pool_gpu[s]), oracle.load(wl.initial_pool(w)[s], w.state_dtype))


LENS = [0, 1, 15, 16, 17, 33, 50]


@pytest.mark.parametrize("sdt,idt", [("f32", "f32"), ("f32", "bf16"), ("bf16", "bf16"), ("f16", "f16")])
@pytest.mark.parametrize("interval", [1, 5, 16, 64])
def test_prefill_small_all_elements(sdt, idt, interval):
    w = wl.Workload("pf", B=len(LENS), Hk=2, Hv=4, dk=128, dv=128, steps=1, state_dtype=sdt, in_dtype=idt, seed=61)
    _check_all(w, LENS, wl.slots(w), interval)


@pytest.mark.parametrize("dk,dv,Hk,Hv", [(64, 64, 1, 2), (32, 96, 2, 4), (128, 32, 2, 2), (64, 256, 1, 1),
                                         (32, 16, 1, 2)])
@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_prefill_other_head_shapes(dk, dv, Hk, Hv, sdt):
    w = wl.Workload("pfh", B=4, Hk=Hk, Hv=Hv, dk=dk, dv=dv, steps=1, state_dtype=sdt, in_dtype="bf16", seed=62)
    _check_all(w, [3, 16, 40, 0], wl.slots(w), 8)


@pytest.mark.parametrize("sdt,d", [("f32", 64), ("bf16", 64), ("bf16", 128), ("f16", 128)])
def test_prefill_extreme_decays(sdt, d):
    # decays near 1, tiny ones and ones that underflow FP32 (A_log = 5, dt_bias = 5: alpha ~ e^-740); with
    # 16-bit states and d = 128 on the chunked tensor-core kernel, whose decays are ratios within a chunk
    w = wl.Workload("pfx", B=3, Hk=1, Hv=4, dk=d, dv=d, steps=1, state_dtype=sdt, in_dtype="f32", seed=66)
    params = (np.array([-4.0, 1.0, 3.0, 5.0], np.float32), np.array([-6.0, 0.0, 2.0, 5.0], np.float32))
    _check_all(w, [40, 70, 17], wl.slots(w), 16, params=params)


@pytest.mark.parametrize("sdt", ["bf16", "f16"])
def test_prefill_tensor_core_shapes(sdt):
    # d = 128 keys with 16-bit states take the tensor-core kernel: dv = 256 (two row blocks), GQA, ragged
    # lengths, an interval that does not divide the 64-token chunks
    w = wl.Workload("pftc", B=3, Hk=1, Hv=2, dk=128, dv=256, steps=1, state_dtype=sdt, in_dtype="bf16", seed=67)
    _check_all(w, [70, 3, 130], wl.slots(w), 48)


def test_prefill_tensor_core_padding_out_of_range_and_narrow_output():
    w = wl.Workload("pftp", B=4, Hk=1, Hv=2, dk=128, dv=128, steps=1, state_dtype="bf16", in_dtype="bf16",
                    num_slots=6, seed=68)
    _check_all(w, [9, 20, 5, 12], np.array([4, -1, 11, 0], np.int32), 4, out_dtype="bf16",
               expect_err=gdn.DEVERR_SLOT)


def test_prefill_padding_out_of_range_and_narrow_output():
    w = wl.Workload("pfp", B=4, Hk=2, Hv=4, dk=64, dv=64, steps=1, state_dtype="f32", in_dtype="bf16", num_slots=6,
                    seed=63)
    _check_all(w, [9, 20, 5, 12], np.array([4, -1, 11, 0], np.int32), 4, out_dtype="bf16",
               expect_err=gdn.DEVERR_SLOT)


def test_prefill_bad_offsets_are_reported_not_fatal():
    w = wl.Workload("pfe", B=3, Hk=1, Hv=2, dk=32, dv=32, steps=1, state_dtype="f32", in_dtype="f32", seed=64)
    cu = np.array([0, 4, 11, 10], np.int32)  # sequence 1 ends past the 10 tokens, sequence 2 runs backwards
    pool = wl.initial_pool(w)
    pool_gpu = dev(pool, "f32")
    x = wl.prefill_inputs(w, 10)
    out, err = _gpu_prefill(pool_gpu, wl.slots(w), cu, x, w, 4)
    assert err == gdn.DEVERR_SEQLEN
    A_log, dt_bias = wl.head_params(w)
    slots = wl.slots(w)
    sub = {k_: v_[:4] for k_, v_ in x.items()}
    p1 = pool[slots[0]][None].copy()
    ref, _ = oracle.prefill(p1, "f32", np.array([0], np.int32), np.array([0, 4], np.int32), sub["q"], sub["k"],
                            sub["v"], sub["a"], sub["b"], "f32", A_log, dt_bias, 4)
    assert maxabs(to_f64(out[:4]), ref) <= TOL["f32"]  # sequence 0 is still right
    assert maxabs(to_f64(pool_gpu[slots[0]]), p1[0]) <= TOL["f32"]
    for b in (1, 2):  # the refused sequences' states are untouched
        assert np.array_equal(to_f64(pool_gpu[slots[b]]), pool[slots[b]].astype(np.float64))


@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_split_at_a_chunk_boundary_is_bit_identical(sdt):
    w = wl.Workload("pfs", B=3, Hk=2, Hv=4, dk=128, dv=128, steps=1, state_dtype=sdt, in_dtype="bf16", seed=65)
    lens = np.array([48, 80, 33], np.int32)
    first = np.array([32, 16, 32], np.int32)  # multiples of the write-back interval 16
    x = wl.prefill_inputs(w, int(lens.sum()))
    cu = _cu(lens)
    pool = wl.initial_pool(w)
    one = dev(pool, sdt)
    out_one, err = _gpu_prefill(one, wl.slots(w), cu, x, w, 16)
    assert err == 0
    two = dev(pool, sdt)
    idx_a = np.concatenate([np.arange(cu[i], cu[i] + first[i]) for i in range(3)])
    idx_b = np.concatenate([np.arange(cu[i] + first[i], cu[i + 1]) for i in range(3)])
    out_a, e1 = _gpu_prefill(two, wl.slots(w), _cu(first), {k_: v_[idx_a] for k_, v_ in x.items()}, w, 16)
    out_b, e2 = _gpu_prefill(two, wl.slots(w), _cu(lens - first), {k_: v_[idx_b] for k_, v_ in x.items()}, w, 16)
    assert e1 == e2 == 0
    assert torch.equal(one, two)
    assert torch.equal(out_one[torch.from_numpy(idx_a).cuda()], out_a)
    assert torch.equal(out_one[torch.from_numpy(idx_b).cuda()], out_b)


@pytest.mark.slow
@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_prefill_full_size_sampled(sdt):
    w = wl.WORKLOADS["prefill_b19_f32"].with_(state_dtype=sdt)
    lens = np.full(w.B, w.prefill_len, np.int32)
    cu = _cu(lens)
    pool = wl.initial_pool(w)
    pool_gpu = dev(pool, sdt)
    slots = wl.slots(w)
    x = wl.prefill_inputs(w, int(cu[-1]))
    out, err = _gpu_prefill(pool_gpu, slots, cu, x, w, 64)
    assert err == 0
    got = to_f64(out)
    A_log, dt_bias = wl.head_params(w)
    for b, h in sample_units(w.B, w.Hv, 6, seed=11):
        kh = h // (w.Hv // w.Hk)
        sl = slice(cu[b], cu[b + 1])
        al_be = [oracle.gating(A_log[h], dt_bias[h], wl.values(x["a"][t, h], w.in_dtype),
                               wl.values(x["b"][t, h], w.in_dtype)) for t in range(cu[b], cu[b + 1])]
        S = pool[slots[b], h].copy()
        ref = oracle.prefill_head(S, sdt, x["q"][sl, kh], x["k"][sl, kh], x["v"][sl, h], w.in_dtype,
                                  [g[0] for g in al_be], [g[1] for g in al_be], 64)
        assert maxabs(got[sl, h], ref) <= TOL[sdt], (b, h)
        assert maxabs(to_f64(pool_gpu[slots[b], h]), oracle.load(S, sdt)) <= TOL[sdt], (b, h)
