"""Pins of the oracle's two-checkpoint ReplaySSM mode (oracle.ReplayHead with
read_dtype): a high-precision checkpoint for the recurrence and a
low-precision copy for reading. Fixed independently of the mode's code:

- with fp64 for both copies it is the single-checkpoint replay, exactly, through
  folds, verify windows and rollbacks;
- between folds its outputs are those of a single-checkpoint replay whose
  checkpoint is the current read copy;
- after a fold the read copy is the stored master rounded to the read dtype (a value just above a
  bf16 tie shows the fp32 store comes first);
- dk = dv = 1: the fold's closed form, whose prediction comes from the master
  (the AREX ReplaySSM article, section "缓存输入而非状态", precision paragraph:
  the recurrence runs on the high-precision checkpoint); a fold that predicted
  from the read copy gives a different value;
- the master after any sequence of steps, windows, rollbacks and flushes is
  the checkpoint of a single-checkpoint replay in the master's dtype fed the
  same calls: the read copy never enters the recurrence;
- beta = 0: the fold is the pure decay of the master.
"""
import math

import numpy as np
import pytest

import oracle

EPS = 1e-6


def _tokens(r, T, dk, dv):
    return (r.standard_normal((T, dk)), r.standard_normal((T, dk)), r.standard_normal((T, dv)),
            r.standard_normal(T), r.standard_normal(T))


def _drive(heads, steps, dk, dv, seed, A_log=0.4, dt_bias=-0.2, windows=True):
    """Feed the same token stream to every head: steps of one token, and (optionally) T=3 windows
    with rollbacks. Returns the list of per-call outputs of every head."""
    r = np.random.default_rng(seed)
    outs = [[] for _ in heads]
    for s in range(steps):
        T = 3 if windows and s % 4 == 3 else 1
        q, k, v, a, b = _tokens(r, T, dk, dv)
        for i, hd in enumerate(heads):
            outs[i].append(hd.window(q, k, v, a, b, A_log, dt_bias))
        if T > 1:
            acc = int(r.integers(0, T))
            for hd in heads:
                hd.rollback(T, acc)
    return outs


def test_fp64_copies_equal_the_single_checkpoint_replay():
    dk, dv, L = 8, 6, 5
    S0 = np.random.default_rng(1).standard_normal((dv, dk))
    two = oracle.ReplayHead(S0, "f64", "f64", L, read_dtype="f64")
    one = oracle.ReplayHead(S0, "f64", "f64", L)
    o2, o1 = _drive([two, one], 30, dk, dv, seed=2)
    for a, b in zip(o2, o1):
        assert np.array_equal(a, b)
    assert np.array_equal(two.S0, one.S0) and np.array_equal(two.Sr, one.S0)
    two.flush(True), one.flush(True)
    assert np.array_equal(two.S0, one.S0)


@pytest.mark.parametrize("mdt,rdt", [("f32", "bf16"), ("f32", "f16"), ("f64", "bf16")])
def test_outputs_read_the_copy_and_folds_refresh_it(mdt, rdt):
    dk, dv, L = 16, 8, 4
    r = np.random.default_rng(3)
    S0 = oracle.round_to(0.3 * r.standard_normal((dv, dk)), mdt)
    two = oracle.ReplayHead(S0, mdt, "f32", L, read_dtype=rdt)
    assert np.array_equal(two.Sr, oracle.round_to(oracle.load(S0, mdt), rdt))
    mirror = oracle.ReplayHead(two.Sr, rdt, "f32", L)  # a single-checkpoint replay on the read copy
    folds = 0
    for s in range(25):
        q, k, v, a, b = _tokens(r, 1, dk, dv)
        a = a.astype(np.float32).astype(np.float64)  # inputs given in fp32
        if two.count + 1 > L:  # this call folds: the mirror restarts from the refreshed copy afterwards
            out = two.window(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32), a, b, 0.3, 0.1)
            folds += 1
            assert np.array_equal(two.Sr, oracle.round_to(oracle.load(two.S0, mdt), rdt))
            mirror = oracle.ReplayHead(two.Sr, rdt, "f32", L, pos=two.ckpt_pos)
            ref = mirror.window(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32), a, b, 0.3, 0.1)
        else:
            out = two.window(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32), a, b, 0.3, 0.1)
            ref = mirror.window(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32), a, b, 0.3, 0.1)
        assert np.array_equal(out, ref), s
    assert folds >= 4


def test_scalar_fold_predicts_from_the_master():
    """dk = dv = 1 with one buffered entry: the fold gives m' = alpha m + k w with
    w = beta (v - alpha m k), m the master, k = x / sqrt(x^2 + eps)."""
    m = 0.7372654321  # not a bf16 value, so the read copy differs from the master
    two = oracle.ReplayHead(np.array([[m]]), "f64", "f64", 1, read_dtype="bf16")
    r_ = float(oracle.load(two.Sr, "bf16")[0, 0])
    assert r_ != m
    x, v, a_in, b_in = 1.25, -0.6, 0.3, 0.8
    A_log, dt_bias = 0.2, -0.1
    alpha, beta = oracle.gating(A_log, dt_bias, a_in, b_in)
    two.window(np.array([[0.5]]), np.array([[x]]), np.array([[v]]), np.array([a_in]), np.array([b_in]), A_log,
               dt_bias)
    # the next window folds that entry first (L = 1)
    two.window(np.array([[0.5]]), np.array([[x]]), np.array([[v]]), np.array([a_in]), np.array([b_in]), A_log,
               dt_bias)
    kn = x / math.sqrt(x * x + EPS)
    expect = alpha * m + kn * beta * (v - alpha * m * kn)
    assert two.S0[0, 0] == pytest.approx(expect, rel=1e-15)
    wrong = alpha * m + kn * beta * (v - alpha * r_ * kn)  # a prediction from the read copy instead
    assert abs(two.S0[0, 0] - wrong) > 1e-6
    assert float(oracle.load(two.Sr, "bf16")[0, 0]) == float(oracle.load(oracle.round_to(np.array([expect]), "bf16"),
                                                                          "bf16")[0])


@pytest.mark.parametrize("mdt,rdt", [("f32", "bf16"), ("f32", "f16")])
def test_master_is_the_single_checkpoint_replay_in_its_dtype(mdt, rdt):
    """The read copy never enters the recurrence: after every call the master equals the checkpoint
    of a single-checkpoint replay stored in the master's dtype and fed the same calls (steps, T = 3
    windows with rollbacks, forced flushes), bit for bit, although the outputs differ."""
    dk, dv, L = 12, 10, 5
    r = np.random.default_rng(11)
    S0 = oracle.round_to(0.3 * r.standard_normal((dv, dk)), mdt)
    two = oracle.ReplayHead(S0, mdt, "f32", L, read_dtype=rdt)
    one = oracle.ReplayHead(S0, mdt, "f32", L)
    differ = False
    folds = 0
    for s in range(40):
        T = 3 if s % 5 == 4 else 1
        q, k, v, a, b = (x.astype(np.float32) for x in _tokens(r, T, dk, dv))
        a, b = a.astype(np.float64), b.astype(np.float64)
        folds += two.count + T > L
        o2 = two.window(q, k, v, a, b, 0.3, 0.1)
        o1 = one.window(q, k, v, a, b, 0.3, 0.1)
        differ = differ or not np.array_equal(o2, o1)
        if T > 1:
            acc = int(r.integers(0, T))
            two.rollback(T, acc), one.rollback(T, acc)
        if s % 13 == 12:
            two.flush(True), one.flush(True)
            folds += 1
        assert np.array_equal(two.S0, one.S0), s
        assert (two.count, two.ckpt_pos) == (one.count, one.ckpt_pos)
    assert differ and folds >= 6


def test_pure_decay_fold():
    """b = -inf: beta = 0, so a fold scales the master by the product of the buffered alphas."""
    dk, dv, L = 8, 4, 3
    r = np.random.default_rng(5)
    M0 = r.standard_normal((dv, dk))
    two = oracle.ReplayHead(M0, "f64", "f64", L, read_dtype="bf16")
    A_log, dt_bias = 0.0, 0.5
    for _ in range(L + 1):  # L entries, then the fold
        q, k, v, _, _ = _tokens(r, 1, dk, dv)
        two.window(q, k, v, np.array([-dt_bias]), np.array([-np.inf]), A_log, dt_bias)
    assert np.allclose(two.S0, 0.5 ** L * M0, rtol=1e-14, atol=0)
    assert np.array_equal(two.Sr, oracle.round_to(two.S0, "bf16"))


def test_copy_is_the_stored_master_rounded_once_more():
    """The copy is the stored fp32 master rounded to bf16, not the fold's fp64 value rounded to bf16.
    With dk = dv = 1, alpha = 1 (a = -inf), beta = 1/2 (b = 0) and a zero checkpoint, one buffered
    token folds to 1 + 2^-8 + 2^-30, just above the bf16 tie between 1 and 1 + 2^-7. The master stores
    the fp32 tie 1 + 2^-8 itself, which rounds to even: the copy is 1. Rounding the fold value directly
    would give 1 + 2^-7."""
    h = oracle.ReplayHead(np.zeros((1, 1)), "f32", "f64", 1, read_dtype="bf16")
    kn = 1.0 / math.sqrt(1.0 + EPS)  # the normalised key of k = 1
    target = 1.0 + 2.0 ** -8 + 2.0 ** -30
    one, a, b = np.ones((1, 1)), np.array([-np.inf]), np.array([0.0])
    h.window(one, one, np.array([[target / (0.5 * kn)]]), a, b, A_log=0.0, dt_bias=0.0)
    h.window(one, one, np.zeros((1, 1)), a, b, A_log=0.0, dt_bias=0.0)  # 1 + 1 > L: the fold comes first
    assert float(h.S0[0, 0]) == 1.0 + 2.0 ** -8
    assert float(oracle.load(h.Sr, "bf16")[0, 0]) == 1.0
