"""Pins of the oracle's speculative step with one state copy per window token
(oracle.spec_head / oracle.spec_step) -- the baseline that a ReplaySSM verify
window replaces -- against things fixed independently of it:

- with fp64 storage (no rounding anywhere) the window equals the same tokens
  fed one at a time through the oracle's decode step, whose own pins are in
  test_oracle_pins.py; every copy equals the state after its token;
- with narrow storage every copy is the fp64 state after its token rounded
  once, while later tokens still start from the unrounded state;
- beta = 0 leaves only the decay, in closed form;
- a window of one token written back to its own slot is exactly a decode step;
- padding and out-of-range slots.
"""
import math

import numpy as np
import pytest

import oracle

EPS = 1e-6


def _window(B, T, Hk, Hv, dk, dv, seed):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, Hk, dk)).astype(np.float32)
    k = r.standard_normal((B, T, Hk, dk)).astype(np.float32)
    v = r.standard_normal((B, T, Hv, dv)).astype(np.float32)
    a = r.standard_normal((B, T, Hv)).astype(np.float32)
    b = r.standard_normal((B, T, Hv)).astype(np.float32)
    A_log = r.uniform(0, 2, Hv).astype(np.float32)
    dt_bias = r.uniform(-1, 1, Hv).astype(np.float32)
    return q, k, v, a, b, A_log, dt_bias


def test_fp64_window_equals_sequential_decode_steps():
    B, T, Hk, Hv, dk, dv = 3, 4, 2, 4, 16, 8
    q, k, v, a, b, A_log, dt_bias = _window(B, T, Hk, Hv, dk, dv, seed=1)
    r = np.random.default_rng(2)
    pool = r.standard_normal((12, Hv, dv, dk))
    src = np.array([0, 5, 9], np.int32)
    dst = np.array([[1, 2, 3, 4], [6, 7, 8, 10], [11, -1, -1, 9]], np.int32)  # the last one ends in place
    ref = pool.copy()
    out, bad = oracle.spec_step(pool, "f64", src, dst, q, k, v, a, b, "f32", A_log, dt_bias)
    assert bad == 0
    for t in range(T):  # the same tokens, one decode step at a time on the source slots
        o_t, bad = oracle.decode_step(ref, "f64", src, q[:, t], k[:, t], v[:, t], a[:, t], b[:, t], "f32", A_log,
                                      dt_bias)
        assert bad == 0
        assert np.array_equal(out[:, t], o_t)
        for bi in range(B):
            if dst[bi, t] >= 0 and dst[bi, t] != src[bi]:
                assert np.array_equal(pool[dst[bi, t]], ref[src[bi]])
    assert np.array_equal(pool[9], ref[9])  # the copy written back to the source slot is the final state


@pytest.mark.parametrize("sdt", ["f32", "bf16", "f16"])
def test_narrow_copies_are_fp64_states_rounded_once(sdt):
    dk, dv, T = 16, 8, 5
    r = np.random.default_rng(3)
    S64 = (0.3 * r.standard_normal((dv, dk))).astype(np.float64)
    S = oracle.round_to(S64, sdt)
    q, k = r.standard_normal((T, dk)), r.standard_normal((T, dk))
    v = r.standard_normal((T, dv))
    al, be = r.uniform(0.3, 1.0, T), r.uniform(0.1, 0.9, T)
    out, copies = oracle.spec_head(S, sdt, q, k, v, "f64", al, be)
    out64, copies64 = oracle.spec_head(oracle.load(S, sdt).astype(np.float64), "f64", q, k, v, "f64", al, be)
    assert np.array_equal(out, out64)  # outputs come from the unrounded recursion
    for t in range(T):
        assert np.array_equal(copies[t], oracle.round_to(copies64[t], sdt))
    # continuing from a rounded copy is a different computation: the recursion must not
    rounded_restart, _ = oracle.spec_head(copies[1], sdt, q[2:], k[2:], v[2:], "f64", al[2:], be[2:])
    assert not np.array_equal(rounded_restart, out[2:]) or sdt == "f32"


def test_pure_decay_closed_form():
    """b = -inf gives beta = 0: S after token t is (prod_{s<=t} alpha_s) S0, and with q = e_m the
    output of token t is column m of that state, scaled by the normalisation of q."""
    B, T, Hk, Hv, dk, dv = 2, 3, 1, 2, 8, 4
    r = np.random.default_rng(5)
    pool = r.standard_normal((6, Hv, dv, dk))
    pool0 = pool.copy()
    src = np.array([4, 1], np.int32)
    dst = np.array([[0, 2, 3], [5, -1, 1]], np.int32)
    m = 3
    q = np.zeros((B, T, Hk, dk), np.float32)
    q[..., m] = 1.0
    k = r.standard_normal((B, T, Hk, dk)).astype(np.float32)
    v = r.standard_normal((B, T, Hv, dv)).astype(np.float32)
    dt_bias = np.array([0.5, -0.75], np.float32)
    A_log = np.zeros(Hv, np.float32)
    a = np.broadcast_to(-dt_bias, (B, T, Hv)).astype(np.float32)  # softplus(0) = ln 2: alpha = 1/2
    b = np.full((B, T, Hv), -np.inf, np.float32)
    out, bad = oracle.spec_step(pool, "f64", src, dst, q, k, v, a, b, "f32", A_log, dt_bias)
    assert bad == 0
    for bi in range(B):
        for t in range(T):
            scale = 2.0 ** -(t + 1)
            expect = scale * pool0[src[bi]][:, :, m] / math.sqrt(1 + EPS) / math.sqrt(dk)
            assert np.allclose(out[bi, t], expect, rtol=1e-12, atol=1e-300)
            if dst[bi, t] >= 0:
                assert np.allclose(pool[dst[bi, t]], scale * pool0[src[bi]], rtol=1e-14, atol=0)


@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_window_of_one_in_place_is_a_decode_step(sdt):
    B, T, Hk, Hv, dk, dv = 4, 1, 2, 4, 32, 16
    q, k, v, a, b, A_log, dt_bias = _window(B, T, Hk, Hv, dk, dv, seed=6)
    r = np.random.default_rng(7)
    pool = oracle.round_to(0.1 * r.standard_normal((8, Hv, dv, dk)), sdt)
    ref = pool.copy()
    src = np.array([3, 0, 7, 5], np.int32)
    out, bad = oracle.spec_step(pool, sdt, src, src[:, None], q, k, v, a, b, "f32", A_log, dt_bias)
    o1, bad1 = oracle.decode_step(ref, sdt, src, q[:, 0], k[:, 0], v[:, 0], a[:, 0], b[:, 0], "f32", A_log,
                                  dt_bias)
    assert bad == bad1 == 0
    assert np.array_equal(out[:, 0], o1)
    assert np.array_equal(pool.view(np.uint8), ref.view(np.uint8))


def test_padding_and_out_of_range_slots():
    B, T, Hk, Hv, dk, dv = 3, 2, 1, 2, 8, 4
    q, k, v, a, b, A_log, dt_bias = _window(B, T, Hk, Hv, dk, dv, seed=8)
    pool = np.random.default_rng(9).standard_normal((4, Hv, dv, dk))
    pool0 = pool.copy()
    src = np.array([-1, 2, 1], np.int32)
    dst = np.array([[0, 3], [7, 0], [3, -1]], np.int32)  # sequence 1 names slot 7 of 4
    out, bad = oracle.spec_step(pool, "f64", src, dst, q, k, v, a, b, "f32", A_log, dt_bias)
    assert bad == Hv  # every head of sequence 1
    assert np.all(out[0] == 0) and np.all(out[1] == 0) and np.all(out[2] != 0)
    assert np.array_equal(pool[0], pool0[0])  # named only by padding and by the refused sequence
    assert not np.array_equal(pool[3], pool0[3])  # sequence 2's first copy
    assert np.array_equal(pool[2], pool0[2]) and np.array_equal(pool[1], pool0[1])
