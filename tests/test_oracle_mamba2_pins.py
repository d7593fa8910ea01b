"""Pins of the oracle's Mamba2 decode step and Mamba2 ReplaySSM (oracle.m2_*,
oracle.Mamba2ReplayHead) against things fixed independently of them:

- the gates' closed forms (delta = ln 2 and alpha = 1/2 at zero argument, the
  softplus cut-over, the limits);
- B = 0 leaves the pure decay alpha^t S0; S0 = 0 and B = 0 leave y = D x;
- a one-hot B writes one state column, a one-hot C reads one (orientation);
- N = P = 1 equals the closed form of the scalar recurrence;
- random tiny windows equal the quadratic ("dual") form of the same
  recurrence, y_t = sum_{s<=t} decay(s, t) delta_s (C_t . B_s) x_s +
  decay(0, t) S0^T C_t + D x_t, a different order of computation in which a
  swapped B/C, a transposed state or a misplaced decay gives other numbers;
- groups: H = 2G equals duplicated groups, and head h reads group h / (H/G);
- the batch driver's padding and out-of-range slots, narrow rounding once at
  write-back;
- ReplaySSM: with an fp64 checkpoint it equals sequential decode steps
  exactly; a narrow checkpoint changes only at folds, every L steps; a window
  equals its tokens one at a time; a rollback equals a run on the kept tokens;
  the ring holds the raw B and x bits and the gates, and no C.
"""
import math

import numpy as np
import pytest

import oracle


def test_gating_closed_forms():
    al, de = oracle.m2_gating(0.0, 0.0, 0.0)
    assert de == pytest.approx(math.log(2), rel=1e-15) and al == pytest.approx(0.5, rel=1e-15)
    al, de = oracle.m2_gating(math.log(3.0), 0.25, -0.25)  # A = -3, delta = ln 2: alpha = 2^-3
    assert al == pytest.approx(0.125, rel=1e-14)
    al, de = oracle.m2_gating(0.0, 0.0, math.log(15.0))  # below the cut-over: delta = ln 16, alpha = 1/16
    assert de == pytest.approx(4 * math.log(2), rel=1e-14) and al == pytest.approx(1 / 16, rel=1e-14)
    al, de = oracle.m2_gating(0.0, 0.0, math.log(2.0 ** 26 - 1))  # still below it: delta = 26 ln 2
    assert al == pytest.approx(2.0 ** -26, rel=1e-12)
    al, de = oracle.m2_gating(0.0, 10.0, 20.5)  # above the cut-over softplus is the identity
    assert de == 30.5 and al == pytest.approx(math.exp(-30.5), rel=1e-14)
    al, de = oracle.m2_gating(1.0, 0.0, -800.0)
    assert de == 0.0 and al == 1.0
    xs = np.linspace(-5, 5, 41)
    g = np.array([oracle.m2_gating(0.5, 0.1, x) for x in xs])
    assert np.all(np.diff(g[:, 1]) > 0) and np.all(np.diff(g[:, 0]) < 0)


def _head(N, P, seed, sdt="f64"):
    r = np.random.default_rng(seed)
    return oracle.round_to(r.standard_normal((P, N)), sdt), r


def test_pure_decay_and_skip_term():
    N, P = 8, 4
    S, r = _head(N, P, 1)
    S0 = S.copy()
    m = 5
    C = np.zeros(N)
    C[m] = 1.0
    x = r.standard_normal(P)
    for t in range(1, 6):
        y = oracle.m2_decode_head(S, "f64", x, np.zeros(N), C, "f64", 0.5, 0.7, 1.25)
        assert np.array_equal(S, 0.5 ** t * S0)
        assert np.allclose(y, 0.5 ** t * S0[:, m] + 1.25 * x, rtol=1e-15, atol=0)
    Z = np.zeros((P, N))
    y = oracle.m2_decode_head(Z, "f64", x, np.zeros(N), r.standard_normal(N), "f64", 0.3, 0.9, -0.75)
    assert np.array_equal(y, -0.75 * x) and np.all(Z == 0)


def test_one_hot_input_and_readout_orientation():
    N, P = 6, 5
    x = np.random.default_rng(2).standard_normal(P)
    i, j = 2, 4
    Bv, Ci, Cj = np.zeros(N), np.zeros(N), np.zeros(N)
    Bv[i], Ci[i], Cj[j] = 1.0, 1.0, 1.0
    S = np.zeros((P, N))
    y = oracle.m2_decode_head(S, "f64", x, Bv, Ci, "f64", 0.9, 0.4, 0.0)
    assert np.allclose(y, 0.4 * x, rtol=1e-15, atol=0)  # written to column i, read from column i
    assert np.allclose(S[:, i], 0.4 * x, rtol=1e-15, atol=0) and np.all(np.delete(S, i, axis=1) == 0)
    S = np.zeros((P, N))
    y = oracle.m2_decode_head(S, "f64", x, Bv, Cj, "f64", 0.9, 0.4, 0.0)
    assert np.all(y == 0)  # read from another column


def test_scalar_recurrence_closed_form():
    """N = P = 1, constant gates: s_t = a s + d b x, so s_t = a^t s_0 + d b x (1 - a^t)/(1 - a)."""
    a, d, b, x, c, D = 0.8, 0.35, 1.5, -0.6, 0.7, 0.2
    s0 = 0.9
    S = np.array([[s0]])
    for t in range(1, 41):
        y = oracle.m2_decode_head(S, "f64", [x], [b], [c], "f64", a, d, D)
        st = a ** t * s0 + d * b * x * (1 - a ** t) / (1 - a)
        assert S[0, 0] == pytest.approx(st, rel=1e-12)
        assert y[0] == pytest.approx(st * c + D * x, rel=1e-12)


def _dual_form(S0, C, Bm, x, al, de, D):
    """Outputs of T tokens through the quadratic form of the recurrence."""
    T = C.shape[0]
    y = np.zeros((T, S0.shape[0]))
    for t in range(T):
        for s in range(t + 1):
            decay = np.prod(al[s + 1:t + 1])
            y[t] += decay * de[s] * float(C[t] @ Bm[s]) * x[s]
        y[t] += np.prod(al[:t + 1]) * (S0 @ C[t]) + D * x[t]
    return y


@pytest.mark.parametrize("seed", range(6))
def test_windows_equal_the_dual_form(seed):
    r = np.random.default_rng(10 + seed)
    N, P, T = int(r.integers(1, 7)), int(r.integers(1, 7)), int(r.integers(1, 7))
    S0 = r.standard_normal((P, N))
    C, Bm, x = r.standard_normal((T, N)), r.standard_normal((T, N)), r.standard_normal((T, P))
    al, de, D = r.uniform(0.2, 1.0, T), r.uniform(0.05, 1.5, T), float(r.standard_normal())
    S = S0.copy()
    got = np.stack([oracle.m2_decode_head(S, "f64", x[t], Bm[t], C[t], "f64", al[t], de[t], D) for t in range(T)])
    assert np.allclose(got, _dual_form(S0, C, Bm, x, al, de, D), rtol=1e-12, atol=1e-12)


def _batch(B, G, H, N, P, seed, idt="f32"):
    r = np.random.default_rng(seed)
    x = r.standard_normal((B, H, P)).astype(np.float32)
    dt = r.standard_normal((B, H)).astype(np.float32)
    Bm = r.standard_normal((B, G, N)).astype(np.float32)
    Cm = r.standard_normal((B, G, N)).astype(np.float32)
    A_log = r.uniform(0, 2, H).astype(np.float32)
    dt_bias = r.uniform(-1, 1, H).astype(np.float32)
    D = r.uniform(0.5, 1.5, H).astype(np.float32)
    return x, dt, Bm, Cm, A_log, dt_bias, D


def test_groups_map_heads_to_group_h_over_heads_per_group():
    B, G, H, N, P = 2, 2, 4, 8, 4
    x, dt, Bm, Cm, A_log, dt_bias, D = _batch(B, G, H, N, P, 3)
    pool = np.random.default_rng(4).standard_normal((B, H, P, N))
    slots = np.arange(B, dtype=np.int32)
    p1 = pool.copy()
    o1, _ = oracle.m2_decode_step(p1, "f64", slots, x, dt, Bm, Cm, "f32", A_log, dt_bias, D)
    # the same with one group per head (duplicated): H/G = 1
    p2 = pool.copy()
    o2, _ = oracle.m2_decode_step(p2, "f64", slots, x, dt, np.repeat(Bm, 2, axis=1), np.repeat(Cm, 2, axis=1), "f32",
                                  A_log, dt_bias, D)
    assert np.array_equal(o1, o2) and np.array_equal(p1, p2)
    # swapping the groups changes heads 0-1 (group 0) and 2-3 (group 1)
    p3 = pool.copy()
    o3, _ = oracle.m2_decode_step(p3, "f64", slots, x, dt, Bm[:, ::-1].copy(), Cm[:, ::-1].copy(), "f32", A_log,
                                  dt_bias, D)
    assert not np.allclose(o3[:, 0], o1[:, 0]) and not np.allclose(o3[:, 3], o1[:, 3])
    # head h against the single-head step with group h // 2 and its own gates
    for b in range(B):
        for h in range(H):
            al, de = oracle.m2_gating(A_log[h], dt_bias[h], dt[b, h])
            S = pool[b, h].copy()
            y = oracle.m2_decode_head(S, "f64", x[b, h], Bm[b, h // 2], Cm[b, h // 2], "f32", al, de, D[h])
            assert np.array_equal(y, o1[b, h]) and np.array_equal(S, p1[b, h])


def test_padding_and_out_of_range_slots():
    B, G, H, N, P = 3, 1, 2, 4, 4
    x, dt, Bm, Cm, A_log, dt_bias, D = _batch(B, G, H, N, P, 5)
    pool = np.random.default_rng(6).standard_normal((3, H, P, N))
    pool0 = pool.copy()
    slots = np.array([-1, 7, 1], np.int32)
    out, bad = oracle.m2_decode_step(pool, "f64", slots, x, dt, Bm, Cm, "f32", A_log, dt_bias, D)
    assert bad == H
    assert np.all(out[:2] == 0) and np.all(out[2] != 0)
    assert np.array_equal(pool[0], pool0[0]) and np.array_equal(pool[2], pool0[2])
    assert not np.array_equal(pool[1], pool0[1])


@pytest.mark.parametrize("sdt", ["f32", "bf16", "f16"])
def test_narrow_state_rounds_once_at_write_back(sdt):
    N, P = 16, 8
    S, r = _head(N, P, 7, sdt)
    S64 = oracle.load(S, sdt).copy()
    x, Bv, Cv = r.standard_normal(P), r.standard_normal(N), r.standard_normal(N)
    y = oracle.m2_decode_head(S, sdt, x, Bv, Cv, "f64", 0.7, 0.3, 0.5)
    y64 = oracle.m2_decode_head(S64, "f64", x, Bv, Cv, "f64", 0.7, 0.3, 0.5)
    assert np.array_equal(y, y64)
    assert np.array_equal(S, oracle.round_to(S64, sdt))


def _tokens(r, T, N, P):
    return r.standard_normal((T, N)), r.standard_normal((T, N)), r.standard_normal((T, P)), r.standard_normal(T)


def test_replay_fp64_checkpoint_equals_sequential_decode():
    N, P, L = 8, 6, 4
    S0 = np.random.default_rng(8).standard_normal((P, N))
    hd = oracle.Mamba2ReplayHead(S0, "f64", "f64", L)
    S = S0.copy()
    r = np.random.default_rng(9)
    A_log, dt_bias, D = 0.3, -0.2, 0.8
    for step in range(3 * L + 1):
        C, Bv, x, dt = _tokens(r, 1, N, P)
        y = hd.window(C, Bv, x, dt, A_log, dt_bias, D)
        al, de = oracle.m2_gating(A_log, dt_bias, dt[0])
        y_ref = oracle.m2_decode_head(S, "f64", x[0], Bv[0], C[0], "f64", al, de, D)
        assert np.array_equal(y[0], y_ref), step
    hd.flush(True)
    assert np.array_equal(hd.S0, S)


@pytest.mark.parametrize("sdt", ["f32", "bf16"])
def test_replay_narrow_checkpoint_changes_only_at_folds(sdt):
    N, P, L = 8, 4, 5
    S0 = oracle.round_to(np.random.default_rng(11).standard_normal((P, N)), sdt)
    hd = oracle.Mamba2ReplayHead(S0, sdt, "f32", L)
    r = np.random.default_rng(12)
    prev = hd.S0.copy()
    for step in range(1, 4 * L + 1):
        C, Bv, x, dt = _tokens(r, 1, N, P)
        hd.window(C.astype(np.float32), Bv.astype(np.float32), x.astype(np.float32), dt, 0.1, 0.0, 1.0)
        folded = (step - 1) % L == 0 and step > 1
        assert (not np.array_equal(hd.S0, prev)) == folded, step
        assert hd.count == (step - 1) % L + 1
        prev = hd.S0.copy()


def test_replay_window_equals_its_tokens_one_at_a_time_and_rollback():
    N, P, L, T = 6, 5, 8, 4
    S0 = np.random.default_rng(13).standard_normal((P, N))
    r = np.random.default_rng(14)
    C, Bv, x, dt = _tokens(r, T, N, P)
    win = oracle.Mamba2ReplayHead(S0, "f64", "f64", L, pos=3)
    one = oracle.Mamba2ReplayHead(S0, "f64", "f64", L, pos=3)
    yw = win.window(C, Bv, x, dt, 0.2, 0.1, 0.9)
    ys = np.concatenate([one.window(C[t:t + 1], Bv[t:t + 1], x[t:t + 1], dt[t:t + 1], 0.2, 0.1, 0.9)
                         for t in range(T)])
    assert np.array_equal(yw, ys)
    # the ring holds the raw inputs and gates of the window, no C
    assert np.array_equal(win.eB[:T], Bv) and np.array_equal(win.ex[:T], x)
    for t in range(T):
        assert (win.ea[t], win.ed[t]) == oracle.m2_gating(0.2, 0.1, dt[t])
    # keep 1 + accepted tokens: the next output equals a run that saw only those
    acc = 1
    win.rollback(T, acc)
    assert win.count == 1 + acc and win.pos == 3 + 1 + acc
    kept = oracle.Mamba2ReplayHead(S0, "f64", "f64", L, pos=3)
    kept.window(C[:1 + acc], Bv[:1 + acc], x[:1 + acc], dt[:1 + acc], 0.2, 0.1, 0.9)
    C2, B2, x2, dt2 = _tokens(r, 1, N, P)
    assert np.array_equal(win.window(C2, B2, x2, dt2, 0.2, 0.1, 0.9), kept.window(C2, B2, x2, dt2, 0.2, 0.1, 0.9))
