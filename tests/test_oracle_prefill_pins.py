"""Pins of the oracle's chunked prefill (oracle.prefill_head / oracle.prefill):
the tokens of a sequence run through the gated delta rule in order, and the
state is rounded to its storage dtype at every chunk write-back (every
`interval` tokens) and after the last token. Fixed independently of it:

- interval 1 equals the same tokens through the pinned decode step, exactly;
- with fp64 storage the result does not depend on the interval, and it equals
  the chunked (UT-transform) form of the rule computed with numpy linear
  algebra: per chunk, W = (I + A)^-1 diag(beta) (V - diag(G) K S0) with
  A_ij = beta_i (G_i / G_j) (k_i . k_j) for j < i, outputs
  o_t = G_t S0^T q_t + sum_{i<=t} (G_t / G_i) (k_i . q_t) w_i and the final
  state G_C S0 + sum_i (G_C / G_i) k_i w_i^T -- a different order of
  computation in which a dropped decay, a wrong sign or a transposed
  operand gives other numbers;
- an interval of at least T rounds once: the fp64 run rounded at the end;
- two calls split at a chunk boundary equal one call, bit for bit;
- variable lengths: empty sequences leave their state alone; padding and
  out-of-range slots.
"""
import numpy as np
import pytest

import oracle


def _seq(T, dk, dv, seed):
    r = np.random.default_rng(seed)
    return (r.standard_normal((T, dk)), r.standard_normal((T, dk)), r.standard_normal((T, dv)),
            r.uniform(0.3, 1.0, T), r.uniform(0.05, 0.95, T))


@pytest.mark.parametrize("sdt", ["f32", "bf16", "f16"])
def test_interval_one_equals_decode_steps(sdt):
    dk, dv, T = 16, 8, 9
    q, k, v, al, be = _seq(T, dk, dv, 1)
    S = oracle.round_to(0.3 * np.random.default_rng(2).standard_normal((dv, dk)), sdt)
    Sd = S.copy()
    out = oracle.prefill_head(S, sdt, q, k, v, "f64", al, be, 1)
    for t in range(T):
        o = oracle.decode_head(Sd, sdt, q[t], k[t], v[t], "f64", al[t], be[t])
        assert np.array_equal(out[t], o)
    assert np.array_equal(S.view(np.uint8), Sd.view(np.uint8))


def _chunk_form(S0, q, k, v, al, be, C):
    """The chunked (UT-transform) form, fp64 numpy; S0 is dk x dv."""
    dk = S0.shape[0]
    T = q.shape[0]
    kn = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
    qn = q / np.sqrt((q * q).sum(1, keepdims=True) + 1e-6) / np.sqrt(dk)
    S = S0.copy()
    out = np.zeros((T, S0.shape[1]))
    for c0 in range(0, T, C):
        sl = slice(c0, min(T, c0 + C))
        K, Q, V, a, b = kn[sl], qn[sl], v[sl], al[sl], be[sl]
        n = K.shape[0]
        G = np.cumprod(a)
        A = np.zeros((n, n))
        for i in range(n):
            for j in range(i):
                A[i, j] = b[i] * G[i] / G[j] * (K[i] @ K[j])
        W = np.linalg.solve(np.eye(n) + A, b[:, None] * (V - G[:, None] * (K @ S)))
        for t in range(n):
            o = G[t] * (S.T @ Q[t])
            for i in range(t + 1):
                o += G[t] / G[i] * (K[i] @ Q[t]) * W[i]
            out[c0 + t] = o
        S = G[-1] * S + sum(G[-1] / G[i] * np.outer(K[i], W[i]) for i in range(n))
    return out, S


@pytest.mark.parametrize("seed", range(5))
def test_fp64_equals_the_chunked_form_at_any_interval(seed):
    r = np.random.default_rng(10 + seed)
    dk, dv, T = int(r.integers(2, 9)), int(r.integers(1, 7)), int(r.integers(1, 13))
    q, k, v, al, be = _seq(T, dk, dv, 20 + seed)
    S0 = r.standard_normal((dv, dk))
    for C in (1, 3, 64):
        o_chunk, S_chunk = _chunk_form(S0.T.copy(), q, k, v, al, be, C)
        for interval in (1, 4, 100):
            S = S0.copy()
            out = oracle.prefill_head(S, "f64", q, k, v, "f64", al, be, interval)
            assert np.allclose(out, o_chunk, rtol=1e-10, atol=1e-10)
            assert np.allclose(S, S_chunk.T, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("sdt", ["bf16", "f16", "f32"])
def test_long_interval_rounds_once(sdt):
    dk, dv, T = 16, 8, 12
    q, k, v, al, be = _seq(T, dk, dv, 3)
    S = oracle.round_to(0.3 * np.random.default_rng(4).standard_normal((dv, dk)), sdt)
    S64 = oracle.load(S, sdt).copy()
    out = oracle.prefill_head(S, sdt, q, k, v, "f64", al, be, T)
    out64 = oracle.prefill_head(S64, "f64", q, k, v, "f64", al, be, T)
    assert np.array_equal(out, out64)
    assert np.array_equal(S, oracle.round_to(S64, sdt))


@pytest.mark.parametrize("sdt", ["bf16", "f32"])
def test_split_at_a_chunk_boundary_equals_one_call(sdt):
    dk, dv, T, I = 32, 16, 20, 4
    q, k, v, al, be = _seq(T, dk, dv, 5)
    S_one = oracle.round_to(0.2 * np.random.default_rng(6).standard_normal((dv, dk)), sdt)
    S_two = S_one.copy()
    o_one = oracle.prefill_head(S_one, sdt, q, k, v, "f64", al, be, I)
    o_a = oracle.prefill_head(S_two, sdt, q[:8], k[:8], v[:8], "f64", al[:8], be[:8], I)
    o_b = oracle.prefill_head(S_two, sdt, q[8:], k[8:], v[8:], "f64", al[8:], be[8:], I)
    assert np.array_equal(o_one, np.concatenate([o_a, o_b]))
    assert np.array_equal(S_one.view(np.uint8), S_two.view(np.uint8))
    if sdt == "bf16":  # a split that is not at a chunk boundary rounds at another point
        S_odd = oracle.round_to(0.2 * np.random.default_rng(6).standard_normal((dv, dk)), sdt)
        oracle.prefill_head(S_odd, sdt, q[:7], k[:7], v[:7], "f64", al[:7], be[:7], I)
        oracle.prefill_head(S_odd, sdt, q[7:], k[7:], v[7:], "f64", al[7:], be[7:], I)
        assert not np.array_equal(S_odd.view(np.uint8), S_one.view(np.uint8))


def test_batch_driver_varlen_padding_and_heads():
    Hk, Hv, dk, dv = 2, 4, 16, 8
    lens = np.array([5, 0, 3, 7, 2], np.int32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    r = np.random.default_rng(7)
    q = r.standard_normal((total, Hk, dk)).astype(np.float32)
    k = r.standard_normal((total, Hk, dk)).astype(np.float32)
    v = r.standard_normal((total, Hv, dv)).astype(np.float32)
    a = r.standard_normal((total, Hv)).astype(np.float32)
    b = r.standard_normal((total, Hv)).astype(np.float32)
    A_log = r.uniform(0, 2, Hv).astype(np.float32)
    dt_bias = r.uniform(-1, 1, Hv).astype(np.float32)
    pool = r.standard_normal((6, Hv, dv, dk))
    pool0 = pool.copy()
    slots = np.array([4, 0, -1, 2, 9], np.int32)  # sequence 2 is padding, sequence 4 names slot 9 of 6
    out, bad = oracle.prefill(pool, "f64", slots, cu, q, k, v, a, b, "f32", A_log, dt_bias, 4)
    assert bad == Hv
    assert np.array_equal(pool[0], pool0[0])  # an empty sequence leaves its state alone
    assert np.all(out[cu[2]:cu[3]] == 0) and np.all(out[cu[4]:cu[5]] == 0)
    for s in (1, 3, 5):
        assert np.array_equal(pool[s], pool0[s])
    # sequence 3, head 3 (key head 1) against the single-head prefill with its own gates
    h, kh = 3, 1
    al = np.array([oracle.gating(A_log[h], dt_bias[h], a[t, h], b[t, h])[0] for t in range(cu[3], cu[4])])
    be = np.array([oracle.gating(A_log[h], dt_bias[h], a[t, h], b[t, h])[1] for t in range(cu[3], cu[4])])
    S = pool0[2, h].copy()
    o = oracle.prefill_head(S, "f64", q[cu[3]:cu[4], kh], k[cu[3]:cu[4], kh], v[cu[3]:cu[4], h], "f32", al, be, 4)
    assert np.array_equal(o, out[cu[3]:cu[4], h]) and np.array_equal(S, pool[2, h])
